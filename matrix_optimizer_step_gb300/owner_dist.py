"""The owner-partitioned step over several ranks (one process per GPU).

The pages' system around the owner step ("架构设计" (architecture design), §2
"专属归属权——原语" and §4; "Pure DMuon 路由", route table):

* every "muon"-route and "adamw"-route tensor has exactly one owner rank,
  chosen by one global LPT pass ("架构设计" §3.1); only the owner holds its
  fp32 master and optimizer state and runs its optimizer step;
* gradients reach the owner by a reduce of the mean over the ranks
  (backward bullet of §2), the owner steps with no communication (optimizer
  -step bullet), and the updated bf16 parameter goes back to every rank by a
  broadcast from the owner (forward bullet: here issued right after the
  step, so every rank leaves the step with the full parameters);
* "sharded_adamw"-route tensors (embedding, lm_head) are cut into equal
  pieces, one per rank: gradients by reduce_scatter to the optimizer pieces,
  parameters by all_gather from the pieces.

GB300 layout: every rank keeps the bf16 parameters and the gradients of all
owner-route tensors in one flat buffer each, laid out owner by owner (owner
r's tensors contiguous, every tensor starting on a 256-byte boundary), so the
reduce and the broadcast of an owner are each one call on a contiguous view
with no packing copy.  The sharded tensors live in a second pair of flat
buffers padded to a multiple of the rank count, so the piece of rank r is the
contiguous range [r*P, (r+1)*P) and both collectives run in place.  The
owner's fp32 state is allocated for its own tensors only.

All arithmetic of the step runs in the CUDA library (``OwnerStep``); the
collectives are torch.distributed calls (NCCL between GPUs).  On a gloo
group, CUDA tensors are staged through host memory and the mean is a sum
divided by the rank count on the receiving rank (gloo offers no mean for
reduce); a test may pass its own ``stepper`` with OwnerStep's methods.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch
import torch.distributed as dist

from . import capi
from .optim import OwnerStep

_ALIGN = 128  # elements: 256 bytes of bf16, 512 of fp32


def _up(x, a):
    return (x + a - 1) // a * a


def ns_cost_ps(shape, ns_steps=5):
    """Estimated device time (picoseconds) of one Muon tensor's step: the
    dense Newton-Schulz flops at 1.5 PFLOP/s plus 24 bytes per element at
    7 TB/s.  The LPT cost of a Muon tensor."""
    m, n = int(shape[-2]), int(shape[-1])
    lead = math.prod(int(s) for s in shape[:-2])
    p, q = min(m, n), max(m, n)
    flops = lead * ns_steps * (4 * p * p * q + 2 * p ** 3)
    return flops // 1500 + (lead * m * n * 24) // 7


def adamw_cost_ps(numel):
    """Estimated device time (picoseconds) of an AdamW tensor's step: 28
    bytes per element at 7 TB/s.  The LPT cost of an "adamw"-route tensor."""
    return int(numel) * 4


@dataclass
class OwnerLayout:
    """Owners and flat-buffer offsets of a model's optimizer tensors.

    muon_shapes     shapes (rank >= 2) of the "muon"-route tensors
    adamw_numels    element counts of the "adamw"-route tensors
    sharded_numels  element counts of the "sharded_adamw"-route tensors
    world           number of ranks
    layers          optional layer id per owner-route item (Muon items first,
                    then AdamW items; < 0 = none): the layer-aware LPT with
                    element counts as sizes, as on the pages; without it one
                    global LPT over estimated step times (ns_cost_ps,
                    adamw_cost_ps) balances the owners' compute
    Deterministic: every rank builds the same layout on its own.
    """

    muon_shapes: list
    adamw_numels: list
    sharded_numels: list
    world: int
    owner: list          # per owner-route item (Muon items, then AdamW items)
    offset: list         # per owner-route item: start in the owner flat buffers (elements)
    owner_range: list    # per rank: (start, end) of its tensors in the owner flat buffers
    owner_numel: int     # size of the owner flat buffers
    sharded_offset: list # per sharded tensor: start in the sharded flat buffers
    piece: int           # elements per rank in the sharded flat buffers
    sharded_numel: int   # size of the sharded flat buffers (= world * piece)

    @classmethod
    def build(cls, muon_shapes, adamw_numels=(), sharded_numels=(), world=1, layers=None,
              small_threshold=5_000_000, ns_steps=5):
        muon_shapes = [tuple(int(s) for s in shp) for shp in muon_shapes]
        adamw_numels = [int(n) for n in adamw_numels]
        sharded_numels = [int(n) for n in sharded_numels]
        world = int(world)
        if world < 1:
            raise ValueError("world must be >= 1")
        if any(len(s) < 2 for s in muon_shapes):
            raise ValueError("a Muon-route tensor needs rank >= 2 (route it to AdamW)")
        numels = [math.prod(s) for s in muon_shapes] + adamw_numels
        if layers is not None:
            if len(layers) != len(numels):
                raise ValueError("one layer id per Muon and AdamW tensor")
            owner, _ = capi.dmuon_lpt_assign_layered(numels, [int(x) for x in layers], world, small_threshold)
        else:
            costs = [ns_cost_ps(s, ns_steps) for s in muon_shapes] + [adamw_cost_ps(n) for n in adamw_numels]
            owner, _ = capi.dmuon_lpt_assign(costs, world)
        offset = [0] * len(numels)
        owner_range = []
        o = 0
        for r in range(world):
            start = o
            for i, n in enumerate(numels):
                if owner[i] == r:
                    offset[i] = o
                    o = _up(o + n, _ALIGN)
            owner_range.append((start, o))
        s_off, so = [], 0
        for n in sharded_numels:
            s_off.append(so)
            so = _up(so + n, _ALIGN)
        piece = _up(so, world * _ALIGN) // world if so else 0
        return cls(muon_shapes, adamw_numels, sharded_numels, world, list(owner), offset, owner_range, o,
                   s_off, piece, piece * world)

    def owned(self, rank):
        """Indices of the owner-route items that `rank` owns (Muon items
        are 0 .. len(muon_shapes)-1, AdamW items follow)."""
        return [i for i, r in enumerate(self.owner) if r == rank]


class _Comm:
    """The collectives of the step on one process group.  NCCL: mean by
    ReduceOp.AVG.  gloo: CUDA tensors staged through host memory, mean as a
    sum divided by the rank count on the rank that receives it."""

    def __init__(self, group):
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.nccl = dist.get_backend(group) == "nccl"
        self.ranks = [dist.get_global_rank(group, r) if group is not None else r for r in range(self.world)]

    def _staged(self, t):
        return t if (self.nccl or not t.is_cuda) else t.cpu()

    def reduce_mean(self, t, dst):
        if t.numel() == 0:
            return
        if self.nccl:
            dist.reduce(t, dst=self.ranks[dst], op=dist.ReduceOp.AVG, group=self.group)
            return
        s = self._staged(t)
        dist.reduce(s, dst=self.ranks[dst], op=dist.ReduceOp.SUM, group=self.group)
        if self.rank == dst:
            s.div_(self.world)
            if s is not t:
                t.copy_(s)

    def broadcast(self, t, src):
        if t.numel() == 0:
            return
        s = self._staged(t)
        dist.broadcast(s, src=self.ranks[src], group=self.group)
        if s is not t:
            t.copy_(s)

    def reduce_scatter_mean(self, out, full):
        if full.numel() == 0:
            return
        if self.nccl:
            dist.reduce_scatter_tensor(out, full, op=dist.ReduceOp.AVG, group=self.group)
            return
        # gloo: a separate output (the piece is a view of `full`).
        sf = self._staged(full)
        so = torch.empty(out.shape, dtype=out.dtype, device=sf.device)
        dist.reduce_scatter_tensor(so, sf, op=dist.ReduceOp.SUM, group=self.group)
        so.div_(self.world)
        out.copy_(so)

    def all_gather_pieces(self, full, piece_numel):
        """In-place all-gather: rank r's piece is full[r*P:(r+1)*P]."""
        if full.numel() == 0:
            return
        sf = self._staged(full)
        mine = sf[self.rank * piece_numel:(self.rank + 1) * piece_numel]
        dist.all_gather_into_tensor(sf, mine, group=self.group)
        if sf is not full:
            full.copy_(sf)


class DistributedOwnerStep:
    """One optimizer step of a whole model over the ranks of a process group.

    Every rank allocates the bf16 parameters and the gradients of every
    tensor (flat buffers; ``params()`` / ``grads()`` give per-tensor views for
    the model), and fp32 master and optimizer state for the tensors it owns
    and for its piece of the sharded tensors.  ``load_masters`` initialises
    them from the full fp32 weights (the same on every rank).  ``step`` runs
    reduce -> owner step -> broadcast for the owner routes and reduce_scatter
    -> piece step -> all_gather for the sharded route.
    """

    def __init__(self, layout, group=None, device=None, grad_dtype=torch.bfloat16, stepper=None):
        self.layout = layout
        self.comm = _Comm(group)
        if self.comm.world != layout.world:
            raise ValueError(f"layout is for {layout.world} ranks, the group has {self.comm.world}")
        self.rank = self.comm.rank
        if device is None:
            device = torch.device("cuda", torch.cuda.current_device())
        self.device = torch.device(device)
        L = layout
        dev = self.device
        self.param_flat = torch.zeros(L.owner_numel, dtype=torch.bfloat16, device=dev)
        self.grad_flat = torch.zeros(L.owner_numel, dtype=grad_dtype, device=dev)
        self.sp_param_flat = torch.zeros(L.sharded_numel, dtype=torch.bfloat16, device=dev)
        self.sp_grad_flat = torch.zeros(L.sharded_numel, dtype=grad_dtype, device=dev)
        n_muon = len(L.muon_shapes)
        self._mine = L.owned(self.rank)
        self._mine_muon = [i for i in self._mine if i < n_muon]
        self._mine_adam = [i for i in self._mine if i >= n_muon]
        own_numel = sum(self._numel(i) for i in self._mine)
        # Owner state: Muon (master, momentum) and AdamW (master, m, v) per owned
        # tensor, carved from one fp32 allocation.
        k = 2 * sum(self._numel(i) for i in self._mine_muon) + 3 * sum(self._numel(i) for i in self._mine_adam)
        self._state = torch.zeros(k + 3 * L.piece, dtype=torch.float32, device=dev)
        self._own_numel = own_numel
        o = 0

        def take(n, shape):
            nonlocal o
            v = self._state[o:o + n].view(shape)
            o += n
            return v

        self.masters, self.momenta = {}, {}
        for i in self._mine_muon:
            shp = L.muon_shapes[i]
            self.masters[i] = take(self._numel(i), shp)
            self.momenta[i] = take(self._numel(i), shp)
        self.exp_avg, self.exp_avg_sq = {}, {}
        for i in self._mine_adam:
            self.masters[i] = take(self._numel(i), (self._numel(i),))
            self.exp_avg[i] = take(self._numel(i), (self._numel(i),))
            self.exp_avg_sq[i] = take(self._numel(i), (self._numel(i),))
        P = L.piece
        self.sp_master = take(P, (P,))
        self.sp_exp_avg = take(P, (P,))
        self.sp_exp_avg_sq = take(P, (P,))
        self.stepper = stepper if stepper is not None else OwnerStep(self.device.index or 0)
        self._registered = False

    # ------------------------------------------------------------- views
    def _numel(self, i):
        L = self.layout
        n_muon = len(L.muon_shapes)
        return math.prod(L.muon_shapes[i]) if i < n_muon else L.adamw_numels[i - n_muon]

    def _shape(self, i):
        L = self.layout
        n_muon = len(L.muon_shapes)
        return L.muon_shapes[i] if i < n_muon else (L.adamw_numels[i - n_muon],)

    def _view(self, flat, i):
        o = self.layout.offset[i]
        return flat[o:o + self._numel(i)].view(self._shape(i))

    def params(self):
        """bf16 parameter views: Muon tensors, then AdamW, then sharded."""
        L = self.layout
        out = [self._view(self.param_flat, i) for i in range(len(L.owner))]
        out += [self.sp_param_flat[o:o + n] for o, n in zip(L.sharded_offset, L.sharded_numels)]
        return out

    def grads(self):
        """Gradient views (where backward writes), in the order of params()."""
        L = self.layout
        out = [self._view(self.grad_flat, i) for i in range(len(L.owner))]
        out += [self.sp_grad_flat[o:o + n] for o, n in zip(L.sharded_offset, L.sharded_numels)]
        return out

    def load_masters(self, full_weights):
        """Initialise from the full fp32 weights (a list in params() order,
        the same on every rank): owned masters, this rank's sharded piece,
        every bf16 parameter; optimizer state zero."""
        if len(full_weights) != len(self.layout.owner) + len(self.layout.sharded_numels):
            raise ValueError("one weight per tensor, in params() order")
        with torch.no_grad():
            self._state.zero_()
        for i, w in enumerate(full_weights):
            self.load_weight(i, w)

    def load_weight(self, i, w):
        """Initialise tensor i (params() order) from its full fp32 weight:
        its bf16 parameter on every rank, its master on its owner, the part
        of a sharded tensor that falls in this rank's piece.  Optimizer
        state is left as it is (zero after construction)."""
        L = self.layout
        n_own = len(L.owner)
        with torch.no_grad():
            p = self.params()[i]
            p.copy_(w.reshape(p.shape).to(torch.bfloat16))
            if i < n_own:
                if i in self.masters:
                    self.masters[i].copy_(w.reshape(self.masters[i].shape))
                return
            k = i - n_own
            o, n = L.sharded_offset[k], L.sharded_numels[k]
            r0, r1 = self.rank * L.piece, (self.rank + 1) * L.piece
            a, b = max(o, r0), min(o + n, r1)
            if a < b:
                self.sp_master[a - r0:b - r0].copy_(w.reshape(-1)[a - o:b - o])

    def _register(self):
        L = self.layout
        pv, gv = self.params(), self.grads()
        st = self.stepper
        if self._mine_muon:
            st.set_muon([self.masters[i] for i in self._mine_muon], [self.momenta[i] for i in self._mine_muon],
                        [gv[i] for i in self._mine_muon], [pv[i] for i in self._mine_muon])
        r0, r1 = self.rank * L.piece, (self.rank + 1) * L.piece
        vm = [self.masters[i] for i in self._mine_adam]
        ve = [self.exp_avg[i] for i in self._mine_adam]
        vv = [self.exp_avg_sq[i] for i in self._mine_adam]
        vg = [gv[i].reshape(-1) for i in self._mine_adam]
        vp = [pv[i].reshape(-1) for i in self._mine_adam]
        if L.piece > 0:
            vm.append(self.sp_master)
            ve.append(self.sp_exp_avg)
            vv.append(self.sp_exp_avg_sq)
            vg.append(self.sp_grad_flat[r0:r1])
            vp.append(self.sp_param_flat[r0:r1])
        self._has_adam = len(vm) > 0
        if self._has_adam:
            st.set_adamw(vm, ve, vv, vg, vp)
        self._registered = True

    # -------------------------------------------------------------- step
    def reduce_grads(self):
        """Mean gradient of every owner-route tensor onto its owner; the mean
        of every sharded piece onto its rank."""
        L = self.layout
        for r, (a, b) in enumerate(L.owner_range):
            self.comm.reduce_mean(self.grad_flat[a:b], r)
        if L.piece > 0:
            r0, r1 = self.rank * L.piece, (self.rank + 1) * L.piece
            self.comm.reduce_scatter_mean(self.sp_grad_flat[r0:r1], self.sp_grad_flat)

    def local_step(self, muon, adamw, stream=None):
        """The owner's step of its tensors and its sharded piece (no
        communication).  ``muon`` / ``adamw``: keyword dicts of
        OwnerStep.muon_step / adamw_step."""
        if not self._registered:
            self._register()
        if self._mine_muon:
            self.stepper.muon_step(stream=stream, **muon)
        if self._has_adam and adamw is not None:
            self.stepper.adamw_step(stream=stream, **adamw)

    def publish_params(self):
        """Owners broadcast their updated bf16 parameters; the sharded pieces
        are gathered on every rank."""
        L = self.layout
        for r, (a, b) in enumerate(L.owner_range):
            self.comm.broadcast(self.param_flat[a:b], r)
        if L.piece > 0:
            self.comm.all_gather_pieces(self.sp_param_flat, L.piece)

    def step(self, muon, adamw=None, stream=None):
        """reduce -> owner step -> publish.  The collectives are ordered on
        torch's current stream; a ``stream`` (torch.cuda.Stream) other than
        that one runs the owner step after the reduce and before the
        broadcast.  A raw stream handle must be the current stream."""
        self.reduce_grads()
        if isinstance(stream, torch.cuda.Stream):
            cur = torch.cuda.current_stream(self.device)
            stream.wait_stream(cur)
            self.local_step(muon, adamw, stream=stream)
            cur.wait_stream(stream)
        else:
            self.local_step(muon, adamw, stream=stream)
        self.publish_params()

    def close(self):
        close = getattr(self.stepper, "close", None)
        if close is not None:
            close()
