"""The owner-partitioned step's choreography on two gloo ranks (CPU).

"架构设计" §2 (专属归属权): every owner-route tensor has one owner; the mean
gradient is reduced to it, only it steps, and it broadcasts the updated
parameter.  "Pure DMuon 路由": the sharded_adamw route reduce-scatters the
gradients to equal pieces and all-gathers the parameters.  Here the local
step is the float64 oracle behind OwnerStep's interface (a test stepper on
CPU tensors), so the test checks the data movement: after two steps every
rank holds the same parameters, and they equal, bit for bit, one process
stepping every tensor with the same stepper on the mean gradients.
"""

import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUON = [(64, 96), (3, 40, 24), (128, 64), (32, 32), (2, 16, 48)]
ADAMW = [100, 7, 64]
SHARDED = [1000, 333]
MUON_KW = dict(lr=0.02, momentum=0.95, wd=0.01, ns_steps=5, a=3.4445, b=-4.7750, c=2.0315)
ADAM_KW = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1)


class OracleStepper:
    """OwnerStep's interface over CPU tensors, stepping with the oracle."""

    def set_muon(self, masters, momenta, grads, params):
        self.m = (masters, momenta, grads, params)

    def set_adamw(self, masters, exp_avgs, exp_avg_sqs, grads, params):
        self.a = (masters, exp_avgs, exp_avg_sqs, grads, params)

    def muon_step(self, lr, momentum, wd, ns_steps, a, b, c, stream=None):
        from oracle import muon as omuon

        for W, B, G, P in zip(*self.m):
            out = omuon.muon_step(W.double().numpy(), B.double().numpy(), G.double().numpy(), lr, momentum, wd,
                                  ns_steps, a, b, c)
            W.copy_(torch.from_numpy(out["W"]).float())
            B.copy_(torch.from_numpy(out["buf"]).float())
            P.copy_(W.to(torch.bfloat16))

    def adamw_step(self, lr, beta1, beta2, eps, wd, step, stream=None):
        from oracle import adamw as oadamw

        for W, M, V, G, P in zip(*self.a):
            out = oadamw.adamw_step(W.double().numpy(), M.double().numpy(), V.double().numpy(), G.double().numpy(),
                                    lr, beta1, beta2, eps, wd, step)
            W.copy_(torch.from_numpy(np.asarray(out["W"])).float())
            M.copy_(torch.from_numpy(np.asarray(out["m"])).float())
            V.copy_(torch.from_numpy(np.asarray(out["v"])).float())
            P.copy_(W.to(torch.bfloat16))


def _weights():
    g = torch.Generator().manual_seed(11)
    shapes = MUON + [(n,) for n in ADAMW] + [(n,) for n in SHARDED]
    return [torch.randn(s, generator=g) * 0.02 for s in shapes]


def _grads(rank, step):
    g = torch.Generator().manual_seed(1000 * step + rank)
    shapes = MUON + [(n,) for n in ADAMW] + [(n,) for n in SHARDED]
    return [torch.randn(s, generator=g) for s in shapes]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q, layered):
    import sys

    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from matrix_optimizer_step_gb300 import build
        from matrix_optimizer_step_gb300.owner_dist import DistributedOwnerStep, OwnerLayout

        build.build()
        layers = [0, 0, 1, 1, 2, 0, 1, 2] if layered else None
        L = OwnerLayout.build(MUON, ADAMW, SHARDED, world, layers=layers)
        ds = DistributedOwnerStep(L, device="cpu", grad_dtype=torch.float32, stepper=OracleStepper())
        ds.load_masters(_weights())
        for step in (1, 2):
            for gv, gh in zip(ds.grads(), _grads(rank, step)):
                gv.copy_(gh.reshape(gv.shape))
            ds.step(MUON_KW, dict(ADAM_KW, step=step))
        q.put((rank, L.owner, ds.param_flat.view(torch.int16).numpy().copy(),
               ds.sp_param_flat.view(torch.int16).numpy().copy(),
               {i: ds.masters[i].numpy().copy() for i in ds.masters}, ds.sp_master.numpy().copy()))
    except Exception as e:
        q.put((rank, repr(e), None, None, None, None))
        raise
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("layered", [False, True])
def test_two_gloo_ranks_owner_step_equals_one_process(layered):
    from matrix_optimizer_step_gb300.owner_dist import OwnerLayout

    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q, layered)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted((q.get(timeout=300) for _ in procs), key=lambda o: o[0])
    for p in procs:
        p.join(timeout=60)
    assert all(o[2] is not None for o in out), [o[1] for o in out]
    assert all(p.exitcode == 0 for p in procs)
    owners = out[0][1]
    assert owners == out[1][1] and sorted(set(owners)) == [0, 1]
    # Every rank leaves the step with the same parameters.
    assert np.array_equal(out[0][2], out[1][2]) and np.array_equal(out[0][3], out[1][3])
    # Each owner-route tensor's master lives on its owner only.
    assert set(out[0][4]) | set(out[1][4]) == set(range(len(owners)))
    assert not (set(out[0][4]) & set(out[1][4]))

    # One process, one rank, the same stepper, the mean gradients.
    W = _weights()
    n_own = len(MUON) + len(ADAMW)
    ref_state = [w.clone().float() for w in W]
    mom = [torch.zeros(s) for s in MUON]
    ema = [torch.zeros(w.numel()) for w in W[len(MUON):]]
    emv = [torch.zeros(w.numel()) for w in W[len(MUON):]]
    params = [w.to(torch.bfloat16) for w in W]
    st = OracleStepper()
    for step in (1, 2):
        g0, g1 = _grads(0, step), _grads(1, step)
        mean = [(a + b) / 2 for a, b in zip(g0, g1)]
        st.set_muon(ref_state[:len(MUON)], mom, mean[:len(MUON)], params[:len(MUON)])
        st.muon_step(**MUON_KW)
        st.set_adamw(ref_state[len(MUON):], ema, emv, mean[len(MUON):], params[len(MUON):])
        st.adamw_step(**ADAM_KW, step=step)
    # Distributed params, per tensor, in params() order.
    L = OwnerLayout.build(MUON, ADAMW, SHARDED, world, layers=[0, 0, 1, 1, 2, 0, 1, 2] if layered else None)
    pf, sp = out[0][2], out[0][3]

    def bits(t):
        return t.reshape(-1).view(torch.int16).numpy()

    for i in range(n_own):
        n = params[i].numel()
        assert np.array_equal(pf[L.offset[i]:L.offset[i] + n], bits(params[i])), i
        owner = L.owner[i]
        assert np.array_equal(out[owner][4][i].reshape(-1), ref_state[i].reshape(-1).numpy()), i
    for k, (o, n) in enumerate(zip(L.sharded_offset, L.sharded_numels)):
        assert np.array_equal(sp[o:o + n], bits(params[n_own + k])), n_own + k
    # Sharded masters: the pieces, in rank order, rebuild the full masters.
    full = np.concatenate([out[r][5] for r in range(world)])
    for k, (o, n) in enumerate(zip(L.sharded_offset, L.sharded_numels)):
        assert np.array_equal(full[o:o + n], ref_state[n_own + k].reshape(-1).numpy()), k


def test_owner_layout_properties():
    from matrix_optimizer_step_gb300.owner_dist import OwnerLayout

    for world in (1, 2, 3, 8):
        L = OwnerLayout.build(MUON * 4, ADAMW, SHARDED, world)
        numels = [math.prod(s) for s in L.muon_shapes] + list(L.adamw_numels)
        # Owner ranges tile the owner buffer in rank order; each tensor lies in its owner's range,
        # starts on a 128-element boundary and overlaps no other tensor.
        assert L.owner_range[0][0] == 0 and L.owner_range[-1][1] == L.owner_numel
        for r in range(world - 1):
            assert L.owner_range[r][1] == L.owner_range[r + 1][0]
        spans = sorted((L.offset[i], L.offset[i] + n) for i, n in enumerate(numels))
        for (a0, a1), (b0, _) in zip(spans, spans[1:]):
            assert a1 <= b0
        for i, n in enumerate(numels):
            a, b = L.owner_range[L.owner[i]]
            assert a <= L.offset[i] and L.offset[i] + n <= b and L.offset[i] % 128 == 0
        assert L.sharded_numel == world * L.piece and L.piece % 128 == 0
        assert L.sharded_offset[-1] + L.sharded_numels[-1] <= L.sharded_numel
    with pytest.raises(ValueError):
        OwnerLayout.build([(5,)], [], [], 2)


def test_owner_partition_balances_the_llama_set():
    """On the Llama-3-8B set the owners' estimated step times stay within
    the greedy list-scheduling bound (mean + largest item) and, for 2-8
    ranks, within 1 % of the mean; every tensor has exactly one owner."""
    from matrix_optimizer_step_gb300 import workloads as W
    from matrix_optimizer_step_gb300.owner_dist import OwnerLayout, adamw_cost_ps, ns_cost_ps

    wl = W.workload("llama3_8b")
    shapes = [s.shape for s in wl.matrices]
    adam = [v.numel for v in wl.vectors if "embed" not in v.name and "lm_head" not in v.name]
    costs = [ns_cost_ps(s) for s in shapes] + [adamw_cost_ps(n) for n in adam]
    for world in (2, 3, 4, 8):
        L = OwnerLayout.build(shapes, adam, [], world)
        assert len(L.owner) == len(costs) and set(L.owner) == set(range(world))
        load = [0] * world
        for i, r in enumerate(L.owner):
            load[r] += costs[i]
        mean, top = sum(costs) / world, max(costs)
        assert max(load) <= mean + top
        # 224 tensors of 7 shapes: LPT evens the owners out to well under 1 %.
        assert max(load) <= 1.01 * mean, (world, max(load) / mean)


def test_nccl_branch_issues_the_pages_collectives(monkeypatch):
    """The NCCL branch (which needs one GPU per rank, so it cannot run here)
    checked by recording its calls as rank 1 of 2: a mean reduce of each
    owner's contiguous gradient range to that owner, an in-place mean
    reduce_scatter of the sharded gradients onto this rank's piece, a
    broadcast of each owner's parameter range from it, and an in-place
    all_gather of the pieces; every call on a view of the flat buffers."""
    from matrix_optimizer_step_gb300.owner_dist import DistributedOwnerStep, OwnerLayout

    calls = []
    monkeypatch.setattr(dist, "get_world_size", lambda group=None: 2)
    monkeypatch.setattr(dist, "get_rank", lambda group=None: 1)
    monkeypatch.setattr(dist, "get_backend", lambda group=None: "nccl")
    monkeypatch.setattr(dist, "reduce", lambda t, dst, op, group=None: calls.append(("reduce", t, dst, op)))
    monkeypatch.setattr(dist, "broadcast", lambda t, src, group=None: calls.append(("broadcast", t, src, None)))
    monkeypatch.setattr(dist, "reduce_scatter_tensor",
                        lambda out, inp, op, group=None: calls.append(("reduce_scatter", (out, inp), None, op)))
    monkeypatch.setattr(dist, "all_gather_into_tensor",
                        lambda out, inp, group=None: calls.append(("all_gather", (out, inp), None, None)))
    L = OwnerLayout.build(MUON, ADAMW, SHARDED, 2)
    ds = DistributedOwnerStep(L, device="cpu", grad_dtype=torch.float32, stepper=OracleStepper())
    ds.reduce_grads()
    ds.publish_params()
    elt = ds.grad_flat.element_size()
    kinds = [c[0] for c in calls]
    assert kinds == ["reduce", "reduce", "reduce_scatter", "broadcast", "broadcast", "all_gather"]
    for r in range(2):
        a, b = L.owner_range[r]
        _, t, dst, op = calls[r]
        assert dst == r and op == dist.ReduceOp.AVG
        assert t.data_ptr() == ds.grad_flat.data_ptr() + a * elt and t.numel() == b - a
        _, t, src, _ = calls[3 + r]
        assert src == r
        assert t.data_ptr() == ds.param_flat.data_ptr() + a * ds.param_flat.element_size() and t.numel() == b - a
    (out, inp), op = calls[2][1], calls[2][3]
    assert op == dist.ReduceOp.AVG and inp.data_ptr() == ds.sp_grad_flat.data_ptr()
    assert out.data_ptr() == ds.sp_grad_flat.data_ptr() + 1 * L.piece * elt and out.numel() == L.piece
    out, inp = calls[5][1]
    assert out.data_ptr() == ds.sp_param_flat.data_ptr() and out.numel() == 2 * L.piece
    assert inp.data_ptr() == ds.sp_param_flat.data_ptr() + L.piece * ds.sp_param_flat.element_size()
