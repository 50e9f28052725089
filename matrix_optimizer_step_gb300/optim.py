"""User-facing wrapper: one owner's Muon and AdamW tensors on one GPU.

``OwnerStep`` keeps a library context and the descriptor arrays of a fixed
set of torch tensors, so a training loop calls ``muon_step`` /
``adamw_step`` without re-marshalling pointers every step.  It only
marshals: every step runs in the CUDA library through the C ABI.
"""

from __future__ import annotations

import ctypes

import torch

from . import capi


def _check_tensor(t, name, dtypes, like=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if like is not None and tuple(t.shape) != tuple(like.shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(like.shape)}")


class OwnerStep:
    """Muon-route matrices and AdamW-route tensors owned by this process."""

    def __init__(self, device=0):
        self.device = int(device)
        self.ctx = capi.dmuon_context_create(self.device)
        self._mats = None
        self._n_mats = 0
        self._vecs = None
        self._n_vecs = 0
        self._keep = []

    # -------------------------------------------------------------- Muon
    def set_muon(self, masters, momenta, grads, params=None):
        """Register the Muon tensors: fp32 masters/momenta, bf16 or fp32 grads,
        optional bf16 params (same shapes, rank >= 2, contiguous)."""
        params = params if params is not None else [None] * len(masters)
        descs = []
        for i, (w, b, g, p) in enumerate(zip(masters, momenta, grads, params)):
            _check_tensor(w, f"master[{i}]", (torch.float32,))
            _check_tensor(b, f"momentum[{i}]", (torch.float32,), like=w)
            _check_tensor(g, f"grad[{i}]", (torch.float32, torch.bfloat16), like=w)
            if p is not None:
                _check_tensor(p, f"param[{i}]", (torch.bfloat16,), like=w)
            if w.dim() > 4:
                raise ValueError(f"master[{i}] has rank {w.dim()} > 4")
            descs.append(capi.matrix_desc(w, b, g, p))
        self._mats = capi.descriptor_array(descs, capi.DmuonMatrix)
        self._n_mats = len(descs)
        self._keep = [masters, momenta, grads, params]

    def muon_step(self, lr, momentum, wd, ns_steps=5, a=3.4445, b=-4.7750, c=2.0315,
                  nesterov=True, fp32_ns=False, stream=None):
        if self._mats is None:
            raise RuntimeError("set_muon() first")
        flags = (capi.DMUON_FLAG_NESTEROV if nesterov else 0) | (capi.DMUON_FLAG_FP32_NS if fp32_ns else 0)
        capi._check(capi.load_library().dmuon_muon_step(
            self.ctx, self._mats, self._n_mats, float(lr), float(momentum), float(wd), int(ns_steps),
            float(a), float(b), float(c), flags, capi._stream_handle(stream)))

    # ------------------------------------------------------------- AdamW
    def set_adamw(self, masters, exp_avgs, exp_avg_sqs, grads, params=None):
        params = params if params is not None else [None] * len(masters)
        descs = []
        for i, (w, m, v, g, p) in enumerate(zip(masters, exp_avgs, exp_avg_sqs, grads, params)):
            _check_tensor(w, f"master[{i}]", (torch.float32,))
            _check_tensor(m, f"exp_avg[{i}]", (torch.float32,), like=w)
            _check_tensor(v, f"exp_avg_sq[{i}]", (torch.float32,), like=w)
            _check_tensor(g, f"grad[{i}]", (torch.float32, torch.bfloat16), like=w)
            if p is not None:
                _check_tensor(p, f"param[{i}]", (torch.bfloat16,), like=w)
            descs.append(capi.vector_desc(w, m, v, g, p))
        self._vecs = capi.descriptor_array(descs, capi.DmuonVector)
        self._n_vecs = len(descs)
        self._keep_adam = [masters, exp_avgs, exp_avg_sqs, grads, params]

    def adamw_step(self, lr, beta1, beta2, eps, wd, step, stream=None):
        if self._vecs is None:
            raise RuntimeError("set_adamw() first")
        capi._check(capi.load_library().dmuon_adamw_step(
            self.ctx, self._vecs, self._n_vecs, float(lr), float(beta1), float(beta2), float(eps),
            float(wd), int(step), capi._stream_handle(stream)))

    # ------------------------------------------------------ both routes
    def step(self, muon, adamw, stream=None):
        """One optimizer step of every registered tensor: the Muon step on
        ``stream`` and, concurrently, the AdamW step on a side stream (the two
        share no workspace; AdamW is HBM-bound while the Newton-Schulz
        products are tensor-bound).  ``muon`` / ``adamw`` are keyword dicts for
        muon_step / adamw_step (adamw may be None).  On return ``stream`` is
        ordered after both."""
        main = stream if stream is not None else torch.cuda.current_stream(self.device)
        if adamw is None or self._vecs is None:
            self.muon_step(stream=main, **muon)
            return
        if getattr(self, "_side", None) is None:
            self._side = torch.cuda.Stream(device=self.device)
            self._ev_fork = torch.cuda.Event()
            self._ev_join = torch.cuda.Event()
        self._ev_fork.record(main)
        self._side.wait_event(self._ev_fork)
        self.adamw_step(stream=self._side, **adamw)
        self.muon_step(stream=main, **muon)
        self._ev_join.record(self._side)
        main.wait_event(self._ev_join)

    # ------------------------------------------------- host-side buffers
    def set_host_io(self, grads_host, params_host=None, v_grads_host=None, v_params_host=None):
        """Register page-locked CPU tensors for ``step_host``: per Muon tensor
        a gradient (same shape and dtype as its device grad) and optionally a
        bf16 parameter; the same per AdamW tensor."""
        def check(t, name, like, dtype):
            if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_pinned():
                raise TypeError(f"{name} must be a page-locked CPU tensor")
            if t.dtype != dtype or not t.is_contiguous() or t.numel() != like.numel():
                raise ValueError(f"{name}: expected a contiguous {dtype} tensor of {like.numel()} elements")

        def ios(host_g, host_p, grads, params, tag):
            host_p = host_p if host_p is not None else [None] * len(host_g)
            if len(host_g) != len(grads) or len(host_p) != len(grads):
                raise ValueError(f"{tag}: one host buffer per registered tensor")
            out = []
            for i, (hg, hp) in enumerate(zip(host_g, host_p)):
                check(hg, f"{tag} grad_host[{i}]", grads[i], grads[i].dtype)
                if hp is not None:
                    if params[i] is None:
                        raise ValueError(f"{tag} param_host[{i}] given but no device param registered")
                    check(hp, f"{tag} param_host[{i}]", grads[i], torch.bfloat16)
                out.append(capi.DmuonHostIO(hg.data_ptr(), None if hp is None else hp.data_ptr()))
            return capi.descriptor_array(out, capi.DmuonHostIO)

        if self._mats is None:
            raise RuntimeError("set_muon() first")
        self._mat_io = ios(grads_host, params_host, self._keep[2], self._keep[3], "muon")
        if v_grads_host is not None:
            if self._vecs is None:
                raise RuntimeError("set_adamw() first")
            self._vec_io = ios(v_grads_host, v_params_host, self._keep_adam[3], self._keep_adam[4], "adamw")
        else:
            self._vec_io = None
        self._keep_host = [grads_host, params_host, v_grads_host, v_params_host]

    def step_host(self, muon, adamw=None, n_groups=8, stream=None):
        """One step from host gradients to host bf16 parameters
        (``dmuon_step_host``): the registered host gradients are copied in,
        every tensor steps, the parameters are copied out, with the copies of
        ``n_groups`` groups overlapping the compute of the others.  ``muon`` /
        ``adamw``: keyword dicts as for muon_step / adamw_step."""
        if getattr(self, "_mat_io", None) is None:
            raise RuntimeError("set_host_io() first")
        mh = capi.muon_hparams(**muon)
        use_adam = adamw is not None and self._vecs is not None and self._vec_io is not None
        ah = capi.adamw_hparams(**adamw) if use_adam else None
        capi._check(capi.load_library().dmuon_step_host(
            self.ctx, self._mats, self._mat_io, self._n_mats, ctypes.byref(mh),
            self._vecs if use_adam else None, self._vec_io if use_adam else None,
            self._n_vecs if use_adam else 0, ctypes.byref(ah) if use_adam else None,
            int(n_groups), capi._stream_handle(stream)))

    # ------------------------------------------------------------ misc
    def sync(self, stream=None):
        capi.dmuon_sync(self.ctx, stream)

    def profile(self, enable=True):
        capi.dmuon_profile(self.ctx, enable)

    def profile_read(self):
        return capi.dmuon_profile_read(self.ctx)

    def set_tuning(self, key, value):
        """One tuning key of this context (dmuon_context_set_tuning)."""
        capi.dmuon_context_set_tuning(self.ctx, key, value)

    def host_timeline(self):
        """Timeline of the last step_host call made while profiling."""
        return capi.dmuon_profile_host_timeline(self.ctx)

    def kernel_launches(self):
        return capi.dmuon_kernel_launches(self.ctx)

    def close(self):
        if self.ctx is not None:
            capi.dmuon_context_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def owner_partition(numels, n_owners, layers=None, small_threshold=5_000_000):
    """Owner rank of each Muon tensor: one global LPT pass over all tensors
    ("架构设计" §3.1), element count as the cost; with ``layers`` (a layer id
    per tensor) the layer-aware pass (same-layer tensors on distinct owners,
    a layer's tensors below ``small_threshold`` merged).  Deterministic, so
    every rank computes the same map on its own and each tensor has exactly
    one owner.  Returns (owner per tensor, elements per owner)."""
    numels = [int(n) for n in numels]
    if layers is None:
        return capi.dmuon_lpt_assign(numels, int(n_owners))
    return capi.dmuon_lpt_assign_layered(numels, layers, int(n_owners), small_threshold)


def adamw_shard_ranges(numels, n_ranks, align=8):
    """The `sharded_adamw` route ("Pure DMuon 路由"): every AdamW-route element
    is stepped by exactly one rank.  The tensors are laid end to end and the
    concatenation is cut into n_ranks contiguous pieces of equal size
    (boundaries rounded to multiples of `align` elements, so each piece keeps
    16-byte alignment in fp32 and bf16).  Returns, per rank, a list of
    (tensor index, start, count) runs in concatenation order; the pieces
    partition every tensor exactly once.  Deterministic, so each rank computes
    the same split on its own; gathering the pieces in rank order rebuilds
    the concatenation."""
    numels = [int(n) for n in numels]
    n_ranks = int(n_ranks)
    if n_ranks < 1 or align < 1 or any(n < 0 for n in numels):
        raise ValueError("need n_ranks >= 1, align >= 1 and non-negative sizes")
    total = sum(numels)
    cuts = [min(total, (total * r // n_ranks + align - 1) // align * align) for r in range(n_ranks + 1)]
    cuts[0], cuts[-1] = 0, total
    out = []
    for r in range(n_ranks):
        lo, hi = cuts[r], max(cuts[r], cuts[r + 1])
        runs, base = [], 0
        for i, n in enumerate(numels):
            a, b = max(lo, base), min(hi, base + n)
            if a < b:
                runs.append((i, a - base, b - a))
            base += n
        out.append(runs)
    return out


def adamw_shard_views(tensors, runs):
    """Views of `tensors` (flattened) for one rank's runs, in order: the
    arguments of OwnerStep.set_adamw for that rank's piece."""
    return [tensors[i].reshape(-1)[start:start + count] for i, start, count in runs]

