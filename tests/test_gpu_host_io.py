"""The host-buffer step (``dmuon_step_host``) against the device entry points.

``dmuon_step_host`` copies gradients in from page-locked host memory, runs
the same Muon and AdamW kernels as ``dmuon_muon_step`` / ``dmuon_adamw_step``
group by group, and copies the bf16 parameters out.  Each group is planned
on its own, but every output element is computed by the same kernel code
with the same reduction order, so the results must be bit-identical to the
device path on the same inputs (itself held to the oracle in
test_gpu_parity); one tensor is also checked against the oracle here.
"""

import numpy as np
import pytest
import torch

from oracle import muon as omuon

pytestmark = pytest.mark.gpu

HP = dict(lr=0.02, momentum=0.95, wd=0.01, ns_steps=5, a=3.4445, b=-4.7750, c=2.0315, nesterov=True)
SHAPES = [(256, 512), (512, 256), (3, 128, 96), (24, 320), (1000, 130), (512, 512), (64, 64), (130, 1000),
          (384, 128), (8, 16)]
VEC_NUMELS = [4096, 77, 100000]


def _state(seed, shapes, vec_numels, dev):
    g = torch.Generator().manual_seed(seed)
    W = [(torch.randn(s, generator=g) * 0.02).to(dev) for s in shapes]
    Bf = [torch.zeros(s, device=dev) for s in shapes]
    gdt = [torch.float32 if i == 4 else torch.bfloat16 for i in range(len(shapes))]
    G = [torch.empty(s, device=dev, dtype=d) for s, d in zip(shapes, gdt)]
    P = [torch.empty(s, device=dev, dtype=torch.bfloat16) for s in shapes]
    vW = [(torch.randn(n, generator=g) * 0.02).to(dev) for n in vec_numels]
    vm = [torch.zeros(n, device=dev) for n in vec_numels]
    vv = [torch.zeros(n, device=dev) for n in vec_numels]
    vG = [torch.empty(n, device=dev, dtype=torch.bfloat16) for n in vec_numels]
    vP = [torch.empty(n, device=dev, dtype=torch.bfloat16) for n in vec_numels]
    return dict(W=W, B=Bf, G=G, P=P, vW=vW, vm=vm, vv=vv, vG=vG, vP=vP)


def _host_grads(seed, st):
    g = torch.Generator().manual_seed(seed)
    hg = [torch.randn(t.shape, generator=g).to(t.dtype).pin_memory() for t in st["G"]]
    hv = [torch.randn(t.shape, generator=g).to(t.dtype).pin_memory() for t in st["vG"]]
    return hg, hv


@pytest.fixture
def small_host_groups(cuda_lib):
    # These lists are far below the default smallest group: allow groups of
    # 1 Ki elements so that the requested group counts are formed.
    cuda_lib.dmuon_set_tuning(11, 1)
    yield cuda_lib
    cuda_lib.dmuon_set_tuning(11, 32768)


@pytest.mark.parametrize("n_groups", [1, 3, 8])
def test_step_host_bit_identical_to_device_path(small_host_groups, n_groups):
    cuda_lib = small_host_groups
    dev = torch.device("cuda")
    a = _state(5, SHAPES, VEC_NUMELS, dev)
    b = _state(5, SHAPES, VEC_NUMELS, dev)
    sa, sb = cuda_lib.OwnerStep(0), cuda_lib.OwnerStep(0)
    for s, st in ((sa, a), (sb, b)):
        s.set_muon(st["W"], st["B"], st["G"], st["P"])
        s.set_adamw(st["vW"], st["vm"], st["vv"], st["vG"], st["vP"])
    # Host-side parameters of the host path; tensor 2 keeps its parameter on the device only.
    hp = [torch.empty(t.shape, dtype=torch.bfloat16).pin_memory() for t in b["P"]]
    hp[2] = None
    hvp = [torch.empty(t.shape, dtype=torch.bfloat16).pin_memory() for t in b["vP"]]
    for k in range(2):
        hg, hv = _host_grads(100 + k, a)
        adam = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1, step=k + 1)
        # device path: the caller copies
        for d, h in zip(a["G"] + a["vG"], hg + hv):
            d.copy_(h)
        sa.muon_step(**HP)
        sa.adamw_step(**adam)
        # host path: one call
        sb.set_host_io(hg, hp, hv, hvp)
        sb.step_host(HP, adam, n_groups=n_groups)
        torch.cuda.synchronize()
        sa.sync()
        sb.sync()
        for key in ("W", "B", "P", "vW", "vm", "vv", "vP"):
            for i, (x, y) in enumerate(zip(a[key], b[key])):
                assert torch.equal(x, y), (k, key, i)
        for i, h in enumerate(hp):
            if h is not None:
                assert torch.equal(h, a["P"][i].cpu()), (k, "param_host", i)
        for i, h in enumerate(hvp):
            assert torch.equal(h, a["vP"][i].cpu()), (k, "vec param_host", i)
    sa.close()
    sb.close()


def test_step_host_against_oracle(small_host_groups):
    cuda_lib = small_host_groups
    dev = torch.device("cuda")
    shape = (256, 768)
    g = torch.Generator().manual_seed(11)
    W0 = torch.randn(shape, generator=g) * 0.02
    grad = torch.randn(shape, generator=g).to(torch.bfloat16)
    W = W0.to(dev)
    Bf = torch.zeros(shape, device=dev)
    Gd = torch.empty(shape, device=dev, dtype=torch.bfloat16)
    Pd = torch.empty(shape, device=dev, dtype=torch.bfloat16)
    s = cuda_lib.OwnerStep(0)
    s.set_muon([W], [Bf], [Gd], [Pd])
    hp = torch.empty(shape, dtype=torch.bfloat16).pin_memory()
    s.set_host_io([grad.pin_memory()], [hp])
    s.step_host(HP, None, n_groups=2)
    torch.cuda.synchronize()
    f = lambda x: float(np.float32(x))  # noqa: E731
    ref = omuon.muon_step(W0.double().numpy(), np.zeros(shape), grad.double().numpy(), f(HP["lr"]),
                          f(HP["momentum"]), f(HP["wd"]), 5, f(HP["a"]), f(HP["b"]), f(HP["c"]), nesterov=True)
    scale = omuon.shape_scale(*shape)
    O = (W0.double().numpy() * (1 - f(HP["lr"]) * f(HP["wd"])) - W.double().cpu().numpy()) / (f(HP["lr"]) * scale)
    assert np.linalg.norm(O - ref["O"]) / np.linalg.norm(ref["O"]) <= 2e-2
    assert torch.equal(hp, W.cpu().to(torch.bfloat16))
    s.close()


def test_step_host_refuses_pageable_host_memory(cuda_lib):
    capi = cuda_lib.capi
    dev = torch.device("cuda")
    shape = (128, 256)
    W = torch.randn(shape, device=dev)
    W0 = W.clone()
    Bf = torch.zeros(shape, device=dev)
    Gd = torch.zeros(shape, device=dev, dtype=torch.bfloat16)
    pageable = torch.randn(shape).to(torch.bfloat16)  # not page-locked
    ctx = cuda_lib.dmuon_context_create(0)
    try:
        m = capi.matrix_desc(W, Bf, Gd)
        io = capi.DmuonHostIO(pageable.data_ptr(), None)
        with pytest.raises(cuda_lib.DmuonError) as ei:
            capi.dmuon_step_host(ctx, [m], [io], capi.muon_hparams(**HP))
        assert ei.value.status == capi.DMUON_ERR_INVALID_ARG
        assert "page-locked" in str(ei.value)
        torch.cuda.synchronize()
        assert torch.equal(W, W0)
    finally:
        cuda_lib.dmuon_context_destroy(ctx)


def test_step_host_timeline_is_ordered(small_host_groups):
    """With profiling on, dmuon_step_host records when each group's gradient
    copies, compute and parameter copies ended; the times follow the
    pipeline's order: a group computes after its gradients arrived and after
    the previous group computed, its parameters leave after it computed,
    and the step ends with the last copy."""
    mos = small_host_groups
    dev = torch.device("cuda")
    st = _state(31, SHAPES, VEC_NUMELS, dev)
    hg, hv = _host_grads(32, st)
    hp = [torch.empty(t.shape, dtype=torch.bfloat16).pin_memory() for t in st["P"]]
    hvp = [torch.empty(t.shape, dtype=torch.bfloat16).pin_memory() for t in st["vP"]]
    step = mos.OwnerStep(0)
    step.set_muon(st["W"], st["B"], st["G"], st["P"])
    step.set_adamw(st["vW"], st["vm"], st["vv"], st["vG"], st["vP"])
    step.set_host_io(hg, hp, hv, hvp)
    adam = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.0, step=1)
    assert step.host_timeline() is None
    step.profile(True)
    step.step_host(HP, adam, n_groups=3)
    tl = step.host_timeline()
    step.profile_read()
    step.profile(False)
    step.sync()
    assert tl is not None and len(tl["groups"]) == 3
    prev_compute = 0.0
    for h2d, comp, d2h in tl["groups"]:
        assert 0.0 <= h2d <= tl["h2d_done"] + 1e-3
        assert comp >= max(h2d, prev_compute) - 1e-3
        assert d2h >= comp - 1e-3 and d2h <= tl["end"] + 1e-3
        # Parameter copies wait for the last gradient copy.
        assert d2h >= tl["h2d_done"] - 1e-3
        prev_compute = comp
    # Without profiling nothing new is recorded: the last timeline stays.
    step.step_host(HP, dict(adam, step=2), n_groups=3)
    step.sync()
    assert step.host_timeline() == tl
    step.close()
