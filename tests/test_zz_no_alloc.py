"""The allocation-free Muon entry point against the float64 oracle.

``dmuon_muon_step_noalloc`` serves callers that cannot call cudaMalloc: code
inside a framework that owns every device allocation through its own pool,
or code that must not grow its memory or risk an implicit device
synchronisation after start-up.  Its scratch is one static device array
inside the library, shared by every call.

Each case calls it through the C ABI for two steps in a row (the momentum
buffer carried from the first call into the second) and compares every 2-D
slice with ``oracle.muon.muon_step`` on the same inputs, with the tolerances
of the parity tests: NS output 2e-2 relative Frobenius where the slice runs
on the bf16 tensor cores (min(m, n) >= 64), 1e-4 where it runs on the fp32
CUDA-core kernel (min(m, n) < 64, or DMUON_FLAG_FP32_NS); momentum buffer
1e-6 max-norm relative; bf16 parameter the exact rounding of the fp32
master.  The same calls go to the context entry point ``dmuon_muon_step``
and both must agree within those tolerances too.  A bounded device-side
wait that runs out must be reported by ``dmuon_muon_step_noalloc_sync``.

This file is collected last, so a failure here cannot hide the other
tests' results.
"""

import numpy as np
import pytest
import torch

from oracle import muon as omuon

pytestmark = pytest.mark.gpu

A, B, C = 3.4445, -4.7750, 2.0315
F32 = np.float32


def _f(x):
    return float(F32(x))


def _frob(x, y):
    d = np.linalg.norm(y)
    return float(np.linalg.norm(x - y) / (d if d > 0 else 1.0))


def _maxrel(x, y):
    d = np.max(np.abs(y))
    return float(np.max(np.abs(x - y)) / (d if d > 0 else 1.0))


CASES = [
    ((256, 512), False),     # bf16 tensor cores, wide
    ((3, 384, 128), False),  # bf16, tall, three slices
    ((200, 72), False),      # bf16, ragged tiles
    ((3, 4), False),         # fp32 kernel: min(m, n) < 64
    ((24, 256), False),      # fp32 kernel
    ((2, 40, 24), False),    # fp32 kernel, tall, two slices
    ((160, 96), True),       # fp32 validation mode on a shape the tensor cores would take
]


@pytest.mark.parametrize("shape,fp32_ns", CASES)
def test_noalloc_matches_oracle_on_two_calls(cuda_lib, shape, fp32_ns):
    mos = cuda_lib
    capi = mos.capi
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(42)
    W = torch.randn(shape, generator=g) * 0.02
    lr, mu, wd = 0.02, 0.95, 0.01
    flags = capi.DMUON_FLAG_NESTEROV | (capi.DMUON_FLAG_FP32_NS if fp32_ns else 0)
    m, n = shape[-2], shape[-1]
    fp32_path = fp32_ns or min(m, n) < 64
    tol = 1e-4 if fp32_path else 2e-2
    sides = []
    for _ in range(2):  # [0] the allocation-free entry, [1] the context entry
        sides.append({"W": W.to(dev), "buf": torch.zeros(shape, device=dev),
                      "g": torch.empty(shape, device=dev, dtype=torch.bfloat16),
                      "p": torch.empty(shape, device=dev, dtype=torch.bfloat16)})
    ref_buf = np.zeros(shape)
    ctx = mos.dmuon_context_create(0)
    try:
        descs = [capi.matrix_desc(s["W"], s["buf"], s["g"], s["p"]) for s in sides]
        for call in range(2):
            grad = torch.randn(shape, generator=g).to(torch.bfloat16)
            for s in sides:
                s["g"].copy_(grad)
            W0 = sides[0]["W"].double().cpu().numpy()
            mos.dmuon_muon_step_noalloc(descs[0], lr, mu, wd, 5, A, B, C, flags=flags)
            mos.dmuon_muon_step_noalloc_sync()
            mos.dmuon_muon_step(ctx, [descs[1]], lr, mu, wd, 5, A, B, C, flags=flags)
            mos.dmuon_sync(ctx)
            ref = omuon.muon_step(W0, ref_buf, grad.double().numpy(), _f(lr), _f(mu), _f(wd), 5,
                                  _f(A), _f(B), _f(C))
            scale = omuon.shape_scale(m, n)
            O = [((W0 * (1 - _f(lr) * _f(wd)) - s["W"].double().cpu().numpy()) / (_f(lr) * scale))
                 .reshape(-1, m, n) for s in sides]
            O_ref = ref["O"].reshape(-1, m, n)
            for k in range(O_ref.shape[0]):
                assert _frob(O[0][k], O_ref[k]) <= tol, (shape, call, k, "noalloc vs oracle")
                assert _frob(O[0][k], O[1][k]) <= tol, (shape, call, k, "noalloc vs context entry")
            buf = sides[0]["buf"].double().cpu().numpy()
            assert _maxrel(buf, ref["buf"]) <= 1e-6, (shape, call)
            assert torch.equal(sides[0]["p"], sides[0]["W"].to(torch.bfloat16)), (shape, call)
            ref_buf = buf  # the next call continues from the GPU's own buffer
    finally:
        mos.dmuon_context_destroy(ctx)


@pytest.mark.parametrize("shape,ns_steps", [((1, 300), 5), ((130, 1), 5), ((7, 7), 5), ((96, 160), 0),
                                            ((2, 20, 33), 0), ((1, 1), 3)])
def test_noalloc_edge_shapes_and_no_iterations(cuda_lib, shape, ns_steps):
    """Degenerate shapes (one row, one column, tiny) and ns_steps = 0 (the
    update then applies the normalised momentum direction): the same bits as
    dmuon_muon_step where both run the same kernels (min(m, n) < 64: the
    fp32 kernels; no iteration: momentum, norm and update only), and the
    oracle within the parity tolerances."""
    mos = cuda_lib
    capi = mos.capi
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(7)
    W = torch.randn(shape, generator=g) * 0.02
    grad = torch.randn(shape, generator=g).to(torch.bfloat16)
    lr, mu, wd = 0.02, 0.95, 0.01
    sides = []
    for _ in range(2):
        sides.append({"W": W.to(dev), "buf": torch.zeros(shape, device=dev), "g": grad.to(dev),
                      "p": torch.empty(shape, device=dev, dtype=torch.bfloat16)})
    ctx = mos.dmuon_context_create(0)
    try:
        d = [capi.matrix_desc(s["W"], s["buf"], s["g"], s["p"]) for s in sides]
        mos.dmuon_muon_step_noalloc(d[0], lr, mu, wd, ns_steps, A, B, C)
        mos.dmuon_muon_step_noalloc_sync()
        mos.dmuon_muon_step(ctx, [d[1]], lr, mu, wd, ns_steps, A, B, C)
        mos.dmuon_sync(ctx)
    finally:
        mos.dmuon_context_destroy(ctx)
    m, n = shape[-2], shape[-1]
    if min(m, n) < 64 or ns_steps == 0:
        assert torch.equal(sides[0]["W"], sides[1]["W"]) and torch.equal(sides[0]["p"], sides[1]["p"])
    W0 = W.double().numpy()
    ref = omuon.muon_step(W0, np.zeros(shape), grad.double().numpy(), _f(lr), _f(mu), _f(wd), ns_steps,
                          _f(A), _f(B), _f(C))
    O = ((W0 * (1 - _f(lr) * _f(wd)) - sides[0]["W"].double().cpu().numpy())
         / (_f(lr) * omuon.shape_scale(m, n))).reshape(-1, m, n)
    # bf16 classes hold X0 in bf16 even with no iteration (2e-2); fp32 classes 1e-4.
    tol = 1e-4 if min(m, n) < 64 else 2e-2
    for k in range(O.shape[0]):
        assert _frob(O[k], ref["O"].reshape(-1, m, n)[k]) <= tol, (shape, ns_steps, k)
    assert torch.equal(sides[0]["p"], sides[0]["W"].to(torch.bfloat16))


def test_noalloc_reports_a_wait_that_ran_out(cuda_lib):
    """A bounded wait given a barrier nothing completes records its site in
    the static array's error word; the sync query reports it once, clears
    it, and the next step runs normally."""
    mos = cuda_lib
    capi = mos.capi
    mos.dmuon_muon_step_noalloc_sync()  # nothing pending
    mos.dmuon_selftest_wait_timeout(None, 2000)  # ctx NULL: the allocation-free error word
    with pytest.raises(mos.DmuonError) as e:
        mos.dmuon_muon_step_noalloc_sync()
    assert e.value.status == capi.DMUON_ERR_TIMEOUT
    mos.dmuon_muon_step_noalloc_sync()  # cleared
    dev = torch.device("cuda")
    W = torch.zeros(64, 64, device=dev)
    buf = torch.zeros(64, 64, device=dev)
    G = torch.ones(64, 64, device=dev, dtype=torch.bfloat16)
    d = capi.matrix_desc(W, buf, G, None)
    mos.dmuon_muon_step_noalloc(d, 0.02, 0.95, 0.0, 5, A, B, C)
    mos.dmuon_muon_step_noalloc_sync()
    assert torch.isfinite(W).all() and bool((buf == 1).all())


def test_noalloc_rejects_tensor_over_the_static_limit(cuda_lib):
    mos = cuda_lib
    capi = mos.capi
    d = capi.DmuonMatrix()
    d.rank = 2
    d.shape[0], d.shape[1] = 4096, 4096  # needs ~192 MiB of scratch
    d.grad_dtype = capi.DMUON_DTYPE_BF16
    d.master, d.momentum, d.grad = 1 << 30, 2 << 30, 3 << 30  # never dereferenced: rejected first
    with pytest.raises(mos.DmuonError) as e:
        mos.dmuon_muon_step_noalloc(d, 0.02, 0.95, 0.01, 5, A, B, C)
    assert e.value.status == capi.DMUON_ERR_SHAPE
    assert "static limit" in str(e.value)
