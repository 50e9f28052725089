"""The allocation-free Muon entry point against the context-based one.

``dmuon_muon_step_noalloc`` serves callers that cannot call cudaMalloc (code
inside a framework that owns all device memory, or that must not grow or
synchronise the device after start-up): its scratch is a static device
array inside the library.  Here it is called through the C ABI on the same
inputs as ``dmuon_muon_step`` for two steps in a row (momentum carried), and
its outputs must agree within the tolerances the parity tests use: NS
output 2e-2 relative Frobenius, momentum 1e-6 max-norm relative, bf16 param
the exact rounding of the fp32 master.  This file is collected last so a
failure here cannot hide the other tests' results.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

A, B, C = 3.4445, -4.7750, 2.0315


def _frob(x, y):
    d = np.linalg.norm(y)
    return float(np.linalg.norm(x - y) / (d if d > 0 else 1.0))


@pytest.mark.parametrize("shape", [(256, 512), (3, 384, 128), (200, 72)])
def test_noalloc_matches_context_entry_point_on_two_calls(cuda_lib, shape):
    mos = cuda_lib
    capi = mos.capi
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(42)
    W = torch.randn(shape, generator=g) * 0.02
    lr, mu, wd = 0.02, 0.95, 0.01
    sides = []
    for _ in range(2):  # one copy per entry point
        sides.append({"W": W.to(dev), "buf": torch.zeros(shape, device=dev),
                      "g": torch.empty(shape, device=dev, dtype=torch.bfloat16),
                      "p": torch.empty(shape, device=dev, dtype=torch.bfloat16)})
    ctx = mos.dmuon_context_create(0)
    try:
        descs = [capi.matrix_desc(s["W"], s["buf"], s["g"], s["p"]) for s in sides]
        for call in range(2):
            grad = torch.randn(shape, generator=g).to(torch.bfloat16)
            for s in sides:
                s["g"].copy_(grad)
            W0 = sides[0]["W"].double().cpu().numpy()
            mos.dmuon_muon_step(ctx, [descs[0]], lr, mu, wd, 5, A, B, C)
            mos.dmuon_muon_step_noalloc(descs[1], lr, mu, wd, 5, A, B, C)
            torch.cuda.synchronize()
            m, n = shape[-2], shape[-1]
            scale = max(1.0, m / n) ** 0.5
            O = [((W0 * (1 - np.float32(lr) * np.float32(wd)) - s["W"].double().cpu().numpy())
                  / (np.float32(lr) * scale)).reshape(-1, m, n) for s in sides]
            for k in range(O[0].shape[0]):
                assert _frob(O[1][k], O[0][k]) <= 2e-2, (shape, call, k)
            b0 = sides[0]["buf"].double().cpu().numpy()
            b1 = sides[1]["buf"].double().cpu().numpy()
            assert np.max(np.abs(b1 - b0)) <= 1e-6 * np.max(np.abs(b0)), (shape, call)
            for s in sides:
                assert torch.equal(s["p"], s["W"].to(torch.bfloat16))
    finally:
        mos.dmuon_context_destroy(ctx)


def test_noalloc_rejects_tensor_over_the_static_limit(cuda_lib):
    mos = cuda_lib
    capi = mos.capi
    d = capi.DmuonMatrix()
    d.rank = 2
    d.shape[0], d.shape[1] = 4096, 4096  # needs ~256 MiB of scratch
    d.grad_dtype = capi.DMUON_DTYPE_BF16
    d.master, d.momentum, d.grad = 1 << 30, 2 << 30, 3 << 30  # never dereferenced: rejected first
    with pytest.raises(mos.DmuonError) as e:
        mos.dmuon_muon_step_noalloc(d, 0.02, 0.95, 0.01, 5, A, B, C)
    assert e.value.status == capi.DMUON_ERR_SHAPE
    assert "static limit" in str(e.value)
