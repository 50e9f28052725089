"""The Muon step at the largest slice the C ABI accepts (m * n just under
2^31, ragged in both dimensions, both orientations), checked element by
element against a closed form that holds at any size.

The gradient is a signed partial permutation: G[i, pi(i)] = +-1 for every
row i (m <= n; every column j when m > n), zeros elsewhere.  Its values are
exact in bf16 and its rows (columns) are orthonormal, so after the momentum
step and the normalisation every singular value of X0 is the same s, the
Newton-Schulz iteration acts on each of them as the scalar map
s -> a s + b s^3 + c s^5 ("架构设计" §1), and the orthogonalised update is
O = (p5(s) / s) * X0: the same sparsity pattern, every non-zero equal to
+-p5(s).  p5(s) comes from the oracle's iteration on the 1 x 1 matrix [[s]].
Every output tile is written, so a misplaced row, column or tile shows up
as a non-zero off the pattern or a missing one on it.
"""

import gc
import math

import numpy as np
import pytest
import torch

from oracle import muon as omuon

pytestmark = pytest.mark.gpu

A, B, C = 3.4445, -4.7750, 2.0315
F32 = np.float32


def _f(x):
    return float(F32(x))


@pytest.mark.slow
@pytest.mark.parametrize("m,n", [(40003, 53681), (53681, 40003)])
def test_largest_slice_closed_form(cuda_lib, m, n):
    assert m * n < 2 ** 31
    dev = torch.device("cuda")
    lr, mu, wd = 0.02, 0.95, 0.01
    g = torch.Generator(device=dev).manual_seed(m)
    p = min(m, n)
    # The signed partial permutation: one +-1 per row (m <= n) or column.
    perm = torch.randperm(max(m, n), generator=g, device=dev)[:p]
    sign = torch.randint(0, 2, (p,), generator=g, device=dev).float() * 2 - 1
    idx = torch.arange(p, device=dev)
    rows, cols = (idx, perm) if m <= n else (perm, idx)
    G = torch.zeros((m, n), device=dev, dtype=torch.bfloat16)
    G[rows, cols] = sign.to(torch.bfloat16)
    W = torch.randn((m, n), device=dev, generator=g) * 0.02
    W0 = W.clone()
    buf = torch.zeros((m, n), device=dev)
    P = torch.empty((m, n), device=dev, dtype=torch.bfloat16)

    step = cuda_lib.OwnerStep(0)
    step.set_muon([W], [buf], [G], [P])
    step.muon_step(lr, mu, wd, 5, A, B, C)
    step.sync()
    step.close()

    # Closed form: u = (1 + mu) G, X0 = u / (||u|| + eps), all singular values
    # s; O = +-p5(s) on the pattern.
    nrm = (1.0 + _f(mu)) * math.sqrt(p)
    s = (1.0 + _f(mu)) / (nrm + omuon.NS_EPS)
    p5 = float(omuon.ns_iterate(np.array([[s]]), _f(A), _f(B), _f(C), 5)[0, 0])
    assert 0.6 < p5 < 1.25
    scale = omuon.shape_scale(m, n)
    decay = float(F32(1.0) - F32(lr) * F32(wd))

    # Momentum buffer: mu * 0 + G, exactly.
    assert torch.equal(buf, G.float())
    # bf16 parameter: exactly the rounding of the fp32 master.
    assert torch.equal(P, W.to(torch.bfloat16))

    # O recovered from the master, compared in row chunks.
    on_pattern_err = 0.0
    off_pattern_max = 0.0
    chunk = 2048
    for r0 in range(0, m, chunk):
        r1 = min(m, r0 + chunk)
        O = (W0[r0:r1].double() * decay - W[r0:r1].double()) / (_f(lr) * scale)
        expect = torch.zeros_like(O)
        sel = (rows >= r0) & (rows < r1)
        expect[rows[sel] - r0, cols[sel]] = sign[sel].double() * p5
        mask = torch.zeros_like(O, dtype=torch.bool)
        mask[rows[sel] - r0, cols[sel]] = True
        d = (O - expect).abs()
        if mask.any():
            on_pattern_err = max(on_pattern_err, float(d[mask].max()))
        off_pattern_max = max(off_pattern_max, float(d.masked_fill(mask, 0.0).max()))
        del O, expect, mask, d
    assert on_pattern_err <= 2e-2 * p5, (on_pattern_err, p5)
    assert off_pattern_max <= 1e-4 * p5, off_pattern_max

    del W, W0, buf, G, P, perm, sign, idx, rows, cols
    gc.collect()
    torch.cuda.empty_cache()
