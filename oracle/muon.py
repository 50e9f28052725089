"""Float64 oracle of the owner-side Muon step (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference leg may use this module.

The step an owner runs on its own full matrix, with no communication (DMuon
docs, "架构设计", §2 "专属归属权——原语", optimizer-step bullet; "HSDP 训练（多机）",
"底层发生了什么" step 3): momentum, Newton-Schulz orthogonalisation, decoupled
weight decay and the parameter update.  The pages name the parts but give a
formula only for the Newton-Schulz iteration ("架构设计" §1, the NS equation
X <- aX + bXX^T X + cX(X^T X)^2).  Readings taken where the pages are silent:

* momentum: Nesterov with no dampening, buf <- mu*buf + g, u <- g + mu*buf
  (plain heavy-ball u <- buf when ``nesterov`` is False);
* normalisation: X0 = u / (||u||_F + eps), eps = 1e-7, per 2-D slice;
* orientation: when m > n the iteration runs on u^T (so X X^T is p x p with
  p = min(m, n)) and the result is transposed back;
* iteration: each step forms A = X X^T, B = b*A + c*A*A, X <- a*X + B*X,
  which is the NS equation with its two right-hand terms grouped as
  (b*A + c*A^2) X;
* update: W <- W*(1 - lr*wd) - lr*sqrt(max(1, m/n))*O, both terms from the
  old W; the bf16 parameter is W rounded to nearest-even;
* rank >= 2 tensors act on their last two dimensions, every leading index a
  separate matrix; rank < 2 is an error (MindSpore hyper-parallel
  "分布式 Muon 优化器 — 参数分组设计文档（v2）", §2.1 and §2.2, §6 table).
"""

from __future__ import annotations

import math

import numpy as np

NS_EPS = 1e-7


def bf16_round(x):
    """Round to the nearest bfloat16 value, ties to even, returned as float64.

    The value is first rounded to float32 (as a float32 datapath would hold
    it) and then to the 8-bit-mantissa bfloat16 grid by adding half an ulp
    of the kept part plus the tie-breaking bit and truncating.  Finite
    inputs only.
    """
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    keep_lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + keep_lsb) & np.uint64(0xFFFF0000)
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def momentum_update(buf, g, mu, nesterov=True):
    """One momentum step.  Returns (new buffer, direction u fed to NS).

    buf <- mu*buf + g ; u <- g + mu*buf (Nesterov) or u <- buf.
    The pages only name momentum ("动量", "架构设计" §2 and §3.3); the form is
    the reading stated in the module docstring.
    """
    buf = np.asarray(buf, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    new_buf = mu * buf + g
    u = g + mu * new_buf if nesterov else new_buf.copy()
    return new_buf, u


def ns_iterate(X, a, b, c, steps, emulate_bf16=False):
    """Run ``steps`` Newton-Schulz iterations on a p x q matrix (p <= q).

    Each iteration: A = X X^T; B = b*A + c*(A A); X <- a*X + B X.  With
    ``emulate_bf16`` the products A, B and the new X are rounded to bfloat16,
    mirroring where a bf16-storage datapath keeps them.
    ("架构设计" §1, NS iteration equation.)
    """
    X = np.array(X, dtype=np.float64)
    for _ in range(int(steps)):
        A = X @ X.T
        if emulate_bf16:
            A = bf16_round(A)
        B = b * A + c * (A @ A)
        if emulate_bf16:
            B = bf16_round(B)
        X = a * X + B @ X
        if emulate_bf16:
            X = bf16_round(X)
    return X


def newton_schulz(G, a, b, c, steps, eps=NS_EPS, emulate_bf16=False):
    """Orthogonalise one m x n matrix: normalise, iterate, restore orientation."""
    G = np.asarray(G, dtype=np.float64)
    if G.ndim != 2:
        raise ValueError("newton_schulz takes one 2-D matrix")
    m, n = G.shape
    transposed = m > n
    X = G.T if transposed else G
    X = X / (np.linalg.norm(X) + eps)
    if emulate_bf16:
        X = bf16_round(X)
    X = ns_iterate(X, a, b, c, steps, emulate_bf16=emulate_bf16)
    return X.T if transposed else X


def shape_scale(m, n):
    """sqrt(max(1, m/n)) for an m x n matrix (rows x cols of the last two dims)."""
    return math.sqrt(max(1.0, m / n))


def apply_update(W, O, lr, wd, m, n):
    """Decoupled weight decay plus the scaled orthogonalised update.

    W <- W*(1 - lr*wd) - lr*sqrt(max(1, m/n))*O ("架构设计" §2: "权重衰减 +
    参数更新" on the owner's own copy; the fp32 master / bf16 parameter split
    follows "Pure DMuon 路由", dtype paragraph).
    """
    W = np.asarray(W, dtype=np.float64)
    return W * (1.0 - lr * wd) - lr * shape_scale(m, n) * np.asarray(O, dtype=np.float64)


def muon_step(W, buf, g, lr, mu, wd, ns_steps, a, b, c, nesterov=True,
              eps=NS_EPS, emulate_bf16=False):
    """One owner-side Muon step on a tensor of rank >= 2.

    Returns a dict with the new master ``W``, the new momentum ``buf``, the
    orthogonalised update ``O`` and the bf16-rounded parameter ``param``
    (all float64, same shape as W).  Leading dimensions are independent
    matrices (hyper-parallel §2.2 "last two dims"); rank < 2 raises
    ValueError (§2.1).
    """
    W = np.asarray(W, dtype=np.float64)
    buf = np.asarray(buf, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    if W.ndim < 2:
        raise ValueError("Muon needs a tensor of rank >= 2; route rank-1 tensors to AdamW")
    if W.shape != buf.shape or W.shape != g.shape:
        raise ValueError("W, momentum and grad shapes differ")
    m, n = W.shape[-2], W.shape[-1]
    lead = W.shape[:-2]
    Wf = W.reshape((-1, m, n))
    bf = buf.reshape((-1, m, n))
    gf = g.reshape((-1, m, n))
    W_out = np.empty_like(Wf)
    buf_out = np.empty_like(bf)
    O_out = np.empty_like(Wf)
    for s in range(Wf.shape[0]):
        nb, u = momentum_update(bf[s], gf[s], mu, nesterov=nesterov)
        O = newton_schulz(u, a, b, c, ns_steps, eps=eps, emulate_bf16=emulate_bf16)
        buf_out[s] = nb
        O_out[s] = O
        W_out[s] = apply_update(Wf[s], O, lr, wd, m, n)
    shape = lead + (m, n)
    W_out = W_out.reshape(shape)
    return {
        "W": W_out,
        "buf": buf_out.reshape(shape),
        "O": O_out.reshape(shape),
        "param": bf16_round(W_out),
    }

