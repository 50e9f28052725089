"""Float64 oracle of the element-wise AdamW step (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference leg may use this module.

The ``adamw`` and ``sharded_adamw`` routes both run AdamW and differ only in
where parameters and gradients live (DMuon docs, "Pure DMuon 路由", route
table); the state is fp32 master/optimizer storage with a bf16 parameter
("Pure DMuon 路由", dtype paragraph: master_dtype / optim_dtype vs
param_dtype).  The pages do not print the AdamW formula; the reading taken
is the usual bias-corrected form with decoupled weight decay:

    m <- b1*m + (1-b1)*g
    v <- b2*v + (1-b2)*g^2
    W <- W*(1 - lr*wd) - lr * (m/(1-b1^t)) / (sqrt(v/(1-b2^t)) + eps)

with the step counter t >= 1 supplied by the caller, and both W terms taken
from the old W.
"""

from __future__ import annotations

import numpy as np

from .muon import bf16_round


def adamw_step(W, m, v, g, lr, beta1, beta2, eps, wd, t):
    """One AdamW step in float64.  Returns dict(W, m, v, param)."""
    if int(t) < 1:
        raise ValueError("AdamW step counter starts at 1")
    W = np.asarray(W, dtype=np.float64)
    m = np.asarray(m, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    m_new = beta1 * m + (1.0 - beta1) * g
    v_new = beta2 * v + (1.0 - beta2) * g * g
    m_hat = m_new / (1.0 - beta1 ** t)
    v_hat = v_new / (1.0 - beta2 ** t)
    W_new = W * (1.0 - lr * wd) - lr * m_hat / (np.sqrt(v_hat) + eps)
    return {"W": W_new, "m": m_new, "v": v_new, "param": bf16_round(W_new)}
