"""Float64 CPU oracle for the owner-side Muon / AdamW optimizer step.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import, call or execute anything in this package.  The CUDA
library never calls it and it never calls the CUDA library: the two share no
code.  Inputs reach both sides from the seeded generators in
``matrix_optimizer_step_gb300.workloads``, which hold none of the method's
arithmetic.

What the oracle computes, and the passages it follows:

* ``muon``   -- momentum, Frobenius normalisation, the Newton-Schulz
  iteration on the last two dimensions, decoupled weight decay and the
  parameter update (DMuon docs, "架构设计" (architecture), §1 NS iteration
  equation and §2 "optimizer step" bullet; "HSDP 训练（多机）", "底层发生了什么"
  step 3; MindSpore hyper-parallel "分布式 Muon 优化器 — 参数分组设计文档（v2）"
  §2.1, §2.2, §6).
* ``adamw``  -- the element-wise AdamW step of the ``adamw`` and
  ``sharded_adamw`` routes (DMuon docs, "Pure DMuon 路由", route table and
  the dtype paragraph).
* ``lpt``    -- the longest-processing-time greedy assignment and Graham's
  bound (DMuon docs, "架构设计" §3.1 "分区（全局 LPT）").

Everything is float64 numpy (host BLAS for the matrix products) or pure
Python; there is no blocking, fusion or reordering beyond the definitions.

Parity status per function (what pins it is in ``tests/test_oracle.py``):

* ``muon.newton_schulz``      pinned (SVD closed form, band invariant,
  transpose equivariance, scale invariance, unfactored-formula identity).
* ``muon.momentum_update``    pinned (torch.optim.SGD Nesterov buffer on CPU,
  zero-buffer closed form).
* ``muon.apply_update``       pinned (closed forms: lr=0, wd=0, shape scale).
* ``muon.muon_step``          pinned through its parts plus the slice rule;
  the composition of the parts has no printed worked example on the pages.
* ``adamw.adamw_step``        pinned (torch.optim.AdamW float64 on CPU,
  constant-gradient closed form).
* ``lpt.lpt_assign``          pinned (brute-force optimum + Graham bound,
  equal-size balance, the pages' 7-items/8-slots idle example).
* ``muon.bf16_round``         pinned (torch bfloat16 cast on CPU).
"""

from . import adamw, lpt, muon  # noqa: F401

__all__ = ["adamw", "lpt", "muon"]
