"""Seeded synthetic inputs for the owner-side Muon / AdamW step.

This module only draws inputs and counts work: it holds none of the
optimizer's arithmetic, so both the CUDA path and the float64 oracle can take
their inputs from it without sharing any of the method.

Five workloads, named for what they are:

* ``single_256x512``  one fp32 matrix W 256x512 (W~N(0,0.02^2), G~N(0,1),
  momentum zeros), plus tiny 3x4 and 8x16 matrices for closed-form checks;
* ``gpt2_small``      12 layers x {q,k,v,o 768x768, fc 3072x768, proj
  768x3072} = 72 Muon matrices with bf16 grads N(0,1e-2^2) plus a rank-16
  spike whose Frobenius norm is 10x the noise's; 50 LayerNorm vectors (768)
  on AdamW; three consecutive steps with fresh grads;
* ``many_small``      4096 bf16-grad matrices, m and n drawn independently
  and uniformly from {64,...,2048}, grads N(0,1) times a per-matrix scale
  with log10 uniform in [-4,-1];
* ``llama3_8b``       32 layers x {q 4096^2, k 1024x4096, v 1024x4096,
  o 4096^2, gate 14336x4096, up 14336x4096, down 4096x14336} = 224 Muon
  matrices, bf16 grads 1e-3*Student-t(3) plus a rank-8 part of equal
  Frobenius norm; embedding and lm_head 128256x4096 and 65 RMSNorm vectors
  (4096) on AdamW;
* ``moe_experts``     4 layers x {w1 [8,14336,4096], w3 [8,14336,4096],
  w2 [8,4096,14336]}, bf16 grads N(0,1e-3^2) times a per-expert scale
  U[0.1,10].

Random draws use ``torch.Generator`` seeded per tensor, so every tensor can
be regenerated alone (that is how the oracle gets sampled matrices of the
full-size workloads).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

NS_COEFFS = (3.4445, -4.7750, 2.0315)

WORKLOADS = ("single_256x512", "gpt2_small", "many_small", "llama3_8b", "moe_experts")
# Small stand-in used only to profile kernels on Llama-3-8B's shapes: one layer
# (7 matrices, 2.18e8 elements) plus its two norm vectors.
PROFILE_WORKLOADS = ("llama3_8b_layer",)

_SMALL_SIDES = (64, 128, 256, 512, 1024, 2048)


@dataclass(frozen=True)
class MatrixSpec:
    """One Muon tensor (rank >= 2; NS acts on the last two dims)."""

    name: str
    shape: tuple
    grad_dtype: torch.dtype = torch.bfloat16
    grad_scale: float = 1.0          # many_small: per-matrix scale
    slice_scales: tuple = ()         # moe_experts: per-leading-index scale

    @property
    def numel(self):
        return math.prod(self.shape)

    @property
    def mn(self):
        return self.shape[-2], self.shape[-1]

    @property
    def n_slices(self):
        return math.prod(self.shape[:-2]) if len(self.shape) > 2 else 1


@dataclass(frozen=True)
class VectorSpec:
    """One AdamW-route tensor (flattened)."""

    name: str
    shape: tuple

    @property
    def numel(self):
        return math.prod(self.shape)


@dataclass
class Workload:
    name: str
    matrices: list
    vectors: list
    hyper: dict = field(default_factory=dict)
    grad_kind: str = "normal"
    steps: int = 1

    @property
    def muon_numel(self):
        return sum(s.numel for s in self.matrices)

    @property
    def adamw_numel(self):
        return sum(v.numel for v in self.vectors)


def _hyper(**kw):
    h = dict(lr=0.02, momentum=0.95, wd=0.01, ns_steps=5, a=NS_COEFFS[0],
             b=NS_COEFFS[1], c=NS_COEFFS[2], nesterov=True, fp32_ns=False,
             adam_lr=1e-3, beta1=0.9, beta2=0.95, adam_eps=1e-8, adam_wd=0.0)
    h.update(kw)
    return h


def workload(name, tiny_extra=True):
    """Return the spec of one named workload."""
    if name == "single_256x512":
        mats = [MatrixSpec("W", (256, 512), torch.float32)]
        if tiny_extra:
            mats += [MatrixSpec("tiny_3x4", (3, 4), torch.float32),
                     MatrixSpec("tiny_8x16", (8, 16), torch.float32)]
        return Workload(name, mats, [], _hyper(fp32_ns=True), grad_kind="normal")
    if name == "gpt2_small":
        mats, vecs = [], []
        for l in range(12):
            for p in ("q", "k", "v", "o"):
                mats.append(MatrixSpec(f"h{l}.attn.{p}", (768, 768)))
            mats.append(MatrixSpec(f"h{l}.mlp.fc", (3072, 768)))
            mats.append(MatrixSpec(f"h{l}.mlp.proj", (768, 3072)))
            for ln in ("ln_1", "ln_2"):
                vecs.append(VectorSpec(f"h{l}.{ln}.weight", (768,)))
                vecs.append(VectorSpec(f"h{l}.{ln}.bias", (768,)))
        vecs += [VectorSpec("ln_f.weight", (768,)), VectorSpec("ln_f.bias", (768,))]
        return Workload(name, mats, vecs, _hyper(), grad_kind="spiked16", steps=3)
    if name == "many_small":
        g = torch.Generator().manual_seed(0)
        idx = torch.randint(0, len(_SMALL_SIDES), (4096, 2), generator=g)
        logs = torch.rand(4096, generator=g, dtype=torch.float64) * 3.0 - 4.0
        mats = [MatrixSpec(f"m{i}", (_SMALL_SIDES[int(idx[i, 0])], _SMALL_SIDES[int(idx[i, 1])]),
                           grad_scale=float(10.0 ** logs[i]))
                for i in range(4096)]
        return Workload(name, mats, [], _hyper(), grad_kind="normal")
    if name in ("llama3_8b", "llama3_8b_layer"):
        layers = 32 if name == "llama3_8b" else 1
        mats, vecs = [], []
        shapes = (("q", (4096, 4096)), ("k", (1024, 4096)), ("v", (1024, 4096)),
                  ("o", (4096, 4096)), ("gate", (14336, 4096)), ("up", (14336, 4096)),
                  ("down", (4096, 14336)))
        for l in range(layers):
            for p, s in shapes:
                mats.append(MatrixSpec(f"layers.{l}.{p}", s))
            vecs.append(VectorSpec(f"layers.{l}.input_norm", (4096,)))
            vecs.append(VectorSpec(f"layers.{l}.post_norm", (4096,)))
        if layers == 32:
            vecs += [VectorSpec("norm", (4096,)),
                     VectorSpec("embed_tokens", (128256, 4096)),
                     VectorSpec("lm_head", (128256, 4096))]
        else:
            # One layer's share of the step, with a 16384-row slice of the
            # embedding on the AdamW route (67M elements, 1.9 GB of AdamW
            # traffic: larger than L2, small enough for a profiler capture).
            vecs.append(VectorSpec("embed_tokens_rows_0_16383", (16384, 4096)))
        return Workload(name, mats, vecs, _hyper(), grad_kind="student_t_rank8")
    if name == "moe_experts":
        g = torch.Generator().manual_seed(5)
        mats = []
        for l in range(4):
            for w, s in (("w1", (8, 14336, 4096)), ("w3", (8, 14336, 4096)), ("w2", (8, 4096, 14336))):
                scales = tuple(float(x) for x in (torch.rand(8, generator=g, dtype=torch.float64) * 9.9 + 0.1))
                mats.append(MatrixSpec(f"layers.{l}.experts.{w}", s, slice_scales=scales))
        return Workload(name, mats, [], _hyper(), grad_kind="normal_1e-3")
    raise KeyError(name)


# --------------------------------------------------------------------------
# Seeded tensor draws
# --------------------------------------------------------------------------

def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def master_init(spec, index, device="cpu"):
    """fp32 master weight ~ N(0, 0.02^2), seed 1_000_000 + index."""
    g = _gen(device, 1_000_000 + index)
    return torch.randn(spec.shape, generator=g, device=device, dtype=torch.float32) * 0.02


def vector_init(spec, index, device="cpu"):
    """AdamW-route master: RMS/LayerNorm-like vectors start near 1, big tables ~N(0,0.02^2)."""
    g = _gen(device, 2_000_000 + index)
    x = torch.randn(spec.shape, generator=g, device=device, dtype=torch.float32) * 0.02
    if len(spec.shape) == 1:
        x += 1.0
    return x.reshape(-1)


def _orthonormal(rows, k, g, device):
    # Drawn on `device` (seeded stream), factored on the host: a rows x k QR
    # is tiny, and the host routine needs no optional GPU linear-algebra
    # library at run time.
    a = torch.randn(rows, k, generator=g, device=device, dtype=torch.float32)
    q, _ = torch.linalg.qr(a.cpu())
    return q.to(device)


def muon_grad(wl, spec, index, step=0, device="cpu"):
    """Gradient of one Muon tensor for step ``step`` (fresh per step)."""
    seed = index + 1000 * step
    g = _gen(device, seed)
    shape = spec.shape
    kind = wl.grad_kind
    if kind == "normal":
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * spec.grad_scale
    elif kind == "normal_1e-3":
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * 1e-3
        if spec.slice_scales:
            sc = torch.tensor(spec.slice_scales, device=device, dtype=torch.float32)
            x = x * sc.reshape((-1,) + (1,) * (len(shape) - 1))
    elif kind == "spiked16":
        m, n = shape
        noise = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * 1e-2
        u = _orthonormal(m, 16, g, device)
        v = _orthonormal(n, 16, g, device)
        spike = u @ v.T  # 16 unit singular values, Frobenius norm 4
        x = noise + spike * (10.0 * noise.norm() / 4.0)
    elif kind == "student_t_rank8":
        m, n = shape
        z = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        chi = torch.zeros(shape, device=device, dtype=torch.float32)
        for _ in range(3):
            e = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
            chi.addcmul_(e, e)
        t = z * torch.rsqrt(chi / 3.0) * 1e-3
        del z, chi
        lo = torch.randn(m, 8, generator=g, device=device, dtype=torch.float32) @ \
            torch.randn(8, n, generator=g, device=device, dtype=torch.float32)
        x = t + lo * (t.norm() / lo.norm())
        del t, lo
    else:
        raise KeyError(kind)
    return x.to(spec.grad_dtype)


def vector_grad(spec, index, step=0, device="cpu"):
    """bf16 gradient of one AdamW-route tensor, N(0, 1e-2^2), flattened."""
    g = _gen(device, 3_000_000 + index + 1000 * step)
    return (torch.randn(spec.numel, generator=g, device=device, dtype=torch.float32) * 1e-2).to(torch.bfloat16)


# --------------------------------------------------------------------------
# Work accounting (used for roofline figures; not part of the method)
# --------------------------------------------------------------------------

def ns_flops(m, n, steps):
    """Dense flop count of ``steps`` NS iterations on one m x n matrix.

    Per iteration with p = min(m,n), q = max(m,n): the Gram product
    2p^2q, the square of the Gram 2p^3 and the final product 2p^2q.
    """
    p, q = min(m, n), max(m, n)
    return steps * (4 * p * p * q + 2 * p ** 3)


def ns_flops_algorithmic(m, n, steps):
    """Algorithmic flops of the symmetric iteration: the Gram X X^T and the
    square A A are symmetric, so only their upper triangle needs forming
    (p(p+1)/2 dot products each), while B X is computed in full.  The
    tensor-core kernels form whole 256-blocks on the diagonal, so they
    execute slightly more than this count."""
    p, q = min(m, n), max(m, n)
    return steps * (p * (p + 1) * q + p * (p + 1) * p + 2 * p * p * q)


def workload_ns_flops_algorithmic(wl):
    return sum(ns_flops_algorithmic(*s.mn, wl.hyper["ns_steps"]) * s.n_slices for s in wl.matrices)


def workload_ns_flops(wl):
    return sum(ns_flops(*s.mn, wl.hyper["ns_steps"]) * s.n_slices for s in wl.matrices)


def momentum_bytes(wl):
    """HBM bytes of the momentum pass: grad read, momentum read+write, X0
    write (4 bytes per element either way: the bf16 operand plus its bf16
    low half on the bf16 path, fp32 in the fp32 mode and for the small
    classes that run in fp32)."""
    xb = 4
    return sum(s.numel * ((2 if s.grad_dtype == torch.bfloat16 else 4) + 8 + xb) for s in wl.matrices)


def momentum_bytes_algorithmic(wl):
    """Algorithmic HBM bytes of the momentum pass: grad read, momentum
    read+write, X0 write in the Newton-Schulz operand type (2 bytes bf16,
    4 in the fp32 mode); the X0 low half the bf16 path also writes is a
    design choice, not counted."""
    xb = 4 if wl.hyper["fp32_ns"] else 2
    return sum(s.numel * ((2 if s.grad_dtype == torch.bfloat16 else 4) + 8 + xb) for s in wl.matrices)


def update_bytes(wl):
    """HBM bytes of a separate update pass: X read, master read+write, bf16
    param write (on the bf16 path the update is fused into the last NS
    product instead)."""
    xb = 4 if wl.hyper["fp32_ns"] else 2
    return wl.muon_numel * (xb + 8 + 2)


def muon_elementwise_bytes(wl):
    """Minimal HBM bytes of the streaming work of the Muon step (momentum
    pass plus the update, wherever it runs)."""
    return momentum_bytes(wl) + update_bytes(wl)


def adamw_bytes(wl):
    """bf16 grad read, fp32 master/m/v read+write, bf16 param write."""
    return wl.adamw_numel * (2 + 24 + 2)


# --------------------------------------------------------------------------
# Device-resident materialisation (flat buffers, per-tensor views)
# --------------------------------------------------------------------------

@dataclass
class Materialized:
    """A workload's tensors as views into a few flat device buffers.

    One flat buffer per role keeps every gradient in one contiguous block
    (one host-to-device copy per step) and every bf16 parameter in another
    (one device-to-host copy).  Views start on 256-byte boundaries.
    """

    wl: Workload
    masters: list
    momenta: list
    grads: list
    params: list
    v_masters: list
    v_exp_avg: list
    v_exp_avg_sq: list
    v_grads: list
    v_params: list
    flats: dict


def _layout(sizes, align=128):
    offs, o = [], 0
    for s in sizes:
        offs.append(o)
        o += (s + align - 1) // align * align
    return offs, max(o, align)


def _views(flat, offs, shapes):
    return [flat[o:o + math.prod(s)].view(s) for o, s in zip(offs, shapes)]


def materialize(wl, device="cuda", step=0, progress=None):
    """Allocate and fill every tensor of ``wl`` on ``device`` (seeded)."""
    mshapes = [s.shape for s in wl.matrices]
    vshapes = [(v.numel,) for v in wl.vectors]
    gdt = wl.matrices[0].grad_dtype if wl.matrices else torch.bfloat16
    moffs, mtot = _layout([math.prod(s) for s in mshapes])
    voffs, vtot = _layout([math.prod(s) for s in vshapes])
    f32 = dict(device=device, dtype=torch.float32)
    flats = {
        "master": torch.empty(mtot, **f32),
        "momentum": torch.zeros(mtot, **f32),
        "grad": torch.empty(mtot + vtot, device=device, dtype=gdt),
        "param": torch.empty(mtot + vtot, device=device, dtype=torch.bfloat16),
        "v_master": torch.empty(vtot, **f32),
        "v_m": torch.zeros(vtot, **f32),
        "v_v": torch.zeros(vtot, **f32),
    }
    masters = _views(flats["master"], moffs, mshapes)
    momenta = _views(flats["momentum"], moffs, mshapes)
    grads = _views(flats["grad"], moffs, mshapes)
    params = _views(flats["param"], moffs, mshapes)
    v_grads = _views(flats["grad"][mtot:], voffs, vshapes)
    v_params = _views(flats["param"][mtot:], voffs, vshapes)
    for i, spec in enumerate(wl.matrices):
        masters[i].copy_(master_init(spec, i, device))
        grads[i].copy_(muon_grad(wl, spec, i, step, device))
        if progress:
            progress(i)
    v_masters = _views(flats["v_master"], voffs, vshapes)
    for i, spec in enumerate(wl.vectors):
        v_masters[i].copy_(vector_init(spec, i, device))
        v_grads[i].copy_(vector_grad(spec, i, step, device).to(gdt))
    return Materialized(wl, masters, momenta, grads, params, v_masters,
                        _views(flats["v_m"], voffs, vshapes), _views(flats["v_v"], voffs, vshapes),
                        v_grads, v_params, flats)
