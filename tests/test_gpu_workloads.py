"""The named workloads at full size, through the same OwnerStep calls bench.py
times, checked against the float64 oracle on sampled tensors.

Inputs are drawn on the device; the sampled tensors' inputs are copied back
before the step, so the oracle sees exactly what the GPU saw.  Tolerances as
in test_gpu_parity: NS output 2e-2 (relative Frobenius, bf16 path) or 1e-4
(fp32 path), momentum and AdamW state 1e-6 (max-norm relative), bf16 params
bit-exact against the fp32 master.
"""

import gc

import numpy as np
import pytest
import torch

from matrix_optimizer_step_gb300 import workloads as W
from oracle import adamw as oadamw
from oracle import muon as omuon

pytestmark = pytest.mark.gpu
F32 = np.float32


def _f(x):
    return float(F32(x))


def _frob(got, want):
    d = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (d if d > 0 else 1.0))


def _maxrel(got, want):
    d = np.max(np.abs(want))
    return float(np.max(np.abs(got - want)) / (d if d > 0 else 1.0))


def _run(mos, name, sample_names, steps=1, adam_sample=0, slice_pick=None):
    wl = W.workload(name)
    h = wl.hyper
    dev = torch.device("cuda")
    mat = W.materialize(wl, dev)
    step = mos.OwnerStep(0)
    step.set_muon(mat.masters, mat.momenta, mat.grads, mat.params)
    if wl.vectors:
        step.set_adamw(mat.v_masters, mat.v_exp_avg, mat.v_exp_avg_sq, mat.v_grads, mat.v_params)
    idx = [i for i, s in enumerate(wl.matrices) if s.name in sample_names]
    assert len(idx) == len(sample_names)
    tol = 1e-4 if h["fp32_ns"] else 2e-2
    gen = torch.Generator().manual_seed(123)
    results = []
    for t in range(1, steps + 1):
        if t > 1:  # fresh gradients each step
            for i, spec in enumerate(wl.matrices):
                mat.grads[i].copy_(W.muon_grad(wl, spec, i, t - 1, dev))
            for i, spec in enumerate(wl.vectors):
                mat.v_grads[i].copy_(W.vector_grad(spec, i, t - 1, dev).to(mat.v_grads[i].dtype))
        torch.cuda.synchronize()
        before = {i: (mat.masters[i].double().cpu().numpy(), mat.momenta[i].double().cpu().numpy(),
                      mat.grads[i].double().cpu().numpy()) for i in idx}
        vpick = {}
        for j, v in enumerate(wl.vectors):
            n = v.numel
            sel = torch.arange(n) if (adam_sample == 0 or n <= adam_sample) else \
                torch.randperm(n, generator=gen)[:adam_sample]
            sel = sel.to(dev)
            vpick[j] = (sel, mat.v_masters[j][sel].double().cpu().numpy(),
                        mat.v_exp_avg[j][sel].double().cpu().numpy(),
                        mat.v_exp_avg_sq[j][sel].double().cpu().numpy(),
                        mat.v_grads[j][sel].double().cpu().numpy())
        step.muon_step(h["lr"], h["momentum"], h["wd"], h["ns_steps"], h["a"], h["b"], h["c"],
                       nesterov=h["nesterov"], fp32_ns=h["fp32_ns"])
        if wl.vectors:
            step.adamw_step(h["adam_lr"], h["beta1"], h["beta2"], h["adam_eps"], h["adam_wd"], t)
        step.sync()
        for i in idx:
            spec = wl.matrices[i]
            W0, B0, G = before[i]
            m, n = spec.mn
            W1 = mat.masters[i].double().cpu().numpy()
            B1 = mat.momenta[i].double().cpu().numpy()
            slices = range(spec.n_slices) if slice_pick is None else slice_pick
            W0s, B0s, Gs = (x.reshape(-1, m, n) for x in (W0, B0, G))
            W1s, B1s = W1.reshape(-1, m, n), B1.reshape(-1, m, n)
            for s in slices:
                ref = omuon.muon_step(W0s[s], B0s[s], Gs[s], _f(h["lr"]), _f(h["momentum"]), _f(h["wd"]),
                                      h["ns_steps"], _f(h["a"]), _f(h["b"]), _f(h["c"]), nesterov=h["nesterov"])
                O = (W0s[s] * (1 - _f(h["lr"]) * _f(h["wd"])) - W1s[s]) / (_f(h["lr"]) * omuon.shape_scale(m, n))
                r = {"tensor": spec.name, "slice": s, "t": t, "O": _frob(O, ref["O"]),
                     "buf": _maxrel(B1s[s], ref["buf"])}
                results.append(r)
                assert r["O"] <= tol and r["buf"] <= 1e-6, r
            assert torch.equal(mat.params[i].cpu(), mat.masters[i].cpu().to(torch.bfloat16)), spec.name
        for j, (sel, w0, m0, v0, g) in vpick.items():
            ref = oadamw.adamw_step(w0, m0, v0, g, _f(h["adam_lr"]), _f(h["beta1"]), _f(h["beta2"]),
                                    _f(h["adam_eps"]), _f(h["adam_wd"]), t)
            got_w = mat.v_masters[j][sel].double().cpu().numpy()
            got_m = mat.v_exp_avg[j][sel].double().cpu().numpy()
            got_v = mat.v_exp_avg_sq[j][sel].double().cpu().numpy()
            for a_, b_ in ((got_w, ref["W"]), (got_m, ref["m"]), (got_v, ref["v"])):
                assert _maxrel(a_, b_) <= 1e-6, (wl.vectors[j].name, t)
            assert torch.equal(mat.v_params[j][sel], mat.v_masters[j][sel].to(torch.bfloat16))
    step.close()
    del mat, step
    gc.collect()
    torch.cuda.empty_cache()
    return results


def test_single_256x512_fp32(cuda_lib):
    res = _run(cuda_lib, "single_256x512", ["W", "tiny_3x4", "tiny_8x16"])
    assert len(res) == 3


def test_gpt2_small_three_steps(cuda_lib):
    names = [s.name for s in W.workload("gpt2_small").matrices]
    res = _run(cuda_lib, "gpt2_small", names, steps=3)
    assert len(res) == 72 * 3


def test_many_small_sampled(cuda_lib):
    wl = W.workload("many_small")
    # 48 sampled matrices spread over the list, both aspect ratios.
    names = [wl.matrices[i].name for i in range(0, 4096, 85)]
    res = _run(cuda_lib, "many_small", names)
    assert len(res) == len(names)


@pytest.mark.slow
def test_llama3_8b_sampled(cuda_lib):
    names = ["layers.0.k", "layers.17.q", "layers.3.gate", "layers.30.down"]
    res = _run(cuda_lib, "llama3_8b", names, adam_sample=1 << 20)
    assert len(res) == 4


@pytest.mark.slow
def test_llama3_8b_sampled_wide_tiles(cuda_lib):
    """Every launch that can (all but the fused last product) on 256 x 512
    tiles of the CTA-pair kernel."""
    cuda_lib.dmuon_set_tuning(12, 1)
    try:
        res = _run(cuda_lib, "llama3_8b", ["layers.1.v", "layers.12.o", "layers.5.up", "layers.21.down"])
    finally:
        cuda_lib.dmuon_set_tuning(12, 128)
    assert len(res) == 4


@pytest.mark.slow
def test_moe_experts_sampled(cuda_lib):
    names = ["layers.0.experts.w1", "layers.2.experts.w2"]
    res = _run(cuda_lib, "moe_experts", names, slice_pick=[3, 7])
    assert len(res) == 4
