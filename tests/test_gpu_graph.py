"""A steady-state step enqueues kernel launches only (its plan, pointer
tables and tensor maps are reused unchanged), so it can be captured into a
CUDA graph and replayed; replays must match eager steps bit for bit."""

import pytest
import torch

pytestmark = pytest.mark.gpu

A, B, C = 3.4445, -4.7750, 2.0315
SHAPES = [(256, 512), (384, 128), (3, 64, 96), (24, 320), (1000, 130)]


def _state(seed, dev):
    g = torch.Generator().manual_seed(seed)
    W = [(torch.randn(s, generator=g) * 0.02).to(dev) for s in SHAPES]
    Bf = [torch.zeros(s, device=dev) for s in SHAPES]
    G = [torch.empty(s, device=dev, dtype=torch.bfloat16) for s in SHAPES]
    P = [torch.empty(s, device=dev, dtype=torch.bfloat16) for s in SHAPES]
    vW = [(torch.randn(n, generator=g) * 0.02).to(dev) for n in (4096, 77)]
    vm = [torch.zeros(n, device=dev) for n in (4096, 77)]
    vv = [torch.zeros(n, device=dev) for n in (4096, 77)]
    vG = [torch.empty(n, device=dev, dtype=torch.bfloat16) for n in (4096, 77)]
    vP = [torch.empty(n, device=dev, dtype=torch.bfloat16) for n in (4096, 77)]
    return dict(W=W, B=Bf, G=G, P=P, vW=vW, vm=vm, vv=vv, vG=vG, vP=vP)


def test_steady_state_step_replays_from_a_cuda_graph(cuda_lib):
    dev = torch.device("cuda")
    a, b = _state(7, dev), _state(7, dev)
    sa, sb = cuda_lib.OwnerStep(0), cuda_lib.OwnerStep(0)
    for s, st in ((sa, a), (sb, b)):
        s.set_muon(st["W"], st["B"], st["G"], st["P"])
        s.set_adamw(st["vW"], st["vm"], st["vv"], st["vG"], st["vP"])
    g = torch.Generator().manual_seed(8)
    grads = [[torch.randn(t.shape, generator=g).to(t.dtype) for t in a["G"] + a["vG"]] for _ in range(5)]
    adam = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1, step=1)

    def load(st, k):
        for d, h in zip(st["G"] + st["vG"], grads[k]):
            d.copy_(h)

    # Two eager steps on both sides build the plans and upload the tables.
    for k in range(2):
        for s, st in ((sa, a), (sb, b)):
            load(st, k)
            s.muon_step(0.02, 0.95, 0.01, 5, A, B, C)
            s.adamw_step(**adam)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(graph, stream=side):
        sb.muon_step(0.02, 0.95, 0.01, 5, A, B, C, stream=side)
        sb.adamw_step(stream=side, **adam)
    torch.cuda.synchronize()
    for k in range(2, 5):
        load(a, k)
        sa.muon_step(0.02, 0.95, 0.01, 5, A, B, C)
        sa.adamw_step(**adam)
        load(b, k)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
    sa.sync()
    sb.sync()
    for key in ("W", "B", "P", "vW", "vm", "vv", "vP"):
        for i, (x, y) in enumerate(zip(a[key], b[key])):
            assert torch.equal(x, y), (key, i)
    sa.close()
    sb.close()
