"""The owner-partitioned step with the CUDA kernels, two ranks on one GPU.

Two processes share cuda:0 and a gloo group (the collectives run on the
host; no kernel of one process waits for the other).  Each rank steps only
the tensors it owns and its piece of the sharded AdamW tensors, after the
mean gradients have been reduced to it, and publishes the bf16 parameters
("架构设计" §2 and §4; "Pure DMuon 路由" route table).  After two steps:

* both ranks hold the same bf16 parameters;
* they equal, bit for bit, one process stepping every tensor with
  OwnerStep on the same mean gradients (gathered from the owners), and so
  do the owners' fp32 masters and momenta and the AdamW pieces;
* the Newton-Schulz outputs and the AdamW state match the float64 oracle
  within the parity tolerances (2e-2 / 1e-4 relative Frobenius for bf16 /
  fp32 slices, 1e-6 for the AdamW master).
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUON = [(256, 512), (384, 128), (2, 128, 192), (24, 256), (640, 320)]
ADAMW = [768, 4096]
SHARDED = [64000, 12345]
MUON_KW = dict(lr=0.02, momentum=0.95, wd=0.01, ns_steps=5, a=3.4445, b=-4.7750, c=2.0315)
ADAM_KW = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1)


def _shapes():
    return MUON + [(n,) for n in ADAMW] + [(n,) for n in SHARDED]


def _weights():
    g = torch.Generator().manual_seed(21)
    return [torch.randn(s, generator=g) * 0.02 for s in _shapes()]


def _grads(rank, step):
    g = torch.Generator().manual_seed(500 * step + rank)
    return [torch.randn(s, generator=g).to(torch.bfloat16) for s in _shapes()]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q, backend="gloo"):
    import sys

    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    os.environ["NCCL_NVLS_ENABLE"] = "0"
    import torch.distributed as dist

    if backend == "nccl":
        torch.cuda.set_device(0)
    dist.init_process_group(backend, rank=rank, world_size=world)
    try:
        torch.cuda.set_device(0)
        from matrix_optimizer_step_gb300.owner_dist import DistributedOwnerStep, OwnerLayout

        L = OwnerLayout.build(MUON, ADAMW, SHARDED, world)
        ds = DistributedOwnerStep(L, device="cuda:0")
        ds.load_masters([w.cuda() for w in _weights()])
        mean = []  # per step: this rank's reduced gradients (its owner range, its sharded piece)
        r0, r1 = rank * L.piece, (rank + 1) * L.piece
        for step in (1, 2):
            for gv, gh in zip(ds.grads(), _grads(rank, step)):
                gv.copy_(gh.reshape(gv.shape))
            ds.step(MUON_KW, dict(ADAM_KW, step=step))
            torch.cuda.synchronize()
            ds.stepper.sync()
            a, b = L.owner_range[rank]
            mean.append((ds.grad_flat[a:b].view(torch.int16).cpu().numpy(),
                         ds.sp_grad_flat[r0:r1].view(torch.int16).cpu().numpy()))
        q.put((rank, ds.param_flat.view(torch.int16).cpu().numpy(), ds.sp_param_flat.view(torch.int16).cpu().numpy(),
               {i: ds.masters[i].cpu().numpy() for i in ds.masters},
               {i: ds.momenta[i].cpu().numpy() for i in ds.momenta}, ds.sp_master.cpu().numpy(), mean))
        ds.close()
    except Exception as e:
        q.put((rank, repr(e), None, None, None, None, None))
        raise
    finally:
        dist.destroy_process_group()


def _frob(x, y):
    d = np.linalg.norm(y)
    return float(np.linalg.norm(x - y) / (d if d > 0 else 1.0))


def _run_ranks(world, backend):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q, backend)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted((q.get(timeout=600) for _ in procs), key=lambda o: o[0])
    for p in procs:
        p.join(timeout=120)
    assert all(o[1] is not None and not isinstance(o[1], str) for o in out), [o[1] for o in out]
    assert all(p.exitcode == 0 for p in procs)
    return out


def test_two_ranks_on_one_gpu_equal_one_process(cuda_lib):
    out = _run_ranks(2, "gloo")
    assert np.array_equal(out[0][1], out[1][1]) and np.array_equal(out[0][2], out[1][2])
    _check_against_one_process(cuda_lib, out, 2)


def test_nccl_group_of_one_equals_one_process(cuda_lib):
    """The NCCL branch of the collectives (mean by ReduceOp.AVG, in-place
    reduce_scatter and all_gather on views of the flat buffers, broadcast)
    on a group of one rank: the only NCCL group one GPU can hold without
    ranks that wait on one another.  Every collective is then an identity,
    so the step must equal one process stepping every tensor, bit for bit."""
    out = _run_ranks(1, "nccl")
    _check_against_one_process(cuda_lib, out, 1)


def _check_against_one_process(mos, out, world):
    from matrix_optimizer_step_gb300.owner_dist import OwnerLayout
    from oracle import adamw as oadamw
    from oracle import muon as omuon

    L = OwnerLayout.build(MUON, ADAMW, SHARDED, world)
    n_muon, n_own = len(MUON), len(MUON) + len(ADAMW)
    shapes = _shapes()

    def mean_grads(step):
        """The mean gradients as the owners received them, per tensor."""
        flat = np.zeros(L.owner_numel, dtype=np.int16)
        sp = np.zeros(L.sharded_numel, dtype=np.int16)
        for r in range(world):
            a, b = L.owner_range[r]
            flat[a:b] = out[r][6][step][0]
            sp[r * L.piece:(r + 1) * L.piece] = out[r][6][step][1]
        flat = torch.from_numpy(flat).view(torch.bfloat16)
        sp = torch.from_numpy(sp).view(torch.bfloat16)
        g = [flat[L.offset[i]:L.offset[i] + int(np.prod(shapes[i]))].reshape(shapes[i]) for i in range(n_own)]
        g += [sp[o:o + n] for o, n in zip(L.sharded_offset, L.sharded_numels)]
        return g

    # One process, every tensor, the same mean gradients.
    dev = torch.device("cuda")
    W = _weights()
    Wd = [w.to(dev) for w in W]
    Bd = [torch.zeros(s, device=dev) for s in MUON]
    Md = [torch.zeros(w.numel(), device=dev) for w in W[n_muon:]]
    Vd = [torch.zeros(w.numel(), device=dev) for w in W[n_muon:]]
    Gd = [torch.empty(s, device=dev, dtype=torch.bfloat16) for s in shapes]
    Pd = [torch.empty(s, device=dev, dtype=torch.bfloat16) for s in shapes]
    st = mos.OwnerStep(0)
    st.set_muon(Wd[:n_muon], Bd, Gd[:n_muon], Pd[:n_muon])
    st.set_adamw([w.reshape(-1) for w in Wd[n_muon:]], Md, Vd, [g.reshape(-1) for g in Gd[n_muon:]],
                 [p.reshape(-1) for p in Pd[n_muon:]])
    ref_W = [w.double().numpy() for w in W]
    ref_B = [np.zeros(s) for s in MUON]
    ref_M = [np.zeros(w.numel()) for w in W[n_muon:]]
    ref_V = [np.zeros(w.numel()) for w in W[n_muon:]]
    f = lambda x: float(np.float32(x))  # noqa: E731
    for step in (1, 2):
        G = mean_grads(step - 1)
        for gd, gh in zip(Gd, G):
            gd.copy_(gh)
        W_before = [w.double().cpu().numpy() for w in Wd[:n_muon]]
        st.muon_step(**MUON_KW)
        st.adamw_step(**ADAM_KW, step=step)
        st.sync()
        for i, s in enumerate(MUON):
            ref = omuon.muon_step(W_before[i], ref_B[i], G[i].double().numpy(), f(0.02), f(0.95), f(0.01), 5,
                                  f(3.4445), f(-4.7750), f(2.0315))
            m, n = s[-2], s[-1]
            O = (W_before[i] * (1 - f(0.02) * f(0.01)) - Wd[i].double().cpu().numpy()) / (f(0.02) * omuon.shape_scale(m, n))
            tol = 1e-4 if min(m, n) < 64 else 2e-2
            Os, Rs = O.reshape(-1, m, n), ref["O"].reshape(-1, m, n)
            for k in range(Os.shape[0]):
                assert _frob(Os[k], Rs[k]) <= tol, (s, step, k)
            ref_B[i] = Bd[i].double().cpu().numpy()
        for k, w in enumerate(W[n_muon:]):
            ref = oadamw.adamw_step(ref_W[n_muon + k].reshape(-1), ref_M[k], ref_V[k], G[n_muon + k].double().numpy().reshape(-1),
                                    f(1e-3), f(0.9), f(0.95), f(1e-8), f(0.1), step)
            got = Wd[n_muon + k].double().cpu().numpy().reshape(-1)
            assert np.max(np.abs(got - ref["W"])) <= 1e-6 * np.max(np.abs(ref["W"])), (k, step)
            ref_W[n_muon + k] = got
            ref_M[k] = Md[k].double().cpu().numpy()
            ref_V[k] = Vd[k].double().cpu().numpy()

    # Distributed result, bit for bit against the one-process result.
    pf = out[0][1]
    sp = out[0][2]
    for i in range(n_own):
        n = int(np.prod(shapes[i]))
        assert np.array_equal(pf[L.offset[i]:L.offset[i] + n], Pd[i].reshape(-1).view(torch.int16).cpu().numpy()), i
        owner = L.owner[i]
        assert np.array_equal(out[owner][3][i].reshape(-1), Wd[i].reshape(-1).cpu().numpy()), i
        if i < n_muon:
            assert np.array_equal(out[owner][4][i].reshape(-1), Bd[i].reshape(-1).cpu().numpy()), i
    full_master = np.concatenate([out[r][5] for r in range(world)])
    for k, (o, n) in enumerate(zip(L.sharded_offset, L.sharded_numels)):
        i = n_own + k
        assert np.array_equal(sp[o:o + n], Pd[i].view(torch.int16).cpu().numpy()), i
        assert np.array_equal(full_master[o:o + n], Wd[i].cpu().numpy()), i
    st.close()


def test_bench_owner_mode_on_two_ranks_of_one_gpu(cuda_lib):
    """bench.py's owner-partitioned mode end to end under torchrun: two ranks
    on one GPU over gloo (a check of the code path; its timings mean
    nothing).  One JSON line from rank 0, strong scaling, both ranks own
    tensors and launched kernels."""
    import json
    import subprocess
    import sys

    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--gpus", "2", "--workload", "gpt2_small", "--steps", "2", "--warmup", "3", "--dist-backend", "gloo"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and d["scaling"] == "strong" and d["ms_per_step"] > 0
    per = d["owner"]["per_rank"]
    assert len(per) == 2 and all(p["launches"] > 0 and p["ns_ms"] > 0 for p in per)
    assert all(n > 0 for n in d["owner"]["owned_elements"])


def test_bench_owner_mode_on_an_nccl_group_of_one(cuda_lib):
    """bench.py's owner-partitioned mode under torchrun with one rank on
    NCCL: the process-group code of the mode (collectives of the step,
    gathers of the per-rank statistics, barriers, the max over ranks) on
    the NCCL backend, on the hardware (a group of one: nothing waits on
    another rank)."""
    import json
    import subprocess
    import sys

    port = _free_port()
    env = dict(os.environ, NCCL_NVLS_ENABLE="0")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "1",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--gpus", "1", "--mode", "owner", "--workload", "gpt2_small", "--steps", "2", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900, env=env)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["n_gpus"] == 1 and d["scaling"] == "strong" and d["ms_per_step"] > 0
    assert d["config"]["backend"] == "nccl" and len(d["owner"]["per_rank"]) == 1
