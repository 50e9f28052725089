"""Host logic of the multi-rank path, as two gloo ranks on the CPU.

* bench.py's slowest-rank reduction of the step time;
* the owner partition: every rank computes the LPT owner map of the Muon
  tensors on its own and all ranks agree, so each tensor has exactly one
  owner ("架构设计" §3.1, and invariant I1 of §8: a single global owner).
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys

    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import matrix_optimizer_step_gb300 as mos
        from matrix_optimizer_step_gb300 import build, workloads

        build.build()
        slowest = bench.reduce_max_over_ranks(10.0 + 5.0 * rank, dist, torch.device("cpu"))
        wl = workloads.workload("llama3_8b")
        owners, loads = mos.owner_partition([s.numel for s in wl.matrices], world)
        mine = torch.tensor(owners, dtype=torch.int64)
        gathered = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(gathered, mine)
        agree = all(torch.equal(g, mine) for g in gathered)
        q.put((rank, slowest, agree, owners, loads))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_slowest_time_and_owner_map():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=300) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    assert [o[1] for o in out] == [15.0, 15.0]
    assert all(o[2] for o in out)
    owners, loads = out[0][3], out[0][4]
    assert sorted(set(owners)) == [0, 1]
    # 224 tensors over 2 owners: LPT is within 4/3 - 1/6 of the perfect split.
    assert max(loads) <= (4 / 3 - 1 / 6) * sum(loads) / 2 + 1


def _shard_worker(rank, world, port, q):
    import sys

    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import numpy as np

        from matrix_optimizer_step_gb300.optim import adamw_shard_ranges, adamw_shard_views
        from oracle import adamw as oadamw

        numels = [4096, 77, 0, 100003, 768, 5]
        g = torch.Generator().manual_seed(3)
        W = [torch.randn(n, generator=g, dtype=torch.float64) * 0.02 for n in numels]
        m = [torch.randn(n, generator=g, dtype=torch.float64) * 1e-3 for n in numels]
        v = [torch.rand(n, generator=g, dtype=torch.float64) * 1e-6 for n in numels]
        G = [torch.randn(n, generator=g, dtype=torch.float64) for n in numels]
        runs = adamw_shard_ranges(numels, world)[rank]
        hyper = (1e-3, 0.9, 0.95, 1e-8, 0.1, 3)
        mine = []
        for w_, m_, v_, g_ in zip(*(adamw_shard_views(t, runs) for t in (W, m, v, G))):
            out = oadamw.adamw_step(w_.numpy(), m_.numpy(), v_.numpy(), g_.numpy(), *hyper)
            mine.append(np.concatenate([np.asarray(out[k]).reshape(-1) for k in ("W", "m", "v")]))
        sizes = [int(c) for _, _, c in runs]
        gathered = [None] * world
        dist.all_gather_object(gathered, (sizes, [x.tolist() for x in mine]))
        q.put((rank, gathered, runs))
    except Exception as e:  # report instead of leaving the parent waiting
        q.put((rank, repr(e), None))
        raise
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_sharded_adamw_rebuilds_the_full_step():
    """`sharded_adamw` route: each rank steps its contiguous piece of the
    AdamW tensors; gathering the pieces in rank order gives the full step."""
    import numpy as np

    from matrix_optimizer_step_gb300.optim import adamw_shard_ranges
    from oracle import adamw as oadamw

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted((q.get(timeout=300) for _ in procs), key=lambda o: o[0])
    for p in procs:
        p.join(timeout=60)
    assert all(o[2] is not None for o in out), out
    assert all(p.exitcode == 0 for p in procs)
    numels = [4096, 77, 0, 100003, 768, 5]
    # The pieces partition every tensor exactly once.
    seen = [np.zeros(n, dtype=int) for n in numels]
    for _, _, runs in out:
        for i, start, count in runs:
            seen[i][start:start + count] += 1
    assert all((s == 1).all() for s in seen)
    # Gathered pieces equal the full step, element by element.
    g = torch.Generator().manual_seed(3)
    W = [torch.randn(n, generator=g, dtype=torch.float64) * 0.02 for n in numels]
    m = [torch.randn(n, generator=g, dtype=torch.float64) * 1e-3 for n in numels]
    v = [torch.rand(n, generator=g, dtype=torch.float64) * 1e-6 for n in numels]
    G = [torch.randn(n, generator=g, dtype=torch.float64) for n in numels]
    full = {}
    for i in range(len(numels)):
        full[i] = oadamw.adamw_step(W[i].numpy(), m[i].numpy(), v[i].numpy(), G[i].numpy(), 1e-3, 0.9, 0.95, 1e-8,
                                    0.1, 3)
    gathered = out[0][1]
    assert gathered == out[1][1]
    for rank, (sizes, pieces) in enumerate(gathered):
        for (i, start, count), piece in zip(adamw_shard_ranges(numels, 2)[rank], pieces):
            want = np.concatenate([np.asarray(full[i][k]).reshape(-1)[start:start + count] for k in ("W", "m", "v")])
            assert np.array_equal(np.asarray(piece), want), (rank, i)
    sizes = [sum(s) for s, _ in gathered]
    assert abs(sizes[0] - sizes[1]) < 2 * 8  # one cut, moved by less than the alignment


def test_adamw_shard_ranges_edge_cases():
    from matrix_optimizer_step_gb300.optim import adamw_shard_ranges

    assert adamw_shard_ranges([], 3) == [[], [], []]
    assert adamw_shard_ranges([5], 4) == [[(0, 0, 5)], [], [], []]
    r = adamw_shard_ranges([10, 0, 7, 33], 3, align=4)
    assert [sum(c for _, _, c in x) for x in r] == [16, 20, 14]
    with pytest.raises(ValueError):
        adamw_shard_ranges([1], 0)
