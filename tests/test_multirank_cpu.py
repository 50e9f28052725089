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
