"""The multi-process side of bench.py on the CPU: two gloo ranks, as `torchrun
--nproc-per-node 2 bench.py` would start them on two GPUs. Each GPU compresses its own
replica of the workload (no data-path collective); the ranks only agree on the slowest
rank's time, and the whole-job rate counts every rank's words."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist
    r, w, l = bench.dist_init("gloo")
    ms = 10.0 * (rank + 1)  # rank 1 is the slower one
    bench.barrier()
    slowest = bench.reduce_max(ms)
    gbs = bench.whole_job_gbs(4e9, w, 5, slowest)
    # the reference arm: only rank 0 runs the oracle and prints; the others exit at once
    class A:
        gpus, steps, warmup, chunk_elems = w, 1, 0, 4096
    ref_rc = bench.run_reference(A) if rank != 0 else None
    q.put((r, w, l, slowest, gbs, ref_rc))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_count_every_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r, w, l, slowest, gbs, ref_rc) in enumerate(got):
        assert (r, w, l) == (rank, 2, rank)
        assert slowest == 20.0  # max over ranks, on every rank
        # 4 GB per rank per step, 2 ranks, 5 steps in 20 ms
        assert gbs == pytest.approx(4e9 * 2 * 5 / 0.020 / 1e9)
    assert got[1][5] == 0  # rank 1 of the reference arm exits 0 without work


def test_one_process_needs_no_process_group():
    assert bench.reduce_max(3.5) == 3.5
    assert bench.whole_job_gbs(1e9, 1, 2, 1000.0) == pytest.approx(2.0)
