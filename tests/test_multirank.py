"""The multi-process path of bench.py on CPU: world size 2 over gloo (127.0.0.1).
Each rank is an independent replica; the only cross-rank traffic is the timing
barrier and the max / sum reductions of the per-rank timings and byte counts,
and the reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, local, pg = bench.dist_setup(world)
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(pg)
    mx = bench.max_over_ranks(pg, float(rank + 1) * 1.5)     # the slowest rank's time
    sm = bench.sum_over_ranks(pg, 1000.0 * (rank + 1))        # bytes moved by all ranks
    # the reference arm prints on rank 0 only; other ranks return without work
    ran = None
    if rank != 0:
        class A:
            steps, warmup = 1, 0
        ran = bench.main_reference(A()) is None
    out.put((rank, mx, sm, ran))
    pg.destroy_process_group()


def test_two_rank_gloo_barrier_and_reductions():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [3.0, 3.0]
    assert [r[2] for r in res] == [3000.0, 3000.0]
    assert res[1][3] is True
