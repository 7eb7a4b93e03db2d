"""The multi-rank path of the benchmark on CPU: two gloo ranks on 127.0.0.1.

The attention path shards into independent (batch, head) problems, so ranks
share no data and exchange only the timing: a barrier around the timed
region and the slowest rank's time (max over ranks).  These tests run that
host logic with world_size 2 (no GPU)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, lr = bench.dist_setup()
        assert (w, r, lr) == (world, rank, rank)
        bench.barrier(w)
        ms = [2.0, 5.0][rank]                       # rank 1 is the slow one
        slowest = bench.max_over_ranks(ms, w)
        value = bench.weak_scaling_value(1.0e9, ms, w)
        seeds = (bench.rank_seed(7, 0), bench.rank_seed(7, 1))
        # the reference arm runs on rank 0 only; the other ranks leave without work
        class A:                                        # noqa: N801 - argparse stand-in
            steps, warmup, gpus = 1, 0, world
        ref_rc = bench.run_reference(A, w, r) if r != 0 else None
        q.put((rank, slowest, value, seeds, ref_rc))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_weak_scaling():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, slowest, value, seeds, ref_rc in res:
        assert slowest == 5.0                      # both ranks see the slowest time
        assert value == pytest.approx(2 * 1.0e9 / 5.0e-3)
        assert seeds[0] == 7 and seeds[0] != seeds[1]
    assert res[1][4] == 0                          # rank 1 of the reference arm exits 0 without work
