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


# ---------------------------------------------------------------- KV-range sharded decode
def _states(q, rho, k, v, L, k0, k1, scale, splits):
    """Online-softmax states of positions [k0, min(k1, L)) of one (b, h), in
    ``splits`` equal parts, as the kernels lay them out: (m, l, C, 0, A[d],
    U[d]) with m in log2 units (an empty part: m = -inf, l = 0)."""
    import numpy as np
    q, rho, k, v = (np.asarray(a, np.float64) for a in (q, rho, k, v))
    d = q.shape[0]
    hi = min(k1, max(L, 0))
    n = max(hi - k0, 0)
    per = -(-n // splits) if n else 0
    out = np.zeros((splits, 2 * d + 4))
    for s in range(splits):
        a, b = k0 + s * per, min(k0 + (s + 1) * per, k0 + n)
        if b <= a:
            out[s, 0] = -np.inf
            continue
        sc = (k[a:b] @ q) * scale / np.log(2.0)
        m = sc.max()
        w = np.exp2(sc - m)
        r = k[a:b] @ rho
        out[s, 0], out[s, 1], out[s, 2] = m, w.sum(), (w * r).sum()
        out[s, 4:4 + d] = w @ v[a:b]
        out[s, 4 + d:] = (w * r) @ v[a:b]
    return out


def _merge(parts, d):
    """The log-sum-exp merge of (m, l, C, 0, A, U) states -> (o, lse)."""
    import numpy as np
    live = parts[parts[:, 0] > -np.inf]
    if len(live) == 0:
        return np.zeros(d), -np.inf
    M = live[:, 0].max()
    w = np.exp2(live[:, 0] - M)
    L, C = w @ live[:, 1], w @ live[:, 2]
    A, U = w @ live[:, 4:4 + d], w @ live[:, 4 + d:]
    vbar = A / L
    return (1 + C / L) * vbar - U / L, (M + np.log2(L)) * np.log(2.0)


def _kv_rank_main(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import numpy as np
    import torch
    import torch.distributed as dist
    import plx_inputs
    from parameterized_local_linear_02_b300 import kv_sharded
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, H, d, S = 4, 2, 8, 96
        x = plx_inputs.decode(B, H, d, S, seed=91, seqlens=np.array([96, 40, 1, 0]), rho_std=0.5)
        bounds = [(0, 50), (50, 96)]
        k0, k1 = bounds[rank]
        # ranks propose different split counts; both must use the larger
        n = kv_sharded.agree_num_splits([1, 2][rank])
        mine = np.stack([_states(x.q[b, h], x.rho[b, h], x.k_cache[b, h], x.v_cache[b, h], int(x.seqlens[b]),
                                 k0, k1, x.scale, n) for b in range(B) for h in range(H)])
        allp = kv_sharded.gather_partials(torch.from_numpy(mine.reshape(-1)))
        allp = allp.numpy().reshape(world, B * H, n, 2 * d + 4)
        res = {}
        for bh in range(B * H):
            res[divmod(bh, H)] = _merge(allp[:, bh].reshape(-1, 2 * d + 4), d)
        q.put((rank, n, allp[rank].reshape(-1).tolist() == mine.reshape(-1).tolist(),
               {k: (v[0].tolist(), float(v[1])) for k, v in res.items()}))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_the_decode_key_range_and_merge_exactly():
    """Each rank holds half of every sequence's cache positions; the ranks agree
    on a split count, all-gather their online-softmax states in rank order, and
    the log-sum-exp merge of them equals the oracle's decode over the whole
    range (lengths that end in the first shard, a length of one, and an empty
    sequence included)."""
    import numpy as np
    import oracle
    import plx_inputs
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_kv_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted((q.get(timeout=5) for _ in range(2)), key=lambda t: t[0])
    x = plx_inputs.decode(4, 2, 8, 96, seed=91, seqlens=np.array([96, 40, 1, 0]), rho_std=0.5)
    ref = oracle.decode("stream", x.q, x.rho, x.k_cache, x.v_cache, x.seqlens, x.scale)
    for rank, n, own_slot_is_own_rank, got in res:
        assert n == 2
        assert own_slot_is_own_rank                  # the gathered buffer is rank-major
        for bh, (o, lse) in got.items():
            ro, rl = ref[bh]
            assert np.allclose(o, ro, rtol=1e-10, atol=1e-12), (rank, bh)
            if np.isinf(rl):
                assert np.isinf(lse) and lse < 0
            else:
                assert abs(lse - rl) < 1e-10, (rank, bh)
