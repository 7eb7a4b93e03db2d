"""plx_fwd_cached: T new query tokens per sequence against a bf16 KV cache on
the tensor cores, against the fp64 oracle (query row i of sequence b at
position seqlens[b] - T + i).  Cache rows past each sequence hold NaN: they
must not reach the output."""
import numpy as np
import pytest

import oracle
import plx_inputs
from parity import LSE_BF16, assert_bf16, assert_lse

pytestmark = pytest.mark.gpu

NAN_BF16 = np.int16(0x7FC0)


def make(B, H, T, S_cap, d, seqlens, seed):
    rng = np.random.default_rng(seed)
    x = plx_inputs.prefill(B, H, S_cap, d, seed=seed, dtype="bf16", rho="normal", rho_std=0.3)
    kb = x.bits["k"].view(np.int16).copy()
    vb = x.bits["v"].view(np.int16).copy()
    for b in range(B):
        kb[b, :, seqlens[b]:, :] = NAN_BF16
        vb[b, :, seqlens[b]:, :] = NAN_BF16
    # the T newest positions of each sequence carry the queries and probes
    qb = np.zeros((B, H, T, d), np.int16)
    rb = np.zeros((B, H, T, d), np.int16)
    for b in range(B):
        qb[b] = x.bits["q"].view(np.int16)[b, :, seqlens[b] - T:seqlens[b], :]
        rb[b] = x.bits["rho"].view(np.int16)[b, :, seqlens[b] - T:seqlens[b], :]
    return x, qb, rb, kb, vb


def run(B, H, T, S_cap, d, seqlens, seed, rho=True):
    import torch
    import parameterized_local_linear_02_b300 as plx
    x, qb, rb, kb, vb = make(B, H, T, S_cap, d, seqlens, seed)
    dev = lambda a: torch.from_numpy(a).view(torch.bfloat16).cuda()
    out, lse = plx.plx_fwd_cached(dev(qb), dev(rb) if rho else None, dev(kb), dev(vb),
                                  torch.tensor(seqlens, dtype=torch.int32, device="cuda"), scale=x.scale,
                                  out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert plx.plx_last_device_error() == 0
    got, lg = out.cpu().numpy(), lse.cpu().numpy()
    exp, le = np.zeros_like(got), np.zeros_like(lg)
    form = "stream" if rho else "sa"
    for b in range(B):
        rows = np.arange(seqlens[b] - T, seqlens[b])
        res = oracle.prefill(form, x.q[b:b + 1], x.k[b:b + 1], x.v[b:b + 1], x.rho[b:b + 1], x.scale, rows=rows)
        for h in range(H):
            exp[b, h], le[b, h] = res[(0, h)][0], res[(0, h)][1]
    assert np.all(np.isfinite(got))
    return got, exp, lg, le


@pytest.mark.parametrize("T,S_cap,seqlens", [(16, 512, [512, 300, 16]), (200, 640, [600, 200, 457]),
                                             (1, 256, [256, 1, 77]), (128, 384, [383, 128, 129]),
                                             (64, 512, [512, 64, 100]), (65, 512, [512, 65, 400]),
                                             (33, 300, [300, 33, 250])])
def test_cached_matches_oracle(T, S_cap, seqlens):
    got, exp, lg, le = run(3, 2, T, S_cap, 128, seqlens, seed=T + S_cap)
    assert_bf16(got, exp, f"cached T={T}")
    assert_lse(lg, le, LSE_BF16, f"cached lse T={T}")


def test_cached_softmax_attention_and_d64():
    got, exp, lg, le = run(2, 3, 40, 300, 64, [300, 45], seed=9, rho=False)
    assert_bf16(got, exp, "cached SA d=64")
    assert_lse(lg, le, LSE_BF16, "cached SA lse")


def test_cached_full_cache_equals_prefill():
    """T = N = S_cap with seqlens = N is the self-attention prefill: the same
    kernel gives the same bits."""
    import torch
    import parameterized_local_linear_02_b300 as plx
    x = plx_inputs.prefill(1, 2, 300, 128, seed=3, dtype="bf16", rho="normal", rho_std=0.3)
    t = x.device_tensors()
    o1, l1 = plx.plx_fwd(t["q"], t["k"], t["v"], t["rho"], scale=x.scale, out_dtype=torch.float32)
    o2, l2 = plx.plx_fwd_cached(t["q"], t["rho"], t["k"], t["v"], torch.tensor([300], dtype=torch.int32,
                                device="cuda"), scale=x.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
