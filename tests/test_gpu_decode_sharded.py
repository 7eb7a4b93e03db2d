"""plx_decode_partials + plx_decode_combine: the decode with its key range in
several shards (as on several GPUs), merged by the log-sum-exp combine, equals
plx_decode over the whole cache and the fp64 oracle.  The shards here live on
one GPU; the exchange between ranks is tested on CPU (test_multirank_cpu)."""
import numpy as np
import pytest

import oracle
import plx_inputs
from parity import LSE_F32, assert_f32, assert_lse


@pytest.mark.gpu
@pytest.mark.parametrize("d,with_rho,splits", [(128, True, 2), (64, False, 1), (128, True, 5)])
def test_sharded_key_range_merges_to_the_whole_decode(d, with_rho, splits):
    import torch
    import parameterized_local_linear_02_b300 as plx
    S = 700
    x = plx_inputs.decode(4, 4, d, S, seed=93, seqlens=np.array([700, 333, 1, 0]))
    t = x.device_tensors("cuda")
    rho = t["rho"] if with_rho else None
    bounds = [(0, 256), (256, 512), (512, 700)]       # the last shard is shorter
    n = plx.plx_decode_partials_size(4, 4, d, splits) // 4
    buf = torch.full((len(bounds) * n,), float("nan"), dtype=torch.float32, device="cuda")
    for g, (a, b) in enumerate(bounds):
        plx.plx_decode_partials(t["q"], rho, t["k_cache"][:, :, a:b].contiguous(),
                                t["v_cache"][:, :, a:b].contiguous(), t["seqlens"], key_begin=a,
                                num_splits=splits, out=buf[g * n:(g + 1) * n])
    out, lse = plx.plx_decode_combine(buf, groups=len(bounds), num_splits=splits, B=4, H=4, d=d,
                                      with_rho=with_rho, out_dtype=torch.float32)
    ref_out, ref_lse = plx.plx_decode(t["q"], rho, t["k_cache"], t["v_cache"], t["seqlens"],
                                      out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert plx.plx_last_device_error() == 0
    got, got_lse = out.cpu().numpy(), lse.cpu().numpy()
    assert_f32(got, ref_out.cpu().numpy(), "sharded vs plx_decode")
    assert_lse(got_lse, ref_lse.cpu().numpy(), LSE_F32, "sharded vs plx_decode")
    res = oracle.decode("stream", x.q, x.rho if with_rho else None, x.k_cache, x.v_cache, x.seqlens, x.scale)
    ref = np.stack([res[(b, h)][0] for b in range(4) for h in range(4)]).reshape(4, 4, d)
    rl = np.array([res[(b, h)][1] for b in range(4) for h in range(4)]).reshape(4, 4)
    assert_f32(got, ref, "sharded vs oracle")
    assert_lse(got_lse, rl, LSE_F32, "sharded vs oracle")
    assert np.all(got[3] == 0.0) and np.all(np.isneginf(got_lse[3]))    # the empty sequence


@pytest.mark.gpu
def test_a_shard_past_every_sequence_contributes_nothing():
    # a fourth shard beyond every length: its partials are the empty state and
    # the merge is unchanged bit for bit
    import torch
    import parameterized_local_linear_02_b300 as plx
    x = plx_inputs.decode(2, 2, 128, 300, seed=94, seqlens=np.array([300, 120]))
    t = x.device_tensors("cuda")
    n = plx.plx_decode_partials_size(2, 2, 128, 1) // 4
    kc, vc = t["k_cache"], t["v_cache"]
    far = torch.zeros((2, 2, 64, 128), dtype=torch.bfloat16, device="cuda")
    buf3 = torch.empty(2 * n, dtype=torch.float32, device="cuda")
    buf4 = torch.empty(3 * n, dtype=torch.float32, device="cuda")
    for g, (a, b) in enumerate([(0, 150), (150, 300)]):
        plx.plx_decode_partials(t["q"], t["rho"], kc[:, :, a:b].contiguous(), vc[:, :, a:b].contiguous(),
                                t["seqlens"], key_begin=a, num_splits=1, out=buf3[g * n:(g + 1) * n])
    buf4[:2 * n] = buf3
    plx.plx_decode_partials(t["q"], t["rho"], far, far, t["seqlens"], key_begin=300, num_splits=1,
                            out=buf4[2 * n:])
    o3, l3 = plx.plx_decode_combine(buf3, groups=2, num_splits=1, B=2, H=2, d=128, out_dtype=torch.float32)
    o4, l4 = plx.plx_decode_combine(buf4, groups=3, num_splits=1, B=2, H=2, d=128, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(o3, o4) and torch.equal(l3, l4)
    assert torch.all(torch.isneginf(buf4[2 * n:].view(4, -1)[:, 0]))
