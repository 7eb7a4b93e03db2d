"""plx_decode_noalloc: decode without a caller workspace.

Some callers cannot allocate device memory at the point where they decode:
they run under an allocator that owns all of the device memory, or in a
process whose footprint must not grow after start-up. plx_decode_noalloc
serves them. It keeps its split partials in a static device array that the
library holds. These tests call it through the C ABI and compare it with
plx_decode on the same inputs and the same split count. They make two calls
in a row with different data, so a call that read partials left behind by
the previous call would fail. The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest

import plx_inputs
from parity import LSE_F32, assert_f32, assert_lse

SCRATCH_BYTES = 4 << 20


def _decode_pair(x, splits):
    import torch
    import parameterized_local_linear_02_b300 as plx
    t = x.device_tensors("cuda")
    ref_out, ref_lse = plx.plx_decode(t["q"], t["rho"], t["k_cache"], t["v_cache"], t["seqlens"],
                                      num_splits=splits, out_dtype=torch.float32)
    out = torch.full_like(ref_out, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    plx.plx_decode_noalloc(t["q"], t["rho"], t["k_cache"], t["v_cache"], t["seqlens"],
                           num_splits=splits, out=out, lse=lse)
    torch.cuda.synchronize()
    assert plx.plx_last_device_error() == 0
    return (out.cpu().numpy(), lse.cpu().numpy()), (ref_out.cpu().numpy(), ref_lse.cpu().numpy())


@pytest.mark.gpu
@pytest.mark.parametrize("splits", [5, 0])
def test_noalloc_matches_plx_decode_on_two_calls_in_a_row(splits):
    # two different problems back to back: the second must not see the
    # first call's partials, which stay in the shared scratch
    first = plx_inputs.decode(3, 4, 128, 700, seed=71, seqlens=np.array([700, 13, 400]))
    second = plx_inputs.decode(2, 4, 128, 900, seed=72, seqlens=np.array([1, 900]))
    for n, x in enumerate((first, second)):
        (out, lse), (ref_out, ref_lse) = _decode_pair(x, splits)
        assert_f32(out, ref_out, f"noalloc call {n + 1}, splits={splits}")
        assert_lse(lse, ref_lse, LSE_F32, f"noalloc call {n + 1}, splits={splits}")


# (B, H, S_cap) at d = 128 whose automatic split count is above what the
# scratch holds for some plausible resident-block count of the split kernel
CAPPED_CANDIDATES = [(85, 16, 2048), (25, 16, 8192), (28, 16, 8192), (56, 16, 4096), (98, 16, 2048),
                     (100, 16, 2048)]


@pytest.mark.gpu
def test_noalloc_caps_the_automatic_split_count_to_the_scratch():
    # a shape where plx_decode would pick more splits than 4 MiB holds: the
    # automatic count must come down to the largest that fits, and the result
    # must equal plx_decode run with exactly that count
    import torch
    import parameterized_local_linear_02_b300 as plx
    d = 128
    chosen = None
    for B, H, S_cap in CAPPED_CANDIDATES:
        fit = SCRATCH_BYTES // (B * H * (2 * d + 4) * 4)
        auto = plx.plx_decode_num_splits(B, H, d, S_cap)
        if fit >= 2 and auto > fit:
            chosen = (B, H, S_cap, fit, auto)
            break
    assert chosen is not None, "no candidate shape needs more splits than the scratch holds"
    B, H, S_cap, fit, auto = chosen
    t = plx_inputs.decode_device(B, H, d, S_cap, seed=73, seqlens="ragged", device="cuda")
    ref_out, ref_lse = plx.plx_decode(t["q"], t["rho"], t["k_cache"], t["v_cache"], t["seqlens"],
                                      num_splits=fit, out_dtype=torch.float32)
    auto_out, _ = plx.plx_decode(t["q"], t["rho"], t["k_cache"], t["v_cache"], t["seqlens"],
                                 num_splits=0, out_dtype=torch.float32)
    out = torch.full_like(ref_out, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    plx.plx_decode_noalloc(t["q"], t["rho"], t["k_cache"], t["v_cache"], t["seqlens"],
                           num_splits=0, out=out, lse=lse)
    torch.cuda.synchronize()
    assert plx.plx_last_device_error() == 0
    where = f"noalloc B={B} H={H} S_cap={S_cap}: {auto} splits capped to {fit}"
    # the same kernels with the same split count: the same bits
    assert torch.equal(out, ref_out), where
    assert torch.equal(lse, ref_lse), where
    # and within fp32 rounding of plx_decode's own (larger) split count
    assert_f32(out.cpu().numpy(), auto_out.cpu().numpy(), where)


def test_noalloc_rejects_a_split_count_beyond_the_scratch():
    # host-side check before any device access (fake, never dereferenced pointers)
    import parameterized_local_linear_02_b300 as plx
    lib = plx.library()
    p = ctypes.c_void_p(0x10000)
    B, H, d = 64, 16, 128
    splits = SCRATCH_BYTES // (B * H * (2 * d + 4) * 4) + 1
    st = lib.plx_decode_noalloc(p, p, p, p, p, p, p, B, H, d, 4096, 0.088, splits, 1, None)
    assert st == 2, plx.plx_strerror(st)
