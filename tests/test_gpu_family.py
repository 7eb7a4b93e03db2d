"""Family switches (plx_fwd_family, plx_decode_family) against the fp64
oracle: the no-intercept member, o = -(sum_j w_ij v_j k_j^T) rho_i, and with
uniform weights linear attention with probe -rho (zhichai.net section 2.1)."""
import numpy as np
import pytest

import oracle
import plx_inputs
from parity import LSE_BF16, assert_bf16, assert_lse

pytestmark = pytest.mark.gpu

UNIFORM, NOINT = 0x1, 0x2


def fwd(x, flags):
    import torch
    import parameterized_local_linear_02_b300 as plx
    t = x.device_tensors()
    out, lse = plx.plx_fwd_family(t["q"], t["k"], t["v"], t["rho"], flags=flags, scale=x.scale,
                                  out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert plx.plx_last_device_error() == 0
    return out.cpu().numpy(), lse.cpu().numpy()


def ref(x, form, scale):
    res = oracle.prefill(form, x.q, x.k, x.v, x.rho, scale)
    B, H = x.q.shape[:2]
    return (np.stack([np.stack([res[(b, h)][0] for h in range(H)]) for b in range(B)]),
            np.stack([np.stack([res[(b, h)][1] for h in range(H)]) for b in range(B)]))


@pytest.mark.parametrize("shape", [(1, 2, 200, 128), (2, 1, 129, 64)])
def test_no_intercept_prefill(shape):
    B, H, N, d = shape
    x = plx_inputs.prefill(B, H, N, d, seed=N + 3, dtype="bf16", rho="normal", rho_std=0.3)
    got, lg = fwd(x, NOINT)
    exp, le = ref(x, "noint", x.scale)
    assert_bf16(got, exp, f"no intercept {shape}")
    assert_lse(lg, le, LSE_BF16, "no intercept lse")


def test_uniform_no_intercept_is_linear_attention():
    x = plx_inputs.prefill(1, 2, 150, 128, seed=77, dtype="bf16", rho="normal", rho_std=0.3)
    got, lg = fwd(x, UNIFORM | NOINT)
    exp, _ = ref(x, "noint", 0.0)
    assert_bf16(got, exp, "uniform + no intercept")
    # lse of uniform weights: ln(i + 1)
    n = np.arange(1, 151, dtype=np.float64)
    assert_lse(lg, np.broadcast_to(np.log(n), lg.shape), LSE_BF16, "uniform lse")
    # uniform weights alone: PLX at scale 0
    got_u, _ = fwd(x, UNIFORM)
    exp_u, _ = ref(x, "stream", 0.0)
    assert_bf16(got_u, exp_u, "uniform weights")


def test_no_intercept_decode():
    import torch
    import parameterized_local_linear_02_b300 as plx
    dd = plx_inputs.decode(3, 2, 128, 700, seed=12, seqlens=np.array([700, 1, 333]))
    t = dd.device_tensors()
    for splits in (1, 3):
        o, l = plx.plx_decode_family(t["q"], t["rho"], t["k_cache"], t["v_cache"], t["seqlens"], flags=NOINT,
                                     num_splits=splits, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert plx.plx_last_device_error() == 0
        res = oracle.decode("noint", dd.q, dd.rho, dd.k_cache, dd.v_cache, dd.seqlens, dd.scale)
        exp = np.stack([np.stack([res[(b, h)][0] for h in range(2)]) for b in range(3)])
        got = o.cpu().numpy()
        err = np.abs(got - exp).max() / np.sqrt(np.mean(exp ** 2))
        assert err <= 1e-4, f"decode no intercept splits={splits}: {err:.2e}"
