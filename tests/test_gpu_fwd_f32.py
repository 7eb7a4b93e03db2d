"""plx_fwd_f32 (fp32 CUDA-core path) against the fp64 oracle."""
import numpy as np
import pytest

import oracle
import plx_inputs
from parity import LSE_F32, assert_f32, assert_lse

pytestmark = pytest.mark.gpu


def run(x, rho=True):
    import torch
    import parameterized_local_linear_02_b300 as plx
    t = {n: torch.from_numpy(getattr(x, n)).cuda() for n in ("q", "k", "v", "rho")}
    out, lse = plx.plx_fwd_f32(t["q"], t["k"], t["v"], t["rho"] if rho else None, scale=x.scale)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


def oracle_all(x, form):
    res = oracle.prefill(form, x.q, x.k, x.v, x.rho, x.scale)
    out = np.stack([np.stack([res[(b, h)][0] for h in range(x.H)]) for b in range(x.B)])
    lse = np.stack([np.stack([res[(b, h)][1] for h in range(x.H)]) for b in range(x.B)])
    return out, lse


def test_tiny_f32_workload_matches_oracle():
    """B=1, H=2, N=128, d=64, fp32, rho ~ N(0, 0.1^2), seed 0: every row."""
    cfg = plx_inputs.CONFIGS["tiny_f32"]
    x = plx_inputs.prefill(cfg["B"], cfg["H"], cfg["N"], cfg["d"], seed=cfg["seed"], dtype="f32",
                           rho="normal", rho_std=cfg["rho_std"])
    out, lse = run(x)
    ref, lref = oracle_all(x, "explicit")
    assert_f32(out, ref, "tiny fp32 PLX")
    assert_lse(lse, lref, LSE_F32, "tiny fp32 lse")


def test_tiny_f32_zero_probe_is_softmax_attention():
    cfg = plx_inputs.CONFIGS["tiny_f32"]
    x = plx_inputs.prefill(cfg["B"], cfg["H"], cfg["N"], cfg["d"], seed=cfg["seed"], dtype="f32",
                           rho="zero")
    out0, lse0 = run(x, rho=True)
    out_sa, lse_sa = run(x, rho=False)
    assert np.array_equal(out0, out_sa), "rho = 0 must equal the SA instantiation bit for bit"
    ref, lref = oracle_all(x, "sa")
    assert_f32(out_sa, ref, "tiny fp32 SA")
    assert_lse(lse_sa, lref, LSE_F32, "tiny fp32 SA lse")


@pytest.mark.parametrize("shape", [(2, 3, 77, 32), (1, 1, 1, 64), (1, 2, 200, 128), (1, 1, 40, 256)])
def test_f32_ragged_shapes(shape):
    B, H, N, d = shape
    x = plx_inputs.prefill(B, H, N, d, seed=N + d, dtype="f32", rho="normal", rho_std=0.3)
    out, lse = run(x)
    ref, lref = oracle_all(x, "stream")
    assert_f32(out, ref, f"fp32 {shape}")
    assert_lse(lse, lref, LSE_F32, f"fp32 lse {shape}")
