"""plx_bwd_f32 (fp32 backward on the CUDA cores) against the fp64 autograd
oracle of the explicit-covariance forward."""
import numpy as np
import pytest

import plx_inputs
from oracle.backward import plx_backward
from parity import assert_f32

pytestmark = pytest.mark.gpu

GRAD_TOL = 1e-4      # fp32 arithmetic: max and mean |err| / RMS(oracle gradient)


def assert_grad(got, ref, what):
    """fp32 tolerance relative to the oracle gradient's RMS; a gradient that is
    exactly zero (e.g. dq, dk, drho at N = 1, where o_0 = v_0) must come out
    zero to within fp32 rounding."""
    if float(np.sqrt(np.mean(np.asarray(ref, np.float64) ** 2))) == 0.0:
        assert float(np.max(np.abs(got))) <= 1e-6, f"{what}: expected zero, max {np.max(np.abs(got)):.2e}"
    else:
        assert_f32(got, ref, what, tol=GRAD_TOL)


def _run(x, dout, rho=True):
    import torch
    import parameterized_local_linear_02_b300 as plx
    t = {n: torch.from_numpy(np.ascontiguousarray(getattr(x, n), np.float32)).cuda() for n in ("q", "k", "v", "rho")}
    r = t["rho"] if rho else None
    out, lse = plx.plx_fwd_f32(t["q"], t["k"], t["v"], r, scale=x.scale)
    g = plx.plx_bwd_f32(t["q"], t["k"], t["v"], r, out, lse, torch.from_numpy(dout).cuda(), scale=x.scale)
    torch.cuda.synchronize()
    assert plx.plx_last_device_error() == 0
    return [None if a is None else a.cpu().numpy() for a in g]


@pytest.mark.parametrize("shape", [(1, 2, 70, 64), (2, 1, 129, 128), (1, 1, 1, 32), (1, 2, 200, 96)])
def test_bwd_matches_oracle(shape):
    B, H, N, d = shape
    x = plx_inputs.prefill(B, H, N, d, seed=N + d, dtype="f32", rho="normal", rho_std=0.3)
    dout = np.random.default_rng(N).standard_normal((B, H, N, d)).astype(np.float32)
    got = _run(x, dout)
    ref = plx_backward(x.q, x.k, x.v, x.rho, dout, x.scale)[:4]
    for name, g, r in zip(("dq", "dk", "dv", "drho"), got, ref):
        assert_grad(g, r, f"{name} {shape}")


def test_bwd_softmax_attention_instantiation():
    """rho = NULL: the softmax-attention gradients, equal to PLX's at rho = 0."""
    x = plx_inputs.prefill(1, 2, 150, 64, seed=41, dtype="f32", rho="zero")
    dout = np.random.default_rng(41).standard_normal(x.q.shape).astype(np.float32)
    got = _run(x, dout, rho=False)
    ref = plx_backward(x.q, x.k, x.v, np.zeros_like(x.q), dout, x.scale)[:3]
    for name, g, r in zip(("dq", "dk", "dv"), got[:3], ref):
        assert_grad(g, r, f"SA {name}")
    assert got[3] is None


def test_bwd_projection_probe():
    """rho = W_R x: unit-variance probe components, the correction dominates."""
    x = plx_inputs.prefill(1, 1, 160, 128, seed=42, dtype="f32", rho="proj", x_width=128)
    dout = np.random.default_rng(42).standard_normal(x.q.shape).astype(np.float32)
    got = _run(x, dout)
    ref = plx_backward(x.q, x.k, x.v, x.rho, dout, x.scale)[:4]
    for name, g, r in zip(("dq", "dk", "dv", "drho"), got, ref):
        assert_grad(g, r, f"proj {name}")
