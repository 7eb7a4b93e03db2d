"""plx_bwd (tcgen05 tensor-core backward, bf16) against the fp64 autograd
oracle of the explicit-covariance forward, on the same bf16-rounded inputs.

The GPU path recomputes the forward's row statistics with the bf16 forward
kernel and feeds ds, dr and the dv weights to its GEMMs as fp16; the bar is
the bf16 one of the forward (max 2e-2, mean 2e-3 of each gradient's RMS)."""
import numpy as np
import pytest

import plx_inputs
from oracle.backward import plx_backward
from parity import assert_bf16, canary

pytestmark = pytest.mark.gpu


def _bf16_round(a):
    """Round float32 to bf16 (round to nearest even) and back, on the host."""
    b = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return (b.astype(np.uint32) << 16).view(np.float32)


def run_bwd(x, dout, rho=True):
    import torch
    import parameterized_local_linear_02_b300 as plx
    t = x.device_tensors()
    r = t["rho"] if rho else None
    do = torch.from_numpy(dout).to("cuda").to(torch.bfloat16)
    # NaN-filled gradients and a 0xFF-filled workspace inside sentinel guards:
    # every gradient element must be written, and nothing around them
    shape = (x.B, x.H, x.N, x.d)
    bufs = [canary(shape, torch.float32) for _ in range(4 if rho else 3)]
    grads = tuple(b[0] for b in bufs) + ((None,) if not rho else ())
    ws, ws_ok = canary((plx.plx_bwd_bf16_workspace_size(x.B, x.H, x.N, x.d),), torch.uint8)
    g = plx.plx_bwd(t["q"], t["k"], t["v"], r, do, scale=x.scale, workspace=ws, grads=grads)
    torch.cuda.synchronize()
    assert plx.plx_last_device_error() == 0
    assert all(ok() for _, ok in bufs) and ws_ok(), "plx_bwd wrote outside its gradients or workspace"
    assert not any(bool(torch.isnan(a).any()) for a in g if a is not None), "a gradient element was not written"
    return [None if a is None else a.cpu().numpy() for a in g]


def check(got, ref, names, what):
    for name, g, r in zip(names, got, ref):
        mx, mn = assert_bf16(g, r, f"{what} {name}")
        print(f"{what} {name}: max {mx:.2e} mean {mn:.2e}")


@pytest.mark.parametrize("shape", [(1, 2, 70, 64), (2, 1, 129, 128), (1, 1, 1, 128), (1, 2, 200, 64),
                                   (1, 1, 300, 128), (1, 1, 64, 128)])
def test_bwd_tc_matches_oracle(shape):
    B, H, N, d = shape
    x = plx_inputs.prefill(B, H, N, d, seed=N + d + 7, dtype="bf16", rho="normal", rho_std=0.3)
    dout = _bf16_round(np.random.default_rng(N + 1).standard_normal((B, H, N, d)).astype(np.float32))
    got = run_bwd(x, dout)
    ref = plx_backward(x.q, x.k, x.v, x.rho, dout, x.scale)[:4]
    if N == 1:
        # o_0 = v_0: only dv is non-zero
        assert float(np.max(np.abs(got[0]))) <= 1e-6 and float(np.max(np.abs(got[1]))) <= 1e-6
        check(got[2:3], ref[2:3], ("dv",), f"{shape}")
        return
    check(got, ref, ("dq", "dk", "dv", "drho"), f"{shape}")


def test_bwd_tc_projection_probe():
    """rho = W_R x (unit-variance components): the correction dominates o."""
    x = plx_inputs.prefill(1, 2, 256, 128, seed=43, dtype="bf16", rho="proj", x_width=256)
    dout = _bf16_round(np.random.default_rng(43).standard_normal(x.q.shape).astype(np.float32))
    got = run_bwd(x, dout)
    ref = plx_backward(x.q, x.k, x.v, x.rho, dout, x.scale)[:4]
    check(got, ref, ("dq", "dk", "dv", "drho"), "proj")


def test_bwd_tc_softmax_attention_instantiation():
    """rho = NULL: softmax-attention gradients, PLX's at rho = 0."""
    x = plx_inputs.prefill(1, 2, 190, 128, seed=44, dtype="bf16", rho="zero")
    dout = _bf16_round(np.random.default_rng(44).standard_normal(x.q.shape).astype(np.float32))
    got = run_bwd(x, dout, rho=False)
    ref = plx_backward(x.q, x.k, x.v, np.zeros_like(x.q), dout, x.scale)[:3]
    check(got[:3], ref, ("dq", "dk", "dv"), "SA")
    assert got[3] is None


@pytest.mark.parametrize("shape", [(2, 2, 390, 64), (1, 3, 257, 128)])
def test_bwd_tc_several_items_ragged(shape):
    """Several 128-row items per head in both passes, the last one ragged,
    and more items than one wave of some CTAs' share."""
    B, H, N, d = shape
    x = plx_inputs.prefill(B, H, N, d, seed=N * 3 + d, dtype="bf16", rho="normal", rho_std=0.3)
    dout = _bf16_round(np.random.default_rng(N + 5).standard_normal((B, H, N, d)).astype(np.float32))
    got = run_bwd(x, dout)
    ref = plx_backward(x.q, x.k, x.v, x.rho, dout, x.scale)[:4]
    check(got, ref, ("dq", "dk", "dv", "drho"), f"{shape}")


def test_bwd_tc_full_size_sampled_heads():
    """The bench's backward workload (B=4, H=16, N=2048, d=128, rho = W_R x) in
    the launch configuration the bench times (every head in one plx_bwd call);
    three whole heads against the closed-form fp64 gradients."""
    import torch
    import parameterized_local_linear_02_b300 as plx
    from oracle.backward import plx_backward_closed
    pc = plx_inputs.CONFIGS["prefill_b4_h16_n2048_d128"]
    B, H, N, d = pc["B"], pc["H"], pc["N"], pc["d"]
    x = plx_inputs.prefill(B, H, N, d, seed=pc["seed"], dtype="bf16", rho=pc["rho"], keys=pc["keys"])
    dout = _bf16_round(np.random.default_rng(2048).standard_normal((B, H, N, d)).astype(np.float32))
    got = run_bwd(x, dout)
    heads = [(0, 0), (1, 7), (3, 15)]
    ref = plx_backward_closed(x.q, x.k, x.v, x.rho, dout, x.scale, heads=heads)
    for (b, h), grads in ref.items():
        for name, g, r in zip(("dq", "dk", "dv", "drho"), got, grads):
            mx, mn = assert_bf16(g[b, h], r, f"full size ({b}, {h}) {name}")
            print(f"full size ({b}, {h}) {name}: max {mx:.2e} mean {mn:.2e}")
