"""plx_fwd_train + plx_bwd_saved: the training forward also returns vbar (the
softmax-attention output of the same weights) and c_i = sum_j w_ij rho_i.k_j,
and the backward forms its row statistics from them instead of recomputing
them with an attention pass.

Checks, on the same bf16-rounded inputs as the oracle:
- plx_fwd_train's o and lse are plx_fwd's, bit for bit;
- vbar is the oracle's softmax attention, and c is rho_i . kbar_i with kbar
  the oracle's softmax attention over the keys used as values;
- the gradients match the fp64 autograd oracle at the bf16 bar (max 2e-2,
  mean 2e-3 of each gradient's RMS), as plx_bwd's do;
- every output element is written and nothing around the outputs."""
import numpy as np
import pytest

import oracle
import plx_inputs
from oracle.backward import plx_backward
from parity import assert_bf16, canary

pytestmark = pytest.mark.gpu


def _bf16_round(a):
    b = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return (b.astype(np.uint32) << 16).view(np.float32)


def run_train(x, out_dtype="f32"):
    import torch
    import parameterized_local_linear_02_b300 as plx
    t = x.device_tensors()
    shape = (x.B, x.H, x.N, x.d)
    odt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    o, o_ok = canary(shape, odt)
    lse, l_ok = canary(shape[:3], torch.float32)
    vbar, v_ok = canary(shape, torch.float32)
    c, c_ok = canary(shape[:3], torch.float32)
    plx.plx_fwd_train(t["q"], t["k"], t["v"], t["rho"], scale=x.scale, out=o, lse=lse, vbar=vbar, c=c)
    ref_o, ref_lse = plx.plx_fwd(t["q"], t["k"], t["v"], t["rho"], scale=x.scale, out_dtype=odt)
    torch.cuda.synchronize()
    assert plx.plx_last_device_error() == 0
    assert o_ok() and l_ok() and v_ok() and c_ok(), "plx_fwd_train wrote outside its outputs"
    assert not bool(torch.isnan(vbar).any()) and not bool(torch.isnan(c).any()), "an element was not written"
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse), "o or lse differs from plx_fwd"
    return t, o, lse, vbar, c


def run_saved(x, t, o, lse, vbar, c, dout, rho=True):
    import torch
    import parameterized_local_linear_02_b300 as plx
    shape = (x.B, x.H, x.N, x.d)
    do = torch.from_numpy(dout).to("cuda").to(torch.bfloat16)
    bufs = [canary(shape, torch.float32) for _ in range(4 if rho else 3)]
    grads = tuple(b[0] for b in bufs) + ((None,) if not rho else ())
    ws, ws_ok = canary((plx.plx_bwd_bf16_workspace_size(x.B, x.H, x.N, x.d),), torch.uint8)
    g = plx.plx_bwd_saved(t["q"], t["k"], t["v"], t["rho"] if rho else None, do, o, lse, vbar, c,
                          scale=x.scale, workspace=ws, grads=grads)
    torch.cuda.synchronize()
    assert plx.plx_last_device_error() == 0
    assert all(ok() for _, ok in bufs) and ws_ok(), "plx_bwd_saved wrote outside its gradients or workspace"
    assert not any(bool(torch.isnan(a).any()) for a in g if a is not None), "a gradient element was not written"
    return [None if a is None else a.cpu().numpy() for a in g]


def _sa(x, values):
    """The oracle's softmax attention of (q, k) over ``values``, [B, H, N, d] fp64."""
    res = oracle.prefill("sa", x.q, x.k, values, np.zeros_like(x.q), x.scale)
    out = np.zeros(np.shape(x.q))
    for (b, h), (o, _, rows) in res.items():
        out[b, h, rows] = o
    return out


def _oracle_vbar_c(x):
    """vbar = softmax attention; kbar = softmax attention with the keys as
    values; c = rho . kbar (fp64)."""
    vbar = _sa(x, x.v)
    kbar = _sa(x, x.k)
    c = np.einsum("bhnd,bhnd->bhn", np.asarray(x.rho, np.float64), kbar)
    return vbar, c


@pytest.mark.parametrize("shape", [(1, 2, 70, 64), (2, 1, 257, 128), (1, 1, 1, 128), (1, 2, 390, 64)])
def test_fwd_train_and_bwd_saved_match_oracle(shape):
    B, H, N, d = shape
    x = plx_inputs.prefill(B, H, N, d, seed=N + d + 11, dtype="bf16", rho="normal", rho_std=0.3)
    t, o, lse, vbar, c = run_train(x)
    ref_vbar, ref_c = _oracle_vbar_c(x)
    assert_bf16(vbar.cpu().numpy(), ref_vbar, f"{shape} vbar")
    assert_bf16(c.cpu().numpy(), ref_c, f"{shape} c")
    dout = _bf16_round(np.random.default_rng(N + 3).standard_normal((B, H, N, d)).astype(np.float32))
    got = run_saved(x, t, o, lse, vbar, c, dout)
    ref = plx_backward(x.q, x.k, x.v, x.rho, dout, x.scale)[:4]
    if N == 1:
        assert float(np.max(np.abs(got[0]))) <= 1e-6 and float(np.max(np.abs(got[1]))) <= 1e-6
        assert_bf16(got[2], ref[2], f"{shape} dv")
        return
    for name, g, r in zip(("dq", "dk", "dv", "drho"), got, ref):
        mx, mn = assert_bf16(g, r, f"{shape} {name}")
        print(f"{shape} {name}: max {mx:.2e} mean {mn:.2e}")


def test_bwd_saved_with_bf16_output_and_projection_probe():
    """rho = W_R x (the correction dominates o), o saved in bf16."""
    x = plx_inputs.prefill(1, 2, 256, 128, seed=47, dtype="bf16", rho="proj", x_width=256)
    t, o, lse, vbar, c = run_train(x, out_dtype="bf16")
    dout = _bf16_round(np.random.default_rng(47).standard_normal(x.q.shape).astype(np.float32))
    got = run_saved(x, t, o, lse, vbar, c, dout)
    ref = plx_backward(x.q, x.k, x.v, x.rho, dout, x.scale)[:4]
    for name, g, r in zip(("dq", "dk", "dv", "drho"), got, ref):
        assert_bf16(g, r, f"proj {name}")


def test_bwd_saved_softmax_attention():
    """rho = NULL: plx_fwd's o and lse are the saved values (vbar = o, c = 0)."""
    import torch
    import parameterized_local_linear_02_b300 as plx
    x = plx_inputs.prefill(1, 2, 190, 128, seed=48, dtype="bf16", rho="zero")
    t = x.device_tensors()
    o, lse = plx.plx_fwd(t["q"], t["k"], t["v"], None, scale=x.scale, out_dtype=torch.float32)
    dout = _bf16_round(np.random.default_rng(48).standard_normal(x.q.shape).astype(np.float32))
    got = run_saved(x, t, o, lse, None, None, dout, rho=False)
    ref = plx_backward(x.q, x.k, x.v, np.zeros_like(x.q), dout, x.scale)[:3]
    for name, g, r in zip(("dq", "dk", "dv"), got[:3], ref):
        assert_bf16(g, r, f"SA {name}")
    assert got[3] is None


def test_bwd_saved_full_size_against_sampled_oracle_heads_and_plx_bwd():
    """The bench's backward workload (B=4, H=16, N=2048, d=128, rho = W_R x):
    two whole heads against the closed-form fp64 gradients at the bf16 bar;
    then every head against plx_bwd's gradients.  The two paths are
    independent approximations of the same gradients, each within the bar of
    the exact values, so they may differ by up to twice the bar's maximum;
    their mean difference must stay within the bar."""
    import torch
    import parameterized_local_linear_02_b300 as plx
    from oracle.backward import plx_backward_closed
    from parity import BF16_MAX, BF16_MEAN, rel_errors
    pc = plx_inputs.CONFIGS["prefill_b4_h16_n2048_d128"]
    B, H, N, d = pc["B"], pc["H"], pc["N"], pc["d"]
    x = plx_inputs.prefill(B, H, N, d, seed=pc["seed"], dtype="bf16", rho=pc["rho"], keys=pc["keys"])
    t, o, lse, vbar, c = run_train(x)
    dout = _bf16_round(np.random.default_rng(2049).standard_normal((B, H, N, d)).astype(np.float32))
    got = run_saved(x, t, o, lse, vbar, c, dout)
    heads = [(0, 0), (2, 9)]
    ref = plx_backward_closed(x.q, x.k, x.v, x.rho, dout, x.scale, heads=heads)
    for (b, h), grads in ref.items():
        for name, g, r in zip(("dq", "dk", "dv", "drho"), got, grads):
            mx, mn = assert_bf16(g[b, h], r, f"full size ({b}, {h}) {name}")
            print(f"full size ({b}, {h}) {name}: max {mx:.2e} mean {mn:.2e}")
    do = torch.from_numpy(dout).to("cuda").to(torch.bfloat16)
    base = [a.cpu().numpy() for a in plx.plx_bwd(t["q"], t["k"], t["v"], t["rho"], do, scale=x.scale)]
    for name, g, r in zip(("dq", "dk", "dv", "drho"), got, base):
        mx, mn = rel_errors(g, r)
        print(f"full size vs plx_bwd {name}: max {mx:.2e} mean {mn:.2e}")
        assert mx <= 2 * BF16_MAX and mn <= BF16_MEAN, f"full size vs plx_bwd {name}: max {mx:.2e} mean {mn:.2e}"
