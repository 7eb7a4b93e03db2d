"""plx_probe_proj (tcgen05 probe projection, bf16 in and out) against the fp64
oracle rho = W_R x split into heads, on the same bf16-rounded inputs.

The kernel accumulates the Dx products of each output in fp32 (each product
of two bf16 values is exact in fp32) and rounds the sum once to bf16.  Per
element, |got - ref| <= 2^-8 |ref| (the final rounding) + Dx 2^-23 sum_k
|W_R[r, k] x[k]| (fp32 accumulation, with a factor 2 of slack), and almost
every element equals the oracle's value rounded to bf16."""
import numpy as np
import pytest

import plx_inputs
from oracle.projection import probe_projection, probe_projection_rows

pytestmark = pytest.mark.gpu


def bf16_rne(a):
    b = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return (b.astype(np.uint32) << 16).view(np.float32)


def run_proj(inp):
    import torch
    import parameterized_local_linear_02_b300 as plx
    t = inp.device_tensors()
    rho = plx.plx_probe_proj(t["x"], t["w_r"], heads=inp.H)
    torch.cuda.synchronize()
    assert plx.plx_last_device_error() == 0
    return rho.float().cpu().numpy()


def check(got, ref, absdot, Dx, what, min_exact=0.98):
    got = np.asarray(got, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    bound = 2.0 ** -8 * np.abs(ref) + Dx * 2.0 ** -23 * absdot
    err = np.abs(got - ref)
    worst = float(np.max(err - bound))
    assert worst <= 0.0, f"{what}: {int(np.sum(err > bound))} elements outside the bound (worst excess {worst:.2e})"
    exact = float(np.mean(got == bf16_rne(ref)))
    assert exact >= min_exact, f"{what}: only {exact:.4f} of the elements equal the rounded fp64 value"
    print(f"{what}: max err {float(err.max()):.2e}, {exact:.4f} equal to bf16(fp64)")


@pytest.mark.parametrize("shape", [
    (2, 300, 3, 128, 200),     # ragged token tail, half-filled second column group, ragged Dx
    (1, 129, 5, 64, 64),       # d = 64: four heads per group, second group holds one head
    (1, 1, 1, 64, 8),          # one token, one head, Dx = 8
    (2, 2048, 16, 128, 256),   # 256 items: several items per CTA, both accumulators reused
    (3, 77, 2, 64, 1032),      # Dx of 17 stages (one of 8 columns), tiny N
    # more items than CTAs with a last wave of at most half the grid: those items run as two
    # 128-column halves (148 SMs: 160 items -> 148 whole + 24 halves; 152 -> 148 + 8)
    (2, 1280, 16, 128, 128),
    (2, 2048, 20, 64, 64),     # d = 64: each half holds two heads
    (4, 2432, 3, 128, 64),     # H d = 384: the second half of the last group lies past H
])
def test_proj_matches_oracle(shape):
    B, N, H, d, Dx = shape
    inp = plx_inputs.probe(B, N, H, d, Dx, seed=B * 1000 + N + Dx)
    got = run_proj(inp)
    ref = probe_projection(inp.x, inp.w_r, H)
    absdot = probe_projection(np.abs(inp.x), np.abs(inp.w_r), H)
    check(got, ref, absdot, Dx, f"{shape}")


def test_proj_full_size():
    """The bench workload in the launch configuration the bench times:
    x [4, 2048, 1024], W_R [16 * 128, 1024] (512 items on a persistent grid).
    Every output element against the fp64 oracle."""
    B, N, H, d, Dx = 4, 2048, 16, 128, 1024
    inp = plx_inputs.probe(B, N, H, d, Dx, seed=11)
    got = run_proj(inp)
    ref = probe_projection(inp.x, inp.w_r, H)
    absdot = probe_projection(np.abs(inp.x), np.abs(inp.w_r), H)
    check(got, ref, absdot, Dx, "full size")


def test_proj_large_values_and_rows_helper():
    """x with std 30 (outputs far from 1) checked on sampled tokens with the
    oracle's row helper, plus one call's determinism."""
    import torch
    import parameterized_local_linear_02_b300 as plx
    B, N, H, d, Dx = 2, 640, 4, 128, 384
    inp = plx_inputs.probe(B, N, H, d, Dx, seed=12, x_std=30.0)
    t = inp.device_tensors()
    r1 = plx.plx_probe_proj(t["x"], t["w_r"], heads=H)
    r2 = plx.plx_probe_proj(t["x"], t["w_r"], heads=H)
    torch.cuda.synchronize()
    assert plx.plx_last_device_error() == 0
    assert torch.equal(r1, r2)
    got = r1.float().cpu().numpy()
    rows = [0, 1, 127, 128, 383, 639]
    for b in range(B):
        ref = probe_projection_rows(inp.x, inp.w_r, H, b, rows)
        absdot = probe_projection_rows(np.abs(inp.x), np.abs(inp.w_r), H, b, rows)
        check(got[b][:, rows], ref, absdot, Dx, f"x std 30, batch {b}")


def test_proj_feeds_plx_fwd():
    """rho from plx_probe_proj drives plx_fwd: the chained result against the
    fp64 oracle's explicit PLX forward on the oracle's own rho, rounded to
    bf16 as the kernel stores it (x std 0.3, so the probe has the size of the
    attention tests' rho)."""
    import torch
    import oracle
    import parameterized_local_linear_02_b300 as plx
    from parity import assert_bf16
    B, H, N, d, Dx = 1, 2, 256, 128, 256
    att = plx_inputs.prefill(B, H, N, d, seed=21, dtype="bf16", rho="zero")
    inp = plx_inputs.probe(B, N, H, d, Dx, seed=22, x_std=0.3)
    t = att.device_tensors()
    ti = inp.device_tensors()
    rho = plx.plx_probe_proj(ti["x"], ti["w_r"], heads=H)
    out, _ = plx.plx_fwd(t["q"], t["k"], t["v"], rho, scale=att.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert plx.plx_last_device_error() == 0
    rho_ref = bf16_rne(probe_projection(inp.x, inp.w_r, H))
    res = oracle.prefill("explicit", att.q, att.k, att.v, rho_ref, att.scale)
    got = out.cpu().numpy()
    for (b, h), (o_ref, _, rows) in res.items():
        assert_bf16(got[b, h][rows], o_ref, f"proj -> fwd ({b}, {h})")
