"""plx_fwd (tcgen05 tensor-core prefill, bf16) against the fp64 oracle."""
import numpy as np
import pytest

import oracle
import plx_inputs
from parity import LSE_BF16, assert_bf16, assert_bf16_output, assert_lse, canary

pytestmark = pytest.mark.gpu


def run(x, rho=True, out_dtype="f32"):
    """plx_fwd into NaN-filled outputs inside sentinel guards: every output
    element must be written, and nothing around them."""
    import torch
    import parameterized_local_linear_02_b300 as plx
    t = x.device_tensors()
    od = torch.float32 if out_dtype == "f32" else torch.bfloat16
    out, out_ok = canary((x.B, x.H, x.N, x.d), od)
    lse, lse_ok = canary((x.B, x.H, x.N), torch.float32)
    plx.plx_fwd(t["q"], t["k"], t["v"], t["rho"] if rho else None, scale=x.scale, out=out, lse=lse)
    torch.cuda.synchronize()
    assert plx.plx_last_device_error() == 0
    assert out_ok() and lse_ok(), "plx_fwd wrote outside its outputs"
    assert not bool(torch.isnan(out).any()) and not bool(torch.isnan(lse).any()), "an output element was not written"
    return out.float().cpu().numpy(), lse.cpu().numpy()


def oracle_rows(x, form, heads=None, rows=None):
    res = oracle.prefill(form, x.q, x.k, x.v, x.rho, x.scale, heads=heads, rows=rows)
    return res


def gather(out, lse, res):
    keys = sorted(res)
    got = np.concatenate([out[b, h][res[(b, h)][2]] for b, h in keys])
    ref = np.concatenate([res[(b, h)][0] for b, h in keys])
    lg = np.concatenate([lse[b, h][res[(b, h)][2]] for b, h in keys])
    lr = np.concatenate([res[(b, h)][1] for b, h in keys])
    return got, ref, lg, lr


@pytest.mark.parametrize("shape", [(1, 2, 300, 128), (2, 1, 129, 128), (1, 1, 1, 128),
                                   (1, 1, 64, 128), (1, 3, 200, 64), (1, 1, 513, 64)])
def test_fwd_small_shapes_all_rows(shape):
    """Several query/key tiles plus a ragged tail; every row vs the oracle."""
    B, H, N, d = shape
    x = plx_inputs.prefill(B, H, N, d, seed=N * 7 + d, dtype="bf16", rho="normal", rho_std=0.3)
    out, lse = run(x)
    got, ref, lg, lr = gather(out, lse, oracle_rows(x, "stream"))
    assert_bf16(got, ref, f"fwd {shape}")
    assert_lse(lg, lr, LSE_BF16, f"fwd lse {shape}")


def test_fwd_projection_probe():
    """rho = W_R x with unit-variance components: the correction dominates
    and early rows reach 15-20x the output RMS."""
    x = plx_inputs.prefill(1, 2, 384, 128, seed=31, dtype="bf16", rho="proj", x_width=256)
    out, lse = run(x)
    got, ref, lg, lr = gather(out, lse, oracle_rows(x, "explicit", rows=np.arange(0, 384, 3)))
    assert_bf16(got, ref, "fwd projection probe")
    assert_lse(lg, lr, LSE_BF16, "fwd projection lse")
    # bf16 output: the same arithmetic, plus the rounding of the stored result
    outb, _ = run(x, out_dtype="bf16")
    gotb, _, _, _ = gather(outb, lse, oracle_rows(x, "explicit", rows=np.arange(0, 384, 3)))
    assert_bf16_output(gotb, ref, "fwd projection probe, bf16 out")


def test_fwd_planted_keys():
    x = plx_inputs.prefill(1, 2, 640, 128, seed=32, dtype="bf16", rho="normal", rho_std=0.1,
                           keys="planted")
    out, lse = run(x)
    got, ref, lg, lr = gather(out, lse, oracle_rows(x, "stream"))
    assert_bf16(got, ref, "fwd planted keys")
    assert_lse(lg, lr, LSE_BF16, "fwd planted lse")


def test_fwd_zero_probe_equals_softmax_instantiation_bitwise():
    x = plx_inputs.prefill(2, 2, 300, 128, seed=33, dtype="bf16", rho="zero")
    out0, lse0 = run(x, rho=True)
    out_sa, lse_sa = run(x, rho=False)
    assert np.array_equal(out0, out_sa)
    assert np.array_equal(lse0, lse_sa)
    got, ref, lg, lr = gather(out_sa, lse_sa, oracle_rows(x, "sa"))
    assert_bf16(got, ref, "fwd SA")
    assert_lse(lg, lr, LSE_BF16, "fwd SA lse")


def test_fwd_large_scores_rescale_path():
    """Scores that keep growing along the sequence force the lazy rescale of
    O, U, l and C (row maxima rise by more than 2^8 between tiles)."""
    x = plx_inputs.prefill(1, 1, 512, 128, seed=34, dtype="bf16", rho="normal", rho_std=0.2)
    ramp = np.linspace(0.2, 4.0, 512, dtype=np.float32)[:, None]
    k = x.k * ramp
    bits, vals = plx_inputs.bf16_round(k)
    x.bits["k"], x.k = bits, vals
    out, lse = run(x)
    got, ref, lg, lr = gather(out, lse, oracle_rows(x, "stream"))
    assert_bf16(got, ref, "fwd rescale path")
    assert_lse(lg, lr, LSE_BF16, "fwd rescale lse")


def _sample_rows(N, rng, n_rand=256):
    return np.unique(np.concatenate([[0, 1, 2, N - 3, N - 2, N - 1], rng.integers(0, N, n_rand)]))


@pytest.mark.slow
@pytest.mark.parametrize("name", ["prefill_b4_h16_n2048_d128", "prefill_b2_h16_n8192_d128_planted"])
def test_fwd_full_size_sampled(name):
    """The prefill workloads at full size, in the benchmark's launch
    configuration (fp32 output); 4 heads x (first 3, last 3, 256 random rows)."""
    cfg = plx_inputs.CONFIGS[name]
    x = plx_inputs.prefill(cfg["B"], cfg["H"], cfg["N"], cfg["d"], seed=cfg["seed"], dtype="bf16",
                           rho=cfg["rho"], rho_std=cfg.get("rho_std", 0.1), keys=cfg["keys"])
    out, lse = run(x, out_dtype="f32")
    rng = np.random.default_rng(1)
    heads = [(0, 0), (cfg["B"] - 1, cfg["H"] - 1), (0, cfg["H"] // 2), (cfg["B"] // 2, 3)]
    rows = {hd: _sample_rows(cfg["N"], rng) for hd in heads}
    got, ref, lg, lr = gather(out, lse, oracle_rows(x, "stream", heads=heads, rows=rows))
    assert_bf16(got, ref, name)
    assert_lse(lg, lr, LSE_BF16, name + " lse")
    assert np.all(np.isfinite(out))


def test_fwd_zero_scale_uniform_weights():
    """scale = 0: uniform causal weights (the h -> infinity end of the family);
    masked keys must contribute exactly nothing."""
    x = plx_inputs.prefill(1, 2, 200, 128, seed=35, dtype="bf16", rho="normal", rho_std=0.3, scale=0.0)
    out, lse = run(x)
    got, ref, lg, lr = gather(out, lse, oracle_rows(x, "stream"))
    assert_bf16(got, ref, "fwd scale 0")
    assert_lse(lg, lr, LSE_BF16, "fwd scale 0 lse")


def test_fwd_out_of_range_probe_is_flagged():
    """|rho.k| far beyond the fp16 range of P o R gives a non-finite output,
    which the kernel reports through the device status word."""
    import torch
    import parameterized_local_linear_02_b300 as plx
    x = plx_inputs.prefill(1, 1, 128, 128, seed=36, dtype="bf16", rho="normal", rho_std=1.0)
    t = x.device_tensors()
    big = (t["rho"].float() * 3.0e4).to(torch.bfloat16)
    plx.plx_last_device_error()
    out, _ = plx.plx_fwd(t["q"], t["k"], t["v"], big, out_dtype=torch.float32)
    assert plx.plx_last_device_error() == 7
    out, _ = plx.plx_fwd(t["q"], t["k"], t["v"], t["rho"], out_dtype=torch.float32)
    assert plx.plx_last_device_error() == 0
    assert torch.isfinite(out).all()
