"""plx_decode (split-KV bf16 decode + LSE combine) against the fp64 oracle."""
import numpy as np
import pytest

import oracle
import plx_inputs
from parity import LSE_BF16, assert_bf16, assert_f32, assert_lse, canary

pytestmark = pytest.mark.gpu


def device(x):
    return x.device_tensors("cuda")


def run(t, rho=True, **kw):
    """plx_decode into NaN-filled outputs and a 0xFF-filled workspace, each
    inside sentinel guards: every output element must be written, every
    partial read must have been written first, and nothing outside is touched."""
    import torch
    import parameterized_local_linear_02_b300 as plx
    B, H, S_cap, d = t["k_cache"].shape
    od = kw.pop("out_dtype", torch.bfloat16)
    out, out_ok = canary((B, H, d), od)
    lse, lse_ok = canary((B, H), torch.float32)
    ws_ok = lambda: True
    need = plx.plx_decode_workspace_size(B, H, d, S_cap, kw.get("num_splits", 0))
    if need > 0 and "workspace" not in kw:
        kw["workspace"], ws_ok = canary((need,), torch.uint8)
    plx.plx_decode(t["q"], t["rho"] if rho else None, t["k_cache"], t["v_cache"], t["seqlens"], out=out, lse=lse,
                   **kw)
    torch.cuda.synchronize()
    assert out_ok() and lse_ok() and ws_ok(), "plx_decode wrote outside its outputs or workspace"
    assert not bool(torch.isnan(out).any()) and not bool(torch.isnan(lse).any()), "an output element was not written"
    return out.float().cpu().numpy(), lse.cpu().numpy()


def oracle_dec(x, form, heads=None, rho=True):
    res = oracle.decode(form, x.q, x.rho if rho else None, x.k_cache, x.v_cache, x.seqlens,
                        x.scale, heads=heads)
    return res


def compare(out, lse, res, strict, what):
    keys = sorted(res)
    got = np.stack([out[b, h] for b, h in keys])
    ref = np.stack([res[k][0] for k in keys])
    if strict:
        assert_f32(got, ref, what)        # fp32 output: nothing is rounded to bf16 inside the kernel
    else:
        assert_bf16(got, ref, what)
    assert_lse(np.array([lse[b, h] for b, h in keys]), np.array([res[k][1] for k in keys]),
               LSE_BF16, what)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_decode_small_ragged(d, splits):
    import torch
    x = plx_inputs.decode(3, 2, d, 200, seed=10 + d, seqlens=np.array([200, 1, 77]))
    t = device(x)
    out, lse = run(t, num_splits=splits, out_dtype=torch.float32)
    compare(out, lse, oracle_dec(x, "explicit"), True, f"decode d={d} splits={splits}")


def test_decode_bf16_output_and_softmax_instantiation():
    import torch
    x = plx_inputs.decode(2, 4, 128, 333, seed=21, seqlens=np.array([333, 129]))
    t = device(x)
    out, lse = run(t, num_splits=2)
    compare(out, lse, oracle_dec(x, "stream"), False, "decode bf16 out")
    out_sa, lse_sa = run(t, rho=False, num_splits=2, out_dtype=torch.float32)
    compare(out_sa, lse_sa, oracle_dec(x, "sa", rho=False), True, "decode SA")


def test_decode_split_count_invariance():
    import torch
    x = plx_inputs.decode(2, 3, 128, 1000, seed=22, seqlens="ragged")
    t = device(x)
    base, lb = run(t, num_splits=1, out_dtype=torch.float32)
    for s in (2, 5, 16, 40):
        o, l = run(t, num_splits=s, out_dtype=torch.float32)
        rms = np.sqrt(np.mean(base ** 2))
        assert np.max(np.abs(o - base)) / rms < 1e-5, s
        assert np.max(np.abs(l - lb)) < 1e-5, s


def test_decode_empty_and_clamped_lengths():
    import torch
    import parameterized_local_linear_02_b300 as plx
    x = plx_inputs.decode(3, 2, 128, 64, seed=23, seqlens=np.array([0, 64, 1000]))
    t = device(x)
    assert plx.plx_last_device_error() == 0
    out, lse = run(t, num_splits=2, out_dtype=torch.float32)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert plx.plx_last_device_error() == 1        # length above capacity was clamped and flagged
    assert plx.plx_last_device_error() == 0        # and the flag was cleared
    res = oracle_dec(x, "explicit", heads=[(1, 0), (1, 1), (2, 0), (2, 1)])
    compare(out, lse, res, True, "decode clamped")


def test_decode_matches_prefill_last_row():
    """Decode at length L over a cache equals the causal prefill row L-1."""
    import torch
    import parameterized_local_linear_02_b300 as plx
    p = plx_inputs.prefill(1, 2, 190, 128, seed=24, dtype="bf16", rho="normal", rho_std=0.5)
    t = p.device_tensors()
    L = 150
    out_p, lse_p = plx.plx_fwd(t["q"], t["k"], t["v"], t["rho"], out_dtype=torch.float32)
    sl = torch.full((1,), L, dtype=torch.int32, device="cuda")
    out_d, lse_d = plx.plx_decode(t["q"][:, :, L - 1].contiguous(), t["rho"][:, :, L - 1].contiguous(),
                                  t["k"], t["v"], sl, out_dtype=torch.float32, num_splits=3)
    torch.cuda.synchronize()
    ref = np.stack([oracle.query("explicit", p.q[0, h, L - 1], p.rho[0, h, L - 1], p.k[0, h, :L],
                                 p.v[0, h, :L], p.scale)[0] for h in range(2)])
    assert_f32(out_d[0].cpu().numpy(), ref, "decode vs oracle prefill row")
    assert_bf16(out_p[0, :, L - 1].cpu().numpy(), out_d[0].cpu().numpy(), "prefill row vs decode")


@pytest.mark.slow
def test_decode_full_size_b64_h16_ctx4096_sampled():
    """The decode workload at full size (B=64, H=16, d=128, every length 4096),
    in the launch configuration the benchmark times; 12 sampled heads."""
    import torch
    import parameterized_local_linear_02_b300 as plx
    cfg = plx_inputs.CONFIGS["decode_b64_h16_ctx4096_d128"]
    t = plx_inputs.decode_device(cfg["B"], cfg["H"], cfg["d"], cfg["S_cap"], seed=cfg["seed"],
                                 seqlens=cfg["seqlens"], rho_std=cfg["rho_std"])
    out, lse = plx.plx_decode(t["q"], t["rho"], t["k_cache"], t["v_cache"], t["seqlens"])
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    heads = [(0, 0), (63, 15)] + [(int(b), int(h)) for b, h in
                                  zip(rng.integers(0, 64, 10), rng.integers(0, 16, 10))]
    got, ref, lg, lr = [], [], [], []
    for b, h in heads:
        L = int(t["seqlens_host"][b])
        f = lambda name: t[name][b, h].float().cpu().numpy()
        kc = t["k_cache"][b, h, :L].float().cpu().numpy()
        vc = t["v_cache"][b, h, :L].float().cpu().numpy()
        o, l = oracle.query("stream", f("q"), f("rho"), kc, vc, 1 / np.sqrt(cfg["d"]))
        got.append(out[b, h].float().cpu().numpy())
        ref.append(o)
        lg.append(float(lse[b, h]))
        lr.append(l)
    assert_bf16(np.stack(got), np.stack(ref), "decode full size")
    assert_lse(lg, lr, LSE_BF16, "decode full size lse")
    assert torch.isfinite(out.float()).all()


@pytest.mark.slow
@pytest.mark.parametrize("B,ctx", [(8, 32768), (1, 131072), (256, 2048)])
def test_decode_sweep_cells_sampled(B, ctx):
    """Cells of the decode sweep at full size: lengths drawn from [ctx/2, ctx],
    the split count the library picks for this GPU; sampled heads vs the
    oracle, every output finite."""
    import torch
    import parameterized_local_linear_02_b300 as plx
    cfg = plx_inputs.CONFIGS["decode_sweep"]
    t = plx_inputs.decode_device(B, cfg["H"], cfg["d"], ctx, seed=cfg["seed"] + B, seqlens="ragged",
                                 rho_std=cfg["rho_std"])
    out, lse = plx.plx_decode(t["q"], t["rho"], t["k_cache"], t["v_cache"], t["seqlens"],
                              out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert plx.plx_last_device_error() == 0
    rng = np.random.default_rng(B + ctx)
    heads = sorted({(0, 0), (B - 1, cfg["H"] - 1)} |
                   {(int(b), int(h)) for b, h in zip(rng.integers(0, B, 4), rng.integers(0, cfg["H"], 4))})
    got, ref, lg, lr = [], [], [], []
    for b, h in heads:
        L = int(t["seqlens_host"][b])
        f = lambda name: t[name][b, h].float().cpu().numpy()
        kc = t["k_cache"][b, h, :L].float().cpu().numpy()
        vc = t["v_cache"][b, h, :L].float().cpu().numpy()
        o, l = oracle.query("stream", f("q"), f("rho"), kc, vc, 1 / np.sqrt(cfg["d"]))
        got.append(out[b, h].cpu().numpy())
        ref.append(o)
        lg.append(float(lse[b, h]))
        lr.append(l)
    assert_f32(np.stack(got), np.stack(ref), f"decode sweep B={B} ctx={ctx}")
    assert_lse(lg, lr, LSE_BF16, f"decode sweep B={B} ctx={ctx} lse")
    assert torch.isfinite(out).all()
