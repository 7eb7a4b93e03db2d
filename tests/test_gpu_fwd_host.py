"""plx_fwd_host: the forward on host buffers, streamed through a device
workspace in chunks of heads with the copies overlapping the kernels.  Its
out and lse must be plx_fwd's on the same values, bit for bit (each 128-row
item is computed the same way whatever the chunk), for page-locked and for
pageable host memory, and two calls in a row that share the workspace must
not see each other's data."""
import pytest

import plx_inputs

pytestmark = pytest.mark.gpu


def _host(t, pinned=True):
    h = t.cpu()
    return h.pin_memory() if pinned else h


def _check(B, H, N, d, seed, rho=True, f32=True, pinned=True, with_lse=True, workspace=None):
    import torch
    import parameterized_local_linear_02_b300 as plx
    x = plx_inputs.prefill(B, H, N, d, seed=seed, dtype="bf16", rho="normal" if rho else "zero", rho_std=0.3)
    t = x.device_tensors()
    odt = torch.float32 if f32 else torch.bfloat16
    ref_o, ref_lse = plx.plx_fwd(t["q"], t["k"], t["v"], t["rho"] if rho else None, scale=x.scale, out_dtype=odt)
    hq, hk, hv = _host(t["q"], pinned), _host(t["k"], pinned), _host(t["v"], pinned)
    hr = _host(t["rho"], pinned) if rho else None
    out = torch.full((B, H, N, d), float("nan"), dtype=odt)
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32) if with_lse else None
    if pinned:
        out = out.pin_memory()
        lse = lse.pin_memory() if lse is not None else None
    if workspace is None:
        workspace = torch.empty(plx.plx_fwd_host_workspace_size(B, H, N, d, odt), dtype=torch.uint8, device="cuda")
    plx.plx_fwd_host(hq, hk, hv, hr, out, lse, workspace=workspace, scale=x.scale)
    torch.cuda.synchronize()
    assert plx.plx_last_device_error() == 0
    assert torch.equal(out, ref_o.cpu()), f"out differs from plx_fwd ({B}, {H}, {N}, {d})"
    if with_lse:
        assert torch.equal(lse, ref_lse.cpu()), f"lse differs from plx_fwd ({B}, {H}, {N}, {d})"
    return workspace


@pytest.mark.parametrize("shape", [(1, 2, 300, 64), (2, 3, 257, 128), (1, 1, 1, 128), (3, 7, 130, 64)])
def test_fwd_host_equals_plx_fwd(shape):
    _check(*shape, seed=sum(shape))


def test_fwd_host_softmax_attention_bf16_out_no_lse():
    _check(2, 9, 200, 128, seed=5, rho=False, f32=False, with_lse=False)


def test_fwd_host_pageable_memory():
    _check(2, 5, 190, 128, seed=6, pinned=False)


def test_fwd_host_two_calls_share_the_workspace():
    """Two calls enqueued back to back on one stream with one workspace, no
    synchronisation between them: each must return its own problem's result."""
    import torch
    import parameterized_local_linear_02_b300 as plx
    B, H, N, d = 2, 20, 256, 128
    ws = torch.empty(plx.plx_fwd_host_workspace_size(B, H, N, d, torch.float32), dtype=torch.uint8, device="cuda")
    runs = []
    for seed in (7, 8):
        x = plx_inputs.prefill(B, H, N, d, seed=seed, dtype="bf16", rho="normal", rho_std=0.3)
        t = x.device_tensors()
        ref_o, ref_lse = plx.plx_fwd(t["q"], t["k"], t["v"], t["rho"], scale=x.scale, out_dtype=torch.float32)
        host = {n: _host(t[n]) for n in ("q", "k", "v", "rho")}
        out = torch.full((B, H, N, d), float("nan")).pin_memory()
        lse = torch.full((B, H, N), float("nan")).pin_memory()
        runs.append((x, host, out, lse, ref_o.cpu(), ref_lse.cpu()))
    torch.cuda.synchronize()
    for x, host, out, lse, _, _ in runs:
        plx.plx_fwd_host(host["q"], host["k"], host["v"], host["rho"], out, lse, workspace=ws, scale=x.scale)
    torch.cuda.synchronize()
    assert plx.plx_last_device_error() == 0
    for n, (_, _, out, lse, ref_o, ref_lse) in enumerate(runs):
        assert torch.equal(out, ref_o) and torch.equal(lse, ref_lse), f"call {n + 1} differs from plx_fwd"


def test_fwd_host_bench_shape():
    """The bench's prefill workload (B=4, H=16, N=2048, d=128), fp32 out and lse."""
    pc = plx_inputs.CONFIGS["prefill_b4_h16_n2048_d128"]
    _check(pc["B"], pc["H"], pc["N"], pc["d"], seed=9)
