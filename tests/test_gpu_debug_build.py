"""The bounds-checking debug build (libplx_debug.so, compiled with
-DPLX_DEBUG): every checked index of the small test shapes stays inside its
buffer, so the status word stays clear, and the results equal those of the
normal build.  A failing check would record PLX_ERR_BOUNDS and skip the
access; it never traps.  This stands in for a memory checker, which is not
available here."""
import contextlib

import numpy as np
import pytest

import plx_inputs

pytestmark = pytest.mark.gpu


@contextlib.contextmanager
def debug_library():
    """Route the binding's calls to the debug build for the block."""
    from parameterized_local_linear_02_b300 import binding, build
    path = build.build(debug=True)          # prebuilt next to the package; rebuilt only if stale
    dbg = binding.load(path)
    saved = binding.library()
    binding._lib = dbg
    try:
        yield dbg
    finally:
        binding._lib = saved


def both(fn):
    """fn() with the normal build, then with the debug build (status checked)."""
    import torch
    import parameterized_local_linear_02_b300 as plx
    ref = fn()
    torch.cuda.synchronize()
    with debug_library():
        plx.plx_last_device_error()
        got = fn()
        torch.cuda.synchronize()
        st = plx.plx_last_device_error()
    assert st == 0, f"debug build: {plx.plx_strerror(st)}"
    return ref, got


def same(ref, got):
    """Equal results: bit for bit, or within 1e-5 of the RMS where the compiler
    contracted the arithmetic around the checks differently."""
    import torch
    for a, b in zip(ref, got):
        if a is None:
            continue
        if torch.equal(a, b):
            continue
        a64, b64 = a.double(), b.double()
        fin = torch.isfinite(a64)
        assert torch.equal(fin, torch.isfinite(b64)), "the debug build computed something else"
        rms = float(a64[fin].pow(2).mean().sqrt()) or 1.0
        err = float((a64[fin] - b64[fin]).abs().max()) / rms
        assert err <= 1e-5, f"the debug build computed something else ({err:.2e} of the RMS)"


@pytest.mark.parametrize("shape", [(1, 2, 300, 128), (1, 1, 1, 128), (1, 3, 200, 64)])
def test_debug_build_prefill(shape):
    import torch
    import parameterized_local_linear_02_b300 as plx
    B, H, N, d = shape
    x = plx_inputs.prefill(B, H, N, d, seed=N + d, dtype="bf16", rho="normal", rho_std=0.3)
    t = x.device_tensors()
    ref, got = both(lambda: plx.plx_fwd(t["q"], t["k"], t["v"], t["rho"], out_dtype=torch.float32))
    same(ref, got)


def test_debug_build_decode_contiguous_and_paged():
    import torch
    import parameterized_local_linear_02_b300 as plx
    x = plx_inputs.decode(3, 2, 128, 320, seed=95, seqlens=np.array([320, 1, 77]))
    t = x.device_tensors("cuda")
    ref, got = both(lambda: plx.plx_decode(t["q"], t["rho"], t["k_cache"], t["v_cache"], t["seqlens"], num_splits=3,
                                           out_dtype=torch.float32))
    same(ref, got)
    # the same cache as 32-row pages in a shuffled block table
    page, nb = 32, 10
    perm = torch.randperm(3 * nb, generator=torch.Generator().manual_seed(5)).to("cuda")
    kp = torch.empty((3 * nb, 2, page, 128), dtype=torch.bfloat16, device="cuda")
    vp = torch.empty_like(kp)
    table = torch.empty((3, nb), dtype=torch.int32, device="cuda")
    for b in range(3):
        for j in range(nb):
            blk = int(perm[b * nb + j])
            table[b, j] = blk
            kp[blk] = t["k_cache"][b, :, j * page:(j + 1) * page]
            vp[blk] = t["v_cache"][b, :, j * page:(j + 1) * page]
    refp, gotp = both(lambda: plx.plx_decode_paged(t["q"], t["rho"], kp, vp, table, t["seqlens"], num_splits=3,
                                                  out_dtype=torch.float32))
    same(refp, gotp)


def test_debug_build_backward():
    import torch
    import parameterized_local_linear_02_b300 as plx
    x = plx_inputs.prefill(1, 2, 200, 64, seed=96, dtype="bf16", rho="normal", rho_std=0.3)
    t = x.device_tensors()
    do = torch.randn((1, 2, 200, 64), generator=torch.Generator().manual_seed(6)).to("cuda").to(torch.bfloat16)
    ref, got = both(lambda: plx.plx_bwd(t["q"], t["k"], t["v"], t["rho"], do, scale=x.scale))
    same(ref, got)


def test_debug_build_lla():
    import torch
    import parameterized_local_linear_02_b300 as plx
    x = plx_inputs.prefill(1, 2, 96, 64, seed=97, dtype="f32", rho="zero")
    tl = {n: torch.from_numpy(getattr(x, n)).to("cuda") for n in ("q", "k", "v")}
    ref, got = both(lambda: plx.plx_lla_f32(tl["q"], tl["k"], tl["v"], lam=0.1, max_iters=8, tol=1e-6,
                                           scale=x.scale))
    same(ref[:1], got[:1])


@pytest.mark.parametrize("shape", [(1, 2, 300, 128), (2, 1, 130, 64)])
def test_debug_build_training_pair(shape):
    """plx_fwd_train and plx_bwd_saved under the bounds checks."""
    import torch
    import parameterized_local_linear_02_b300 as plx
    B, H, N, d = shape
    x = plx_inputs.prefill(B, H, N, d, seed=N + d + 1, dtype="bf16", rho="normal", rho_std=0.3)
    t = x.device_tensors()
    dout = torch.randn((B, H, N, d), device="cuda").to(torch.bfloat16)

    def run():
        o, lse, vbar, c = plx.plx_fwd_train(t["q"], t["k"], t["v"], t["rho"])
        g = plx.plx_bwd_saved(t["q"], t["k"], t["v"], t["rho"], dout, o, lse, vbar, c)
        return (o, lse, vbar, c) + tuple(g)
    ref, got = both(run)
    same(ref, got)


def test_debug_build_host_forward():
    """plx_fwd_host (chunked copies around the forward) under the bounds checks."""
    import torch
    import parameterized_local_linear_02_b300 as plx
    B, H, N, d = 2, 5, 200, 128
    x = plx_inputs.prefill(B, H, N, d, seed=97, dtype="bf16", rho="normal", rho_std=0.3)
    t = x.device_tensors()
    host = {n: t[n].cpu().pin_memory() for n in ("q", "k", "v", "rho")}
    ws = torch.empty(plx.plx_fwd_host_workspace_size(B, H, N, d, torch.float32), dtype=torch.uint8, device="cuda")

    def run():
        out = torch.empty((B, H, N, d)).pin_memory()
        lse = torch.empty((B, H, N)).pin_memory()
        plx.plx_fwd_host(host["q"], host["k"], host["v"], host["rho"], out, lse, workspace=ws)
        torch.cuda.synchronize()
        return out, lse
    ref, got = both(run)
    same(ref, got)
