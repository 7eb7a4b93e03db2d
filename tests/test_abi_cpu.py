"""The C ABI library loads on a host without a GPU and exports every entry
point include/plx.h declares; argument validation runs before any device
access (CPU only, no compute calls)."""
import ctypes
import os
import re

import pytest

import parameterized_local_linear_02_b300 as plx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(plx_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("plx_fwd", "plx_fwd_f32", "plx_decode", "plx_decode_workspace_size",
                 "plx_decode_num_splits", "plx_strerror", "plx_last_device_error", "plx_version"):
        assert must in names


def test_library_exports_every_declared_symbol():
    lib = plx.library()
    for name in declared_functions():
        assert hasattr(lib, name), f"libplx.so does not export {name}"


def test_version_and_strerror():
    assert plx.plx_version() >= 100
    assert plx.plx_strerror(0) == "ok"
    assert "misaligned" in plx.plx_strerror(3)
    assert plx.plx_strerror(99) == "unknown status"


P16 = ctypes.c_void_p(0x10000)        # aligned fake device address (never dereferenced)
P_ODD = ctypes.c_void_p(0x10008)      # 8-byte aligned only


def test_fwd_rejects_bad_arguments_before_launch():
    lib = plx.library()
    f = lib.plx_fwd
    # null required pointer
    assert f(None, P16, P16, None, P16, None, 1, 1, 8, 128, 0.1, 0, None) == 1
    # non-positive sizes, bad scale, bad dtype
    assert f(P16, P16, P16, None, P16, None, 0, 1, 8, 128, 0.1, 0, None) == 1
    assert f(P16, P16, P16, None, P16, None, 1, 1, 0, 128, 0.1, 0, None) == 1
    assert f(P16, P16, P16, None, P16, None, 1, 1, 8, 128, -1.0, 0, None) == 1
    assert f(P16, P16, P16, None, P16, None, 1, 1, 8, 128, float("nan"), 0, None) == 1
    assert f(P16, P16, P16, None, P16, None, 1, 1, 8, 128, 0.1, 7, None) == 1
    # head dims without a kernel
    assert f(P16, P16, P16, None, P16, None, 1, 1, 8, 96, 0.1, 0, None) == 2
    assert f(P16, P16, P16, None, P16, None, 1, 1, 8, 256, 0.1, 0, None) == 2
    # misaligned pointers
    assert f(P_ODD, P16, P16, None, P16, None, 1, 1, 8, 128, 0.1, 0, None) == 3
    assert f(P16, P16, P16, P_ODD, P16, None, 1, 1, 8, 128, 0.1, 0, None) == 3


def test_fwd_f32_rejects_bad_arguments_before_launch():
    f = plx.library().plx_fwd_f32
    assert f(None, P16, P16, None, P16, None, 1, 1, 8, 64, 0.1, None) == 1
    assert f(P16, P16, P16, None, P16, None, 1, 1, 8, 48, 0.1, None) == 2
    assert f(P16, P16, P16, None, P16, None, 1, 1, 8, 288, 0.1, None) == 2
    assert f(P16, P16, P16, None, P_ODD, None, 1, 1, 8, 64, 0.1, None) == 3


def test_decode_rejects_bad_arguments_before_launch():
    f = plx.library().plx_decode
    args = lambda **kw: [kw.get("q", P16), kw.get("rho", None), kw.get("kc", P16), kw.get("vc", P16),
                         kw.get("sl", P16), kw.get("out", P16), None, kw.get("B", 2), 16,
                         kw.get("d", 128), kw.get("S", 64), 0.1, kw.get("ns", 1), None, 0,
                         kw.get("dt", 0), None]
    assert f(*args(q=None)) == 1
    assert f(*args(sl=None)) == 1
    assert f(*args(B=0)) == 1
    assert f(*args(ns=-1)) == 1
    assert f(*args(ns=5000)) == 1
    assert f(*args(dt=3)) == 1
    assert f(*args(d=96)) == 2
    assert f(*args(kc=P_ODD)) == 3


def test_decode_workspace_size_arithmetic():
    ws = plx.library().plx_decode_workspace_size
    assert ws(2, 16, 128, 4096, 1) == 0                         # one split: no partials
    assert ws(2, 16, 128, 4096, 4) == 2 * 16 * 4 * (2 * 128 + 4) * 4
    assert ws(3, 8, 64, 100, 7) == 3 * 8 * 7 * (2 * 64 + 4) * 4
    assert ws(2, 16, 96, 4096, 4) == 0                          # unsupported head dim
    assert ws(2, 16, 128, 4096, 2000) == 0                      # out of range


def test_bwd_rejects_bad_arguments_before_launch():
    lib = plx.library()
    P, WS = P16, ctypes.c_void_p(0x20000)
    args = [P] * 11
    # head dim not a multiple of 32
    assert lib.plx_bwd_f32(*args, WS, 1 << 20, 1, 1, 64, 48, 0.1, None) == 2
    # workspace missing or too small
    assert lib.plx_bwd_f32(*args, None, 0, 1, 1, 64, 64, 0.1, None) == 6
    need = lib.plx_bwd_workspace_size(2, 3, 64, 64)
    assert need == 2 * 3 * 64 * 16
    assert lib.plx_bwd_f32(*args, WS, need - 16, 2, 3, 64, 64, 0.1, None) == 6
    # misaligned gradient output
    bad = args[:]
    bad[8] = P_ODD
    assert lib.plx_bwd_f32(*bad, WS, need, 2, 3, 64, 64, 0.1, None) == 3
    # rho given without drho
    bad = args[:]
    bad[10] = None
    assert lib.plx_bwd_f32(*bad, WS, need, 2, 3, 64, 64, 0.1, None) == 1


def test_bwd_tc_rejects_bad_arguments_before_launch():
    """plx_bwd validates everything on the host and launches nothing on error
    (so these calls are safe without a GPU)."""
    lib = plx.library()
    P, WS = P16, ctypes.c_void_p(0x20000)
    ins = [P] * 5           # q, k, v, rho, dout
    outs = [P] * 4          # dq, dk, dv, drho
    need = lib.plx_bwd_bf16_workspace_size(2, 3, 64, 128)
    assert need == 2 * 3 * 64 * 16
    assert lib.plx_bwd_bf16_workspace_size(2, 3, 64, 96) == 0
    # head dim without a tensor-core kernel
    assert lib.plx_bwd(*ins, *outs, WS, need, 2, 3, 64, 96, 0.1, None) == 2
    # workspace missing or too small
    assert lib.plx_bwd(*ins, *outs, None, 0, 2, 3, 64, 128, 0.1, None) == 6
    assert lib.plx_bwd(*ins, *outs, WS, need - 16, 2, 3, 64, 128, 0.1, None) == 6
    # misaligned dout and dv
    bad = ins[:]
    bad[4] = P_ODD
    assert lib.plx_bwd(*bad, *outs, WS, need, 2, 3, 64, 128, 0.1, None) == 3
    bad = outs[:]
    bad[2] = P_ODD
    assert lib.plx_bwd(*ins, *bad, WS, need, 2, 3, 64, 128, 0.1, None) == 3
    # rho given without drho; missing dout
    bad = outs[:]
    bad[3] = None
    assert lib.plx_bwd(*ins, *bad, WS, need, 2, 3, 64, 128, 0.1, None) == 1
    bad = ins[:]
    bad[4] = None
    assert lib.plx_bwd(*bad, *outs, WS, need, 2, 3, 64, 128, 0.1, None) == 1
    # non-positive sizes, negative scale
    assert lib.plx_bwd(*ins, *outs, WS, need, 0, 3, 64, 128, 0.1, None) == 1
    assert lib.plx_bwd(*ins, *outs, WS, need, 2, 3, 64, 128, -1.0, None) == 1

def test_family_entry_points_reject_bad_flags_before_launch():
    """plx_fwd_family / plx_decode_family: unknown flag bits and the
    no-intercept switch without a probe are rejected on the host."""
    lib = plx.library()
    P = P16
    F32 = 1
    # unknown bit
    assert lib.plx_fwd_family(P, P, P, P, P, P, 1, 1, 64, 128, 0.1, 0x4, F32, None) == 1
    # no intercept without rho
    assert lib.plx_fwd_family(P, P, P, None, P, P, 1, 1, 64, 128, 0.1, 0x2, F32, None) == 1
    # still validated like plx_fwd: head dim
    assert lib.plx_fwd_family(P, P, P, P, P, P, 1, 1, 64, 96, 0.1, 0x1, F32, None) == 2
    SL = ctypes.c_void_p(0x30000)
    assert lib.plx_decode_family(P, P, P, P, SL, P, P, 1, 1, 128, 64, 0.1, 1, None, 0, 0x8, F32, None) == 1
    assert lib.plx_decode_family(P, None, P, P, SL, P, P, 1, 1, 128, 64, 0.1, 1, None, 0, 0x2, F32, None) == 1


def test_decode_paged_rejects_bad_arguments_before_launch():
    lib = plx.library()
    P = P16
    F32 = 1
    T = ctypes.c_void_p(0x40000)
    SL = ctypes.c_void_p(0x30000)
    args = lambda table, page, maxb, nblk: (P, P, P, P, table, SL, P, P, 2, 2, 128, page, maxb, nblk, 0.1, 1,
                                            None, 0, F32, None)
    assert lib.plx_decode_paged(*args(None, 64, 4, 8)) == 1            # no block table
    assert lib.plx_decode_paged(*args(T, 48, 4, 8)) == 1               # page not a multiple of 32
    assert lib.plx_decode_paged(*args(T, 64, 0, 8)) == 1               # no blocks per sequence
    assert lib.plx_decode_paged(*args(T, 64, 4, 0)) == 1               # empty cache
    assert lib.plx_decode_paged(*args(ctypes.c_void_p(0x40002), 64, 4, 8)) == 3   # misaligned table


def test_fwd_cached_rejects_bad_arguments_before_launch():
    lib = plx.library()
    P = P16
    SL = ctypes.c_void_p(0x30000)
    F32 = 1
    assert lib.plx_fwd_cached(P, P, P, P, None, P, P, 1, 2, 16, 64, 128, 0.1, F32, None) == 1   # no seqlens
    assert lib.plx_fwd_cached(P, P, P, P, SL, P, P, 1, 2, 65, 64, 128, 0.1, F32, None) == 1     # T > S_cap
    assert lib.plx_fwd_cached(P, P, P, P, SL, P, P, 1, 2, 0, 64, 128, 0.1, F32, None) == 1      # T < 1
    assert lib.plx_fwd_cached(P, P, P, P, SL, P, P, 1, 2, 16, 64, 96, 0.1, F32, None) == 2      # head dim
    assert lib.plx_fwd_cached(P, P, P, P, ctypes.c_void_p(0x30002), P, P, 1, 2, 16, 64, 128, 0.1, F32,
                              None) == 3                                                        # misaligned seqlens


def test_probe_proj_rejects_bad_arguments_before_launch():
    lib = plx.library()
    P = P16
    assert lib.plx_probe_proj(None, P, P, 1, 64, 2, 128, 256, None) == 1                      # no x
    assert lib.plx_probe_proj(P, P, None, 1, 64, 2, 128, 256, None) == 1                      # no rho
    assert lib.plx_probe_proj(P, P, P, 0, 64, 2, 128, 256, None) == 1                         # B < 1
    assert lib.plx_probe_proj(P, P, P, 1, 64, 2, 128, 0, None) == 1                           # Dx < 1
    assert lib.plx_probe_proj(P, P, P, 1, 64, 2, 96, 256, None) == 2                          # head dim
    assert lib.plx_probe_proj(P, P, P, 1, 64, 2, 128, 250, None) == 2                         # Dx % 8
    assert lib.plx_probe_proj(P, ctypes.c_void_p(0x40008), P, 1, 64, 2, 128, 256, None) == 3  # misaligned W_R


def test_lla_rejects_bad_arguments_before_launch():
    lib = plx.library()
    P = P16
    WS = ctypes.c_void_p(0x100000)
    need = lib.plx_lla_workspace_size(2, 3, 64, 64)
    assert need >= 2 * 3 * 64 * (4 * 64 + 4) * 4
    assert lib.plx_lla_workspace_size(2, 3, 64, 48) == 0
    args = lambda ws, nbytes, d, lam, iters, tol: (P, P, P, P, None, None, None, ws, nbytes, 2, 3, 64, d, 0.1, lam,
                                                   iters, tol, None)
    assert lib.plx_lla_f32(*args(WS, need, 64, -0.1, 8, 0.0)) == 1                  # negative lambda
    assert lib.plx_lla_f32(*args(WS, need, 64, 0.1, -1, 0.0)) == 1                  # negative iterations
    assert lib.plx_lla_f32(*args(WS, need, 64, 0.1, 8, float("nan"))) == 1          # tol not finite
    assert lib.plx_lla_f32(*args(WS, need, 48, 0.1, 8, 0.0)) == 2                   # head dim
    assert lib.plx_lla_f32(*args(None, 0, 64, 0.1, 8, 0.0)) == 6                    # no workspace
    assert lib.plx_lla_f32(*args(WS, need - 256, 64, 0.1, 8, 0.0)) == 6             # workspace too small
    assert lib.plx_lla_f32(*args(ctypes.c_void_p(0x100010), need, 64, 0.1, 8, 0.0)) == 3   # misaligned workspace
    assert lib.plx_lla_f32(None, P, P, P, None, None, None, WS, need, 2, 3, 64, 64, 0.1, 0.1, 8, 0.0, None) == 1


def test_decode_partials_and_combine_reject_bad_arguments_before_launch():
    lib = plx.library()
    P = P16
    assert lib.plx_decode_partials_size(2, 3, 128, 2) == 2 * 3 * 2 * (2 * 128 + 4) * 4
    assert lib.plx_decode_partials_size(2, 3, 96, 2) == 0
    assert lib.plx_decode_partials_size(2, 3, 128, 0) == 0
    need = lib.plx_decode_partials_size(2, 3, 128, 2)
    ok = (P, P, P, P, P, 0, P, need, 2, 3, 128, 64, 0.1, 2, None)

    def call(**kw):
        names = ("q", "rho", "k", "v", "sl", "kb", "parts", "bytes", "B", "H", "d", "S", "scale", "n", "st")
        a = dict(zip(names, ok))
        a.update(kw)
        return lib.plx_decode_partials(*[a[n] for n in names])
    assert call(q=None) == 1
    assert call(kb=-1) == 1
    assert call(n=0) == 1
    assert call(S=0) == 1
    assert call(d=96) == 2
    assert call(parts=P_ODD) == 3
    assert call(bytes=need - 4) == 6
    assert lib.plx_decode_combine(None, 2, 2, P, None, 2, 3, 128, 1, 0, 0, None) == 1
    assert lib.plx_decode_combine(P, 0, 2, P, None, 2, 3, 128, 1, 0, 0, None) == 1
    assert lib.plx_decode_combine(P, 2, 2, P, None, 2, 3, 128, 0, 2, 0, None) == 1     # no intercept without rho
    assert lib.plx_decode_combine(P, 2, 2, P, None, 2, 3, 128, 1, 1, 0, None) == 1     # uniform weights is not a combine flag
    assert lib.plx_decode_combine(P, 2, 2, P, None, 2, 3, 96, 1, 0, 0, None) == 2
    assert lib.plx_decode_combine(P_ODD, 2, 2, P, None, 2, 3, 128, 1, 0, 0, None) == 3


def test_selftest_wait_rejects_a_limit_out_of_range_before_launch():
    lib = plx.library()
    assert lib.plx_selftest_wait(0, 0, None) == 1
    assert lib.plx_selftest_wait(1000001, 1, None) == 1


def test_no_cpu_fallback_without_a_device():
    """With no CUDA device every entry point raises; none computes on the host.
    (Skipped on a GPU host: CPU tensors must never reach the library there.)"""
    import torch
    if torch.cuda.is_available():
        pytest.skip("checks the behaviour without a CUDA device")
    x = torch.zeros((1, 64, 64), dtype=torch.bfloat16)
    w = torch.zeros((128, 64), dtype=torch.bfloat16)
    qb = torch.zeros((1, 1, 8, 64), dtype=torch.bfloat16)
    qf = torch.zeros((1, 1, 8, 64), dtype=torch.float32)
    calls = [
        lambda: plx.plx_probe_proj(x, w, heads=1),
        lambda: plx.plx_lla_f32(qf, qf, qf, lam=0.1, max_iters=1),
        lambda: plx.plx_fwd(qb, qb, qb, qb),
        lambda: plx.plx_bwd(qb, qb, qb, qb, qb),
    ]
    for call in calls:
        with pytest.raises((RuntimeError, plx.PlxError)):
            call()


def test_fwd_train_and_bwd_saved_reject_bad_arguments_before_launch():
    lib = plx.library()
    f = lib.plx_fwd_train
    # q, k, v, rho, out, lse, vbar, c, B, H, N, d, scale, out_dtype, stream
    assert f(P16, P16, P16, None, P16, P16, P16, P16, 1, 1, 8, 128, 0.1, 1, None) == 1   # rho required
    assert f(P16, P16, P16, P16, P16, None, P16, P16, 1, 1, 8, 128, 0.1, 1, None) == 1   # lse required
    assert f(P16, P16, P16, P16, P16, P16, None, P16, 1, 1, 8, 128, 0.1, 1, None) == 1   # vbar required
    assert f(P16, P16, P16, P16, P16, P16, P16, None, 1, 1, 8, 128, 0.1, 1, None) == 1   # c required
    assert f(P16, P16, P16, P16, P16, P16, P16, P16, 1, 1, 0, 128, 0.1, 1, None) == 1
    assert f(P16, P16, P16, P16, P16, P16, P16, P16, 1, 1, 8, 128, 0.1, 9, None) == 1
    assert f(P16, P16, P16, P16, P16, P16, P16, P16, 1, 1, 8, 96, 0.1, 1, None) == 2
    assert f(P16, P16, P16, P16, P16, P16, P_ODD, P16, 1, 1, 8, 128, 0.1, 1, None) == 3
    g = lib.plx_bwd_saved
    ws = plx.plx_bwd_bf16_workspace_size(1, 1, 8, 128)
    # q, k, v, rho, dout, out, out_dtype, lse, vbar, c, dq, dk, dv, drho, ws, ws_bytes, B, H, N, d, scale, stream
    ok = [P16] * 6 + [1] + [P16] * 8 + [ws, 1, 1, 8, 128, 0.1, None]
    bad = list(ok); bad[8] = None                           # vbar missing while rho is given
    assert g(*bad) == 1
    bad = list(ok); bad[6] = 5                              # unknown out dtype
    assert g(*bad) == 1
    bad = list(ok); bad[19] = 96                            # head dim without a kernel
    assert g(*bad) == 2
    bad = list(ok); bad[5] = P_ODD                          # misaligned out
    assert g(*bad) == 3
    bad = list(ok); bad[15] = ws - 1                        # workspace too small
    assert g(*bad) == 6


def test_fwd_host_rejects_bad_arguments_before_launch():
    lib = plx.library()
    f = lib.plx_fwd_host
    ws = plx.plx_fwd_host_workspace_size(1, 2, 64, 128)
    assert ws > 0
    assert plx.plx_fwd_host_workspace_size(1, 2, 64, 96) == 0
    assert plx.plx_fwd_host_workspace_size(0, 2, 64, 128) == 0
    # more heads than chunks: the workspace holds three chunks of ceil(B H / 16) heads
    assert plx.plx_fwd_host_workspace_size(4, 16, 2048, 128) < 64 * 2048 * 128 * 12
    W = ctypes.c_void_p(0x100000)                    # 256-byte aligned fake device address
    # q, k, v, rho, out, lse, workspace, ws_bytes, B, H, N, d, scale, out_dtype, stream
    ok = [P16, P16, P16, None, P16, None, W, ws, 1, 2, 64, 128, 0.1, 1, None]
    bad = list(ok); bad[0] = None
    assert f(*bad) == 1
    bad = list(ok); bad[10] = 0
    assert f(*bad) == 1
    bad = list(ok); bad[13] = 4
    assert f(*bad) == 1
    bad = list(ok); bad[11] = 96
    assert f(*bad) == 2
    bad = list(ok); bad[6] = ctypes.c_void_p(0x100010)  # workspace 16- but not 256-byte aligned
    assert f(*bad) == 3
    bad = list(ok); bad[6] = None
    assert f(*bad) == 6
    bad = list(ok); bad[7] = ws - 1
    assert f(*bad) == 6
