"""ctypes binding of libplx.so (argument marshalling only).

Each function checks tensor dtypes, shapes, devices and contiguity, passes
raw device pointers and the current torch CUDA stream to the C entry point
of the same name (include/plx.h), and raises PlxError on a non-zero status.
Outputs (and the decode workspace) are allocated with torch when the caller
does not pass them.  Nothing here computes any part of the attention.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import build as _build

PLX_BF16, PLX_F32 = 0, 1
# family switches (see plx_fwd_family in include/plx.h)
PLX_FAMILY_UNIFORM_WEIGHTS, PLX_FAMILY_NO_INTERCEPT = 0x1, 0x2
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "misaligned", 4: "CUDA error", 7: "range",
           5: "device-side wait timed out", 6: "workspace too small"}

_lib = None
_lock = threading.Lock()


class PlxError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {plx_strerror(status)} (status {status})")


def library_path() -> str:
    return _build.LIB


def library() -> ctypes.CDLL:
    """Load libplx.so, building it first if it is missing or older than its
    sources.  Raises if it cannot be built or loaded."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if _build.stale():
            _build.build()
        _lib = load(_build.LIB)
        return _lib


def load(path: str) -> ctypes.CDLL:
    """Open a build of the library (libplx.so, or the bounds-checking debug
    build) and declare the argument types of its entry points."""
    lib = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.plx_version.restype = i
    lib.plx_version.argtypes = []
    lib.plx_strerror.restype = ctypes.c_char_p
    lib.plx_strerror.argtypes = [i]
    lib.plx_fwd.restype = i
    lib.plx_fwd.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    lib.plx_fwd_cached.restype = i
    lib.plx_fwd_cached.argtypes = [vp] * 7 + [i] * 5 + [f, i, vp]
    lib.plx_fwd_family.restype = i
    lib.plx_fwd_family.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, f, ctypes.c_uint, i, vp]
    lib.plx_fwd_f32.restype = i
    lib.plx_fwd_f32.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, f, vp]
    lib.plx_decode.restype = i
    lib.plx_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, sz, i, vp]
    lib.plx_decode_paged.restype = i
    lib.plx_decode_paged.argtypes = [vp] * 8 + [i] * 6 + [f, i, vp, sz, i, vp]
    lib.plx_decode_family.restype = i
    lib.plx_decode_family.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, sz, ctypes.c_uint, i, vp]
    lib.plx_decode_num_splits.restype = i
    lib.plx_decode_num_splits.argtypes = [i, i, i, i]
    lib.plx_decode_workspace_size.restype = sz
    lib.plx_decode_workspace_size.argtypes = [i, i, i, i, i]
    lib.plx_bwd_f32.restype = i
    lib.plx_bwd_f32.argtypes = [vp] * 12 + [sz, i, i, i, i, f, vp]
    lib.plx_bwd_workspace_size.restype = sz
    lib.plx_bwd_workspace_size.argtypes = [i, i, i, i]
    lib.plx_bwd.restype = i
    lib.plx_bwd.argtypes = [vp] * 10 + [sz, i, i, i, i, f, vp]
    lib.plx_bwd_bf16_workspace_size.restype = sz
    lib.plx_bwd_bf16_workspace_size.argtypes = [i, i, i, i]
    lib.plx_fwd_host.restype = i
    lib.plx_fwd_host.argtypes = [vp] * 7 + [sz, i, i, i, i, f, i, vp]
    lib.plx_fwd_host_workspace_size.restype = sz
    lib.plx_fwd_host_workspace_size.argtypes = [i, i, i, i, i]
    lib.plx_fwd_train.restype = i
    lib.plx_fwd_train.argtypes = [vp] * 8 + [i, i, i, i, f, i, vp]
    lib.plx_bwd_saved.restype = i
    lib.plx_bwd_saved.argtypes = [vp] * 6 + [i] + [vp] * 8 + [sz, i, i, i, i, f, vp]
    lib.plx_decode_noalloc.restype = i
    lib.plx_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
    lib.plx_probe_proj.restype = i
    lib.plx_lla_f32.restype = i
    lib.plx_lla_f32.argtypes = [vp] * 8 + [sz, i, i, i, i, f, f, i, f, vp]
    lib.plx_lla_workspace_size.restype = sz
    lib.plx_lla_workspace_size.argtypes = [i, i, i, i]
    lib.plx_lla_kept_weights_workspace_size.restype = sz
    lib.plx_lla_kept_weights_workspace_size.argtypes = [i, i, i, i]
    lib.plx_probe_proj.argtypes = [vp, vp, vp, i, i, i, i, i, vp]
    lib.plx_last_device_error.restype = i
    lib.plx_last_device_error.argtypes = [vp]
    lib.plx_selftest_wait.restype = i
    lib.plx_selftest_wait.argtypes = [ctypes.c_uint, i, vp]
    lib.plx_decode_partials_size.restype = sz
    lib.plx_decode_partials_size.argtypes = [i, i, i, i]
    lib.plx_decode_partials.restype = i
    lib.plx_decode_partials.argtypes = [vp, vp, vp, vp, vp, i, vp, sz, i, i, i, i, f, i, vp]
    lib.plx_decode_combine.restype = i
    lib.plx_decode_combine.argtypes = [vp, i, i, vp, vp, i, i, i, i, ctypes.c_uint, i, vp]
    return lib


def plx_version() -> int:
    return library().plx_version()


def plx_strerror(status: int) -> str:
    try:
        return library().plx_strerror(int(status)).decode()
    except OSError:
        return _STATUS.get(int(status), "unknown status")


def _check(status: int, where: str):
    if status != 0:
        raise PlxError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t, name, dtype, shape, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _out_code(dtype) -> int:
    if dtype == torch.bfloat16:
        return PLX_BF16
    if dtype == torch.float32:
        return PLX_F32
    raise TypeError("out dtype must be torch.bfloat16 or torch.float32")


def plx_fwd(q, k, v, rho=None, *, scale=None, out=None, lse=None, out_dtype=torch.bfloat16,
            with_lse=True):
    """Causal PLX forward, bf16 [B, H, N, d] inputs on the tensor cores.

    ``rho=None`` runs the softmax-attention instantiation of the same kernel.
    Returns ``(out, lse)``; ``lse`` is None when ``with_lse`` is False."""
    return _fwd(q, k, v, rho, None, scale, out, lse, out_dtype, with_lse)


def plx_fwd_cached(q, rho, k_cache, v_cache, seqlens, *, scale=None, out=None, lse=None,
                   out_dtype=torch.bfloat16, with_lse=True):
    """T new query tokens per sequence against a bf16 KV cache, on the tensor
    cores: ``q``, ``rho`` bf16 [B, H, T, d]; ``k_cache``, ``v_cache`` bf16
    [B, H, S_cap, d] already holding the new tokens at positions
    seqlens[b] - T .. seqlens[b] - 1; ``seqlens`` int32 [B].  Query row i of
    sequence b attends to cache rows 0 .. seqlens[b] - T + i."""
    B, H, T, d = q.shape
    S_cap = k_cache.shape[2]
    dev = q.device
    _need(q, "q", torch.bfloat16, (B, H, T, d), dev)
    if rho is not None:
        _need(rho, "rho", torch.bfloat16, (B, H, T, d), dev)
    _need(k_cache, "k_cache", torch.bfloat16, (B, H, S_cap, d), dev)
    _need(v_cache, "v_cache", torch.bfloat16, (B, H, S_cap, d), dev)
    _need(seqlens, "seqlens", torch.int32, (B,), dev)
    if out is None:
        out = torch.empty((B, H, T, d), dtype=out_dtype, device=dev)
    else:
        _need(out, "out", out.dtype, (B, H, T, d), dev)
    if lse is None and with_lse:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    elif lse is not None:
        _need(lse, "lse", torch.float32, (B, H, T), dev)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = library().plx_fwd_cached(_ptr(q), _ptr(rho), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens), _ptr(out),
                                  _ptr(lse), B, H, T, S_cap, d, scale, _out_code(out.dtype), _stream(dev))
    _check(st, "plx_fwd_cached")
    return out, lse


def plx_fwd_family(q, k, v, rho=None, *, flags, scale=None, out=None, lse=None, out_dtype=torch.bfloat16,
                   with_lse=True):
    """plx_fwd with family switches: ``flags`` is a bitwise OR of
    PLX_FAMILY_UNIFORM_WEIGHTS and PLX_FAMILY_NO_INTERCEPT (0 is plx_fwd)."""
    return _fwd(q, k, v, rho, int(flags), scale, out, lse, out_dtype, with_lse)


def _fwd(q, k, v, rho, flags, scale, out, lse, out_dtype, with_lse):
    B, H, N, d = q.shape
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v)) + ((("rho", rho),) if rho is not None else ()):
        _need(t, name, torch.bfloat16, (B, H, N, d), dev)
    if out is None:
        out = torch.empty((B, H, N, d), dtype=out_dtype, device=dev)
    else:
        _need(out, "out", out.dtype, (B, H, N, d), dev)
    if lse is None and with_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    elif lse is not None:
        _need(lse, "lse", torch.float32, (B, H, N), dev)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if flags is None:
        st = library().plx_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(rho), _ptr(out), _ptr(lse), B, H, N, d,
                               scale, _out_code(out.dtype), _stream(dev))
        _check(st, "plx_fwd")
    else:
        st = library().plx_fwd_family(_ptr(q), _ptr(k), _ptr(v), _ptr(rho), _ptr(out), _ptr(lse), B, H, N, d,
                                      scale, flags, _out_code(out.dtype), _stream(dev))
        _check(st, "plx_fwd_family")
    return out, lse


def plx_fwd_f32(q, k, v, rho=None, *, scale=None, out=None, lse=None, with_lse=True):
    """Causal PLX forward, fp32 [B, H, N, d] inputs, fp32 arithmetic."""
    B, H, N, d = q.shape
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v)) + ((("rho", rho),) if rho is not None else ()):
        _need(t, name, torch.float32, (B, H, N, d), dev)
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
    else:
        _need(out, "out", torch.float32, (B, H, N, d), dev)
    if lse is None and with_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    elif lse is not None:
        _need(lse, "lse", torch.float32, (B, H, N), dev)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = library().plx_fwd_f32(_ptr(q), _ptr(k), _ptr(v), _ptr(rho), _ptr(out), _ptr(lse), B, H, N, d,
                               scale, _stream(dev))
    _check(st, "plx_fwd_f32")
    return out, lse


def plx_bwd_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return library().plx_bwd_workspace_size(B, H, N, d)


def plx_bwd_f32(q, k, v, rho, out, lse, dout, *, scale=None, workspace=None, grads=None):
    """Gradients (dq, dk, dv, drho) of the causal PLX forward, fp32 on the
    CUDA cores.  ``out`` and ``lse`` are the forward's outputs; ``rho=None``
    gives the softmax-attention gradients (drho is then None).  ``grads`` may
    pass preallocated (dq, dk, dv, drho) tensors."""
    B, H, N, d = q.shape
    dev = q.device
    names = (("q", q), ("k", k), ("v", v), ("out", out), ("dout", dout))
    for name, t in names + ((("rho", rho),) if rho is not None else ()):
        _need(t, name, torch.float32, (B, H, N, d), dev)
    _need(lse, "lse", torch.float32, (B, H, N), dev)
    if grads is None:
        grads = tuple(torch.empty((B, H, N, d), dtype=torch.float32, device=dev) for _ in range(3)) + (
            torch.empty((B, H, N, d), dtype=torch.float32, device=dev) if rho is not None else None,)
    dq, dk, dv, drho = grads
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)) + ((("drho", drho),) if rho is not None else ()):
        _need(t, name, torch.float32, (B, H, N, d), dev)
    need = plx_bwd_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = library().plx_bwd_f32(_ptr(q), _ptr(k), _ptr(v), _ptr(rho), _ptr(out), _ptr(lse), _ptr(dout),
                               _ptr(dq), _ptr(dk), _ptr(dv), _ptr(drho), _ptr(workspace), ws_bytes,
                               B, H, N, d, scale, _stream(dev))
    _check(st, "plx_bwd_f32")
    return dq, dk, dv, drho


def plx_bwd_bf16_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return library().plx_bwd_bf16_workspace_size(B, H, N, d)


def plx_bwd(q, k, v, rho, dout, *, scale=None, workspace=None, grads=None):
    """Gradients (dq, dk, dv, drho), fp32, of the bf16 causal PLX forward, on
    the tensor cores.  q, k, v, rho and dout (dL/do) are bf16 [B, H, N, d];
    the forward's row statistics are recomputed, so o and lse are not needed.
    ``rho=None`` gives the softmax-attention gradients (drho is then None).
    ``grads`` may pass preallocated (dq, dk, dv, drho) tensors."""
    B, H, N, d = q.shape
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("dout", dout)) + ((("rho", rho),) if rho is not None else ()):
        _need(t, name, torch.bfloat16, (B, H, N, d), dev)
    if grads is None:
        grads = tuple(torch.empty((B, H, N, d), dtype=torch.float32, device=dev) for _ in range(3)) + (
            torch.empty((B, H, N, d), dtype=torch.float32, device=dev) if rho is not None else None,)
    dq, dk, dv, drho = grads
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)) + ((("drho", drho),) if rho is not None else ()):
        _need(t, name, torch.float32, (B, H, N, d), dev)
    need = plx_bwd_bf16_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = library().plx_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(rho), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                           _ptr(drho), _ptr(workspace), ws_bytes, B, H, N, d, scale, _stream(dev))
    _check(st, "plx_bwd")
    return dq, dk, dv, drho


def plx_fwd_host_workspace_size(B: int, H: int, N: int, d: int, out_dtype=torch.float32) -> int:
    return library().plx_fwd_host_workspace_size(B, H, N, d, _out_code(out_dtype))


def plx_fwd_host(q, k, v, rho, out, lse=None, *, workspace, scale=None, stream=None):
    """plx_fwd on host tensors (page-locked for overlap): ``q``, ``k``, ``v``,
    ``rho`` bf16 [B, H, N, d] and ``out`` (fp32 or bf16) / ``lse`` (fp32
    [B, H, N] or None) on the CPU; ``workspace`` a CUDA uint8 tensor of
    plx_fwd_host_workspace_size bytes.  Asynchronous on ``stream`` (default:
    the current stream of the workspace's device): synchronize it before
    reading out and lse."""
    B, H, N, d = q.shape
    cpu = torch.device("cpu")
    for name, t in (("q", q), ("k", k), ("v", v)) + ((("rho", rho),) if rho is not None else ()):
        _need(t, name, torch.bfloat16, (B, H, N, d), cpu)
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out must be float32 or bfloat16")
    _need(out, "out", out.dtype, (B, H, N, d), cpu)
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, H, N), cpu)
    if not isinstance(workspace, torch.Tensor) or workspace.device.type != "cuda":
        raise ValueError("workspace must be a CUDA tensor")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st_ = stream if stream is not None else torch.cuda.current_stream(workspace.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(workspace.device):
        st = library().plx_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(rho), _ptr(out), _ptr(lse), _ptr(workspace),
                                    ws_bytes, B, H, N, d, scale, _out_code(out.dtype),
                                    ctypes.c_void_p(st_.cuda_stream))
    _check(st, "plx_fwd_host")
    return out, lse


def plx_fwd_train(q, k, v, rho, *, scale=None, out=None, lse=None, vbar=None, c=None, out_dtype=torch.float32):
    """plx_fwd for training: returns ``(out, lse, vbar, c)``, where vbar (fp32
    [B, H, N, d]) and c (fp32 [B, H, N]) are the per-row values plx_bwd_saved
    forms the gradients' row statistics from.  rho is required."""
    B, H, N, d = q.shape
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("rho", rho)):
        _need(t, name, torch.bfloat16, (B, H, N, d), dev)
    if out is None:
        out = torch.empty((B, H, N, d), dtype=out_dtype, device=dev)
    else:
        _need(out, "out", out.dtype, (B, H, N, d), dev)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    _need(lse, "lse", torch.float32, (B, H, N), dev)
    if vbar is None:
        vbar = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
    _need(vbar, "vbar", torch.float32, (B, H, N, d), dev)
    if c is None:
        c = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    _need(c, "c", torch.float32, (B, H, N), dev)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = library().plx_fwd_train(_ptr(q), _ptr(k), _ptr(v), _ptr(rho), _ptr(out), _ptr(lse), _ptr(vbar), _ptr(c),
                                 B, H, N, d, scale, _out_code(out.dtype), _stream(dev))
    _check(st, "plx_fwd_train")
    return out, lse, vbar, c


def plx_bwd_saved(q, k, v, rho, dout, out, lse, vbar=None, c=None, *, scale=None, workspace=None, grads=None):
    """plx_bwd from the training forward's saved values (plx_fwd_train's out,
    lse, vbar, c; for ``rho=None`` plx_fwd's out and lse, vbar and c unused):
    the row statistics come from a bandwidth-bound kernel instead of an
    attention pass.  Returns (dq, dk, dv, drho), fp32."""
    B, H, N, d = q.shape
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("dout", dout)) + ((("rho", rho),) if rho is not None else ()):
        _need(t, name, torch.bfloat16, (B, H, N, d), dev)
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out must be float32 or bfloat16")
    _need(out, "out", out.dtype, (B, H, N, d), dev)
    _need(lse, "lse", torch.float32, (B, H, N), dev)
    if rho is not None:
        if vbar is None or c is None:
            raise ValueError("vbar and c are required with rho")
        _need(vbar, "vbar", torch.float32, (B, H, N, d), dev)
        _need(c, "c", torch.float32, (B, H, N), dev)
    else:
        vbar = c = None
    if grads is None:
        grads = tuple(torch.empty((B, H, N, d), dtype=torch.float32, device=dev) for _ in range(3)) + (
            torch.empty((B, H, N, d), dtype=torch.float32, device=dev) if rho is not None else None,)
    dq, dk, dv, drho = grads
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)) + ((("drho", drho),) if rho is not None else ()):
        _need(t, name, torch.float32, (B, H, N, d), dev)
    need = plx_bwd_bf16_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = library().plx_bwd_saved(_ptr(q), _ptr(k), _ptr(v), _ptr(rho), _ptr(dout), _ptr(out), _out_code(out.dtype),
                                 _ptr(lse), _ptr(vbar), _ptr(c), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(drho),
                                 _ptr(workspace), ws_bytes, B, H, N, d, scale, _stream(dev))
    _check(st, "plx_bwd_saved")
    return dq, dk, dv, drho


def plx_lla_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return library().plx_lla_workspace_size(B, H, N, d)


def plx_lla_kept_weights_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return library().plx_lla_kept_weights_workspace_size(B, H, N, d)


def plx_lla_f32(q, k, v, *, lam, max_iters, tol=0.0, scale=None, workspace=None, out=None, rho_out=None,
                lse=None, steps=None, with_rho=True, with_steps=True, keep_weights=False):
    """Local linear attention with the probe solved by conjugate gradients
    (fp32 [B, H, N, d] q, k, v; ridge ``lam``; at most ``max_iters`` steps per
    row, a row stopping once |r| <= tol |mu|).  Returns ``(out, rho, lse,
    steps)``; rho (the solved probe) and steps (int32 per row) are None when
    not requested.  ``keep_weights`` allocates the larger workspace with which
    the CG steps keep their softmax weights (B H N^2 fp32 more; for N % 4 == 0
    and d in {64, 128} the steps after the first then run on the tensor cores
    in split tf32, within fp32 rounding of the recomputing path); a
    caller-given ``workspace`` of that size has the same effect."""
    B, H, N, d = q.shape
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.float32, (B, H, N, d), dev)
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
    _need(out, "out", torch.float32, (B, H, N, d), dev)
    if with_rho and rho_out is None:
        rho_out = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
    if rho_out is not None:
        _need(rho_out, "rho_out", torch.float32, (B, H, N, d), dev)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    _need(lse, "lse", torch.float32, (B, H, N), dev)
    if with_steps and steps is None:
        steps = torch.empty((B, H, N), dtype=torch.int32, device=dev)
    if steps is not None:
        _need(steps, "steps", torch.int32, (B, H, N), dev)
    need = plx_lla_kept_weights_workspace_size(B, H, N, d) if keep_weights else plx_lla_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = library().plx_lla_f32(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(rho_out), _ptr(lse), _ptr(steps),
                               _ptr(workspace), ws_bytes, B, H, N, d, scale, float(lam), int(max_iters),
                               float(tol), _stream(dev))
    _check(st, "plx_lla_f32")
    return out, rho_out, lse, steps


def plx_probe_proj(x, w_r, *, heads, out=None):
    """The probe projection rho = W_R x on the tensor cores, written in the
    [B, H, N, d] layout the PLX entry points read.  x is bf16 [B, N, Dx];
    w_r is bf16 [H * d, Dx] (head h in rows h d .. h d + d - 1); ``heads`` = H.
    Returns bf16 rho [B, H, N, d] (``out`` may pass it preallocated)."""
    if x.dim() != 3 or w_r.dim() != 2:
        raise ValueError("x must be [B, N, Dx] and w_r [H * d, Dx]")
    B, N, Dx = x.shape
    H = int(heads)
    if H < 1 or w_r.shape[0] % H != 0:
        raise ValueError(f"w_r has {w_r.shape[0]} rows, not a multiple of heads={H}")
    d = w_r.shape[0] // H
    dev = x.device
    _need(x, "x", torch.bfloat16, (B, N, Dx), dev)
    _need(w_r, "w_r", torch.bfloat16, (H * d, Dx), dev)
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (B, H, N, d), dev)
    st = library().plx_probe_proj(_ptr(x), _ptr(w_r), _ptr(out), B, N, H, d, Dx, _stream(dev))
    _check(st, "plx_probe_proj")
    return out


def plx_decode_num_splits(B: int, H: int, d: int, S_cap: int) -> int:
    return library().plx_decode_num_splits(B, H, d, S_cap)


def plx_decode_workspace_size(B: int, H: int, d: int, S_cap: int, num_splits: int = 0) -> int:
    return library().plx_decode_workspace_size(B, H, d, S_cap, num_splits)


def plx_decode(q, rho, k_cache, v_cache, seqlens, *, scale=None, num_splits=0, workspace=None,
               out=None, lse=None, out_dtype=torch.bfloat16, with_lse=True):
    """One-token PLX decode over a bf16 [B, H, S_cap, d] KV cache.

    ``q``, ``rho``: bf16 [B, H, d] (``rho=None``: softmax attention);
    ``seqlens``: int32 [B] on the device.  Returns ``(out, lse)``."""
    return _decode(q, rho, k_cache, v_cache, seqlens, None, scale, num_splits, workspace, out, lse, out_dtype,
                   with_lse)


def plx_decode_paged(q, rho, k_pages, v_pages, block_table, seqlens, *, scale=None, num_splits=0,
                     workspace=None, out=None, lse=None, out_dtype=torch.bfloat16, with_lse=True):
    """plx_decode over a paged bf16 cache: ``k_pages``, ``v_pages`` are
    [num_blocks, H, page_size, d]; ``block_table`` is int32 [B, max_blocks]
    (row r of sequence b is row r % page_size of block block_table[b, r //
    page_size]); ``q``, ``rho`` bf16 [B, H, d]; ``seqlens`` int32 [B]."""
    num_blocks, H, page, d = k_pages.shape
    B, max_blocks = block_table.shape
    dev = k_pages.device
    _need(q, "q", torch.bfloat16, (B, H, d), dev)
    if rho is not None:
        _need(rho, "rho", torch.bfloat16, (B, H, d), dev)
    _need(k_pages, "k_pages", torch.bfloat16, (num_blocks, H, page, d), dev)
    _need(v_pages, "v_pages", torch.bfloat16, (num_blocks, H, page, d), dev)
    _need(block_table, "block_table", torch.int32, (B, max_blocks), dev)
    _need(seqlens, "seqlens", torch.int32, (B,), dev)
    if out is None:
        out = torch.empty((B, H, d), dtype=out_dtype, device=dev)
    else:
        _need(out, "out", out.dtype, (B, H, d), dev)
    if lse is None and with_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    elif lse is not None:
        _need(lse, "lse", torch.float32, (B, H), dev)
    need = plx_decode_workspace_size(B, H, d, max_blocks * page, num_splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = library().plx_decode_paged(_ptr(q), _ptr(rho), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                    _ptr(seqlens), _ptr(out), _ptr(lse), B, H, d, page, max_blocks, num_blocks,
                                    scale, int(num_splits), _ptr(workspace), ws_bytes, _out_code(out.dtype),
                                    _stream(dev))
    _check(st, "plx_decode_paged")
    return out, lse


def plx_decode_family(q, rho, k_cache, v_cache, seqlens, *, flags, scale=None, num_splits=0, workspace=None,
                      out=None, lse=None, out_dtype=torch.bfloat16, with_lse=True):
    """plx_decode with family switches (``flags`` as for plx_fwd_family)."""
    return _decode(q, rho, k_cache, v_cache, seqlens, int(flags), scale, num_splits, workspace, out, lse,
                   out_dtype, with_lse)


def _decode(q, rho, k_cache, v_cache, seqlens, flags, scale, num_splits, workspace, out, lse, out_dtype,
            with_lse):
    B, H, S_cap, d = k_cache.shape
    dev = k_cache.device
    _need(q, "q", torch.bfloat16, (B, H, d), dev)
    if rho is not None:
        _need(rho, "rho", torch.bfloat16, (B, H, d), dev)
    _need(k_cache, "k_cache", torch.bfloat16, (B, H, S_cap, d), dev)
    _need(v_cache, "v_cache", torch.bfloat16, (B, H, S_cap, d), dev)
    _need(seqlens, "seqlens", torch.int32, (B,), dev)
    if out is None:
        out = torch.empty((B, H, d), dtype=out_dtype, device=dev)
    else:
        _need(out, "out", out.dtype, (B, H, d), dev)
    if lse is None and with_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    elif lse is not None:
        _need(lse, "lse", torch.float32, (B, H), dev)
    need = plx_decode_workspace_size(B, H, d, S_cap, num_splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if flags is None:
        st = library().plx_decode(_ptr(q), _ptr(rho), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens),
                                  _ptr(out), _ptr(lse), B, H, d, S_cap, scale, int(num_splits),
                                  _ptr(workspace), ws_bytes, _out_code(out.dtype), _stream(dev))
        _check(st, "plx_decode")
    else:
        st = library().plx_decode_family(_ptr(q), _ptr(rho), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens),
                                         _ptr(out), _ptr(lse), B, H, d, S_cap, scale, int(num_splits),
                                         _ptr(workspace), ws_bytes, flags, _out_code(out.dtype), _stream(dev))
        _check(st, "plx_decode_family")
    return out, lse


def plx_decode_partials_size(B: int, H: int, d: int, num_splits: int) -> int:
    return library().plx_decode_partials_size(B, H, d, num_splits)


def plx_decode_partials(q, rho, k_shard, v_shard, seqlens, *, key_begin, num_splits, scale=None, out=None):
    """The online-softmax states of one shard of the key range: ``k_shard``,
    ``v_shard`` bf16 [B, H, S_shard, d] hold positions key_begin ..
    key_begin + S_shard - 1.  Returns (or fills) fp32 partials, a flat buffer
    of [B*H][num_splits][2 d + 4] states (include/plx.h)."""
    B, H, S, d = k_shard.shape
    dev = k_shard.device
    _need(q, "q", torch.bfloat16, (B, H, d), dev)
    if rho is not None:
        _need(rho, "rho", torch.bfloat16, (B, H, d), dev)
    _need(k_shard, "k_shard", torch.bfloat16, (B, H, S, d), dev)
    _need(v_shard, "v_shard", torch.bfloat16, (B, H, S, d), dev)
    _need(seqlens, "seqlens", torch.int32, (B,), dev)
    n = plx_decode_partials_size(B, H, d, int(num_splits)) // 4
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=dev)
    else:
        _need(out, "partials", torch.float32, (n,), dev)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = library().plx_decode_partials(_ptr(q), _ptr(rho), _ptr(k_shard), _ptr(v_shard), _ptr(seqlens),
                                       int(key_begin), _ptr(out), out.numel() * 4, B, H, d, S, scale,
                                       int(num_splits), _stream(dev))
    _check(st, "plx_decode_partials")
    return out


def plx_decode_combine(partials, *, groups, num_splits, B, H, d, with_rho=True, flags=0, out=None, lse=None,
                       out_dtype=torch.bfloat16, with_lse=True):
    """Merge ``groups`` shards' partials, concatenated in shard order in the
    flat fp32 tensor ``partials``, into ``(out [B, H, d], lse [B, H])``."""
    dev = partials.device
    n = groups * (plx_decode_partials_size(B, H, d, int(num_splits)) // 4)
    _need(partials, "partials", torch.float32, (n,), dev)
    if out is None:
        out = torch.empty((B, H, d), dtype=out_dtype, device=dev)
    else:
        _need(out, "out", out.dtype, (B, H, d), dev)
    if lse is None and with_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    elif lse is not None:
        _need(lse, "lse", torch.float32, (B, H), dev)
    st = library().plx_decode_combine(_ptr(partials), int(groups), int(num_splits), _ptr(out), _ptr(lse), B, H, d,
                                      1 if with_rho else 0, int(flags), _out_code(out.dtype), _stream(dev))
    _check(st, "plx_decode_combine")
    return out, lse


def plx_decode_noalloc(q, rho, k_cache, v_cache, seqlens, *, scale=None, num_splits=0, out=None, lse=None,
                       out_dtype=torch.bfloat16, with_lse=True):
    """plx_decode through the entry point that takes no workspace: the split
    partials use the library's static device scratch, so the C call
    allocates nothing (for callers that cannot allocate device memory).
    Calls that overlap on the GPU share that scratch and race; this binding
    issues them on the current stream.  ``out`` and ``lse`` are allocated
    here with torch when not passed.  Returns ``(out, lse)``."""
    B, H, S_cap, d = k_cache.shape
    dev = k_cache.device
    _need(q, "q", torch.bfloat16, (B, H, d), dev)
    if rho is not None:
        _need(rho, "rho", torch.bfloat16, (B, H, d), dev)
    _need(k_cache, "k_cache", torch.bfloat16, (B, H, S_cap, d), dev)
    _need(v_cache, "v_cache", torch.bfloat16, (B, H, S_cap, d), dev)
    _need(seqlens, "seqlens", torch.int32, (B,), dev)
    if out is None:
        out = torch.empty((B, H, d), dtype=out_dtype, device=dev)
    else:
        _need(out, "out", out.dtype, (B, H, d), dev)
    if lse is None and with_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    elif lse is not None:
        _need(lse, "lse", torch.float32, (B, H), dev)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = library().plx_decode_noalloc(_ptr(q), _ptr(rho), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens),
                                      _ptr(out), _ptr(lse), B, H, d, S_cap, scale, int(num_splits),
                                      _out_code(out.dtype), _stream(dev))
    _check(st, "plx_decode_noalloc")
    return out, lse


def plx_selftest_wait(limit_us: int, arrive: bool, device=None) -> None:
    """Run the library's bounded device wait once (plx_selftest_wait in
    include/plx.h): with ``arrive=False`` nothing arrives and the wait gives up
    after ``limit_us`` microseconds, which the next plx_last_device_error
    reports as 5 (PLX_ERR_TIMEOUT)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    st = library().plx_selftest_wait(int(limit_us), 1 if arrive else 0, _stream(dev))
    if st != 0:
        raise PlxError(st, "plx_selftest_wait")


def plx_last_device_error(device=None) -> int:
    """Synchronise the current stream and return (and clear) the device
    status: 0 ok, 5 a device wait timed out, 1 a decode length exceeded the
    cache capacity."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    return library().plx_last_device_error(_stream(dev))
