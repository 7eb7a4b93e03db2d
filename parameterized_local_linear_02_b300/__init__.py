"""Parallax (PLX) parameterized local linear attention on B300 (sm_103a).

The compute lives in ``libplx.so`` (hand-written CUDA: tcgen05/TMEM prefill,
backward and probe-projection kernels, fp32 prefill and backward kernels and a
split-KV decode kernel, and fp32 conjugate-gradient kernels for local linear
attention) behind the C ABI declared in ``include/plx.h``.  This package is a thin ctypes
binding with the same entry-point names; torch provides device memory and
streams only.  There is no CPU fallback: every call needs the CUDA library
and a CUDA device, and fails loudly otherwise.
"""
from .binding import (PLX_FAMILY_NO_INTERCEPT, PLX_FAMILY_UNIFORM_WEIGHTS, PlxError, plx_bwd, plx_bwd_bf16_workspace_size, plx_bwd_saved, plx_bwd_f32, plx_bwd_workspace_size, plx_decode, plx_decode_family, plx_decode_noalloc, plx_decode_paged, plx_decode_partials, plx_decode_partials_size, plx_decode_combine, plx_decode_num_splits, plx_decode_workspace_size,
                      plx_fwd, plx_fwd_cached, plx_fwd_host, plx_fwd_host_workspace_size, plx_fwd_train, plx_fwd_f32, plx_fwd_family, plx_last_device_error, plx_selftest_wait, plx_lla_f32, plx_lla_workspace_size, plx_lla_kept_weights_workspace_size, plx_probe_proj, plx_strerror, plx_version,
                      library, library_path)

__all__ = ["PlxError", "PLX_FAMILY_UNIFORM_WEIGHTS", "PLX_FAMILY_NO_INTERCEPT", "plx_fwd", "plx_fwd_cached", "plx_fwd_family", "plx_decode_family", "plx_fwd_f32", "plx_bwd", "plx_bwd_bf16_workspace_size", "plx_bwd_saved", "plx_fwd_train", "plx_fwd_host", "plx_fwd_host_workspace_size", "plx_bwd_f32", "plx_bwd_workspace_size", "plx_decode", "plx_decode_noalloc", "plx_decode_paged", "plx_decode_partials", "plx_decode_partials_size", "plx_decode_combine", "plx_decode_num_splits",
           "plx_decode_workspace_size", "plx_last_device_error", "plx_selftest_wait", "plx_lla_f32", "plx_lla_workspace_size", "plx_lla_kept_weights_workspace_size", "plx_probe_proj", "plx_strerror", "plx_version",
           "library", "library_path"]
