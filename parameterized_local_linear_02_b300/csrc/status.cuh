// status.cuh -- the device status word shared by every kernel of the library.
// Kernels OR PLX_DEV_ERR_* bits into it (a bounded wait that gave up, a decode
// length beyond the cache capacity); plx_last_device_error reads and clears it.
#pragma once
#include "ptx.cuh"

namespace plx {
__device__ unsigned int g_plx_status;

// Bounds checks of the debug build (compiled with -DPLX_DEBUG): a check that
// fails records PLX_DEV_ERR_BOUNDS and the caller skips the access, so a
// wrong index shows up as a status, never as an access outside a buffer.  In
// the normal build the check is the constant true and compiles away.
#ifdef PLX_DEBUG
__device__ __forceinline__ bool in_bounds(bool ok) {
    if (!ok) atomicOr(&g_plx_status, PLX_DEV_ERR_BOUNDS);
    return ok;
}
#else
__device__ __forceinline__ constexpr bool in_bounds(bool) { return true; }
#endif
}  // namespace plx
