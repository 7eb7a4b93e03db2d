// status.cuh -- the device status word shared by every kernel of the library.
// Kernels OR PLX_DEV_ERR_* bits into it (a bounded wait that gave up, a decode
// length beyond the cache capacity); plx_last_device_error reads and clears it.
#pragma once
#include "ptx.cuh"

namespace plx {
__device__ unsigned int g_plx_status;
}  // namespace plx
