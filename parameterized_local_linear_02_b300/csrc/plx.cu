// plx.cu -- the C ABI of the PLX attention library (see include/plx.h).
//
// One translation unit: argument validation, launch configuration, TMA
// tensor-map encoding and the device status word, around the kernels in
// fwd_tc.cuh (tcgen05 prefill), fwd_f32.cuh (fp32 prefill), bwd_tc.cuh (tcgen05
// backward), bwd_f32.cuh (fp32 backward), decode.cuh (split-KV decode +
// combine), proj_tc.cuh (tcgen05 probe projection) and lla_f32.cuh (local
// linear attention, conjugate gradients in fp32).  Every entry point
// validates its arguments before launching anything and never lets a C++
// exception escape.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "plx.h"
#include "bwd_f32.cuh"
#include "decode.cuh"
#include "fwd_f32.cuh"
#include "lla_f32.cuh"
#include "lla_tc.cuh"
#include "fwd_tc.cuh"
#include "bwd_tc.cuh"
#include "proj_tc.cuh"

namespace {

using plx::BwdTcCfg;
using plx::DecodeCfg;
using plx::FwdTcCfg;
using plx::ProjCfg;

constexpr int kMaxDevices = 64;
constexpr float kLog2e = 1.4426950408889634f;

inline bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

struct DeviceInfo {
    int sm_count = 0;
    int decode_blocks_per_sm[2] = {0, 0};   // d = 64, d = 128
    // the decode's split combine runs inside one thread-block cluster of up to
    // kMaxFusedSplits CTAs (false if no such cluster can be resident)
    bool decode_cluster_ok = false;
};

constexpr int kMaxFusedSplits = plx::DECODE_MAX_CLUSTER_SPLITS;

std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ready[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_encode_tried = false;

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// Per-device facts and one-time kernel attributes.  Returns nullptr on error.
const DeviceInfo* device_info() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_dev_ready[dev]) return &g_dev[dev];
    DeviceInfo info;
    if (cudaDeviceGetAttribute(&info.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return nullptr;
    cudaError_t e = cudaSuccess;
    e = e ? e : set_smem(plx::plx_fwd_tc_kernel<128, true>, FwdTcCfg<128, true>::SMEM);
    e = e ? e : set_smem(plx::plx_fwd_tc_kernel<128, false>, FwdTcCfg<128, false>::SMEM);
    e = e ? e : set_smem(plx::plx_fwd_tc_kernel<64, true>, FwdTcCfg<64, true>::SMEM);
    e = e ? e : set_smem(plx::plx_fwd_tc_kernel<64, false>, FwdTcCfg<64, false>::SMEM);
    e = e ? e : set_smem(plx::plx_fwd_tc_kernel<128, true, true>, FwdTcCfg<128, true>::SMEM);
    e = e ? e : set_smem(plx::plx_fwd_tc_kernel<128, false, true>, FwdTcCfg<128, false>::SMEM);
    e = e ? e : set_smem(plx::plx_fwd_tc_kernel<64, true, true>, FwdTcCfg<64, true>::SMEM);
    e = e ? e : set_smem(plx::plx_fwd_tc_kernel<64, false, true>, FwdTcCfg<64, false>::SMEM);
    e = e ? e : set_smem(plx::plx_fwd_tc_kernel<128, true, false, true>, FwdTcCfg<128, true>::SMEM);
    e = e ? e : set_smem(plx::plx_fwd_tc_kernel<64, true, false, true>, FwdTcCfg<64, true>::SMEM);
    e = e ? e : set_smem(plx::plx_bwd_tc_kernel<128, true, plx::BWD_STATS>, BwdTcCfg<128, true, plx::BWD_STATS>::SMEM);
    e = e ? e : set_smem(plx::plx_bwd_tc_kernel<128, false, plx::BWD_STATS>, BwdTcCfg<128, false, plx::BWD_STATS>::SMEM);
    e = e ? e : set_smem(plx::plx_bwd_tc_kernel<64, true, plx::BWD_STATS>, BwdTcCfg<64, true, plx::BWD_STATS>::SMEM);
    e = e ? e : set_smem(plx::plx_bwd_tc_kernel<64, false, plx::BWD_STATS>, BwdTcCfg<64, false, plx::BWD_STATS>::SMEM);
    e = e ? e : set_smem(plx::plx_bwd_tc_kernel<128, true, plx::BWD_DQ>, BwdTcCfg<128, true, plx::BWD_DQ>::SMEM);
    e = e ? e : set_smem(plx::plx_bwd_tc_kernel<128, false, plx::BWD_DQ>, BwdTcCfg<128, false, plx::BWD_DQ>::SMEM);
    e = e ? e : set_smem(plx::plx_bwd_tc_kernel<128, true, plx::BWD_DKV>, BwdTcCfg<128, true, plx::BWD_DKV>::SMEM);
    e = e ? e : set_smem(plx::plx_bwd_tc_kernel<128, false, plx::BWD_DKV>, BwdTcCfg<128, false, plx::BWD_DKV>::SMEM);
    e = e ? e : set_smem(plx::plx_bwd_tc_kernel<64, true, plx::BWD_DQ>, BwdTcCfg<64, true, plx::BWD_DQ>::SMEM);
    e = e ? e : set_smem(plx::plx_bwd_tc_kernel<64, false, plx::BWD_DQ>, BwdTcCfg<64, false, plx::BWD_DQ>::SMEM);
    e = e ? e : set_smem(plx::plx_bwd_tc_kernel<64, true, plx::BWD_DKV>, BwdTcCfg<64, true, plx::BWD_DKV>::SMEM);
    e = e ? e : set_smem(plx::plx_bwd_tc_kernel<64, false, plx::BWD_DKV>, BwdTcCfg<64, false, plx::BWD_DKV>::SMEM);
    e = e ? e : set_smem(plx::plx_lla_cg_gemm_kernel<128>, plx::LlaGemmCfg<128>::SMEM);
    e = e ? e : set_smem(plx::plx_lla_cg_gemm_kernel<64>, plx::LlaGemmCfg<64>::SMEM);
    e = e ? e : set_smem(plx::plx_lla_cg_gemm_kernel<128, 2>, plx::LlaGemmCfg<128>::SMEM);
    e = e ? e : set_smem(plx::plx_lla_cg_gemm_kernel<64, 2>, plx::LlaGemmCfg<64>::SMEM);
    e = e ? e : set_smem(plx::plx_lla_cg_gemm_kernel<128, 3>, plx::LlaGemmCfg<128>::SMEM);
    e = e ? e : set_smem(plx::plx_lla_cg_gemm_kernel<64, 3>, plx::LlaGemmCfg<64>::SMEM);
    e = e ? e : set_smem(plx::plx_lla_kbar_gemm_kernel<128, true>, plx::LlaKbarCfg<128>::SMEM);
    e = e ? e : set_smem(plx::plx_lla_kbar_gemm_kernel<64, true>, plx::LlaKbarCfg<64>::SMEM);
    e = e ? e : set_smem(plx::plx_lla_cg_tc_kernel<128>, plx::LlaTcCfg<128>::SMEM);
    e = e ? e : set_smem(plx::plx_lla_cg_tc_kernel<64>, plx::LlaTcCfg<64>::SMEM);
    e = e ? e : set_smem(plx::plx_lla_out_gemm_kernel<128>, plx::LlaOutCfg<128>::SMEM);
    e = e ? e : set_smem(plx::plx_lla_out_gemm_kernel<64>, plx::LlaOutCfg<64>::SMEM);
    e = e ? e : set_smem(plx::plx_lla_out_gemm_kernel<128, true>, plx::LlaOutCfg<128>::SMEM);
    e = e ? e : set_smem(plx::plx_lla_out_gemm_kernel<64, true>, plx::LlaOutCfg<64>::SMEM);
    e = e ? e : set_smem(plx::plx_lla_kbar_gemm_kernel<128>, plx::LlaKbarCfg<128>::SMEM);
    e = e ? e : set_smem(plx::plx_lla_kbar_gemm_kernel<64>, plx::LlaKbarCfg<64>::SMEM);
    e = e ? e : set_smem(plx::plx_proj_tc_kernel<128>, ProjCfg<128>::SMEM);
    e = e ? e : set_smem(plx::plx_proj_tc_kernel<64>, ProjCfg<64>::SMEM);
    e = e ? e : set_smem(plx::plx_decode_split_kernel<128, true>, DecodeCfg<128>::SMEM);
    e = e ? e : set_smem(plx::plx_decode_split_kernel<128, false>, DecodeCfg<128>::SMEM);
    e = e ? e : set_smem(plx::plx_decode_split_kernel<64, true>, DecodeCfg<64>::SMEM);
    e = e ? e : set_smem(plx::plx_decode_split_kernel<64, false>, DecodeCfg<64>::SMEM);
    e = e ? e : set_smem(plx::plx_decode_split_kernel<128, true, true>, DecodeCfg<128>::SMEM);
    e = e ? e : set_smem(plx::plx_decode_split_kernel<128, false, true>, DecodeCfg<128>::SMEM);
    e = e ? e : set_smem(plx::plx_decode_split_kernel<64, true, true>, DecodeCfg<64>::SMEM);
    e = e ? e : set_smem(plx::plx_decode_split_kernel<64, false, true>, DecodeCfg<64>::SMEM);
    if (e != cudaSuccess) return nullptr;
    // clusters of more than 8 CTAs are opt-in; without the opt-in, or if no
    // cluster of kMaxFusedSplits decode CTAs fits, the combine stays a kernel
    {
        bool ok = true;
        auto allow = [&](auto kernel) {
            ok = ok && cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
        };
        allow(plx::plx_decode_split_kernel<128, true, true>);
        allow(plx::plx_decode_split_kernel<128, false, true>);
        allow(plx::plx_decode_split_kernel<64, true, true>);
        allow(plx::plx_decode_split_kernel<64, false, true>);
        if (ok) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 1;
            attr[0].val.clusterDim.y = kMaxFusedSplits;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(1, kMaxFusedSplits, 1);
            cfg.blockDim = dim3(DecodeCfg<128>::THREADS, 1, 1);
            cfg.dynamicSmemBytes = DecodeCfg<128>::SMEM;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            ok = cudaOccupancyMaxActiveClusters(&clusters, plx::plx_decode_split_kernel<128, true, true>, &cfg) ==
                     cudaSuccess &&
                 clusters > 0;
        }
        cudaGetLastError();   // a refused opt-in is not an error of the library
        info.decode_cluster_ok = ok;
    }
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, plx::plx_decode_split_kernel<64, true>,
                                                      DecodeCfg<64>::THREADS, DecodeCfg<64>::SMEM) != cudaSuccess)
        return nullptr;
    info.decode_blocks_per_sm[0] = nb > 0 ? nb : 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, plx::plx_decode_split_kernel<128, true>,
                                                      DecodeCfg<128>::THREADS, DecodeCfg<128>::SMEM) != cudaSuccess)
        return nullptr;
    info.decode_blocks_per_sm[1] = nb > 0 ? nb : 1;
    g_dev[dev] = info;
    g_dev_ready[dev] = true;
    return &g_dev[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_encode_tried) {
        g_encode_tried = true;
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    return g_encode;
}

// 3-D bf16 tensor map over [BH][N][d] with a {64, box_rows, 1} box, 128B swizzle.
bool make_map(CUtensorMap* map, const void* base, int d, int N, long long BH, int box_rows) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D output tensor map over [BH][N][d] (fp32 or bf16) for the prefill's TMA
// stores: a {32 columns, 32 rows, 1} box, swizzled across its row (128 bytes
// for fp32, 64 for bf16).
bool make_out_map(CUtensorMap* map, void* base, int d, int N, long long BH, bool f32) {
    auto enc = encoder();
    if (!enc) return false;
    const cuuint64_t es = f32 ? 4 : 2;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * es, static_cast<cuuint64_t>(N) * d * es};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

plx_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? PLX_OK : PLX_ERR_CUDA;
}

bool valid_scale(float scale) { return std::isfinite(scale) && scale >= 0.f; }

// The cached mode of the tcgen05 forward: Tq query rows per head (q, rho, out, lse are [BH][Tq]),
// K/V from a cache of N rows per head, query row i at position
// seqlens[b] - Tq + i.  Tq = 0 and seqlens = nullptr: the self-attention
// prefill (Tq = N, query row i at position i).
struct CachedQueries {
    int Tq = 0;
    const int32_t* seqlens = nullptr;
    int H = 1;
};

// The tcgen05 forward: the self-attention prefill, or the cached mode.
// vbar != nullptr: the training forward, which also writes vbar (fp32, the layout of an fp32 o) and
// c (fp32 per row); PLX self-attention prefill only.
template <int D, bool PLX>
plx_status launch_fwd_tc(const void* q, const void* k, const void* v, const void* rho, void* out, float* lse,
                         int N, long long BH, float scale, plx_dtype out_dtype, cudaStream_t stream,
                         int sm_count, bool no_intercept = false, const CachedQueries& cq = CachedQueries(),
                         float* vbar = nullptr, float* c_out = nullptr) {
    using Cfg = FwdTcCfg<D, PLX>;
    const int Tq = cq.Tq > 0 ? cq.Tq : N;
    const long long n_qt = (Tq + Cfg::BM - 1) / Cfg::BM;
    const long long n_items = BH * n_qt;
    if (n_items > INT_MAX || BH > INT_MAX) return PLX_ERR_UNSUPPORTED;
    CUtensorMap mq, mr, mk, mv, mo, mvb;
    if (!make_map(&mq, q, D, Tq, BH, Cfg::BM) || !make_map(&mk, k, D, N, BH, Cfg::BN) ||
        !make_map(&mv, v, D, N, BH, Cfg::BN))
        return PLX_ERR_CUDA;
    if (!make_out_map(&mo, out, D, Tq, BH, out_dtype == PLX_F32)) return PLX_ERR_CUDA;
    const bool train = PLX && vbar != nullptr && !cq.seqlens;
    if (train) {
        if (!make_out_map(&mvb, vbar, D, Tq, BH, true)) return PLX_ERR_CUDA;
    } else {
        mvb = mo;
    }
    if (PLX) {
        if (!make_map(&mr, rho, D, Tq, BH, Cfg::BM)) return PLX_ERR_CUDA;
    } else {
        mr = mq;
    }
    plx::FwdTcParams p;
    p.lse = lse;
    p.N = N;
    p.Tq = Tq;
    p.seqlens = cq.seqlens;
    p.H = cq.H;
    p.BH = static_cast<int>(BH);
    p.n_qt = static_cast<int>(n_qt);
    p.n_items = static_cast<int>(n_items);
    p.scale_log2 = scale * kLog2e;
    p.out_f32 = out_dtype == PLX_F32;
    p.no_intercept = no_intercept ? 1 : 0;
    p.c_out = train ? c_out : nullptr;
    const int grid = static_cast<int>(n_items < sm_count ? n_items : sm_count);
    if (cq.seqlens) {
        plx::plx_fwd_tc_kernel<D, PLX, true><<<grid, Cfg::THREADS, Cfg::SMEM, stream>>>(mq, mr, mk, mv, mo, mvb, p);
    } else if (train) {
        if constexpr (PLX)
            plx::plx_fwd_tc_kernel<D, PLX, false, true><<<grid, Cfg::THREADS, Cfg::SMEM, stream>>>(mq, mr, mk, mv,
                                                                                                    mo, mvb, p);
    } else {
        plx::plx_fwd_tc_kernel<D, PLX, false><<<grid, Cfg::THREADS, Cfg::SMEM, stream>>>(mq, mr, mk, mv, mo, mvb, p);
    }
    return launch_status();
}

// The probe projection on the tensor cores: x is read through a {64, 128}
// box of its [B][N][Dx] view, W_R through a {64, 256} box of its [H d][Dx]
// view, rho written through the [B H][N][d] output map.
template <int D>
plx_status launch_proj_tc(const void* x, const void* w_r, void* rho, int B, int N, int H, int Dx,
                          cudaStream_t stream, int sm_count) {
    using Cfg = ProjCfg<D>;
    const long long n_mt = (N + Cfg::BM - 1) / Cfg::BM;
    const long long n_hg = (static_cast<long long>(H) * D + Cfg::BN - 1) / Cfg::BN;
    const long long n_items = static_cast<long long>(B) * n_mt * n_hg;
    if (2 * n_items > INT_MAX || static_cast<long long>(H) * D > INT_MAX) return PLX_ERR_UNSUPPORTED;
    CUtensorMap mx, mw, mw2, mo;
    if (!make_map(&mx, x, Dx, N, B, Cfg::BM) || !make_map(&mw, w_r, Dx, H * D, 1, Cfg::BN) ||
        !make_map(&mw2, w_r, Dx, H * D, 1, Cfg::BN / 2) ||
        !make_out_map(&mo, rho, D, N, static_cast<long long>(B) * H, false))
        return PLX_ERR_CUDA;
    const int grid = static_cast<int>(n_items < sm_count ? n_items : sm_count);
    // the last wave's items run as two half items when they fill at most half the grid
    const long long tail = n_items % grid;
    const bool split = n_items > grid && tail > 0 && 2 * tail <= grid;
    plx::ProjParams p;
    p.N = N;
    p.H = H;
    p.n_kb = (Dx + Cfg::BK - 1) / Cfg::BK;
    p.n_mt = static_cast<int>(n_mt);
    p.n_hg = static_cast<int>(n_hg);
    p.n_full = static_cast<int>(split ? n_items - tail : n_items);
    p.n_items = static_cast<int>(split ? n_items + tail : n_items);
    plx::plx_proj_tc_kernel<D><<<grid, Cfg::THREADS, Cfg::SMEM, stream>>>(mx, mw, mw2, mo, p);
    return launch_status();
}

// 3-D map over the backward's per-row statistics [BH][N] x float4, for the dkv
// pass: a {4, 64, 1} box, rows past N zero-filled.
bool make_stats_map(CUtensorMap* map, const void* base, int N, long long BH) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {4, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {16, static_cast<cuuint64_t>(N) * 16};
    cuuint32_t box[3] = {4, 64, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Workspace of plx_bwd: the per-row statistics.
size_t bwd_bf16_ws_bytes(long long BH, int N) { return align256(static_cast<size_t>(BH) * N * 16); }

// plx_bwd on the tensor cores: the pre-pass (the forward in statistics mode),
// the dq pass and the dkv pass.
// prep == nullptr: the statistics pass computes the row statistics; otherwise
// plx_bwd_prep_kernel forms them from the training forward's saved values.
template <int D, bool PLX>
plx_status launch_bwd_tc(const void* q, const void* k, const void* v, const void* rho, const void* dout, float* dq,
                         float* dk, float* dv, float* drho, void* workspace, int N, long long BH, float scale,
                         cudaStream_t s, int sm_count, const plx::BwdPrepParams* prep = nullptr) {
    using CfgS = BwdTcCfg<D, PLX, plx::BWD_STATS>;
    using CfgQ = BwdTcCfg<D, PLX, plx::BWD_DQ>;
    using CfgK = BwdTcCfg<D, PLX, plx::BWD_DKV>;
    auto* stats = static_cast<float4*>(workspace);
    const long long n_rt = (N + 127) / 128;
    if (BH * n_rt > INT_MAX) return PLX_ERR_UNSUPPORTED;
    plx::BwdTcParams p;
    p.stats = stats;
    p.stats_out = stats;
    p.N = N;
    p.BH = static_cast<int>(BH);
    p.n_rt = static_cast<int>(n_rt);
    p.n_items = static_cast<int>(BH * n_rt);
    p.scale = scale;
    p.scale_log2 = scale * kLog2e;
    const int grid = static_cast<int>(p.n_items < sm_count ? p.n_items : sm_count);
    CUtensorMap mq_r, mr_r, mo_r, mk_s, mv_s, mk_r, mv_r, mq_s, mr_s, mo_s, mstat, m_dq, m_dr, m_dk, m_dv;
    // dq pass: Q, rho, dO resident (128 rows); K, V streamed (64 rows)
    if (!make_map(&mq_r, q, D, N, BH, 128) || !make_map(&mo_r, dout, D, N, BH, 128) ||
        !make_map(&mk_s, k, D, N, BH, 64) || !make_map(&mv_s, v, D, N, BH, 64) ||
        !make_map(&mk_r, k, D, N, BH, 128) || !make_map(&mv_r, v, D, N, BH, 128) ||
        !make_map(&mq_s, q, D, N, BH, 64) || !make_map(&mo_s, dout, D, N, BH, 64) ||
        !make_stats_map(&mstat, stats, N, BH) || !make_out_map(&m_dq, dq, D, N, BH, true) ||
        !make_out_map(&m_dk, dk, D, N, BH, true) || !make_out_map(&m_dv, dv, D, N, BH, true))
        return PLX_ERR_CUDA;
    if (PLX) {
        if (!make_map(&mr_r, rho, D, N, BH, 128) || !make_map(&mr_s, rho, D, N, BH, 64) ||
            !make_out_map(&m_dr, drho, D, N, BH, true))
            return PLX_ERR_CUDA;
    } else {
        mr_r = mq_r;
        mr_s = mq_s;
        m_dr = m_dq;
    }
    // unused slots get a valid map of the right kind
    if (prep) {
        // the row statistics from the forward's lse, c, vbar and o
        plx::BwdPrepParams pp = *prep;
        pp.stats = stats;
        pp.rows = BH * N;
        const long long blocks = (pp.rows + plx::BWD_PREP_ROWS_PER_BLOCK - 1) / plx::BWD_PREP_ROWS_PER_BLOCK;
        if (blocks > INT_MAX) return PLX_ERR_UNSUPPORTED;
        plx::plx_bwd_prep_kernel<D><<<static_cast<unsigned>(blocks), plx::BWD_PREP_WARPS * 32, 0, s>>>(pp);
    } else {
        // the row statistics (lse, c, a, D) with the weights the two gradient passes use
        plx::plx_bwd_tc_kernel<D, PLX, plx::BWD_STATS><<<grid, CfgS::THREADS, CfgS::SMEM, s>>>(
            mq_r, PLX ? mr_r : mo_r, mo_r, mk_s, mv_s, mv_s, mstat, m_dq, m_dr, p);
    }
    if (cudaGetLastError() != cudaSuccess) return PLX_ERR_CUDA;
    plx::plx_bwd_tc_kernel<D, PLX, plx::BWD_DQ><<<grid, CfgQ::THREADS, CfgQ::SMEM, s>>>(
        mq_r, PLX ? mr_r : mo_r, mo_r, mk_s, mv_s, mv_s, mstat, m_dq, m_dr, p);
    if (cudaGetLastError() != cudaSuccess) return PLX_ERR_CUDA;
    plx::plx_bwd_tc_kernel<D, PLX, plx::BWD_DKV><<<grid, CfgK::THREADS, CfgK::SMEM, s>>>(
        mk_r, mv_r, mv_r, mq_s, PLX ? mr_s : mo_s, mo_s, mstat, m_dv, m_dk, p);
    return launch_status();
}

template <int DPL, bool PLX>
void launch_f32(const plx::FwdF32Params& p, long long BH, cudaStream_t stream) {
    dim3 grid((p.N + plx::F32_ROWS_PER_BLOCK - 1) / plx::F32_ROWS_PER_BLOCK, static_cast<unsigned>(BH));
    plx::plx_fwd_f32_kernel<DPL, PLX><<<grid, plx::F32_WARPS * 32, 0, stream>>>(p);
}

template <bool PLX>
bool dispatch_f32(const plx::FwdF32Params& p, int d, long long BH, cudaStream_t s) {
    switch (d / 32) {
        case 1: launch_f32<1, PLX>(p, BH, s); return true;
        case 2: launch_f32<2, PLX>(p, BH, s); return true;
        case 3: launch_f32<3, PLX>(p, BH, s); return true;
        case 4: launch_f32<4, PLX>(p, BH, s); return true;
        case 5: launch_f32<5, PLX>(p, BH, s); return true;
        case 6: launch_f32<6, PLX>(p, BH, s); return true;
        case 7: launch_f32<7, PLX>(p, BH, s); return true;
        case 8: launch_f32<8, PLX>(p, BH, s); return true;
        default: return false;
    }
}

// Workspace of plx_lla_f32 for R = B H N rows: kbar, x, r, p ([R][d] fp32
// each), lse, rs, rs0 ([R] fp32 each) and the step counts ([R] int32).
struct LlaWorkspace {
    float *kbar, *x, *r, *p, *lse, *rs, *rs0;
    int* steps;
    float* wts;      // the kept softmax weights [B H][N][N], or nullptr
};
size_t lla_ws_bytes(long long R, int d) {
    return 4 * align256(static_cast<size_t>(R) * d * sizeof(float)) + 4 * align256(static_cast<size_t>(R) * 4);
}
LlaWorkspace lla_ws_carve(void* base, long long R, int d) {
    auto* c = static_cast<char*>(base);
    const size_t vec = align256(static_cast<size_t>(R) * d * sizeof(float)), sc = align256(static_cast<size_t>(R) * 4);
    LlaWorkspace w;
    w.kbar = reinterpret_cast<float*>(c);
    w.x = reinterpret_cast<float*>(c + vec);
    w.r = reinterpret_cast<float*>(c + 2 * vec);
    w.p = reinterpret_cast<float*>(c + 3 * vec);
    w.lse = reinterpret_cast<float*>(c + 4 * vec);
    w.rs = reinterpret_cast<float*>(c + 4 * vec + sc);
    w.rs0 = reinterpret_cast<float*>(c + 4 * vec + 2 * sc);
    w.steps = reinterpret_cast<int*>(c + 4 * vec + 3 * sc);
    w.wts = nullptr;
    return w;
}
// The kept weights of every (b, h, i, j), j <= i, dense [B H][N][N] fp32 after
// the rest of the workspace (d = 64, 128: the block form of the CG step).
size_t lla_wts_bytes(long long BH, int N) {
    return align256(static_cast<size_t>(BH) * N * static_cast<size_t>(N) * sizeof(float));
}

// 3-D fp32 tensor map over the kept weights [BH][N][N] for the tensor-core CG
// step: a {32 keys, 128 rows, 1} box, 128B swizzle (rows past N read as 0).
// The row stride N * 4 bytes must be a multiple of 16: N % 4 == 0.
bool make_wts_map(CUtensorMap* map, const float* wts, int N, long long BH) {
    auto enc = encoder();
    if (!enc || N % 4 != 0) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(N) * 4, static_cast<cuuint64_t>(N) * N * 4};
    cuuint32_t box[3] = {32, 128, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(wts), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// plx_lla_f32's launches: kbar and lse (softmax attention of the keys
// themselves), the CG set-up, max_iters CG steps, and Parallax's output with
// the solved probe (centred).
template <int DPL>
void launch_lla(const float* q, const float* k, const float* v, float* out, float* lse, const LlaWorkspace& w,
                int N, long long BH, float scale, float lambda, int max_iters, float tol, cudaStream_t s) {
    plx::LlaParams lp{q, k, w.kbar, w.lse, w.x, w.r, w.p, w.rs, w.rs0, w.steps, N, scale, lambda, tol * tol, w.wts};
    if constexpr (DPL == 2 || DPL == 4) {
        // d = 64, 128: kbar and lse in the block form of the CG step
        using Kc = plx::LlaKbarCfg<DPL * 32>;
        dim3 kgrid((N + Kc::BM - 1) / Kc::BM, static_cast<unsigned>(BH));
        if (w.wts)       // it keeps the scores for the first CG step
            plx::plx_lla_kbar_gemm_kernel<DPL * 32, true><<<kgrid, Kc::THREADS, Kc::SMEM, s>>>(lp, w.kbar, w.lse);
        else
            plx::plx_lla_kbar_gemm_kernel<DPL * 32><<<kgrid, Kc::THREADS, Kc::SMEM, s>>>(lp, w.kbar, w.lse);
    } else {
        plx::FwdF32Params f{q, k, k, nullptr, w.kbar, w.lse, N, scale};
        launch_f32<DPL, false>(f, BH, s);
    }
    dim3 grid((N + plx::LLA_ROWS_PER_BLOCK - 1) / plx::LLA_ROWS_PER_BLOCK, static_cast<unsigned>(BH));
    plx::plx_lla_init_kernel<DPL><<<grid, plx::LLA_WARPS * 32, 0, s>>>(lp);
    if constexpr (DPL == 2 || DPL == 4) {
        // d = 64, 128: the step as two block GEMMs per key tile
        using G = plx::LlaGemmCfg<DPL * 32>;
        using T = plx::LlaTcCfg<DPL * 32>;
        dim3 ggrid((N + G::BM - 1) / G::BM, static_cast<unsigned>(BH));
        // with the weights kept, the later steps run on the tensor cores (split tf32)
        CUtensorMap mw;
        const bool tc = w.wts && make_wts_map(&mw, w.wts, N, BH);
        const int n_blk = (N + T::BM - 1) / T::BM;
        for (int it = 0; it < max_iters; ++it) {
            if (!w.wts)
                plx::plx_lla_cg_gemm_kernel<DPL * 32, 0><<<ggrid, G::THREADS, G::SMEM, s>>>(lp);
            else if (it == 0)      // the first step turns the kept scores into the weights
                plx::plx_lla_cg_gemm_kernel<DPL * 32, 3><<<ggrid, G::THREADS, G::SMEM, s>>>(lp);
            else if (tc)
                plx::plx_lla_cg_tc_kernel<DPL * 32>
                    <<<static_cast<unsigned>(n_blk * BH), T::THREADS, T::SMEM, s>>>(mw, lp, n_blk);
            else
                plx::plx_lla_cg_gemm_kernel<DPL * 32, 2><<<ggrid, G::THREADS, G::SMEM, s>>>(lp);
        }
    } else {
        for (int it = 0; it < max_iters; ++it)
            plx::plx_lla_cg_step_kernel<DPL><<<grid, plx::LLA_WARPS * 32, plx::LlaTile<DPL>::SMEM, s>>>(lp);
    }
    if constexpr (DPL == 2 || DPL == 4) {
        using O = plx::LlaOutCfg<DPL * 32>;
        dim3 ogrid((N + O::BM - 1) / O::BM, static_cast<unsigned>(BH));
        if (w.wts)       // the weights the first step kept serve the blocks whose rows all took a step
            plx::plx_lla_out_gemm_kernel<DPL * 32, true><<<ogrid, O::THREADS, O::SMEM, s>>>(lp, v, out, lse);
        else
            plx::plx_lla_out_gemm_kernel<DPL * 32><<<ogrid, O::THREADS, O::SMEM, s>>>(lp, v, out, lse);
    } else {
        plx::plx_lla_out_kernel<DPL><<<grid, plx::LLA_WARPS * 32, 0, s>>>(lp, v, out, lse);
    }
}

template <int DPL, bool PLX>
void launch_bwd(const plx::BwdF32Params& p, long long BH, cudaStream_t s) {
    dim3 grid((p.N + plx::BWD_ROWS_PER_BLOCK - 1) / plx::BWD_ROWS_PER_BLOCK, static_cast<unsigned>(BH));
    plx::plx_bwd_pre_kernel<DPL, PLX><<<grid, plx::BWD_WARPS * 32, 0, s>>>(p);
    plx::plx_bwd_dq_kernel<DPL, PLX><<<grid, plx::BWD_WARPS * 32, 0, s>>>(p);
    plx::plx_bwd_dkv_kernel<DPL, PLX><<<grid, plx::BWD_WARPS * 32, 0, s>>>(p);
}

template <bool PLX>
bool dispatch_bwd(const plx::BwdF32Params& p, int d, long long BH, cudaStream_t s) {
    switch (d / 32) {
        case 1: launch_bwd<1, PLX>(p, BH, s); return true;
        case 2: launch_bwd<2, PLX>(p, BH, s); return true;
        case 3: launch_bwd<3, PLX>(p, BH, s); return true;
        case 4: launch_bwd<4, PLX>(p, BH, s); return true;
        case 5: launch_bwd<5, PLX>(p, BH, s); return true;
        case 6: launch_bwd<6, PLX>(p, BH, s); return true;
        case 7: launch_bwd<7, PLX>(p, BH, s); return true;
        case 8: launch_bwd<8, PLX>(p, BH, s); return true;
        default: return false;
    }
}

// Split count for plx_decode: each (b, h) row's cache range is cut into s equal
// parts, one thread block each.  The blocks run in waves of `slots` (SMs x
// resident blocks per SM), so the estimated time is
//   ceil(BH s / slots) x (tiles per block + fixed cost per block)
// plus the combine pass when s > 1; pick the s that minimises it, with at least
// 8 tiles (256 cache rows) per block.
struct DecodePlan {
    int splits = 1;
    bool fused = false;   // the combine inside a thread-block cluster (one launch)
};

// Split count and combine form of the decode.  A split combine costs a second
// launch (kCombineCost, in tile units) unless it runs inside a cluster, which
// holds at most kMaxFusedSplits CTAs.
DecodePlan decode_plan(const DeviceInfo& info, long long BH, int d, int S_cap);

int decode_splits(const DeviceInfo& info, long long BH, int d, int S_cap) {
    return decode_plan(info, BH, d, S_cap).splits;
}

// The combine form for a given split count: inside a cluster when the grid is
// a single wave (measured: it saves the combine launch on small grids, about
// 2 us, but co-scheduling the CTAs of a cluster costs 10-20 % of bandwidth on
// grids of several waves).
bool decode_fused(const DeviceInfo& info, long long BH, int splits) {
    const long long slots = static_cast<long long>(info.sm_count) * info.decode_blocks_per_sm[1];
    return info.decode_cluster_ok && splits >= 2 && splits <= kMaxFusedSplits && BH * splits <= slots;
}

DecodePlan decode_plan(const DeviceInfo& info, long long BH, int d, int S_cap) {
    constexpr int T = 32;
    const long long slots = static_cast<long long>(info.sm_count) * info.decode_blocks_per_sm[d == 128 ? 1 : 0];
    const double tiles = static_cast<double>((static_cast<long long>(S_cap) + T - 1) / T);
    constexpr double kBlockCost = 2.0;     // per-block setup and merge, in tile units
    constexpr double kCombineCost = 4.0;   // the combine launch, in tile units
    auto cost = [&](long long s, bool fused) {
        const double waves = static_cast<double>((BH * s + slots - 1) / slots);
        return waves * (tiles / static_cast<double>(s) + kBlockCost) + (s > 1 && !fused ? kCombineCost : 0.0);
    };
    // a split of at least 8 tiles with the combine kernel, of at least 4 in a cluster
    long long smax = (static_cast<long long>(S_cap) + 8 * T - 1) / (8 * T);
    smax = smax > 1024 ? 1024 : (smax < 1 ? 1 : smax);
    DecodePlan best;
    double best_t = cost(1, false);
    for (long long s = 2; s <= smax; ++s) {
        const double t = cost(s, false);
        if (t < best_t) {
            best_t = t;
            best.splits = static_cast<int>(s);
            best.fused = false;
        }
    }
    if (info.decode_cluster_ok) {
        long long fmax = (static_cast<long long>(S_cap) + 4 * T - 1) / (4 * T);
        fmax = fmax > kMaxFusedSplits ? kMaxFusedSplits : fmax;
        for (long long s = 2; s <= fmax && BH * s <= slots; ++s) {
            const double t = cost(s, true);
            if (t < best_t) {
                best_t = t;
                best.splits = static_cast<int>(s);
                best.fused = true;
            }
        }
    }
    // a split count that a cluster holds always runs fused (same result, one launch)
    best.fused = decode_fused(info, BH, best.splits);
    return best;
}

size_t decode_ws_bytes(long long BH, int d, int splits) {
    if (splits <= 1) return 0;
    return static_cast<size_t>(BH) * splits * (2 * d + 4) * sizeof(float);
}

template <int D, bool PLX>
void launch_decode_split(const plx::DecodeParams& p, long long BH, cudaStream_t s) {
    using Cfg = DecodeCfg<D>;
    dim3 grid(static_cast<unsigned>(BH), static_cast<unsigned>(p.splits));
    plx::plx_decode_split_kernel<D, PLX><<<grid, Cfg::THREADS, Cfg::SMEM, s>>>(p);
}

template <int D, bool PLX>
void launch_decode_combine(const plx::DecodeParams& p, long long BH, cudaStream_t s) {
    plx::plx_decode_combine_kernel<D, PLX><<<static_cast<unsigned>(BH), D, 0, s>>>(p);
}

template <int D, bool PLX>
void launch_decode(const plx::DecodeParams& p, long long BH, cudaStream_t s, bool fused) {
    using Cfg = DecodeCfg<D>;
    dim3 grid(static_cast<unsigned>(BH), static_cast<unsigned>(p.splits));
    if (fused) {
        // the splits of one (b, h) form one cluster; its rank 0 merges them
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = static_cast<unsigned>(p.splits);
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = grid;
        cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
        cfg.dynamicSmemBytes = Cfg::SMEM;
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaLaunchKernelEx(&cfg, plx::plx_decode_split_kernel<D, PLX, true>, p);
        return;
    }
    plx::plx_decode_split_kernel<D, PLX><<<grid, Cfg::THREADS, Cfg::SMEM, s>>>(p);
    if (p.splits > 1) plx::plx_decode_combine_kernel<D, PLX><<<static_cast<unsigned>(BH), D, 0, s>>>(p);
}

// Split partials of plx_decode_noalloc: static device memory, one array per
// GPU that loads the library, shared by every call on that GPU.
constexpr size_t kNoallocScratchBytes = PLX_DECODE_NOALLOC_SCRATCH_BYTES;
static_assert(kNoallocScratchBytes % 256 == 0, "scratch size");
float* g_noalloc_scratch[kMaxDevices] = {};
unsigned long long g_noalloc_ctx[kMaxDevices] = {};   // the context the address above belongs to

}  // namespace

static __device__ __align__(256) float plx_decode_scratch[kNoallocScratchBytes / sizeof(float)];

namespace {

// Unique id of the calling thread's current CUDA context, 0 if there is none
// (or the driver cannot tell).
unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    }
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of plx_decode_scratch on the current device (host code cannot
// take the array's address directly: its name there is a host-side stand-in).
// It is looked up once per device and context: cudaDeviceReset gives the
// device a new context, in which the module and its array may sit elsewhere,
// so a call that finds another context than the one of the cached address
// looks it up again.  nullptr on a CUDA error.
float* noalloc_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    const unsigned long long ctx = current_context_id();
    if (!g_noalloc_scratch[dev] || ctx == 0 || ctx != g_noalloc_ctx[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, plx_decode_scratch) != cudaSuccess || !ptr) return nullptr;
        g_noalloc_scratch[dev] = static_cast<float*>(ptr);
        g_noalloc_ctx[dev] = current_context_id();   // now current, if it was not before
    }
    return g_noalloc_scratch[dev];
}

// plx_fwd_host: host buffers streamed through a device workspace in chunks of
// heads.  kHostBuffers chunks are in flight at once (one being copied in, one
// computed, one copied out), each in its own slice of the workspace.
constexpr int kHostBuffers = 3;
// Chunks per call (fewer when B H is smaller).  The copies set the time: every
// cudaMemcpyAsync costs about 2 us beyond its bytes, and the last chunk's
// kernel and copy-out run alone after the last copy-in.  On the bench prefill
// shape 8 chunks took 3.38 ms per call, 16 took 3.48 and 32 took 3.74.
constexpr int kHostChunks = 8;

// The copy streams and the events of the pipeline, one set per device and
// CUDA context (cudaDeviceReset gives the device a new context, in which the
// old handles are gone; they are created again, not destroyed).
struct HostPipe {
    unsigned long long ctx = 0;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t loaded[kHostBuffers] = {}, computed[kHostBuffers] = {}, stored[kHostBuffers] = {};
    std::mutex m;                         // one call's enqueue sequence at a time
};
HostPipe g_pipe[kMaxDevices];

// The pipeline of the current device with its lock held, or nullptr on a CUDA error.
HostPipe* host_pipe(std::unique_lock<std::mutex>& lock) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    HostPipe& hp = g_pipe[dev];
    lock = std::unique_lock<std::mutex>(hp.m);
    const unsigned long long ctx = current_context_id();
    if (hp.h2d && ctx != 0 && ctx == hp.ctx) return &hp;
    bool ok = cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.done, cudaEventDisableTiming) == cudaSuccess;
    for (int b = 0; ok && b < kHostBuffers; ++b)
        ok = cudaEventCreateWithFlags(&hp.loaded[b], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&hp.computed[b], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&hp.stored[b], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        hp.h2d = nullptr;
        return nullptr;
    }
    hp.ctx = current_context_id();
    return &hp;
}

// Heads per chunk and the bytes of one chunk's slice of the workspace.
struct HostChunking {
    long long heads_per_chunk = 0, chunks = 0;
    size_t in_bytes = 0, out_bytes = 0, lse_bytes = 0, slice_bytes = 0;
};
HostChunking host_chunking(long long BH, int N, int d, bool out_f32) {
    HostChunking hc;
    const long long want = BH < kHostChunks ? BH : kHostChunks;
    hc.heads_per_chunk = (BH + want - 1) / want;
    hc.chunks = (BH + hc.heads_per_chunk - 1) / hc.heads_per_chunk;
    const size_t rows = static_cast<size_t>(hc.heads_per_chunk) * N;
    hc.in_bytes = align256(rows * d * 2);
    hc.out_bytes = align256(rows * d * (out_f32 ? 4 : 2));
    hc.lse_bytes = align256(rows * 4);
    hc.slice_bytes = 4 * hc.in_bytes + hc.out_bytes + hc.lse_bytes;
    return hc;
}

// One bounded wait on a fresh barrier (the diagnostic behind
// plx_selftest_wait): a wait that gives up records PLX_DEV_ERR_TIMEOUT.
__global__ void plx_wait_selftest_kernel(unsigned long long limit_ns, int arrive) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    plx::mbar_init(&bar, 1);
    plx::fence_mbar_init();
    if (arrive) plx::mbar_arrive(&bar);
    if (!plx::mbar_wait_for(&bar, 0, limit_ns)) atomicOr(&plx::g_plx_status, plx::PLX_DEV_ERR_TIMEOUT);
}

}  // namespace

extern "C" {

int plx_version(void) { return 100; }

const char* plx_strerror(plx_status status) {
    switch (status) {
        case PLX_OK: return "ok";
        case PLX_ERR_INVALID_ARG: return "invalid argument";
        case PLX_ERR_UNSUPPORTED: return "unsupported size or head dimension";
        case PLX_ERR_MISALIGNED: return "misaligned pointer";
        case PLX_ERR_CUDA: return "CUDA error";
        case PLX_ERR_TIMEOUT: return "device-side wait timed out";
        case PLX_ERR_WORKSPACE: return "workspace missing or too small";
        case PLX_ERR_RANGE: return "non-finite output (inputs outside the supported range)";
        case PLX_ERR_BOUNDS: return "index outside its buffer (debug build)";
        default: return "unknown status";
    }
}

}  // extern "C"

namespace {

// plx_fwd with the family flags (0 = PLX itself).
plx_status fwd_impl(const void* q, const void* k, const void* v, const void* rho, void* out, float* lse, int B,
                    int H, int N, int d, float scale, unsigned flags, plx_dtype out_dtype, void* stream) {
    try {
        if (!q || !k || !v || !out) return PLX_ERR_INVALID_ARG;
        if (B < 1 || H < 1 || N < 1 || !valid_scale(scale)) return PLX_ERR_INVALID_ARG;
        if (out_dtype != PLX_BF16 && out_dtype != PLX_F32) return PLX_ERR_INVALID_ARG;
        if ((flags & ~(PLX_FAMILY_UNIFORM_WEIGHTS | PLX_FAMILY_NO_INTERCEPT)) != 0) return PLX_ERR_INVALID_ARG;
        if ((flags & PLX_FAMILY_NO_INTERCEPT) && !rho) return PLX_ERR_INVALID_ARG;
        if (flags & PLX_FAMILY_UNIFORM_WEIGHTS) scale = 0.f;
        const bool noint = (flags & PLX_FAMILY_NO_INTERCEPT) != 0;
        if (d != 128 && d != 64) return PLX_ERR_UNSUPPORTED;
        if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
            (rho && !aligned(rho, 16)) || (lse && !aligned(lse, 4)))
            return PLX_ERR_MISALIGNED;
        const DeviceInfo* info = device_info();
        if (!info) return PLX_ERR_CUDA;
        const long long BH = static_cast<long long>(B) * H;
        cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        if (d == 128)
            return rho ? launch_fwd_tc<128, true>(q, k, v, rho, out, lse, N, BH, scale, out_dtype, s, info->sm_count,
                                                  noint)
                       : launch_fwd_tc<128, false>(q, k, v, rho, out, lse, N, BH, scale, out_dtype, s,
                                                   info->sm_count);
        return rho ? launch_fwd_tc<64, true>(q, k, v, rho, out, lse, N, BH, scale, out_dtype, s, info->sm_count,
                                             noint)
                   : launch_fwd_tc<64, false>(q, k, v, rho, out, lse, N, BH, scale, out_dtype, s, info->sm_count);
    } catch (...) {
        return PLX_ERR_CUDA;
    }
}

}  // namespace

extern "C" {

plx_status plx_fwd(const void* q, const void* k, const void* v, const void* rho, void* out, float* lse, int B,
                   int H, int N, int d, float scale, plx_dtype out_dtype, void* stream) {
    return fwd_impl(q, k, v, rho, out, lse, B, H, N, d, scale, 0u, out_dtype, stream);
}

plx_status plx_fwd_family(const void* q, const void* k, const void* v, const void* rho, void* out, float* lse,
                          int B, int H, int N, int d, float scale, unsigned flags, plx_dtype out_dtype,
                          void* stream) {
    return fwd_impl(q, k, v, rho, out, lse, B, H, N, d, scale, flags, out_dtype, stream);
}

plx_status plx_fwd_cached(const void* q, const void* rho, const void* k_cache, const void* v_cache,
                          const int32_t* seqlens, void* out, float* lse, int B, int H, int T, int S_cap, int d,
                          float scale, plx_dtype out_dtype, void* stream) {
    try {
        if (!q || !k_cache || !v_cache || !seqlens || !out) return PLX_ERR_INVALID_ARG;
        if (B < 1 || H < 1 || T < 1 || S_cap < T || !valid_scale(scale)) return PLX_ERR_INVALID_ARG;
        if (out_dtype != PLX_BF16 && out_dtype != PLX_F32) return PLX_ERR_INVALID_ARG;
        if (d != 128 && d != 64) return PLX_ERR_UNSUPPORTED;
        if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
            (rho && !aligned(rho, 16)) || !aligned(seqlens, 4) || (lse && !aligned(lse, 4)))
            return PLX_ERR_MISALIGNED;
        const DeviceInfo* info = device_info();
        if (!info) return PLX_ERR_CUDA;
        const long long BH = static_cast<long long>(B) * H;
        cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        CachedQueries cq;
        cq.Tq = T;
        cq.seqlens = seqlens;
        cq.H = H;
        if (d == 128)
            return rho ? launch_fwd_tc<128, true>(q, k_cache, v_cache, rho, out, lse, S_cap, BH, scale, out_dtype, s,
                                                  info->sm_count, false, cq)
                       : launch_fwd_tc<128, false>(q, k_cache, v_cache, rho, out, lse, S_cap, BH, scale, out_dtype,
                                                   s, info->sm_count, false, cq);
        return rho ? launch_fwd_tc<64, true>(q, k_cache, v_cache, rho, out, lse, S_cap, BH, scale, out_dtype, s,
                                             info->sm_count, false, cq)
                   : launch_fwd_tc<64, false>(q, k_cache, v_cache, rho, out, lse, S_cap, BH, scale, out_dtype, s,
                                              info->sm_count, false, cq);
    } catch (...) {
        return PLX_ERR_CUDA;
    }
}

plx_status plx_fwd_f32(const float* q, const float* k, const float* v, const float* rho, float* out, float* lse,
                       int B, int H, int N, int d, float scale, void* stream) {
    try {
        if (!q || !k || !v || !out) return PLX_ERR_INVALID_ARG;
        if (B < 1 || H < 1 || N < 1 || !valid_scale(scale)) return PLX_ERR_INVALID_ARG;
        if (d < 32 || d > 256 || d % 32 != 0) return PLX_ERR_UNSUPPORTED;
        if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
            (rho && !aligned(rho, 16)) || (lse && !aligned(lse, 4)))
            return PLX_ERR_MISALIGNED;
        const long long BH = static_cast<long long>(B) * H;
        if (BH > 65535) return PLX_ERR_UNSUPPORTED;
        plx::FwdF32Params p{q, k, v, rho, out, lse, N, scale};
        cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        const bool ok = rho ? dispatch_f32<true>(p, d, BH, s) : dispatch_f32<false>(p, d, BH, s);
        if (!ok) return PLX_ERR_UNSUPPORTED;
        return launch_status();
    } catch (...) {
        return PLX_ERR_CUDA;
    }
}

size_t plx_bwd_workspace_size(int B, int H, int N, int d) {
    if (B < 1 || H < 1 || N < 1 || d < 32 || d > 256 || d % 32 != 0) return 0;
    return static_cast<size_t>(B) * H * N * 4 * sizeof(float);
}

plx_status plx_bwd_f32(const float* q, const float* k, const float* v, const float* rho, const float* out,
                       const float* lse, const float* dout, float* dq, float* dk, float* dv, float* drho,
                       void* workspace, size_t workspace_bytes, int B, int H, int N, int d, float scale,
                       void* stream) {
    try {
        if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv || (rho && !drho))
            return PLX_ERR_INVALID_ARG;
        if (B < 1 || H < 1 || N < 1 || !valid_scale(scale)) return PLX_ERR_INVALID_ARG;
        if (d < 32 || d > 256 || d % 32 != 0) return PLX_ERR_UNSUPPORTED;
        const void* ptrs16[] = {q, k, v, out, dout, dq, dk, dv, workspace};
        for (const void* ptr : ptrs16)
            if (ptr && !aligned(ptr, 16)) return PLX_ERR_MISALIGNED;
        if ((rho && (!aligned(rho, 16) || !aligned(drho, 16))) || !aligned(lse, 4)) return PLX_ERR_MISALIGNED;
        const long long BH = static_cast<long long>(B) * H;
        if (BH > 65535) return PLX_ERR_UNSUPPORTED;
        const size_t need = plx_bwd_workspace_size(B, H, N, d);
        if (!workspace || workspace_bytes < need) return PLX_ERR_WORKSPACE;
        plx::BwdF32Params p{q, k, v, rho, out, lse, dout, dq, dk, dv, drho, static_cast<float*>(workspace), N, scale};
        cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        const bool ok = rho ? dispatch_bwd<true>(p, d, BH, s) : dispatch_bwd<false>(p, d, BH, s);
        if (!ok) return PLX_ERR_UNSUPPORTED;
        return launch_status();
    } catch (...) {
        return PLX_ERR_CUDA;
    }
}

size_t plx_bwd_bf16_workspace_size(int B, int H, int N, int d) {
    if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return 0;
    return bwd_bf16_ws_bytes(static_cast<long long>(B) * H, N);
}

plx_status plx_bwd(const void* q, const void* k, const void* v, const void* rho, const void* dout, float* dq,
                   float* dk, float* dv, float* drho, void* workspace, size_t workspace_bytes, int B, int H, int N,
                   int d, float scale, void* stream) {
    try {
        if (!q || !k || !v || !dout || !dq || !dk || !dv || (rho && !drho)) return PLX_ERR_INVALID_ARG;
        if (B < 1 || H < 1 || N < 1 || !valid_scale(scale)) return PLX_ERR_INVALID_ARG;
        if (d != 128 && d != 64) return PLX_ERR_UNSUPPORTED;
        const void* ptrs16[] = {q, k, v, dout, dq, dk, dv, workspace};
        for (const void* ptr : ptrs16)
            if (ptr && !aligned(ptr, 16)) return PLX_ERR_MISALIGNED;
        if (rho && (!aligned(rho, 16) || !aligned(drho, 16))) return PLX_ERR_MISALIGNED;
        const size_t need = plx_bwd_bf16_workspace_size(B, H, N, d);
        if (!workspace || workspace_bytes < need) return PLX_ERR_WORKSPACE;
        const DeviceInfo* info = device_info();
        if (!info) return PLX_ERR_CUDA;
        const long long BH = static_cast<long long>(B) * H;
        cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        if (d == 128)
            return rho ? launch_bwd_tc<128, true>(q, k, v, rho, dout, dq, dk, dv, drho, workspace, N, BH, scale, s,
                                                  info->sm_count)
                       : launch_bwd_tc<128, false>(q, k, v, rho, dout, dq, dk, dv, drho, workspace, N, BH, scale, s,
                                                   info->sm_count);
        return rho ? launch_bwd_tc<64, true>(q, k, v, rho, dout, dq, dk, dv, drho, workspace, N, BH, scale, s,
                                             info->sm_count)
                   : launch_bwd_tc<64, false>(q, k, v, rho, dout, dq, dk, dv, drho, workspace, N, BH, scale, s,
                                              info->sm_count);
    } catch (...) {
        return PLX_ERR_CUDA;
    }
}

plx_status plx_fwd_train(const void* q, const void* k, const void* v, const void* rho, void* out, float* lse,
                         float* vbar, float* c, int B, int H, int N, int d, float scale, plx_dtype out_dtype,
                         void* stream) {
    try {
        if (!q || !k || !v || !rho || !out || !lse || !vbar || !c) return PLX_ERR_INVALID_ARG;
        if (B < 1 || H < 1 || N < 1 || !valid_scale(scale)) return PLX_ERR_INVALID_ARG;
        if (out_dtype != PLX_BF16 && out_dtype != PLX_F32) return PLX_ERR_INVALID_ARG;
        if (d != 128 && d != 64) return PLX_ERR_UNSUPPORTED;
        if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(rho, 16) || !aligned(out, 16) ||
            !aligned(vbar, 16) || !aligned(lse, 4) || !aligned(c, 4))
            return PLX_ERR_MISALIGNED;
        const DeviceInfo* info = device_info();
        if (!info) return PLX_ERR_CUDA;
        const long long BH = static_cast<long long>(B) * H;
        cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        if (d == 128)
            return launch_fwd_tc<128, true>(q, k, v, rho, out, lse, N, BH, scale, out_dtype, s, info->sm_count,
                                            false, CachedQueries(), vbar, c);
        return launch_fwd_tc<64, true>(q, k, v, rho, out, lse, N, BH, scale, out_dtype, s, info->sm_count, false,
                                       CachedQueries(), vbar, c);
    } catch (...) {
        return PLX_ERR_CUDA;
    }
}

size_t plx_fwd_host_workspace_size(int B, int H, int N, int d, plx_dtype out_dtype) {
    if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128) || (out_dtype != PLX_BF16 && out_dtype != PLX_F32)) return 0;
    const HostChunking hc = host_chunking(static_cast<long long>(B) * H, N, d, out_dtype == PLX_F32);
    return kHostBuffers * hc.slice_bytes;
}

plx_status plx_fwd_host(const void* q, const void* k, const void* v, const void* rho, void* out, float* lse,
                        void* workspace, size_t workspace_bytes, int B, int H, int N, int d, float scale,
                        plx_dtype out_dtype, void* stream) {
    try {
        if (!q || !k || !v || !out) return PLX_ERR_INVALID_ARG;
        if (B < 1 || H < 1 || N < 1 || !valid_scale(scale)) return PLX_ERR_INVALID_ARG;
        if (out_dtype != PLX_BF16 && out_dtype != PLX_F32) return PLX_ERR_INVALID_ARG;
        if (d != 128 && d != 64) return PLX_ERR_UNSUPPORTED;
        if (!workspace || !aligned(workspace, 256)) return workspace ? PLX_ERR_MISALIGNED : PLX_ERR_WORKSPACE;
        const size_t need = plx_fwd_host_workspace_size(B, H, N, d, out_dtype);
        if (need == 0 || workspace_bytes < need) return PLX_ERR_WORKSPACE;
        const DeviceInfo* info = device_info();
        if (!info) return PLX_ERR_CUDA;
        const long long BH = static_cast<long long>(B) * H;
        const bool f32 = out_dtype == PLX_F32;
        const HostChunking hc = host_chunking(BH, N, d, f32);
        const size_t head_in = static_cast<size_t>(N) * d * 2, head_out = static_cast<size_t>(N) * d * (f32 ? 4 : 2);
        const size_t head_lse = static_cast<size_t>(N) * 4;
        cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        std::unique_lock<std::mutex> lock;
        HostPipe* hp = host_pipe(lock);
        if (!hp) return PLX_ERR_CUDA;
        auto ck = [](cudaError_t e) { return e == cudaSuccess; };
        // the copies start after the caller's earlier work on `stream`
        if (!ck(cudaEventRecord(hp->start, s)) || !ck(cudaStreamWaitEvent(hp->h2d, hp->start, 0)) ||
            !ck(cudaStreamWaitEvent(hp->d2h, hp->start, 0)))
            return PLX_ERR_CUDA;
        const char* in_h[4] = {static_cast<const char*>(q), static_cast<const char*>(k), static_cast<const char*>(v),
                               static_cast<const char*>(rho)};
        for (long long c = 0; c < hc.chunks; ++c) {
            const int b = static_cast<int>(c % kHostBuffers);
            const long long h0 = c * hc.heads_per_chunk;
            const long long g = (BH - h0) < hc.heads_per_chunk ? (BH - h0) : hc.heads_per_chunk;
            char* slice = static_cast<char*>(workspace) + b * hc.slice_bytes;
            char* in_d[4] = {slice, slice + hc.in_bytes, slice + 2 * hc.in_bytes, slice + 3 * hc.in_bytes};
            char* out_d = slice + 4 * hc.in_bytes;
            float* lse_d = reinterpret_cast<float*>(out_d + hc.out_bytes);
            // a slice is reused once its previous chunk has been copied out
            if (c >= kHostBuffers && !ck(cudaStreamWaitEvent(hp->h2d, hp->stored[b], 0))) return PLX_ERR_CUDA;
            for (int a = 0; a < 4; ++a) {
                if (!in_h[a]) continue;
                if (!ck(cudaMemcpyAsync(in_d[a], in_h[a] + h0 * head_in, g * head_in, cudaMemcpyHostToDevice,
                                        hp->h2d)))
                    return PLX_ERR_CUDA;
            }
            if (!ck(cudaEventRecord(hp->loaded[b], hp->h2d)) || !ck(cudaStreamWaitEvent(s, hp->loaded[b], 0)))
                return PLX_ERR_CUDA;
            const void* r_d = rho ? in_d[3] : nullptr;
            float* l_d = lse ? lse_d : nullptr;
            plx_status st;
            if (d == 128)
                st = rho ? launch_fwd_tc<128, true>(in_d[0], in_d[1], in_d[2], r_d, out_d, l_d, N, g, scale, out_dtype,
                                                    s, info->sm_count)
                         : launch_fwd_tc<128, false>(in_d[0], in_d[1], in_d[2], r_d, out_d, l_d, N, g, scale,
                                                     out_dtype, s, info->sm_count);
            else
                st = rho ? launch_fwd_tc<64, true>(in_d[0], in_d[1], in_d[2], r_d, out_d, l_d, N, g, scale, out_dtype,
                                                   s, info->sm_count)
                         : launch_fwd_tc<64, false>(in_d[0], in_d[1], in_d[2], r_d, out_d, l_d, N, g, scale, out_dtype,
                                                    s, info->sm_count);
            if (st != PLX_OK) return st;
            if (!ck(cudaEventRecord(hp->computed[b], s)) || !ck(cudaStreamWaitEvent(hp->d2h, hp->computed[b], 0)))
                return PLX_ERR_CUDA;
            if (!ck(cudaMemcpyAsync(static_cast<char*>(out) + h0 * head_out, out_d, g * head_out,
                                    cudaMemcpyDeviceToHost, hp->d2h)))
                return PLX_ERR_CUDA;
            if (lse && !ck(cudaMemcpyAsync(reinterpret_cast<char*>(lse) + h0 * head_lse, lse_d, g * head_lse,
                                           cudaMemcpyDeviceToHost, hp->d2h)))
                return PLX_ERR_CUDA;
            if (!ck(cudaEventRecord(hp->stored[b], hp->d2h))) return PLX_ERR_CUDA;
        }
        // the caller's stream resumes once the last chunk is back in host memory
        if (!ck(cudaEventRecord(hp->done, hp->d2h)) || !ck(cudaStreamWaitEvent(s, hp->done, 0))) return PLX_ERR_CUDA;
        return PLX_OK;
    } catch (...) {
        return PLX_ERR_CUDA;
    }
}

plx_status plx_bwd_saved(const void* q, const void* k, const void* v, const void* rho, const void* dout,
                         const void* out, plx_dtype out_dtype, const float* lse, const float* vbar, const float* c,
                         float* dq, float* dk, float* dv, float* drho, void* workspace, size_t workspace_bytes, int B,
                         int H, int N, int d, float scale, void* stream) {
    try {
        if (!q || !k || !v || !dout || !out || !lse || !dq || !dk || !dv) return PLX_ERR_INVALID_ARG;
        if (rho && (!drho || !vbar || !c)) return PLX_ERR_INVALID_ARG;
        if (B < 1 || H < 1 || N < 1 || !valid_scale(scale)) return PLX_ERR_INVALID_ARG;
        if (out_dtype != PLX_BF16 && out_dtype != PLX_F32) return PLX_ERR_INVALID_ARG;
        if (d != 128 && d != 64) return PLX_ERR_UNSUPPORTED;
        const void* ptrs16[] = {q, k, v, dout, out, dq, dk, dv, workspace};
        for (const void* ptr : ptrs16)
            if (ptr && !aligned(ptr, 16)) return PLX_ERR_MISALIGNED;
        if (rho && (!aligned(rho, 16) || !aligned(drho, 16) || !aligned(vbar, 16) || !aligned(c, 4)))
            return PLX_ERR_MISALIGNED;
        if (!aligned(lse, 4)) return PLX_ERR_MISALIGNED;
        const size_t need = plx_bwd_bf16_workspace_size(B, H, N, d);
        if (!workspace || workspace_bytes < need) return PLX_ERR_WORKSPACE;
        const DeviceInfo* info = device_info();
        if (!info) return PLX_ERR_CUDA;
        const long long BH = static_cast<long long>(B) * H;
        cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        plx::BwdPrepParams pp{};
        pp.lse = lse;
        pp.c = rho ? c : nullptr;
        pp.vbar = rho ? vbar : nullptr;
        pp.out = out;
        pp.dout = static_cast<const uint16_t*>(dout);
        pp.out_f32 = out_dtype == PLX_F32;
        if (d == 128)
            return rho ? launch_bwd_tc<128, true>(q, k, v, rho, dout, dq, dk, dv, drho, workspace, N, BH, scale, s,
                                                  info->sm_count, &pp)
                       : launch_bwd_tc<128, false>(q, k, v, rho, dout, dq, dk, dv, drho, workspace, N, BH, scale, s,
                                                   info->sm_count, &pp);
        return rho ? launch_bwd_tc<64, true>(q, k, v, rho, dout, dq, dk, dv, drho, workspace, N, BH, scale, s,
                                             info->sm_count, &pp)
                   : launch_bwd_tc<64, false>(q, k, v, rho, dout, dq, dk, dv, drho, workspace, N, BH, scale, s,
                                              info->sm_count, &pp);
    } catch (...) {
        return PLX_ERR_CUDA;
    }
}

int plx_decode_num_splits(int B, int H, int d, int S_cap) {
    try {
        if (B < 1 || H < 1 || S_cap < 1 || (d != 64 && d != 128)) return 0;
        const DeviceInfo* info = device_info();
        if (!info) return 0;
        return decode_splits(*info, static_cast<long long>(B) * H, d, S_cap);
    } catch (...) {
        return 0;
    }
}

size_t plx_decode_workspace_size(int B, int H, int d, int S_cap, int num_splits) {
    if (B < 1 || H < 1 || S_cap < 1 || (d != 64 && d != 128) || num_splits < 0 || num_splits > 1024) return 0;
    const int splits = num_splits > 0 ? num_splits : plx_decode_num_splits(B, H, d, S_cap);
    return decode_ws_bytes(static_cast<long long>(B) * H, d, splits);
}

}  // extern "C"

namespace {

// A paged KV cache: the block table and its sizes (block_table == nullptr: contiguous).
struct PagedCache {
    const int32_t* block_table = nullptr;
    int max_blocks = 0;
    int page = 0;
    int num_blocks = 0;
};

// plx_decode with the family flags (0 = PLX itself), on a contiguous or paged cache.
plx_status decode_impl(const void* q, const void* rho, const void* k_cache, const void* v_cache,
                       const int32_t* seqlens, void* out, float* lse, int B, int H, int d, int S_cap, float scale,
                       int num_splits, void* workspace, size_t workspace_bytes, unsigned flags, plx_dtype out_dtype,
                       void* stream, const PagedCache& paged = PagedCache()) {
    try {
        if (!q || !k_cache || !v_cache || !seqlens || !out) return PLX_ERR_INVALID_ARG;
        if (B < 1 || H < 1 || S_cap < 1 || !valid_scale(scale)) return PLX_ERR_INVALID_ARG;
        if (num_splits < 0 || num_splits > 1024) return PLX_ERR_INVALID_ARG;
        if (out_dtype != PLX_BF16 && out_dtype != PLX_F32) return PLX_ERR_INVALID_ARG;
        if ((flags & ~(PLX_FAMILY_UNIFORM_WEIGHTS | PLX_FAMILY_NO_INTERCEPT)) != 0) return PLX_ERR_INVALID_ARG;
        if ((flags & PLX_FAMILY_NO_INTERCEPT) && !rho) return PLX_ERR_INVALID_ARG;
        if (flags & PLX_FAMILY_UNIFORM_WEIGHTS) scale = 0.f;
        if (d != 64 && d != 128) return PLX_ERR_UNSUPPORTED;
        if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
            (rho && !aligned(rho, 16)) || !aligned(seqlens, 4) || (lse && !aligned(lse, 4)) ||
            (workspace && !aligned(workspace, 16)))
            return PLX_ERR_MISALIGNED;
        const long long BH = static_cast<long long>(B) * H;
        if (BH > INT_MAX) return PLX_ERR_UNSUPPORTED;
        const DeviceInfo* info = device_info();
        if (!info) return PLX_ERR_CUDA;
        const int splits = num_splits > 0 ? num_splits : decode_splits(*info, BH, d, S_cap);
        // a cluster-fused combine keeps the partials on chip: no workspace needed
        const bool fused = decode_fused(*info, BH, splits);
        const size_t need = fused ? 0 : decode_ws_bytes(BH, d, splits);
        if (need > 0 && (!workspace || workspace_bytes < need)) return PLX_ERR_WORKSPACE;
        plx::DecodeParams p;
        p.q = static_cast<const __nv_bfloat16*>(q);
        p.rho = static_cast<const __nv_bfloat16*>(rho);
        p.kc = static_cast<const __nv_bfloat16*>(k_cache);
        p.vc = static_cast<const __nv_bfloat16*>(v_cache);
        p.seqlens = seqlens;
        p.out = out;
        p.lse = lse;
        p.ws = static_cast<float*>(workspace);
        p.H = H;
        p.S_cap = S_cap;
        p.splits = splits;
        p.scale_log2 = scale * kLog2e;
        p.out_f32 = out_dtype == PLX_F32;
        p.no_intercept = (flags & PLX_FAMILY_NO_INTERCEPT) ? 1 : 0;
        p.block_table = paged.block_table;
        p.max_blocks = paged.max_blocks;
        p.page = paged.page;
        p.num_blocks = paged.num_blocks;
        p.key_begin = 0;
        p.partials_only = 0;
        p.groups = 1;
        cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        if (d == 128) {
            if (rho) launch_decode<128, true>(p, BH, s, fused);
            else launch_decode<128, false>(p, BH, s, fused);
        } else {
            if (rho) launch_decode<64, true>(p, BH, s, fused);
            else launch_decode<64, false>(p, BH, s, fused);
        }
        return launch_status();
    } catch (...) {
        return PLX_ERR_CUDA;
    }
}

// plx_decode without a workspace argument.  The split partials live in a
// static device array of PLX_DECODE_NOALLOC_SCRATCH_BYTES per GPU; its device
// address is looked up once per device and handed to plx_decode as the
// workspace, so this path allocates nothing.
}  // namespace

extern "C" {

plx_status plx_decode(const void* q, const void* rho, const void* k_cache, const void* v_cache,
                      const int32_t* seqlens, void* out, float* lse, int B, int H, int d, int S_cap, float scale,
                      int num_splits, void* workspace, size_t workspace_bytes, plx_dtype out_dtype, void* stream) {
    return decode_impl(q, rho, k_cache, v_cache, seqlens, out, lse, B, H, d, S_cap, scale, num_splits, workspace,
                       workspace_bytes, 0u, out_dtype, stream);
}

plx_status plx_decode_family(const void* q, const void* rho, const void* k_cache, const void* v_cache,
                             const int32_t* seqlens, void* out, float* lse, int B, int H, int d, int S_cap,
                             float scale, int num_splits, void* workspace, size_t workspace_bytes, unsigned flags,
                             plx_dtype out_dtype, void* stream) {
    return decode_impl(q, rho, k_cache, v_cache, seqlens, out, lse, B, H, d, S_cap, scale, num_splits, workspace,
                       workspace_bytes, flags, out_dtype, stream);
}

plx_status plx_decode_paged(const void* q, const void* rho, const void* k_pages, const void* v_pages,
                            const int32_t* block_table, const int32_t* seqlens, void* out, float* lse, int B, int H,
                            int d, int page_size, int max_blocks_per_seq, int num_blocks, float scale, int num_splits,
                            void* workspace, size_t workspace_bytes, plx_dtype out_dtype, void* stream) {
    try {
        if (!block_table) return PLX_ERR_INVALID_ARG;
        if (page_size < 32 || page_size % 32 != 0 || max_blocks_per_seq < 1 || num_blocks < 1)
            return PLX_ERR_INVALID_ARG;
        if (!aligned(block_table, 4)) return PLX_ERR_MISALIGNED;
        const long long S_cap = static_cast<long long>(max_blocks_per_seq) * page_size;
        if (S_cap > INT_MAX) return PLX_ERR_UNSUPPORTED;
        PagedCache pc;
        pc.block_table = block_table;
        pc.max_blocks = max_blocks_per_seq;
        pc.page = page_size;
        pc.num_blocks = num_blocks;
        return decode_impl(q, rho, k_pages, v_pages, seqlens, out, lse, B, H, d, static_cast<int>(S_cap), scale,
                           num_splits, workspace, workspace_bytes, 0u, out_dtype, stream, pc);
    } catch (...) {
        return PLX_ERR_CUDA;
    }
}

plx_status plx_decode_noalloc(const void* q, const void* rho, const void* k_cache, const void* v_cache,
                              const int32_t* seqlens, void* out, float* lse, int B, int H, int d, int S_cap,
                              float scale, int num_splits, plx_dtype out_dtype, void* stream) {
    try {
        if (B < 1 || H < 1 || S_cap < 1 || num_splits < 0 || num_splits > 1024) return PLX_ERR_INVALID_ARG;
        if (d != 64 && d != 128) return PLX_ERR_UNSUPPORTED;
        const long long BH = static_cast<long long>(B) * H;
        if (BH > INT_MAX) return PLX_ERR_UNSUPPORTED;
        const size_t per_split = static_cast<size_t>(BH) * (2 * d + 4) * sizeof(float);   // one split's partials
        int splits = num_splits;
        if (splits == 0) {
            const DeviceInfo* info = device_info();
            if (!info) return PLX_ERR_CUDA;
            splits = decode_splits(*info, BH, d, S_cap);
            const size_t fit = kNoallocScratchBytes / per_split;
            if (splits > 1 && static_cast<size_t>(splits) > fit) splits = fit >= 2 ? static_cast<int>(fit) : 1;
        } else if (decode_ws_bytes(BH, d, splits) > kNoallocScratchBytes) {
            return PLX_ERR_UNSUPPORTED;
        }
        float* scratch = noalloc_scratch();
        if (!scratch) return PLX_ERR_CUDA;
        return plx_decode(q, rho, k_cache, v_cache, seqlens, out, lse, B, H, d, S_cap, scale, splits, scratch,
                          kNoallocScratchBytes, out_dtype, stream);
    } catch (...) {
        return PLX_ERR_CUDA;
    }
}

size_t plx_decode_partials_size(int B, int H, int d, int num_splits) {
    if (B < 1 || H < 1 || (d != 64 && d != 128) || num_splits < 1 || num_splits > 1024) return 0;
    return static_cast<size_t>(B) * H * num_splits * (2 * d + 4) * sizeof(float);
}

plx_status plx_decode_partials(const void* q, const void* rho, const void* k_shard, const void* v_shard,
                               const int32_t* seqlens, int key_begin, void* partials, size_t partials_bytes, int B,
                               int H, int d, int S_shard, float scale, int num_splits, void* stream) {
    try {
        if (!q || !k_shard || !v_shard || !seqlens || !partials) return PLX_ERR_INVALID_ARG;
        if (B < 1 || H < 1 || S_shard < 1 || key_begin < 0 || !valid_scale(scale)) return PLX_ERR_INVALID_ARG;
        if (num_splits < 1 || num_splits > 1024) return PLX_ERR_INVALID_ARG;
        if (d != 64 && d != 128) return PLX_ERR_UNSUPPORTED;
        if (!aligned(q, 16) || !aligned(k_shard, 16) || !aligned(v_shard, 16) || (rho && !aligned(rho, 16)) ||
            !aligned(seqlens, 4) || !aligned(partials, 16))
            return PLX_ERR_MISALIGNED;
        const long long BH = static_cast<long long>(B) * H;
        if (BH > INT_MAX) return PLX_ERR_UNSUPPORTED;
        if (partials_bytes < plx_decode_partials_size(B, H, d, num_splits)) return PLX_ERR_WORKSPACE;
        const DeviceInfo* info = device_info();
        if (!info) return PLX_ERR_CUDA;
        plx::DecodeParams p;
        p.q = static_cast<const __nv_bfloat16*>(q);
        p.rho = static_cast<const __nv_bfloat16*>(rho);
        p.kc = static_cast<const __nv_bfloat16*>(k_shard);
        p.vc = static_cast<const __nv_bfloat16*>(v_shard);
        p.seqlens = seqlens;
        p.out = nullptr;
        p.lse = nullptr;
        p.ws = static_cast<float*>(partials);
        p.H = H;
        p.S_cap = S_shard;
        p.splits = num_splits;
        p.scale_log2 = scale * kLog2e;
        p.out_f32 = 1;
        p.no_intercept = 0;
        p.block_table = nullptr;
        p.max_blocks = 0;
        p.page = 0;
        p.num_blocks = 0;
        p.key_begin = key_begin;
        p.partials_only = 1;
        p.groups = 1;
        cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        if (d == 128) {
            if (rho) launch_decode_split<128, true>(p, BH, s);
            else launch_decode_split<128, false>(p, BH, s);
        } else {
            if (rho) launch_decode_split<64, true>(p, BH, s);
            else launch_decode_split<64, false>(p, BH, s);
        }
        return launch_status();
    } catch (...) {
        return PLX_ERR_CUDA;
    }
}

plx_status plx_decode_combine(const void* partials, int groups, int num_splits, void* out, float* lse, int B, int H,
                              int d, int with_rho, unsigned flags, plx_dtype out_dtype, void* stream) {
    try {
        if (!partials || !out) return PLX_ERR_INVALID_ARG;
        if (B < 1 || H < 1 || groups < 1 || num_splits < 1 || num_splits > 1024) return PLX_ERR_INVALID_ARG;
        if (out_dtype != PLX_BF16 && out_dtype != PLX_F32) return PLX_ERR_INVALID_ARG;
        if ((flags & ~static_cast<unsigned>(PLX_FAMILY_NO_INTERCEPT)) != 0) return PLX_ERR_INVALID_ARG;
        if ((flags & PLX_FAMILY_NO_INTERCEPT) && !with_rho) return PLX_ERR_INVALID_ARG;
        if (d != 64 && d != 128) return PLX_ERR_UNSUPPORTED;
        if (!aligned(partials, 16) || !aligned(out, 16) || (lse && !aligned(lse, 4))) return PLX_ERR_MISALIGNED;
        const long long BH = static_cast<long long>(B) * H;
        if (BH > INT_MAX || static_cast<long long>(groups) * num_splits > (1LL << 24)) return PLX_ERR_UNSUPPORTED;
        plx::DecodeParams p;
        p.q = nullptr;
        p.rho = nullptr;
        p.kc = nullptr;
        p.vc = nullptr;
        p.seqlens = nullptr;
        p.out = out;
        p.lse = lse;
        p.ws = static_cast<float*>(const_cast<void*>(partials));
        p.H = H;
        p.S_cap = 0;
        p.splits = num_splits;
        p.scale_log2 = 0.f;
        p.out_f32 = out_dtype == PLX_F32;
        p.no_intercept = (flags & PLX_FAMILY_NO_INTERCEPT) ? 1 : 0;
        p.block_table = nullptr;
        p.max_blocks = 0;
        p.page = 0;
        p.num_blocks = 0;
        p.key_begin = 0;
        p.partials_only = 0;
        p.groups = groups;
        cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        if (d == 128) {
            if (with_rho) launch_decode_combine<128, true>(p, BH, s);
            else launch_decode_combine<128, false>(p, BH, s);
        } else {
            if (with_rho) launch_decode_combine<64, true>(p, BH, s);
            else launch_decode_combine<64, false>(p, BH, s);
        }
        return launch_status();
    } catch (...) {
        return PLX_ERR_CUDA;
    }
}

size_t plx_lla_workspace_size(int B, int H, int N, int d) {
    if (B < 1 || H < 1 || N < 1 || d < 32 || d > 256 || d % 32 != 0) return 0;
    return lla_ws_bytes(static_cast<long long>(B) * H * N, d);
}

size_t plx_lla_kept_weights_workspace_size(int B, int H, int N, int d) {
    const size_t base = plx_lla_workspace_size(B, H, N, d);
    if (base == 0 || (d != 64 && d != 128)) return base;
    return base + lla_wts_bytes(static_cast<long long>(B) * H, N);
}

plx_status plx_lla_f32(const float* q, const float* k, const float* v, float* out, float* rho_out, float* lse,
                       int32_t* steps_out, void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                       float scale, float lambda, int max_iters, float tol, void* stream) {
    try {
        if (!q || !k || !v || !out) return PLX_ERR_INVALID_ARG;
        if (B < 1 || H < 1 || N < 1 || !valid_scale(scale)) return PLX_ERR_INVALID_ARG;
        if (!std::isfinite(lambda) || lambda < 0.f || max_iters < 0 || !std::isfinite(tol) || tol < 0.f)
            return PLX_ERR_INVALID_ARG;
        if (d < 32 || d > 256 || d % 32 != 0) return PLX_ERR_UNSUPPORTED;
        const float* in16[] = {q, k, v, out, rho_out};
        for (const float* ptr : in16)
            if (ptr && !aligned(ptr, 16)) return PLX_ERR_MISALIGNED;
        if ((lse && !aligned(lse, 4)) || (steps_out && !aligned(steps_out, 4)) ||
            (workspace && !aligned(workspace, 256)))
            return PLX_ERR_MISALIGNED;
        const long long BH = static_cast<long long>(B) * H;
        if (BH > 65535) return PLX_ERR_UNSUPPORTED;
        const long long R = BH * N;
        if (!workspace || workspace_bytes < lla_ws_bytes(R, d)) return PLX_ERR_WORKSPACE;
        if (!device_info()) return PLX_ERR_CUDA;          // kernel attributes (shared-memory sizes)
        LlaWorkspace w = lla_ws_carve(workspace, R, d);
        // a workspace with room for the weights keeps them across the CG steps
        if ((d == 64 || d == 128) && workspace_bytes >= lla_ws_bytes(R, d) + lla_wts_bytes(BH, N))
            w.wts = reinterpret_cast<float*>(static_cast<char*>(workspace) + lla_ws_bytes(R, d));
        cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        switch (d / 32) {
            case 1: launch_lla<1>(q, k, v, out, lse, w, N, BH, scale, lambda, max_iters, tol, s); break;
            case 2: launch_lla<2>(q, k, v, out, lse, w, N, BH, scale, lambda, max_iters, tol, s); break;
            case 3: launch_lla<3>(q, k, v, out, lse, w, N, BH, scale, lambda, max_iters, tol, s); break;
            case 4: launch_lla<4>(q, k, v, out, lse, w, N, BH, scale, lambda, max_iters, tol, s); break;
            case 5: launch_lla<5>(q, k, v, out, lse, w, N, BH, scale, lambda, max_iters, tol, s); break;
            case 6: launch_lla<6>(q, k, v, out, lse, w, N, BH, scale, lambda, max_iters, tol, s); break;
            case 7: launch_lla<7>(q, k, v, out, lse, w, N, BH, scale, lambda, max_iters, tol, s); break;
            case 8: launch_lla<8>(q, k, v, out, lse, w, N, BH, scale, lambda, max_iters, tol, s); break;
            default: return PLX_ERR_UNSUPPORTED;
        }
        if (rho_out && cudaMemcpyAsync(rho_out, w.x, static_cast<size_t>(R) * d * sizeof(float),
                                       cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return PLX_ERR_CUDA;
        if (steps_out && cudaMemcpyAsync(steps_out, w.steps, static_cast<size_t>(R) * sizeof(int32_t),
                                         cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return PLX_ERR_CUDA;
        return launch_status();
    } catch (...) {
        return PLX_ERR_CUDA;
    }
}

plx_status plx_probe_proj(const void* x, const void* w_r, void* rho, int B, int N, int H, int d, int Dx,
                          void* stream) {
    try {
        if (!x || !w_r || !rho) return PLX_ERR_INVALID_ARG;
        if (B < 1 || N < 1 || H < 1 || Dx < 1) return PLX_ERR_INVALID_ARG;
        if ((d != 128 && d != 64) || Dx % 8 != 0) return PLX_ERR_UNSUPPORTED;
        if (!aligned(x, 16) || !aligned(w_r, 16) || !aligned(rho, 16)) return PLX_ERR_MISALIGNED;
        const DeviceInfo* info = device_info();
        if (!info) return PLX_ERR_CUDA;
        cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        return d == 128 ? launch_proj_tc<128>(x, w_r, rho, B, N, H, Dx, s, info->sm_count)
                        : launch_proj_tc<64>(x, w_r, rho, B, N, H, Dx, s, info->sm_count);
    } catch (...) {
        return PLX_ERR_CUDA;
    }
}

plx_status plx_selftest_wait(unsigned int limit_us, int arrive, void* stream) {
    try {
        if (limit_us < 1 || limit_us > 1000000) return PLX_ERR_INVALID_ARG;
        plx_wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
            static_cast<unsigned long long>(limit_us) * 1000ull, arrive ? 1 : 0);
        return launch_status();
    } catch (...) {
        return PLX_ERR_CUDA;
    }
}

plx_status plx_last_device_error(void* stream) {
    try {
        if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return PLX_ERR_CUDA;
        unsigned int v = 0, zero = 0;
        if (cudaMemcpyFromSymbol(&v, plx::g_plx_status, sizeof(v)) != cudaSuccess) return PLX_ERR_CUDA;
        if (v && cudaMemcpyToSymbol(plx::g_plx_status, &zero, sizeof(zero)) != cudaSuccess) return PLX_ERR_CUDA;
        if (v & plx::PLX_DEV_ERR_TIMEOUT) return PLX_ERR_TIMEOUT;
        if (v & plx::PLX_DEV_ERR_SEQLEN) return PLX_ERR_INVALID_ARG;
        if (v & plx::PLX_DEV_ERR_BOUNDS) return PLX_ERR_BOUNDS;
        if (v & plx::PLX_DEV_ERR_NONFINITE) return PLX_ERR_RANGE;
        return PLX_OK;
    } catch (...) {
        return PLX_ERR_CUDA;
    }
}

}  // extern "C"
