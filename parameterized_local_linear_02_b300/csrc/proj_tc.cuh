// proj_tc.cuh -- plx_probe_proj: the probe projection rho_i = W_R x_i of
// "Parallax: Parameterized Local Linear Attention for Language Modeling"
// (zhichai.net section 1.3: each token's probe is a learned linear map of its
// hidden state), on the 5th-generation tensor cores.
//
//   x   : bf16 [B][N][Dx]     W_R : bf16 [H d][Dx]     rho : bf16 [B][H][N][d]
//   rho[b, h, n, :] = W_R[h d : (h + 1) d, :] x[b, n, :]    (fp32 accumulation)
//
// A persistent GEMM whose epilogue writes straight into the [B][H][N][d]
// layout the PLX kernels read, so no transpose pass follows it.  A work item
// is (b, 128-token tile, group of 256 output columns = 256 / d heads):
// D = X_tile W_group^T with M = 128, N = 256, K = Dx, both operands K-major,
// 128B-swizzled TMA tiles of 64 K-elements (columns past Dx and rows past N
// or H d are zero-filled by the TMA unit).  Consecutive items share the token
// tile, so the CTAs running at one time read each X tile from L2 several
// times and from HBM once; W_R stays in L2.
//
// Tail split: when the items left for the last wave would fill at most half
// of the CTAs, each of them runs as two half items of 128 columns (W_R
// through a 128-row box), so the last wave takes about two thirds of an item
// time instead of one and no CTA idles for a whole item.
//
// Roles (192 threads, one CTA per SM):
//   warp 0      TMA producer (one lane): X and W tiles through an NSTAGE ring.
//   warp 1      TMEM owner and MMA issuer (whole warp, elected lane).  Two
//               accumulators of 256 columns alternate between items, so the
//               epilogue of one item overlaps the MMAs of the next.
//   warps 2-5   epilogue, one per TMEM lane quadrant: TMEM -> bf16 -> one of
//               two swizzled 2 KB slots -> TMA store (rows past N clipped by
//               the tensor map, heads past H skipped).
#pragma once
#include "status.cuh"

namespace plx {

template <int D>
struct ProjCfg {
    static constexpr int BM = 128;                 // tokens per item
    static constexpr int BN = 256;                 // output columns per item
    static constexpr int HPI = BN / D;             // heads per item
    static constexpr int BK = 64;                  // K elements per stage (one 128-byte row)
    static constexpr int NSTAGE = 4;
    static constexpr int EPI_WARPS = 4;
    static constexpr int THREADS = 64 + EPI_WARPS * 32;
    static constexpr int X_TILE = BM * 128;        // bytes
    static constexpr int W_TILE = BN * 128;
    static constexpr int STAGE_BYTES = X_TILE + W_TILE;
    static constexpr int STG_SLOT = 32 * 64;       // 32 rows x 32 bf16 (64-byte rows)
    static constexpr int OFF_STAGE = 0;
    static constexpr int OFF_STG = NSTAGE * STAGE_BYTES;
    static constexpr int OFF_BAR = OFF_STG + EPI_WARPS * 2 * STG_SLOT;
    // full[NSTAGE], empty[NSTAGE], acc_full[2], acc_empty[2], drain
    static constexpr int NBARS = 2 * NSTAGE + 5;
    static constexpr int SMEM = OFF_BAR + NBARS * 8 + 16 + 1024;
    static constexpr uint32_t TM_COLS = 2 * BN;    // two accumulators
    static_assert(D == 64 || D == 128, "probe projection supports d in {64, 128}");
    static_assert(STAGE_BYTES % 1024 == 0 && OFF_STG % 1024 == 0, "1024-byte tiles");
    static_assert(SMEM <= 232448, "shared memory budget");
};

struct ProjParams {
    int N, H, n_kb, n_mt, n_hg;
    int n_full;      // items 0 .. n_full - 1 are whole (256 columns)
    int n_items;     // n_full + 2 x (split items): item n_full + 2 s + h is half h of item n_full + s
};

template <int D>
__global__ void __launch_bounds__(ProjCfg<D>::THREADS, 1)
plx_proj_tc_kernel(const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapW,
                   const __grid_constant__ CUtensorMap mapW2, const __grid_constant__ CUtensorMap mapO,
                   const ProjParams p) {
    using Cfg = ProjCfg<D>;
    constexpr int BM = Cfg::BM, BN = Cfg::BN, NSTAGE = Cfg::NSTAGE;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    uint64_t* empty = full + NSTAGE;
    uint64_t* acc_full = empty + NSTAGE;     // per accumulator: the item's MMAs have completed
    uint64_t* acc_empty = acc_full + 2;      // per accumulator: the epilogue has read it
    uint64_t* drain = acc_empty + 2;         // every MMA this CTA issued has completed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, c = blockIdx.x;

    if (warp == 1) {
        tmem_alloc(tmem_slot, Cfg::TM_COLS);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], Cfg::EPI_WARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&mapX);
        tma_prefetch_desc(&mapW);
        tma_prefetch_desc(&mapW2);
        tma_prefetch_desc(&mapO);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto fail = [&]() {
        atomicOr(&g_plx_status, PLX_DEV_ERR_TIMEOUT);
        *abort_flag = 1;
    };
    // item u -> column group hg (fastest), token tile mt, batch b, and which
    // columns of the group: half = -1 for all 256, else 128 * half .. + 127
    auto item = [&](int u, int& b, int& mt, int& hg, int& half) {
        half = -1;
        if (u >= p.n_full) {
            half = (u - p.n_full) & 1;
            u = p.n_full + ((u - p.n_full) >> 1);
        }
        hg = u % p.n_hg;
        const int bm = u / p.n_hg;
        mt = bm % p.n_mt;
        b = bm / p.n_mt;
    };
    auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity));
    };

    if (warp == 0) {
        // ===================================================== TMA producer
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int u = c; u < p.n_items && ok; u += G) {
                if (*abort_flag) break;
                int b, mt, hg, half;
                item(u, b, mt, hg, half);
                const uint32_t bytes = half < 0 ? Cfg::STAGE_BYTES : Cfg::X_TILE + Cfg::W_TILE / 2;
                for (int kb = 0; kb < p.n_kb; ++kb, ++it) {
                    const int s = it % NSTAGE;
                    if (it >= NSTAGE && !mbar_wait(&empty[s], ((it / NSTAGE) - 1) & 1)) { ok = false; break; }
                    uint8_t* st = smem + Cfg::OFF_STAGE + s * Cfg::STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[s], bytes);
                    tma_load_3d(st, &mapX, &full[s], kb * Cfg::BK, mt * BM, b);
                    if (half < 0)
                        tma_load_3d(st + Cfg::X_TILE, &mapW, &full[s], kb * Cfg::BK, hg * BN, 0);
                    else
                        tma_load_3d(st + Cfg::X_TILE, &mapW2, &full[s], kb * Cfg::BK, hg * BN + half * (BN / 2), 0);
                }
            }
            if (!ok) fail();
            // no copy may still be in flight when the CTA exits
            for (int i = max(0, it - NSTAGE); i < it; ++i)
                if (!mbar_wait(&full[i % NSTAGE], (i / NSTAGE) & 1)) fail();
        }
    } else if (warp == 1) {
        // ===================================================== MMA issuer (whole warp)
        constexpr uint32_t ID_FULL = idesc_bf16_f32(BM, BN, false, false);
        constexpr uint32_t ID_HALF = idesc_bf16_f32(BM, BN / 2, false, false);
        const uint32_t sBase = smem_u32(smem + Cfg::OFF_STAGE);
        int it = 0, n = 0;
        bool ok = true;
        for (int u = c; u < p.n_items && ok; u += G, ++n) {
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            const uint32_t ID = u < p.n_full ? ID_FULL : ID_HALF;
            const int ab = n & 1;
            // the epilogue has read this accumulator's previous item (item n - 2)
            if (n >= 2 && !wait_warp(&acc_empty[ab], ((n >> 1) - 1) & 1)) { ok = false; break; }
            tc_fence_after();
            const uint32_t acc = tmem + ab * BN;
            for (int kb = 0; kb < p.n_kb; ++kb, ++it) {
                const int s = it % NSTAGE;
                if (!wait_warp(&full[s], (it / NSTAGE) & 1)) { ok = false; break; }
                tc_fence_after();
                const uint32_t xa = sBase + s * Cfg::STAGE_BYTES, wa = xa + Cfg::X_TILE;
#pragma unroll
                for (int kk = 0; kk < Cfg::BK / 16; ++kk)
                    mma_ss_warp(acc, sdesc_sw128(xa + kk * 32, 16, 1024), sdesc_sw128(wa + kk * 32, 16, 1024), ID,
                                (kb > 0 || kk > 0) ? 1u : 0u);
                mma_commit_warp(&empty[s]);
            }
            if (ok) mma_commit_warp(&acc_full[ab]);
        }
        if (!ok) fail();
        // TMEM is freed only after every MMA issued here has completed
        mma_commit_warp(drain);
        if (!wait_warp(drain, 0)) fail();
    } else {
        // ===================================================== epilogue (warps 2..5)
        const int quad = warp & 3;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        uint8_t* stg = smem + Cfg::OFF_STG + (warp - 2) * 2 * Cfg::STG_SLOT;
        const int swz = (lane >> 1) & 3;
        int n = 0, issued = 0;
        bool ok = true;
        for (int u = c; u < p.n_items; u += G, ++n) {
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            int b, mt, hg, half;
            item(u, b, mt, hg, half);
            const int ab = n & 1;
            if (!wait_warp(&acc_full[ab], (n >> 1) & 1)) { ok = false; break; }
            tc_fence_after();
            const int y = mt * BM + quad * 32;
            const int col0 = half < 0 ? 0 : half * (BN / 2);     // first group column of this item
            const int ncol = half < 0 ? BN : BN / 2;
            if (y < p.N) {
#pragma unroll 1
                for (int cb = 0; cb < ncol; cb += 32) {
                    const int head = hg * Cfg::HPI + (col0 + cb) / D;
                    if (head >= p.H) break;
                    uint32_t v[32];
                    tmem_ld32x32b_x32(lane_addr + ab * BN + cb, v);
                    // 32 columns as bf16 = one 64-byte row per thread, in the output
                    // map's 64-byte swizzle (16-byte unit q of row r at q ^ ((r >> 1) & 3));
                    // two slots alternate, so a slot is free once at most one store is pending
                    uint8_t* slot = stg + (issued & 1) * Cfg::STG_SLOT;
                    if (lane == 0) bulk_wait_read<1>();
                    __syncwarp();
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        *reinterpret_cast<uint4*>(slot + lane * 64 + ((q4 ^ swz) << 4)) = make_uint4(
                            pack_bf16x2(__uint_as_float(v[8 * q4]), __uint_as_float(v[8 * q4 + 1])),
                            pack_bf16x2(__uint_as_float(v[8 * q4 + 2]), __uint_as_float(v[8 * q4 + 3])),
                            pack_bf16x2(__uint_as_float(v[8 * q4 + 4]), __uint_as_float(v[8 * q4 + 5])),
                            pack_bf16x2(__uint_as_float(v[8 * q4 + 6]), __uint_as_float(v[8 * q4 + 7])));
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&mapO, slot, (col0 + cb) % D, y, b * p.H + head);
                        bulk_commit_group();
                    }
                    ++issued;
                }
            }
            // the accumulator is read out: the item two ahead may start on it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[ab]);
        }
        if (!ok) fail();
        if (lane == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::TM_COLS);
    }
}

}  // namespace plx
