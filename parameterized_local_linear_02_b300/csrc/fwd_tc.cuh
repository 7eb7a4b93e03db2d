// fwd_tc.cuh -- plx_fwd: causal PLX prefill forward on the 5th-generation
// tensor cores (tcgen05, TMEM accumulators, TMA-fed 128B-swizzled tiles).
//
// Streaming algorithm of "Parallax: Parameterized Local Linear Attention for
// Language Modeling" (gist.science, "Algoritmo Consapevole
// dell'Hardware": about twice the FlashAttention compute on the same K/V
// stream).  For a 128-row query tile and each 64-key K/V tile j:
//   S = Q K_j^T, R = rho K_j^T                  (tensor cores -> TMEM)
//   online softmax of scale*S: m, l, P = 2^(scale*log2e*S - m)
//   PR = P o R,  C += rowsum(PR)
//   O += P V_j,  U += PR V_j                     (A operand from TMEM)
// P, PR and V_j enter the second pair of GEMMs as fp16 (V_j is re-encoded
// from bf16 in shared memory by the softmax warps); l and C are summed from
// the same rounded values.  With bf16 there the rounding of P and PR alone
// gives errors of a few percent of the output RMS, because the correction
// (1 + c) vbar - u cancels; fp16 keeps them near 5e-3.
// and finally vbar = O/l, u = U/l, c = C/l, o = (1 + c) vbar - u, which is
// o^SA - Sigma_KV rho by the identity
//   Sigma_KV rho = sum_j w_j (k_j.rho) v_j - vbar (kbar.rho)
// (zhichai.net section 1.3; gist.science "Meccanismo Principale").
//
// Roles (192 threads, one CTA per SM, persistent over work items):
//   warp 0     TMA producer: Q and rho once per item, K/V through an
//              NSTAGE ring.
//   warp 1     TMEM owner and MMA issuer (one thread).  Issue order per item
//              SR_0, SR_1, PV_0, SR_2, PV_1, ... so the tensor pipe computes
//              S/R of tile j+1 while the softmax works on tile j.
//   warps 2-5  softmax + epilogue, thread r owns query row r of the tile
//              (TMEM lane quadrant = warp % 4).
// TMEM (512 columns): S0 | R0 | S1 | R1 (64 each) | O (D) | U (D).  P and PR
// are written back as bf16 over the first 32 columns of their S/R buffer.
// The running max is refreshed lazily: O, U, l, C are rescaled only when a
// row max grows by more than 2^4, so P <= 16 and P o R stays inside the fp16
// range for |rho.k| < 4094.  A non-finite output sets PLX_DEV_ERR_NONFINITE.
// Work items (b*h, query tile) run longest-first in a snake order over CTAs.
#pragma once
#include "status.cuh"

namespace plx {

template <int D, bool PLX>
struct FwdTcCfg {
    static constexpr int BM = 128;                 // query rows per item
    static constexpr int BN = 64;                  // keys per K/V tile
    static constexpr int NP = D / 64;              // 64-column panels (128 B rows)
    static constexpr int NSTAGE = (D == 128) ? 4 : 6;
    static constexpr int THREADS = 192;
    static constexpr int Q_PANEL = BM * 128;       // bytes per Q/rho panel
    static constexpr int KV_PANEL = BN * 128;      // bytes per K/V panel
    static constexpr int Q_BYTES = NP * Q_PANEL;
    static constexpr int KV_BYTES = NP * KV_PANEL;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_R = OFF_Q + Q_BYTES;
    static constexpr int OFF_K = OFF_R + (PLX ? Q_BYTES : 0);
    static constexpr int OFF_V = OFF_K + NSTAGE * KV_BYTES;
    static constexpr int OFF_BAR = OFF_V + NSTAGE * KV_BYTES;
    // barriers: q_full, q_empty, kv_full[NSTAGE], kv_empty[NSTAGE], s_full[2], p_full[2], pv_done[2], drain
    static constexpr int NBARS = 2 + 2 * NSTAGE + 2 + 2 + 2 + 1;
    static constexpr int SMEM_USED = OFF_BAR + NBARS * 8 + 16;
    static constexpr int SMEM = SMEM_USED + 1024;  // slack for 1024-byte alignment
    // TMEM columns
    static constexpr uint32_t TM_S0 = 0, TM_R0 = 64, TM_S1 = 128, TM_R1 = 192, TM_O = 256, TM_U = 256 + D;
    static constexpr uint32_t TM_COLS = 512;
    static constexpr float RESCALE_THRESH = 4.0f;  // log2 units: P <= 16
    static_assert(D == 64 || D == 128, "tcgen05 forward supports d in {64, 128}");
    static_assert(SMEM <= 232448, "shared memory budget");
};

struct FwdTcParams {
    void* out;
    float* lse;
    int N;
    int BH;
    int n_qt;
    int n_items;
    float scale_log2;
    int out_f32;
};

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// item u of the longest-first order: query tile qt (descending), head bh
__device__ __forceinline__ void item_coords(int u, int BH, int n_qt, int& bh, int& qt) {
    qt = n_qt - 1 - u / BH;
    bh = u % BH;
}
// u for round r of CTA c in a snake over the grid
__device__ __forceinline__ int snake_item(int r, int c, int G) {
    return r * G + ((r & 1) ? (G - 1 - c) : c);
}

template <int D, bool PLX>
__global__ void __launch_bounds__(192, 1)
plx_fwd_tc_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapR,
                  const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                  const FwdTcParams p) {
    using Cfg = FwdTcCfg<D, PLX>;
    constexpr int BM = Cfg::BM, BN = Cfg::BN, NP = Cfg::NP, NSTAGE = Cfg::NSTAGE;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + Cfg::OFF_Q;
    uint8_t* sR = smem + Cfg::OFF_R;
    uint8_t* sK = smem + Cfg::OFF_K;
    uint8_t* sV = smem + Cfg::OFF_V;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    uint64_t* q_full = bars;
    uint64_t* q_empty = bars + 1;
    uint64_t* kv_full = bars + 2;
    uint64_t* kv_empty = kv_full + NSTAGE;
    uint64_t* s_full = kv_empty + NSTAGE;
    uint64_t* p_full = s_full + 2;
    uint64_t* pv_done = p_full + 2;      // one per S/R buffer: PV of tiles g with g % 2 == b
    uint64_t* drain = pv_done + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, c = blockIdx.x;

    if (warp == 1) {
        tmem_alloc(tmem_slot, Cfg::TM_COLS);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&p_full[b], 128);
            mbar_init(&pv_done[b], 1);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&mapQ);
        tma_prefetch_desc(&mapK);
        tma_prefetch_desc(&mapV);
        if (PLX) tma_prefetch_desc(&mapR);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto fail = [&]() {
        atomicOr(&g_plx_status, PLX_DEV_ERR_TIMEOUT);
        *abort_flag = 1;
    };

    if (warp == 0) {
        // ===================================================== TMA producer
        if (lane == 0) {
            int items = 0, kv_it = 0;
            for (int r = 0;; ++r) {
                const int u = snake_item(r, c, G);
                if (u >= p.n_items || *abort_flag) break;
                int bh, qt;
                item_coords(u, p.BH, p.n_qt, bh, qt);
                const int q0 = qt * BM;
                const int n_kv = (min(p.N, q0 + BM) + BN - 1) / BN;
                if (items > 0 && !mbar_wait(q_empty, (items - 1) & 1)) { fail(); break; }
                mbar_arrive_expect_tx(q_full, (PLX ? 2 : 1) * Cfg::Q_BYTES);
                for (int pn = 0; pn < NP; ++pn) {
                    tma_load_3d(sQ + pn * Cfg::Q_PANEL, &mapQ, q_full, pn * 64, q0, bh);
                    if (PLX) tma_load_3d(sR + pn * Cfg::Q_PANEL, &mapR, q_full, pn * 64, q0, bh);
                }
                for (int j = 0; j < n_kv; ++j, ++kv_it) {
                    const int s = kv_it % NSTAGE;
                    if (kv_it >= NSTAGE && !mbar_wait(&kv_empty[s], ((kv_it / NSTAGE) - 1) & 1)) {
                        fail();
                        break;
                    }
                    mbar_arrive_expect_tx(&kv_full[s], 2 * Cfg::KV_BYTES);
                    for (int pn = 0; pn < NP; ++pn) {
                        tma_load_3d(sK + s * Cfg::KV_BYTES + pn * Cfg::KV_PANEL, &mapK, &kv_full[s], pn * 64,
                                    j * BN, bh);
                        tma_load_3d(sV + s * Cfg::KV_BYTES + pn * Cfg::KV_PANEL, &mapV, &kv_full[s], pn * 64,
                                    j * BN, bh);
                    }
                }
                ++items;
                if (*abort_flag) break;
            }
            // never leave with loads in flight into this CTA's shared memory
            for (int i = max(0, kv_it - NSTAGE); i < kv_it; ++i)
                if (!mbar_wait(&kv_full[i % NSTAGE], (i / NSTAGE) & 1)) fail();
            if (items > 0 && !mbar_wait(q_full, (items - 1) & 1)) fail();
        }
    } else if (warp == 1) {
        // ===================================================== MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_S = idesc_bf16_f32(128, BN, false, false);
            constexpr uint32_t ID_PV = idesc_f16_f32(128, D, false, true);
            const uint32_t sQa = smem_u32(sQ), sRa = smem_u32(sR), sKa = smem_u32(sK), sVa = smem_u32(sV);
            int items = 0, kv_it = 0, g_sr = 0, g_pv = 0;
            bool ok = true;
            int pv_stage = 0;
            auto issue_pv = [&](int jj, int stage) -> bool {
                const int b = g_pv & 1;
                if (!mbar_wait(&p_full[b], (g_pv >> 1) & 1)) return false;
                tc_fence_after();
                const uint32_t tS = tmem + (b ? Cfg::TM_S1 : Cfg::TM_S0);
                const uint32_t tR = tmem + (b ? Cfg::TM_R1 : Cfg::TM_R0);
                const uint32_t vbase = sVa + stage * Cfg::KV_BYTES;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint64_t bdesc = sdesc_sw128(vbase + kk * 16 * 128, Cfg::KV_PANEL, 1024);
                    const uint32_t acc = (jj > 0 || kk > 0) ? 1u : 0u;
                    mma_ts(tmem + Cfg::TM_O, tS + kk * 8, bdesc, ID_PV, acc);
                    if (PLX) mma_ts(tmem + Cfg::TM_U, tR + kk * 8, bdesc, ID_PV, acc);
                }
                mma_commit(&kv_empty[stage]);
                mma_commit(&pv_done[b]);
                ++g_pv;
                return true;
            };
            for (int r = 0; ok; ++r) {
                const int u = snake_item(r, c, G);
                if (u >= p.n_items || *abort_flag) break;
                int bh, qt;
                item_coords(u, p.BH, p.n_qt, bh, qt);
                const int q0 = qt * BM;
                const int n_kv = (min(p.N, q0 + BM) + BN - 1) / BN;
                if (!mbar_wait(q_full, items & 1)) { fail(); break; }
                tc_fence_after();
                for (int j = 0; j < n_kv; ++j, ++kv_it, ++g_sr) {
                    const int s = kv_it % NSTAGE;
                    if (!mbar_wait(&kv_full[s], (kv_it / NSTAGE) & 1)) { ok = false; break; }
                    tc_fence_after();
                    const int b = g_sr & 1;
                    const uint32_t tS = tmem + (b ? Cfg::TM_S1 : Cfg::TM_S0);
                    const uint32_t tR = tmem + (b ? Cfg::TM_R1 : Cfg::TM_R0);
                    const uint32_t kbase = sKa + s * Cfg::KV_BYTES;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * Cfg::Q_PANEL + (kk & 3) * 32;
                        const uint32_t koff = (kk >> 2) * Cfg::KV_PANEL + (kk & 3) * 32;
                        const uint64_t bdesc = sdesc_sw128(kbase + koff, 16, 1024);
                        mma_ss(tS, sdesc_sw128(sQa + off, 16, 1024), bdesc, ID_S, kk > 0);
                        if (PLX) mma_ss(tR, sdesc_sw128(sRa + off, 16, 1024), bdesc, ID_S, kk > 0);
                    }
                    mma_commit(&s_full[b]);
                    if (j == n_kv - 1) mma_commit(q_empty);
                    if (j >= 1 && !issue_pv(j - 1, pv_stage)) { ok = false; break; }
                    pv_stage = s;
                }
                if (!ok) { fail(); break; }
                if (!issue_pv(n_kv - 1, pv_stage)) { fail(); break; }
                ++items;
            }
            // drain: every MMA issued by this thread has finished before TMEM is freed
            mma_commit(drain);
            if (!mbar_wait(drain, 0)) fail();
        }
    } else {
        // ===================================================== softmax + epilogue (warps 2..5)
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        int g_sr = 0;
        // all waits and exits are warp-uniform: the tcgen05 loads/stores below are .sync.aligned
        auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity));
        };
        for (int r = 0;; ++r) {
            const int u = snake_item(r, c, G);
            if (u >= p.n_items || __shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            int bh, qt;
            item_coords(u, p.BH, p.n_qt, bh, qt);
            const int q0 = qt * BM;
            const int i = q0 + row;                 // this thread's query row
            const int n_kv = (min(p.N, q0 + BM) + BN - 1) / BN;
            float m = -INFINITY, l = 0.f, C = 0.f;
            bool ok = true;
            for (int j = 0; j < n_kv; ++j, ++g_sr) {
                const int b = g_sr & 1;
                if (!wait_warp(&s_full[b], (g_sr >> 1) & 1)) { ok = false; break; }
                tc_fence_after();
                const uint32_t tS = lane_addr + (b ? Cfg::TM_S1 : Cfg::TM_S0);
                const uint32_t tR = lane_addr + (b ? Cfg::TM_R1 : Cfg::TM_R0);
                uint32_t sraw[64];
                tmem_ld32x32b_x64(tS, sraw);
                float sc[64];
#pragma unroll
                for (int cc = 0; cc < 64; ++cc) sc[cc] = __uint_as_float(sraw[cc]);
                // causal mask on tiles that reach past the first row of the item
                const bool diag = (j + 1) * BN - 1 > q0;
                const int kbase = j * BN;
                if (diag) {
#pragma unroll
                    for (int cc = 0; cc < 64; ++cc)
                        if (kbase + cc > i) sc[cc] = -INFINITY;
                }
                float mt = sc[0];
#pragma unroll
                for (int cc = 1; cc < 64; ++cc) mt = fmaxf(mt, sc[cc]);
                // scaled row max of this tile, log2 units (-inf when every key is masked)
                const float mt2 = mt == -INFINITY ? -INFINITY : mt * p.scale_log2;
                float alpha = 1.f;
                bool rescale_warp = false;
                if (j == 0) {
                    m = mt2;
                } else {
                    const bool need = mt2 > m + Cfg::RESCALE_THRESH;
                    rescale_warp = __any_sync(0xffffffffu, need);
                    if (rescale_warp) {
                        const float m_new = fmaxf(m, mt2);
                        alpha = fast_exp2(m - m_new);
                        m = m_new;
                        l *= alpha;
                        C *= alpha;
                    }
                }
                // P and PR go to the tensor cores as fp16; l and C are summed from
                // the same rounded values, so o = (1 + C/l) O/l - U/l is exactly
                // PLX for the rounded weights (they sum to one) and the rounding
                // errors cancel the way the exact terms do.
                const float neg_m = -m;
                uint32_t pk[32];
                float lsum = 0.f;
                float pe[64];
#pragma unroll
                for (int cc = 0; cc < 64; ++cc) {
                    pe[cc] = fast_exp2(fmaf(sc[cc], p.scale_log2, neg_m));
                    if (diag && kbase + cc > i) pe[cc] = 0.f;     // also covers scale == 0
                }
#pragma unroll
                for (int cc = 0; cc < 32; ++cc) {
                    pk[cc] = pack_f16x2(pe[2 * cc], pe[2 * cc + 1]);
                    float lo, hi;
                    unpack_f16x2(pk[cc], lo, hi);
                    lsum += lo + hi;
                }
                l += lsum;
                tmem_st32x32b_x32(tS, pk);
                if constexpr (PLX) {
                    uint32_t rraw[64];
                    tmem_ld32x32b_x64(tR, rraw);
                    float csum = 0.f;
#pragma unroll
                    for (int cc = 0; cc < 32; ++cc) {
                        const float a0 = pe[2 * cc] * __uint_as_float(rraw[2 * cc]);
                        const float a1 = pe[2 * cc + 1] * __uint_as_float(rraw[2 * cc + 1]);
                        pk[cc] = pack_f16x2(a0, a1);
                        float lo, hi;
                        unpack_f16x2(pk[cc], lo, hi);
                        csum += lo + hi;
                    }
                    C += csum;
                    tmem_st32x32b_x32(tR, pk);
                }
                {
                    // re-encode this tile's V (bf16 -> fp16) in place for the PV GEMMs;
                    // element-wise, so the 128-byte swizzle is unchanged.  The wait on
                    // the stage's load barrier (already complete: the S/R MMA of this
                    // tile waited on it) orders the TMA writes before these reads.
                    const int stage = g_sr % NSTAGE;
                    if (!wait_warp(&kv_full[stage], (g_sr / NSTAGE) & 1)) { ok = false; break; }
                    uint4* vt = reinterpret_cast<uint4*>(sV + stage * Cfg::KV_BYTES);
#pragma unroll
                    for (int k = 0; k < Cfg::KV_BYTES / 16 / 128; ++k) {
                        uint4 w = vt[row + 128 * k];
                        w.x = bf16x2_to_f16x2(w.x);
                        w.y = bf16x2_to_f16x2(w.y);
                        w.z = bf16x2_to_f16x2(w.z);
                        w.w = bf16x2_to_f16x2(w.w);
                        vt[row + 128 * k] = w;
                    }
                    fence_proxy_async_smem();
                }
                if (rescale_warp) {
                    // O and U must hold the previous tile's PV before they are
                    // rescaled.  Only that PV can still be in flight: the S/R MMA
                    // of this tile completed after the PV two tiles back, and the
                    // next PV needs this tile's P.  So the wait on the previous
                    // tile's buffer barrier is unambiguous, and no other tile waits.
                    const int gp = g_sr - 1;
                    if (!wait_warp(&pv_done[gp & 1], (gp >> 1) & 1)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll 1
                    for (int cb = 0; cb < (PLX ? 2 * D : D); cb += 32) {
                        uint32_t o32[32];
                        tmem_ld32x32b_x32(lane_addr + Cfg::TM_O + cb, o32);
#pragma unroll
                        for (int cc = 0; cc < 32; ++cc)
                            o32[cc] = __float_as_uint(__uint_as_float(o32[cc]) * alpha);
                        tmem_st32x32b_x32(lane_addr + Cfg::TM_O + cb, o32);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&p_full[b]);
            }
            if (!ok) { fail(); break; }
            // ---- epilogue: wait for the last PV (by the same argument the one
            // before it on this buffer's barrier is complete), then
            // o = (1 + c) vbar - u
            {
                const int gl = g_sr - 1;
                if (!wait_warp(&pv_done[gl & 1], (gl >> 1) & 1)) { fail(); break; }
            }
            tc_fence_after();
            const float inv_l = 1.f / l;
            const float cc_ = C * inv_l;
            const bool store = i < p.N;
            bool nonfinite_ok = true;
            const size_t orow = (static_cast<size_t>(bh) * p.N + (store ? i : 0)) * D;
#pragma unroll 1
            for (int cb = 0; cb < D; cb += 32) {
                uint32_t o32[32];
                tmem_ld32x32b_x32(lane_addr + Cfg::TM_O + cb, o32);
                float o[32];
                if constexpr (PLX) {
                    uint32_t u32[32];
                    tmem_ld32x32b_x32(lane_addr + Cfg::TM_U + cb, u32);
#pragma unroll
                    for (int cc = 0; cc < 32; ++cc) {
                        const float vbar = __uint_as_float(o32[cc]) * inv_l;
                        o[cc] = fmaf(cc_, vbar, vbar) - __uint_as_float(u32[cc]) * inv_l;
                    }
                } else {
#pragma unroll
                    for (int cc = 0; cc < 32; ++cc) o[cc] = __uint_as_float(o32[cc]) * inv_l;
                }
#pragma unroll
                for (int cc = 0; cc < 32; ++cc) nonfinite_ok &= isfinite(o[cc]);
                if (store) {
                    if (p.out_f32) {
                        float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + orow + cb);
#pragma unroll
                        for (int v4 = 0; v4 < 8; ++v4)
                            dst[v4] = make_float4(o[4 * v4], o[4 * v4 + 1], o[4 * v4 + 2], o[4 * v4 + 3]);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + orow + cb);
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4)
                            dst[v4] = make_uint4(pack_bf16x2(o[8 * v4], o[8 * v4 + 1]),
                                                 pack_bf16x2(o[8 * v4 + 2], o[8 * v4 + 3]),
                                                 pack_bf16x2(o[8 * v4 + 4], o[8 * v4 + 5]),
                                                 pack_bf16x2(o[8 * v4 + 6], o[8 * v4 + 7]));
                    }
                }
            }
            if (store && p.lse) p.lse[static_cast<size_t>(bh) * p.N + i] = (m + __log2f(l)) * 0.69314718055994531f;
            if (__any_sync(0xffffffffu, store && !nonfinite_ok) && lane == 0)
                atomicOr(&g_plx_status, PLX_DEV_ERR_NONFINITE);
            tc_fence_before();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::TM_COLS);
    }
}

}  // namespace plx
