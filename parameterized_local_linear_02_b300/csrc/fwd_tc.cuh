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
// Roles (384 threads, one CTA per SM, persistent over work items):
//   warp 0       TMA producer (one lane): Q and rho once per item (with an L2
//                prefetch of the next item's tile a few K/V tiles ahead), K
//                through a KSTAGE ring and V through an NSTAGE ring.  A K slot
//                frees when its S/R GEMMs finish, a V slot when its PV GEMMs do.
//   warp 1       TMEM owner and MMA issuer.  The whole warp runs the issue
//                loop and one elected lane issues each tcgen05 instruction,
//                so descriptors stay in warp-uniform registers (one elect.sync
//                per batch of MMAs).  The issue order runs across items: SR_{g+1}
//                before PV_g for the CTA's global tile index g, so the tensor
//                pipe computes S/R of the next tile while the softmax works on
//                the current one; at an item boundary the item's last PV goes
//                first, then the next item's S/R as soon as its Q has landed.
//   warps 2-9    softmax + epilogue, two warps per TMEM lane quadrant
//                (quadrant = warp % 4, so both sit on the same scheduler):
//                thread r of the pair owns query row r of the quadrant, the
//                first warp keys 0-31 of each tile and the second keys 32-63.
//                The pair agrees on the row max through shared memory and a
//                per-quadrant mbarrier (bounded waits), once per tile; the
//                exponentials are taken against the running max while that
//                handshake is in flight (again only if a row max jumps).
//                An item's epilogue runs right after its last tile: the pair
//                adds its (l, C) through the same handshake, waits for the
//                item's last PV (issued ahead of the next item's first S/R
//                GEMMs, which run meanwhile) and writes o through a swizzled
//                shared-memory chunk per warp and a TMA store, before the next
//                item's first P (whose PV overwrites O/U) is released.
//   warps 10-11  V re-encode (bf16 -> fp16, in place) of each V stage as
//                soon as it lands, off the softmax's critical path; the PV
//                GEMMs wait for it.
// TMEM (512 columns): S0 | R0 | S1 | R1 (64 each) | O (D) | U (D).  Each softmax
// warp writes its fp16 P (and PR) over the first half of the S (and R) columns
// it read itself: keys [32h, 32h + 32) of the tile go to columns [32h, 32h + 16).
// So no warp writes columns its partner reads.
#pragma once
#include "status.cuh"

namespace plx {

template <int D, bool PLX>
struct FwdTcCfg {
    static constexpr int BM = 128;                 // query rows per item
    static constexpr int BN = 64;                  // keys per K/V tile
    static constexpr int NP = D / 64;              // 64-column panels (128 B rows)
    static constexpr int NSTAGE = (D == 128) ? 4 : 6;   // V ring
    static constexpr int KSTAGE = NSTAGE - 1;      // K ring: its slots free one PV earlier
    static constexpr int SM_WARPS = 8;             // softmax warps: 2 per TMEM lane quadrant
    static constexpr int SM_THREADS = SM_WARPS * 32;
    static constexpr int CV_WARPS = 2;             // V re-encode warps (schedulers 2 and 3)
    static constexpr int CV_THREADS = CV_WARPS * 32;
    static constexpr int THREADS = 64 + SM_THREADS + CV_THREADS;
    static constexpr int HALF = BN / 2;            // keys of a tile per softmax warp
    static constexpr int Q_PANEL = BM * 128;       // bytes per Q/rho panel
    static constexpr int KV_PANEL = BN * 128;      // bytes per K/V panel
    static constexpr int Q_BYTES = NP * Q_PANEL;
    static constexpr int KV_BYTES = NP * KV_PANEL;
    // output staging: one slot per softmax warp for a 32-column block of its 32
    // rows (fp32: 128-byte rows, 128-byte swizzle; bf16: 64-byte rows, 64-byte
    // swizzle), written to global memory by a TMA store
    static constexpr int NCH = D / 64;             // 32-column output blocks per softmax warp
    static constexpr int STG_SLOT_BYTES = 32 * 128;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_R = OFF_Q + Q_BYTES;
    static constexpr int OFF_K = OFF_R + (PLX ? Q_BYTES : 0);
    static constexpr int OFF_V = OFF_K + KSTAGE * KV_BYTES;
    static constexpr int OFF_STG = OFF_V + NSTAGE * KV_BYTES;
    // pair exchange: row max per tile [2 tile parities][2 halves][BM] floats,
    // (l, C) per item [2 item parities][2 halves][BM] float2
    static constexpr int OFF_XMAX = OFF_STG + SM_WARPS * STG_SLOT_BYTES;
    static constexpr int OFF_XLC = OFF_XMAX + 2 * 2 * BM * 4;
    // the training forward's fp32 (l, C) of the unrounded terms, the same shape
    static constexpr int OFF_XLC32 = OFF_XLC + 2 * 2 * BM * 8;
    static constexpr int OFF_BAR = OFF_XLC32 + 2 * 2 * BM * 8;
    // barriers: q_full, q_empty, k_full[KSTAGE], k_empty[KSTAGE], v_full[NSTAGE], v_empty[NSTAGE],
    // v_ready[NSTAGE], s_full[2], p_full[2], pv_done[2], drain, pair[4]
    static constexpr int NBARS = 2 + 2 * KSTAGE + 3 * NSTAGE + 2 + 2 + 2 + 1 + 4;
    static constexpr int SMEM_USED = OFF_BAR + NBARS * 8 + 16;
    static constexpr int SMEM = SMEM_USED + 1024;  // slack for 1024-byte alignment
    // TMEM columns
    static constexpr uint32_t TM_S0 = 0, TM_R0 = 64, TM_S1 = 128, TM_R1 = 192, TM_O = 256, TM_U = 256 + D;
    static constexpr uint32_t TM_COLS = 512;
    static constexpr float RESCALE_THRESH = 4.0f;  // log2 units: P <= 16
    static_assert(D == 64 || D == 128, "tcgen05 forward supports d in {64, 128}");
    static_assert(HALF == 32, "one 32x32b.x32 TMEM load per warp and tile");
    static_assert(OFF_STG % 1024 == 0, "staging chunks start on the swizzle period");
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert((KV_BYTES / 16) % CV_THREADS == 0, "V re-encode splits evenly over its threads");
};

struct FwdTcParams {
    float* lse;
    int N;                 // K/V rows per head (the cache capacity in the cached mode)
    int Tq;                // query rows per head (N for the self-attention prefill)
    // cached mode: queries are the last Tq positions of a cache of seqlens[b]
    // rows (positions seqlens[b] - Tq + i); nullptr: query row i is position i
    const int* seqlens;
    int H;
    int BH;
    int n_qt;
    int n_items;
    float scale_log2;
    int out_f32;
    int no_intercept;      // the family's no-intercept member: o = -u
    float* c_out;          // the training forward: c_i per row, [BH][Tq] (else unused)
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
// Geometry of item u: head bh, first query row q0, the position of query row
// 0 (off: 0 for the self-attention prefill, seqlens[b] - Tq in the cached
// mode, with seqlens[b] clamped to [Tq, N]) and the number of K/V tiles it
// reads.  Every role computes it the same way.
struct ItemSpan {
    int bh, q0, off, n_kv;
};
template <bool CACHED>
__device__ __forceinline__ ItemSpan item_span(const FwdTcParams& p, int u, int BM, int BN, bool flag_bad = false) {
    ItemSpan it;
    int qt;
    item_coords(u, p.BH, p.n_qt, it.bh, qt);
    it.q0 = qt * BM;
    int L = p.N;
    if (CACHED) {
        L = p.seqlens[it.bh / p.H];
        if (L < p.Tq || L > p.N) {
            if (flag_bad) atomicOr(&g_plx_status, PLX_DEV_ERR_SEQLEN);
            L = L < p.Tq ? p.Tq : p.N;
        }
    }
    it.off = CACHED ? L - p.Tq : 0;       // the self-attention prefill: query row i is position i
    it.n_kv = (it.off + min(p.Tq, it.q0 + BM) + BN - 1) / BN;
    // debug build: the head, the query tile and the K/V tiles lie inside the
    // tensors (every role clamps alike, so the barrier phases stay in step)
    if (!in_bounds(it.bh < p.BH && it.q0 < p.Tq && it.n_kv >= 1 && it.n_kv <= (p.N + BN - 1) / BN)) {
        it.bh = min(it.bh, p.BH - 1);
        it.q0 = 0;
        it.n_kv = 1;
    }
    return it;
}
// u for round r of CTA c in a snake over the grid
__device__ __forceinline__ int snake_item(int r, int c, int G) {
    return r * G + ((r & 1) ? (G - 1 - c) : c);
}

// TRAIN: the training forward, which also writes vbar_i = O_i / l_i (fp32,
// through mapVb, the same layout as an fp32 o) and c_i (p.c_out), the values
// the backward's row statistics are formed from.
template <int D, bool PLX, bool CACHED = false, bool TRAIN = false>
__global__ void __launch_bounds__(FwdTcCfg<D, PLX>::THREADS, 1)
plx_fwd_tc_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapR,
                  const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                  const __grid_constant__ CUtensorMap mapO, const __grid_constant__ CUtensorMap mapVb,
                  const FwdTcParams p) {
    using Cfg = FwdTcCfg<D, PLX>;
    static_assert(!TRAIN || (PLX && !CACHED), "the training forward is the PLX prefill");
    constexpr int BM = Cfg::BM, BN = Cfg::BN, NP = Cfg::NP, NSTAGE = Cfg::NSTAGE, KSTAGE = Cfg::KSTAGE,
                  HALF = Cfg::HALF;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + Cfg::OFF_Q;
    uint8_t* sR = smem + Cfg::OFF_R;
    uint8_t* sK = smem + Cfg::OFF_K;
    uint8_t* sV = smem + Cfg::OFF_V;
    float* xmax = reinterpret_cast<float*>(smem + Cfg::OFF_XMAX);
    float2* xlc = reinterpret_cast<float2*>(smem + Cfg::OFF_XLC);
    float2* xlc32 = reinterpret_cast<float2*>(smem + Cfg::OFF_XLC32);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    uint64_t* q_full = bars;
    uint64_t* q_empty = bars + 1;
    uint64_t* k_full = bars + 2;
    uint64_t* k_empty = k_full + KSTAGE;
    uint64_t* v_full = k_empty + KSTAGE;
    uint64_t* v_empty = v_full + NSTAGE;
    uint64_t* v_ready = v_empty + NSTAGE;    // V of the stage re-encoded to fp16
    uint64_t* s_full = v_ready + NSTAGE;
    uint64_t* p_full = s_full + 2;
    uint64_t* pv_done = p_full + 2;      // one per S/R buffer: PV of tiles g with g % 2 == b
    uint64_t* drain = pv_done + 2;
    uint64_t* pair_bar = drain + 1;      // one per TMEM lane quadrant: the two softmax warps on it
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pair_bar + 4);
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
        for (int s = 0; s < KSTAGE; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
            mbar_init(&v_ready[s], Cfg::CV_WARPS);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&p_full[b], Cfg::SM_WARPS);     // one elected arrival per softmax warp
            mbar_init(&pv_done[b], 1);
        }
        mbar_init(drain, 1);
        for (int qd = 0; qd < 4; ++qd) mbar_init(&pair_bar[qd], 2);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&mapQ);
        tma_prefetch_desc(&mapK);
        tma_prefetch_desc(&mapV);
        tma_prefetch_desc(&mapO);
        if (PLX) tma_prefetch_desc(&mapR);
        if (TRAIN) tma_prefetch_desc(&mapVb);
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
            int nq = 0, nk = 0, nv = 0;           // loads issued: Q tiles, K tiles, V tiles
            bool ok = true;
            for (int r = 0; ok; ++r) {
                const int u = snake_item(r, c, G);
                if (u >= p.n_items || *abort_flag) break;
                const ItemSpan it = item_span<CACHED>(p, u, BM, BN, true);
                const int bh = it.bh, q0 = it.q0, n_kv = it.n_kv;
                const int un = snake_item(r + 1, c, G);    // this CTA's next item
                if (nq > 0 && !mbar_wait(q_empty, (nq - 1) & 1)) { ok = false; break; }
                mbar_arrive_expect_tx(q_full, (PLX ? 2 : 1) * Cfg::Q_BYTES);
                for (int pn = 0; pn < NP; ++pn) {
                    tma_load_3d(sQ + pn * Cfg::Q_PANEL, &mapQ, q_full, pn * 64, q0, bh);
                    if (PLX) tma_load_3d(sR + pn * Cfg::Q_PANEL, &mapR, q_full, pn * 64, q0, bh);
                }
                ++nq;
                for (int j = 0; j < n_kv; ++j) {
                    // the next item's Q (and rho) tile is read once, from HBM: start it
                    // into L2 a few tiles before its load
                    if (j == max(0, n_kv - 3) && un < p.n_items) {
                        int nbh, nqt;
                        item_coords(un, p.BH, p.n_qt, nbh, nqt);
                        for (int pn = 0; pn < NP; ++pn) {
                            tma_prefetch_l2_3d(&mapQ, pn * 64, nqt * BM, nbh);
                            if (PLX) tma_prefetch_l2_3d(&mapR, pn * 64, nqt * BM, nbh);
                        }
                    }
                    const int ks = nk % KSTAGE;
                    if (nk >= KSTAGE && !mbar_wait(&k_empty[ks], ((nk / KSTAGE) - 1) & 1)) { ok = false; break; }
                    mbar_arrive_expect_tx(&k_full[ks], Cfg::KV_BYTES);
                    for (int pn = 0; pn < NP; ++pn)
                        tma_load_3d(sK + ks * Cfg::KV_BYTES + pn * Cfg::KV_PANEL, &mapK, &k_full[ks], pn * 64,
                                    j * BN, bh);
                    ++nk;
                    const int vs = nv % NSTAGE;
                    if (nv >= NSTAGE && !mbar_wait(&v_empty[vs], ((nv / NSTAGE) - 1) & 1)) { ok = false; break; }
                    mbar_arrive_expect_tx(&v_full[vs], Cfg::KV_BYTES);
                    for (int pn = 0; pn < NP; ++pn)
                        tma_load_3d(sV + vs * Cfg::KV_BYTES + pn * Cfg::KV_PANEL, &mapV, &v_full[vs], pn * 64,
                                    j * BN, bh);
                    ++nv;
                }
            }
            if (!ok) fail();
            // never leave with loads in flight into this CTA's shared memory
            for (int i = max(0, nk - KSTAGE); i < nk; ++i)
                if (!mbar_wait(&k_full[i % KSTAGE], (i / KSTAGE) & 1)) fail();
            for (int i = max(0, nv - NSTAGE); i < nv; ++i)
                if (!mbar_wait(&v_full[i % NSTAGE], (i / NSTAGE) & 1)) fail();
            if (nq > 0 && !mbar_wait(q_full, (nq - 1) & 1)) fail();
        }
    } else if (warp == 1) {
        // ===================================================== MMA issuer (whole warp)
        constexpr uint32_t ID_S = idesc_bf16_f32(128, BN, false, false);
        constexpr uint32_t ID_PV = idesc_f16_f32(128, D, false, true);
        const uint32_t sKa = smem_u32(sK), sVa = smem_u32(sV);
        // base descriptors of the K-major Q and rho tiles (fixed for the kernel)
        const uint64_t a_q = sdesc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t a_r = sdesc_sw128(smem_u32(sR), 16, 1024);
        auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity));
        };
        // PV GEMMs of global tile pg; the first tile of an item overwrites O and U
        auto issue_pv = [&](int pg, bool first) -> bool {
            const int b = pg & 1;
            const int stage = pg % NSTAGE;
            if (!wait_warp(&p_full[b], (pg >> 1) & 1)) return false;
            if (!wait_warp(&v_ready[stage], (pg / NSTAGE) & 1)) return false;
            tc_fence_after();
            const uint32_t tS = tmem + (b ? Cfg::TM_S1 : Cfg::TM_S0);
            static_assert(Cfg::TM_R0 == Cfg::TM_S0 + 64 && Cfg::TM_R1 == Cfg::TM_S1 + 64, "R sits 64 columns after S");
            // keys [32h, 32h + 32) of the tile sit, as fp16 pairs, in columns [32h, 32h + 16)
            // of S_b (P) and R_b (PR); V is the MN-major B operand
            const uint64_t b_v = sdesc_sw128(sVa + stage * Cfg::KV_BYTES, Cfg::KV_PANEL, 1024);
            mma_pv_batch<PLX, 0, PLX ? 64 : 0>(tmem + Cfg::TM_O, tmem + Cfg::TM_U, tS, b_v, ID_PV, first ? 0u : 1u);
            mma_commit_warp(&v_empty[stage]);
            mma_commit_warp(&pv_done[b]);
            return true;
        };
        int items = 0, g = 0;
        bool ok = true, pend = false, pend_first = false;
        for (int r = 0; ok; ++r) {
            const int u = snake_item(r, c, G);
            // one read of the flag for the whole warp: every lane takes the same branch
            if (u >= p.n_items || __shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            const int n_kv = item_span<CACHED>(p, u, BM, BN).n_kv;
            // the previous item's last PV goes first: its epilogue then runs while
            // the S/R GEMMs of this item's first tiles do
            if (pend && !issue_pv(g - 1, pend_first)) { ok = false; break; }
            pend = false;
            if (!wait_warp(q_full, items & 1)) { ok = false; break; }
            tc_fence_after();
            for (int j = 0; j < n_kv; ++j, ++g) {
                const int ks = g % KSTAGE;
                if (!wait_warp(&k_full[ks], (g / KSTAGE) & 1)) { ok = false; break; }
                tc_fence_after();
                const int b = g & 1;
                const uint32_t tS = tmem + (b ? Cfg::TM_S1 : Cfg::TM_S0);
                const uint32_t tR = tmem + (b ? Cfg::TM_R1 : Cfg::TM_R0);
                static_assert(Cfg::KV_PANEL == 512 * 16, "panel stride of the S/R batch");
                mma_sr_batch<D, PLX, Cfg::Q_PANEL / 16>(tS, tR, a_q, a_r, sdesc_sw128(sKa + ks * Cfg::KV_BYTES, 16, 1024),
                                                        ID_S);
                mma_commit_warp(&k_empty[ks]);
                mma_commit_warp(&s_full[b]);
                if (j == n_kv - 1) mma_commit_warp(q_empty);
                // then the PV of the tile before this one
                if (pend && !issue_pv(g - 1, pend_first)) { ok = false; break; }
                pend = true;
                pend_first = j == 0;
            }
            ++items;
        }
        if (ok && pend && !issue_pv(g - 1, pend_first)) ok = false;
        if (!ok) fail();
        // drain: every MMA issued by this warp has finished before TMEM is freed
        mma_commit_warp(drain);
        if (!wait_warp(drain, 0)) fail();
    } else if (warp < 2 + Cfg::SM_WARPS) {
        // ===================================================== softmax + epilogue (warps 2..9)
        const int sw = warp - 2;                // 0..7
        const int quad = warp & 3;              // TMEM lane quadrant this warp may access
        const int half = sw >> 2;               // 0: keys 0..31 of each tile, 1: keys 32..63
        const int row = quad * 32 + lane;       // query row within the item
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
        uint64_t* pbar = &pair_bar[quad];
        uint8_t* stg = smem + Cfg::OFF_STG + sw * Cfg::STG_SLOT_BYTES;
        int g = 0, n_pair = 0, items = 0;
        // all waits and exits are warp-uniform: the tcgen05 loads/stores below are .sync.aligned
        auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity));
        };
        // The two warps of a quadrant meet here: each has finished its TMEM loads
        // and shared-memory writes before the other passes pair_wait.
        auto pair_arrive = [&]() {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(pbar);
        };
        auto pair_wait = [&]() -> bool {
            const bool ok = wait_warp(pbar, n_pair & 1);
            ++n_pair;
            tc_fence_after();
            return ok;
        };
        // Epilogue of item eu, whose last tile is global tile eg: wait for its
        // last PV (the one before it on the same buffer barrier is complete,
        // and the next cannot start before this warp releases its P), combine
        // the two warps' (l, C) from xe, then o = (1 + c) vbar - u on this
        // warp's 32 rows and half of the columns, one 32-column block at a time
        // through this warp's staging slot and a TMA store.  Thread r writes row
        // r in the tensor map's swizzle (16-byte unit u of row r at u ^ (r & 7)
        // for 128-byte fp32 rows, u ^ ((r >> 1) & 3) for 64-byte bf16 rows), so
        // the eight rows of a quarter-warp hit eight different bank groups.
        auto epilogue = [&](int eu, int eg, float em, const float2* xe, const float2* xe32) -> bool {
            if (!wait_warp(&pv_done[eg & 1], (eg >> 1) & 1)) return false;
            tc_fence_after();
            int ebh, eqt;
            item_coords(eu, p.BH, p.n_qt, ebh, eqt);
            const int eq0 = eqt * BM;
            // rows past N are clipped by the TMA store; a warp whose 32 rows all
            // are past N has nothing to write (both warps of the pair decide alike)
            if (eq0 + quad * 32 >= p.Tq) return true;
            const float2 e0 = xe[row], e1 = xe[BM + row];
            const float l_all = e0.x + e1.x, C_all = e0.y + e1.y;
            const float inv_l = 1.f / l_all;
            const float cc_ = C_all * inv_l;
            // the training forward's c_i: the same weights summed in fp32 before
            // the fp16 rounding of P and P o R.  (o uses the rounded sums, whose
            // rounding cancels against U's; c on its own feeds the backward's
            // 1 + c_i - r_ij, where it would not.)
            float c32 = 0.f;
            if constexpr (TRAIN) {
                const float2 f0 = xe32[row], f1 = xe32[BM + row];
                c32 = (f0.y + f1.y) / (f0.x + f1.x);
            }
            // 0 * o is NaN exactly when o is not finite: one running sum flags them all
            float bad = 0.f;
#pragma unroll 1
            for (int ch = 0; ch < Cfg::NCH; ++ch) {
                const int col = half * (D / 2) + 32 * ch;
                uint32_t ov[32];
                float o[32];
                if constexpr (PLX) {
                    uint32_t uv[32];
                    tmem_ld32x32b_x32_nowait(lane_addr + Cfg::TM_O + col, ov);
                    tmem_ld32x32b_x32_nowait(lane_addr + Cfg::TM_U + col, uv);
                    tmem_ld_wait(ov);
                    tmem_ld_wait(uv);
                    if (p.no_intercept) {
#pragma unroll
                        for (int cc = 0; cc < 32; ++cc) o[cc] = -__uint_as_float(uv[cc]) * inv_l;
                    } else {
#pragma unroll
                        for (int cc = 0; cc < 32; ++cc) {
                            const float vbar = __uint_as_float(ov[cc]) * inv_l;
                            o[cc] = fmaf(cc_, vbar, vbar) - __uint_as_float(uv[cc]) * inv_l;
                        }
                    }
                } else {
                    tmem_ld32x32b_x32(lane_addr + Cfg::TM_O + col, ov);
#pragma unroll
                    for (int cc = 0; cc < 32; ++cc) o[cc] = __uint_as_float(ov[cc]) * inv_l;
                }
#pragma unroll
                for (int cc = 0; cc < 32; ++cc) bad = fmaf(o[cc], 0.f, bad);
                // the slot is free once this warp's previous store has read it
                if (lane == 0) bulk_wait_read<0>();
                __syncwarp();
                if (p.out_f32) {
#pragma unroll
                    for (int u4 = 0; u4 < 8; ++u4)
                        *reinterpret_cast<uint4*>(stg + lane * 128 + ((u4 ^ (lane & 7)) << 4)) =
                            make_uint4(__float_as_uint(o[4 * u4]), __float_as_uint(o[4 * u4 + 1]),
                                       __float_as_uint(o[4 * u4 + 2]), __float_as_uint(o[4 * u4 + 3]));
                } else {
                    const int swz = (lane >> 1) & 3;
#pragma unroll
                    for (int u4 = 0; u4 < 4; ++u4)
                        *reinterpret_cast<uint4*>(stg + lane * 64 + ((u4 ^ swz) << 4)) =
                            make_uint4(pack_bf16x2(o[8 * u4], o[8 * u4 + 1]),
                                       pack_bf16x2(o[8 * u4 + 2], o[8 * u4 + 3]),
                                       pack_bf16x2(o[8 * u4 + 4], o[8 * u4 + 5]),
                                       pack_bf16x2(o[8 * u4 + 6], o[8 * u4 + 7]));
                }
                // the staged rows are read next by the TMA engine (async proxy)
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_3d(&mapO, stg, col, eq0 + quad * 32, ebh);
                    bulk_commit_group();
                }
                if constexpr (TRAIN) {
                    // vbar of the same block, fp32, through the same slot once o's
                    // store has read it
                    if (lane == 0) bulk_wait_read<0>();
                    __syncwarp();
#pragma unroll
                    for (int u4 = 0; u4 < 8; ++u4)
                        *reinterpret_cast<uint4*>(stg + lane * 128 + ((u4 ^ (lane & 7)) << 4)) =
                            make_uint4(__float_as_uint(__uint_as_float(ov[4 * u4]) * inv_l),
                                       __float_as_uint(__uint_as_float(ov[4 * u4 + 1]) * inv_l),
                                       __float_as_uint(__uint_as_float(ov[4 * u4 + 2]) * inv_l),
                                       __float_as_uint(__uint_as_float(ov[4 * u4 + 3]) * inv_l));
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&mapVb, stg, col, eq0 + quad * 32, ebh);
                        bulk_commit_group();
                    }
                }
            }
            const int ei = eq0 + row;
            const bool store = ei < p.Tq;
            if (store && half == 0 && p.lse && in_bounds(ebh < p.BH))
                p.lse[static_cast<size_t>(ebh) * p.Tq + ei] = (em + __log2f(l_all)) * 0.69314718055994531f;
            if (TRAIN && store && half == 0 && in_bounds(ebh < p.BH)) p.c_out[static_cast<size_t>(ebh) * p.Tq + ei] = c32;
            if (__any_sync(0xffffffffu, store && !(bad == 0.f)) && lane == 0)
                atomicOr(&g_plx_status, PLX_DEV_ERR_NONFINITE);
            return true;
        };
        bool ok = true;
        for (int r = 0; ok; ++r) {
            const int u = snake_item(r, c, G);
            if (u >= p.n_items || __shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            const ItemSpan it = item_span<CACHED>(p, u, BM, BN);
            const int q0 = it.q0, n_kv = it.n_kv;
            const int i = q0 + row;                 // this thread's query row
            const int pos = it.off + i;             // its position: keys 0 .. pos
            float m = -INFINITY, l = 0.f, C = 0.f;
            float2 l32 = make_float2(0.f, 0.f), C32 = make_float2(0.f, 0.f);   // training forward only
            // cached mode: a quadrant none of whose 32 rows is a query row (T < 128)
            // stores nothing; its two warps only keep the barrier phases in step,
            // and the garbage left in its lanes stays in its own rows
            const bool idle = CACHED && q0 + quad * 32 >= p.Tq;
            for (int j = 0; j < n_kv; ++j, ++g) {
                const int b = g & 1;
                if (!wait_warp(&s_full[b], (g >> 1) & 1)) { ok = false; break; }
                tc_fence_after();
                if (idle) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&p_full[b]);
                    continue;
                }
                const uint32_t tS = lane_addr + (b ? Cfg::TM_S1 : Cfg::TM_S0);
                const uint32_t tR = lane_addr + (b ? Cfg::TM_R1 : Cfg::TM_R0);
                // S now; R is loaded after the max is published, so its TMEM
                // latency hides under the exponentials
                uint32_t sraw[HALF], rraw[HALF];
                tmem_ld32x32b_x32_nowait(tS + half * HALF, sraw);
                tmem_ld_wait(sraw);
                float sc[HALF];
#pragma unroll
                for (int cc = 0; cc < HALF; ++cc) sc[cc] = __uint_as_float(sraw[cc]);
                // causal mask on tiles that reach past the first position of the item
                const bool diag = (j + 1) * BN - 1 > it.off + q0;
                const int kbase = j * BN + half * HALF;
                if (diag) {
#pragma unroll
                    for (int cc = 0; cc < HALF; ++cc)
                        if (kbase + cc > pos) sc[cc] = -INFINITY;
                }
                // row max over this warp's 32 keys: a tree of three-input maxes
                float mx[11];
#pragma unroll
                for (int t = 0; t < 10; ++t) mx[t] = fmax3(sc[3 * t], sc[3 * t + 1], sc[3 * t + 2]);
                mx[10] = fmaxf(sc[30], sc[31]);
                const float mloc = fmaxf(fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                               fmax3(mx[6], mx[7], mx[8])),
                                         fmaxf(mx[9], mx[10]));
                // The other warp of the quadrant holds the other 32 keys of the row.
                // Publish this warp's max.  While the handshake completes, take the
                // exponentials against the running max m of the earlier tiles: in the
                // usual case this tile raises no row max of the warp by more than
                // 2^4, m stays, and they are final.  The first tile of an item, and a
                // tile that does raise a row max that far (a warp-uniform decision,
                // the same in both warps), take them again against the new m.
                float* xm = xmax + (b * 2) * BM;
                xm[half * BM + row] = mloc;
                pair_arrive();
                if constexpr (PLX) tmem_ld32x32b_x32_nowait(tR + half * HALF, rraw);
                float pe[HALF];
                auto exps = [&](float mref) {
                    const float2 nm2 = make_float2(-mref, -mref);
#pragma unroll
                    for (int cc = 0; cc < HALF; cc += 2) {
                        const float2 x = ffma2(make_float2(sc[cc], sc[cc + 1]), sl2, nm2);
                        pe[cc] = fast_exp2(x.x);
                        pe[cc + 1] = fast_exp2(x.y);
                    }
                };
                if (j > 0) exps(m);
                if (!pair_wait()) { ok = false; break; }
                const float mt = fmaxf(xm[row], xm[BM + row]);   // same operands, same order in both warps
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
                        if constexpr (TRAIN) {
                            l32 = fmul2(l32, make_float2(alpha, alpha));
                            C32 = fmul2(C32, make_float2(alpha, alpha));
                        }
                    }
                }
                // P = 2^(scale S - m) <= 2^4: every score of the tile is within 2^4 of m
                if (j == 0 || rescale_warp) exps(m);
                if (diag) {
#pragma unroll
                    for (int cc = 0; cc < HALF; ++cc)
                        if (kbase + cc > pos) pe[cc] = 0.f;     // also covers scale == 0
                }
                // P and PR go to the tensor cores as fp16; l and C are summed from
                // the same rounded values, so o = (1 + C/l) O/l - U/l is exactly
                // PLX for the rounded weights (they sum to one) and the rounding
                // errors cancel the way the exact terms do.
                uint32_t pk[HALF / 2];
                float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int cc = 0; cc < HALF / 2; ++cc) {
                    pk[cc] = pack_f16x2(pe[2 * cc], pe[2 * cc + 1]);
                    ls[cc & 3] = add_f16x2(ls[cc & 3], pk[cc]);
                }
                l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                if constexpr (TRAIN) {
#pragma unroll
                    for (int cc = 0; cc < HALF; cc += 2) l32 = fadd2(l32, make_float2(pe[cc], pe[cc + 1]));
                }
                tmem_st32x32b_x16(tS + half * HALF, pk);
                if constexpr (PLX) {
                    tmem_ld_wait(rraw);
                    // cached mode: masked keys contribute nothing, even where R is
                    // not finite (cache rows past the sequence)
                    if (CACHED && diag) {
#pragma unroll
                        for (int cc = 0; cc < HALF; ++cc)
                            if (kbase + cc > pos) rraw[cc] = 0u;
                    }
                    float cs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int cc = 0; cc < HALF / 2; ++cc) {
                        const float2 a = fmul2(make_float2(pe[2 * cc], pe[2 * cc + 1]),
                                               make_float2(__uint_as_float(rraw[2 * cc]),
                                                           __uint_as_float(rraw[2 * cc + 1])));
                        pk[cc] = pack_f16x2(a.x, a.y);
                        cs[cc & 3] = add_f16x2(cs[cc & 3], pk[cc]);
                        if constexpr (TRAIN) C32 = fadd2(C32, a);
                    }
                    C += (cs[0] + cs[1]) + (cs[2] + cs[3]);
                    tmem_st32x32b_x16(tR + half * HALF, pk);
                }
                if (rescale_warp) {
                    // O and U must hold the previous tile's PV before they are
                    // rescaled.  Only that PV can still be in flight: the S/R MMA
                    // of this tile completed after the PV two tiles back, and the
                    // next PV needs this tile's P.  So the wait on the previous
                    // tile's buffer barrier is unambiguous, and no other tile waits.
                    // Both warps of the quadrant take the same decision; each
                    // rescales half of the accumulator columns.
                    const int gp = g - 1;
                    if (!wait_warp(&pv_done[gp & 1], (gp >> 1) & 1)) { ok = false; break; }
                    tc_fence_after();
                    constexpr int ACC = PLX ? 2 * D : D;
#pragma unroll 1
                    for (int cb = half * (ACC / 2); cb < (half + 1) * (ACC / 2); cb += 32) {
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
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[b]);
            }
            if (!ok) break;
            // The item's epilogue, right after its last tile: the pair adds its
            // (l, C), then waits for the last PV.  The MMA warp issues that PV
            // before the next item's first S/R GEMMs, which run meanwhile; the
            // next item's first PV, which overwrites O and U, needs this warp's P
            // of that item and so comes after the epilogue.
            if (!idle) {
                float2* xe = xlc + ((items & 1) * 2) * BM;
                float2* xe32 = xlc32 + ((items & 1) * 2) * BM;
                xe[half * BM + row] = make_float2(l, C);
                if constexpr (TRAIN) xe32[half * BM + row] = make_float2(l32.x + l32.y, C32.x + C32.y);
                pair_arrive();
                if (!pair_wait() || !epilogue(u, g - 1, m, xe, xe32)) { ok = false; break; }
            }
            ++items;
        }
        if (!ok) fail();
        // no TMEM store of this warp is still pending (a wait that gave up may
        // have left the tile after its stores), and the output stores have
        // finished (and stopped reading shared memory)
        tmem_st_wait();
        if (lane == 0) bulk_wait_all();
        tc_fence_before();
    } else if (warp >= 2 + Cfg::SM_WARPS) {
        // ===================================================== V re-encode (warps 10..11, on schedulers 2 and 3: scheduler 1 carries the MMA warp)
        // Each stage's V goes bf16 -> fp16 in place for the PV GEMMs as soon as
        // it lands; element-wise, so the 128-byte swizzle is unchanged.
        const int t = (warp - 2 - Cfg::SM_WARPS) * 32 + lane;
        auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity));
        };
        int g = 0;
        bool ok = true;
        for (int r = 0; ok; ++r) {
            const int u = snake_item(r, c, G);
            if (u >= p.n_items || __shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            const ItemSpan it = item_span<CACHED>(p, u, BM, BN);
            const int n_kv = it.n_kv;
            const int L = it.off + p.Tq;          // keys at L and beyond are masked for every row
            for (int j = 0; j < n_kv; ++j, ++g) {
                const int stage = g % NSTAGE;
                if (!wait_warp(&v_full[stage], (g / NSTAGE) & 1)) { ok = false; break; }
                uint4* vt = reinterpret_cast<uint4*>(sV + stage * Cfg::KV_BYTES);
                if (!CACHED || (j + 1) * BN <= L) {
#pragma unroll
                    for (int k = 0; k < Cfg::KV_BYTES / 16 / Cfg::CV_THREADS; ++k) {
                        uint4 w = vt[t + Cfg::CV_THREADS * k];
                        w.x = bf16x2_to_f16x2(w.x);
                        w.y = bf16x2_to_f16x2(w.y);
                        w.z = bf16x2_to_f16x2(w.z);
                        w.w = bf16x2_to_f16x2(w.w);
                        vt[t + Cfg::CV_THREADS * k] = w;
                    }
                } else {
                    // the item's last tile: 16-byte unit idx lies in key row
                    // (idx mod (64 rows x 8 units)) / 8 of its panel, and rows at or
                    // past L become zeros (P is 0 there, and 0 x a non-finite stale
                    // value would still reach O)
#pragma unroll 4
                    for (int k = 0; k < Cfg::KV_BYTES / 16 / Cfg::CV_THREADS; ++k) {
                        const int idx = t + Cfg::CV_THREADS * k;
                        const int key = j * BN + ((idx % (Cfg::KV_PANEL / 16)) >> 3);
                        uint4 w = vt[idx];
                        if (key >= L) {
                            w = make_uint4(0u, 0u, 0u, 0u);
                        } else {
                            w.x = bf16x2_to_f16x2(w.x);
                            w.y = bf16x2_to_f16x2(w.y);
                            w.z = bf16x2_to_f16x2(w.z);
                            w.w = bf16x2_to_f16x2(w.w);
                        }
                        vt[idx] = w;
                    }
                }
                // the re-encoded V is read next by the tensor cores (async proxy)
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&v_ready[stage]);
            }
        }
        if (!ok) fail();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::TM_COLS);
    }
}

}  // namespace plx
