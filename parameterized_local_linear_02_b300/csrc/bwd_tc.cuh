// bwd_tc.cuh -- plx_bwd: gradients of causal PLX attention on the 5th-generation
// tensor cores (tcgen05, TMEM accumulators, TMA-fed 128B-swizzled tiles).
//
// Forward ("Parallax: Parameterized Local Linear Attention for Language
// Modeling", zhichai.net section 1.3; gist.science "Meccanismo Principale"):
//   w_ij = softmax_{j<=i}(scale q_i.k_j),  r_ij = rho_i.k_j,
//   vbar_i = sum_j w_ij v_j,  c_i = sum_j w_ij r_ij,  o_i = (1 + c_i) vbar_i - u_i.
// The pages give no backward pass.  Differentiating the forward, with
// dO_i = dL/do_i, G_ij = dO_i.v_j, a_i = dO_i.vbar_i, D_i = dO_i.o_i + c_i a_i:
//   ds_ij = w_ij ((1 + c_i - r_ij) G_ij + a_i r_ij - D_i)     (dL/d(scale q_i.k_j))
//   dr_ij = w_ij (a_i - G_ij)                                  (dL/dr_ij)
//   wv_ij = w_ij (1 + c_i - r_ij)                              (dv_j = sum_i wv_ij dO_i)
//   dq_i = scale sum_j ds_ij k_j,   drho_i = sum_j dr_ij k_j,
//   dk_j = scale sum_i ds_ij q_i + sum_i dr_ij rho_i,   dv_j = sum_i wv_ij dO_i,
// with w_ij = 2^(scale log2e s_ij - log2e lse_i).  The row statistics
// (log2e lse_i, c_i, a_i, D_i) come from a third pass of the same template
// (PASS = BWD_STATS): S, R and G per tile, and online fp32 row sums
// c_i = sum w r, a_i = sum w G, e_i = sum w r G with D_i = (1 + 2 c_i) a_i - e_i,
// so the statistics use exactly the weights the two gradient passes use.
//
// Two passes over the causal (i, j) tiles, one kernel template:
//   dq pass  (PASS = BWD_DQ):  a CTA item is 128 query rows; Q, rho and dO of the
//            rows are resident, K and V stream in 64-key tiles.  Per tile
//            S = Q K^T, R = rho K^T, G = dO V^T; then dQ += ds K, dRho += dr K.
//   dkv pass (PASS = BWD_DKV): a CTA item is 128 key rows; K and V are resident,
//            Q, rho, dO and the queries' statistics stream in 64-query tiles.
//            Per tile S^T = K Q^T, R^T = K rho^T, G^T = V dO^T; then
//            dV += wv^T-rows dO, dK += ds Q + dr rho (ds already carries the scale).
// In both, TMEM lane = the CTA's row, TMEM column = the streamed index, so one
// thread owns one row and the elementwise step needs no cross-thread reduction
// and, with lse known, no running max.
//
// Roles (384 threads, one CTA per SM, persistent over items):
//   warp 0       TMA producer (one lane): the resident tiles once per item, the
//                streamed tiles through an NSTAGE ring.
//   warp 1       TMEM owner and MMA issuer (whole warp, elected lane).  Per
//                global step g: S_g, R_g (and in the dq pass G_g) as soon as
//                every elementwise warp has S/R/G of step g - 1 in registers;
//                then the output GEMMs of step g - 1 (dkv: dV_{g-1} before G_g,
//                because wv_{g-1} sits in G's columns).
//   warps 2-9    elementwise + epilogue, two per TMEM lane quadrant (quadrant =
//                warp % 4), each on 32 of the 64 streamed columns.  ds, dr (and
//                wv) go back to TMEM as fp16, the A operands of the output GEMMs.
//   warps 10-11  re-encode the streamed tiles the output GEMMs read (dq: K;
//                dkv: Q, rho, dO) from bf16 to fp16 in place, once the step's
//                S/R/G GEMMs have read them.  With bf16 ds/dr/wv the rounding
//                alone gives gradient errors near 3e-2 of their RMS; fp16 keeps
//                them near 3e-3.
// TMEM (512 columns): S | R | G (64 each) | ds | dr (32 each, fp16 pairs) |
// ACC0 (D) | ACC1 (D); ACC0/ACC1 = dQ/dRho (dq pass) or dV/dK (dkv pass).  In
// the dkv pass wv is written over G: the warp of columns [32h, 32h + 32) puts
// them, as pairs, into G columns [32h, 32h + 16).
#pragma once
#include "status.cuh"

namespace plx {

enum { BWD_DQ = 0, BWD_DKV = 1, BWD_STATS = 2 };

template <int D, bool PLX, int PASS>
struct BwdTcCfg {
    static constexpr int ROWS = 128;               // TMEM lanes: queries (dq) or keys (dkv)
    static constexpr int COLS = 64;                // streamed columns per step
    static constexpr int NP = D / 64;              // 64-element panels (128-byte rows)
    static constexpr int EW_WARPS = 8;
    static constexpr int CV_WARPS = 2;             // bf16 -> fp16 re-encode of the output GEMMs' B tiles
    static constexpr int CV_THREADS = CV_WARPS * 32;
    static constexpr int THREADS = 64 + EW_WARPS * 32 + CV_THREADS;
    static constexpr int HALF = COLS / 2;
    static constexpr int RES_PANEL = ROWS * 128;
    static constexpr int STR_PANEL = COLS * 128;
    static constexpr int RES_TILE = NP * RES_PANEL;
    static constexpr int STR_TILE = NP * STR_PANEL;
    // resident operands: dq and statistics passes -> Q, rho, dO (A of S, R, G); dkv -> K (A of
    // S and R), V (A of G)
    static constexpr int N_RES = PASS != BWD_DKV ? (PLX ? 3 : 2) : 2;
    // streamed operands: dq and statistics passes -> K, V; dkv -> Q, rho, dO (+ the queries'
    // statistics)
    static constexpr int N_STR = PASS != BWD_DKV ? 2 : (PLX ? 3 : 2);
    static constexpr int STATS_BYTES = PASS == BWD_DKV ? COLS * 16 : 0;
    static constexpr int STAGE_BYTES = N_STR * STR_TILE + (STATS_BYTES + 1023) / 1024 * 1024;
    // the streamed tiles the output GEMMs read (dq: K; dkv: Q, rho, dO), re-encoded in place
    static constexpr int CONV_BYTES = PASS == BWD_DQ ? STR_TILE : PASS == BWD_DKV ? N_STR * STR_TILE : 0;
    // a stage is held until its step's output GEMMs finish, late in the step, so
    // the ring needs three stages for the load to run under a whole step
    // (the dkv pass at d = 128 has room for two)
    static constexpr int NSTAGE = (D == 128) ? (PASS != BWD_DKV ? 3 : 2) : 4;
    static constexpr int STG_SLOT_BYTES = 32 * 128;   // per elementwise warp: 32 rows x 32 fp32
    static constexpr int OFF_RES = 0;
    static constexpr int OFF_STR = OFF_RES + N_RES * RES_TILE;
    static constexpr int OFF_STG = OFF_STR + NSTAGE * STAGE_BYTES;
    static constexpr int OFF_BAR = OFF_STG + EW_WARPS * STG_SLOT_BYTES;
    // res_full, res_empty, str_full[NSTAGE], str_empty[NSTAGE], srg_stage[NSTAGE], conv_done[NSTAGE],
    // srg_full, srg_free, ab_full, out_done, drain, pair[4] (statistics pass)
    static constexpr int NBARS = 2 + 4 * NSTAGE + 5 + 4;
    static constexpr int SMEM_USED = OFF_BAR + NBARS * 8 + 16;
    static constexpr int SMEM = SMEM_USED + 1024;
    static constexpr uint32_t TM_S = 0, TM_R = 64, TM_G = 128, TM_DS = 192, TM_DR = 224, TM_ACC0 = 256,
                              TM_ACC1 = 256 + D;
    static constexpr uint32_t TM_COLS = 512;
    static_assert(D == 64 || D == 128, "tcgen05 backward supports d in {64, 128}");
    static_assert(STAGE_BYTES % 1024 == 0 && OFF_STR % 1024 == 0 && OFF_STG % 1024 == 0, "1024-byte tiles");
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert((CONV_BYTES / 16) % CV_THREADS == 0, "re-encode splits evenly over its threads");
    // statistics pass: the pair merge of (m, l, C, A, E) per row, in the idle staging area
    static_assert(2 * 2 * ROWS * 5 * 4 <= EW_WARPS * STG_SLOT_BYTES, "merge area");
};

struct BwdTcParams {
    const float4* stats;   // per row (log2e lse, c, a, D), [BH][N]  (dq pass: read per row)
    float4* stats_out;     // the statistics pass writes them here
    int N;
    int BH;
    int n_rt;              // 128-row tiles per head
    int n_items;
    float scale;
    float scale_log2;      // scale * log2(e)
};

template <int D, bool PLX, int PASS>
__global__ void __launch_bounds__(BwdTcCfg<D, PLX, PASS>::THREADS, 1)
plx_bwd_tc_kernel(const __grid_constant__ CUtensorMap mapRes0, const __grid_constant__ CUtensorMap mapRes1,
                  const __grid_constant__ CUtensorMap mapRes2, const __grid_constant__ CUtensorMap mapStr0,
                  const __grid_constant__ CUtensorMap mapStr1, const __grid_constant__ CUtensorMap mapStr2,
                  const __grid_constant__ CUtensorMap mapStats, const __grid_constant__ CUtensorMap mapOut0,
                  const __grid_constant__ CUtensorMap mapOut1, const BwdTcParams p) {
    using Cfg = BwdTcCfg<D, PLX, PASS>;
    constexpr int ROWS = Cfg::ROWS, COLS = Cfg::COLS, NP = Cfg::NP, NSTAGE = Cfg::NSTAGE, HALF = Cfg::HALF;
    constexpr bool DQ = PASS == BWD_DQ;
    constexpr bool ST = PASS == BWD_STATS;
    constexpr bool QROWS = PASS != BWD_DKV;     // items are query tiles
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sRes = smem + Cfg::OFF_RES;
    uint8_t* sStr = smem + Cfg::OFF_STR;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    uint64_t* res_full = bars;
    uint64_t* res_empty = bars + 1;
    uint64_t* str_full = bars + 2;
    uint64_t* str_empty = str_full + NSTAGE;
    uint64_t* srg_stage = str_empty + NSTAGE;  // per stage: the S/R/G GEMMs reading it have completed
    uint64_t* conv_done = srg_stage + NSTAGE;  // per stage: its output-GEMM B tiles are fp16
    uint64_t* srg_full = conv_done + NSTAGE;   // S/R/G of the current step are in TMEM
    uint64_t* srg_free = srg_full + 1;         // every elementwise warp holds them in registers
    uint64_t* ab_full = srg_free + 1;          // ds/dr/wv of the current step are in TMEM
    uint64_t* out_done = ab_full + 1;          // the output GEMMs of the step have completed
    uint64_t* drain = out_done + 1;
    uint64_t* pair_bar = drain + 1;            // statistics pass: the two warps of a lane quadrant
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pair_bar + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, c = blockIdx.x;

    if (warp == 1) {
        tmem_alloc(tmem_slot, Cfg::TM_COLS);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        mbar_init(res_full, 1);
        mbar_init(res_empty, 1);
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&str_full[s], 1);
            mbar_init(&str_empty[s], 1);
            mbar_init(&srg_stage[s], 1);
            mbar_init(&conv_done[s], Cfg::CV_WARPS);
        }
        mbar_init(srg_full, 1);
        mbar_init(srg_free, Cfg::EW_WARPS);
        mbar_init(ab_full, Cfg::EW_WARPS);
        mbar_init(out_done, 1);
        mbar_init(drain, 1);
        for (int qd = 0; qd < 4; ++qd) mbar_init(&pair_bar[qd], 2);
        *abort_flag = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto fail = [&]() {
        atomicOr(&g_plx_status, PLX_DEV_ERR_TIMEOUT);
        *abort_flag = 1;
    };
    // item u: head bh and 128-row tile rt.  The dq pass runs query tiles
    // longest-first (descending), the dkv pass key tiles longest-first (ascending).
    auto item = [&](int u, int& bh, int& r0, int& n_steps, int& s0) {
        const int t = u / p.BH;
        bh = u % p.BH;
        const int rt = QROWS ? p.n_rt - 1 - t : t;
        r0 = rt * ROWS;
        if (QROWS) {
            s0 = 0;                                                  // keys 0 .. min(N, r0 + 128) - 1
            n_steps = (min(p.N, r0 + ROWS) + COLS - 1) / COLS;
        } else {
            s0 = r0;                                                 // queries r0 .. N - 1
            n_steps = (p.N - r0 + COLS - 1) / COLS;
        }
    };

    if (warp == 0) {
        // ===================================================== TMA producer
        if (lane == 0) {
            int nres = 0, nstr = 0;
            bool ok = true;
            for (int r = 0; ok; ++r) {
                const int u = snake_item(r, c, G);
                if (u >= p.n_items || *abort_flag) break;
                int bh, r0, n_steps, s0;
                item(u, bh, r0, n_steps, s0);
                if (nres > 0 && !mbar_wait(res_empty, (nres - 1) & 1)) { ok = false; break; }
                mbar_arrive_expect_tx(res_full, Cfg::N_RES * Cfg::RES_TILE);
                for (int pn = 0; pn < NP; ++pn) {
                    tma_load_3d(sRes + pn * Cfg::RES_PANEL, &mapRes0, res_full, pn * 64, r0, bh);
                    tma_load_3d(sRes + Cfg::RES_TILE + pn * Cfg::RES_PANEL, &mapRes1, res_full, pn * 64, r0, bh);
                    if (Cfg::N_RES > 2)
                        tma_load_3d(sRes + 2 * Cfg::RES_TILE + pn * Cfg::RES_PANEL, &mapRes2, res_full, pn * 64, r0,
                                    bh);
                }
                ++nres;
                for (int t = 0; t < n_steps; ++t) {
                    const int st = nstr % NSTAGE;
                    if (nstr >= NSTAGE && !mbar_wait(&str_empty[st], ((nstr / NSTAGE) - 1) & 1)) { ok = false; break; }
                    uint8_t* base = sStr + st * Cfg::STAGE_BYTES;
                    const int y = s0 + t * COLS;
                    mbar_arrive_expect_tx(&str_full[st], Cfg::N_STR * Cfg::STR_TILE + Cfg::STATS_BYTES);
                    for (int pn = 0; pn < NP; ++pn) {
                        tma_load_3d(base + pn * Cfg::STR_PANEL, &mapStr0, &str_full[st], pn * 64, y, bh);
                        tma_load_3d(base + Cfg::STR_TILE + pn * Cfg::STR_PANEL, &mapStr1, &str_full[st], pn * 64, y,
                                    bh);
                        if (Cfg::N_STR > 2)
                            tma_load_3d(base + 2 * Cfg::STR_TILE + pn * Cfg::STR_PANEL, &mapStr2, &str_full[st],
                                        pn * 64, y, bh);
                    }
                    if (PASS == BWD_DKV)
                        tma_load_3d(base + Cfg::N_STR * Cfg::STR_TILE, &mapStats, &str_full[st], 0, y, bh);
                    ++nstr;
                }
            }
            if (!ok) fail();
            // never leave with loads in flight into this CTA's shared memory
            for (int i = max(0, nstr - NSTAGE); i < nstr; ++i)
                if (!mbar_wait(&str_full[i % NSTAGE], (i / NSTAGE) & 1)) fail();
            if (nres > 0 && !mbar_wait(res_full, (nres - 1) & 1)) fail();
        }
    } else if (warp == 1) {
        // ===================================================== MMA issuer (whole warp)
        constexpr uint32_t ID_S = idesc_bf16_f32(128, COLS, false, false);
        constexpr uint32_t ID_OUT = idesc_f16_f32(128, D, false, true);
        const uint32_t sResA = smem_u32(sRes), sStrA = smem_u32(sStr);
        auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity));
        };
        // one GEMM over d: D[tmem] (+)= A_res B_str^T, both K-major
        auto gemm_rs = [&](uint32_t d_tmem, uint32_t a_base, uint32_t b_base) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t aoff = (kk >> 2) * Cfg::RES_PANEL + (kk & 3) * 32;
                const uint32_t boff = (kk >> 2) * Cfg::STR_PANEL + (kk & 3) * 32;
                mma_ss_warp(d_tmem, sdesc_sw128(a_base + aoff, 16, 1024), sdesc_sw128(b_base + boff, 16, 1024), ID_S,
                            kk > 0);
            }
        };
        // one output GEMM over the step's 64 columns: ACC (+)= A[tmem, bf16 pairs] B_str (MN-major).
        // Packed A: columns 16kk .. 16kk + 15 of the step at TMEM columns 8kk ..;
        // split A (wv over G): columns [32h, 32h + 32) at TMEM columns [32h, 32h + 16).
        auto gemm_out = [&](uint32_t acc_tmem, uint32_t a_tmem, uint32_t b_base, bool first_acc, bool split) {
#pragma unroll
            for (int kk = 0; kk < COLS / 16; ++kk) {
                const uint64_t bdesc = sdesc_sw128(b_base + kk * 16 * 128, Cfg::STR_PANEL, 1024);
                const uint32_t acol = split ? (kk >> 1) * 32 + (kk & 1) * 8 : kk * 8;
                mma_ts_warp(acc_tmem, a_tmem + acol, bdesc, ID_OUT, (first_acc && kk == 0) ? 0u : 1u);
            }
        };
        int nres = 0, g = 0;
        bool ok = true, prev_first = false;   // step g - 1 exists; was it the first of its item
        // the output GEMMs of step pg may start: ds/dr/wv stored by every
        // elementwise warp, and the stage's B tiles re-encoded to fp16
        auto out_ready = [&](int pg) -> bool {
            if (!wait_warp(ab_full, pg & 1)) return false;
            if (!wait_warp(&conv_done[pg % NSTAGE], (pg / NSTAGE) & 1)) return false;
            tc_fence_after();
            return true;
        };
        auto out_gemms = [&](int pg, bool first) -> bool {
            if (!out_ready(pg)) return false;
            const uint32_t base = sStrA + (pg % NSTAGE) * Cfg::STAGE_BYTES;
            if (DQ) {
                gemm_out(tmem + Cfg::TM_ACC0, tmem + Cfg::TM_DS, base, first, false);          // dQ += ds K
                if (PLX) gemm_out(tmem + Cfg::TM_ACC1, tmem + Cfg::TM_DR, base, first, false); // dRho += dr K
            }
            mma_commit_warp(&str_empty[pg % NSTAGE]);
            mma_commit_warp(out_done);
            return true;
        };
        for (int r = 0; ok; ++r) {
            const int u = snake_item(r, c, G);
            if (u >= p.n_items || __shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            int bh, r0, n_steps, s0;
            item(u, bh, r0, n_steps, s0);
            if (!wait_warp(res_full, nres & 1)) { ok = false; break; }
            tc_fence_after();
            for (int t = 0; t < n_steps; ++t, ++g) {
                const int st = g % NSTAGE;
                if (!wait_warp(&str_full[st], (g / NSTAGE) & 1)) { ok = false; break; }
                // S/R/G of the previous step are in the elementwise warps' registers
                if (g > 0 && !wait_warp(srg_free, (g - 1) & 1)) { ok = false; break; }
                tc_fence_after();
                const uint32_t base = sStrA + st * Cfg::STAGE_BYTES;
                if (ST) {
                    // the statistics pass: S, R, G only; the stage's one reader is done with them
                    gemm_rs(tmem + Cfg::TM_S, sResA, base);
                    if (PLX) gemm_rs(tmem + Cfg::TM_R, sResA + Cfg::RES_TILE, base);
                    gemm_rs(tmem + Cfg::TM_G, sResA + (Cfg::N_RES - 1) * Cfg::RES_TILE, base + Cfg::STR_TILE);
                    mma_commit_warp(srg_full);
                    mma_commit_warp(&str_empty[st]);
                    if (t == n_steps - 1) mma_commit_warp(res_empty);
                } else if (DQ) {
                    gemm_rs(tmem + Cfg::TM_S, sResA, base);                                    // S = Q K^T
                    if (PLX) gemm_rs(tmem + Cfg::TM_R, sResA + Cfg::RES_TILE, base);           // R = rho K^T
                    gemm_rs(tmem + Cfg::TM_G, sResA + (Cfg::N_RES - 1) * Cfg::RES_TILE, base + Cfg::STR_TILE);  // G = dO V^T
                    mma_commit_warp(srg_full);
                    mma_commit_warp(&srg_stage[st]);
                    if (t == n_steps - 1) mma_commit_warp(res_empty);
                    if (g > 0 && !out_gemms(g - 1, prev_first)) { ok = false; break; }
                } else {
                    gemm_rs(tmem + Cfg::TM_S, sResA, base);                                    // S^T = K Q^T
                    if (PLX) gemm_rs(tmem + Cfg::TM_R, sResA, base + Cfg::STR_TILE);           // R^T = K rho^T
                    if (g > 0) {
                        // dV_{g-1} reads wv_{g-1} from G's columns: before G_g overwrites them
                        if (!out_ready(g - 1)) { ok = false; break; }
                        const uint32_t pbase = sStrA + ((g - 1) % NSTAGE) * Cfg::STAGE_BYTES;
                        gemm_out(tmem + Cfg::TM_ACC0, tmem + Cfg::TM_G, pbase + (Cfg::N_STR - 1) * Cfg::STR_TILE,
                                 prev_first, true);                                             // dV += wv dO
                    }
                    gemm_rs(tmem + Cfg::TM_G, sResA + Cfg::RES_TILE, base + (Cfg::N_STR - 1) * Cfg::STR_TILE);  // G^T = V dO^T
                    mma_commit_warp(srg_full);
                    mma_commit_warp(&srg_stage[st]);
                    if (t == n_steps - 1) mma_commit_warp(res_empty);
                    if (g > 0) {
                        // step g - 1 was made ready above
                        const uint32_t pbase = sStrA + ((g - 1) % NSTAGE) * Cfg::STAGE_BYTES;
                        gemm_out(tmem + Cfg::TM_ACC1, tmem + Cfg::TM_DS, pbase, prev_first, false);  // dK += ds Q
                        if (PLX)
                            gemm_out(tmem + Cfg::TM_ACC1, tmem + Cfg::TM_DR, pbase + Cfg::STR_TILE, false, false);  // + dr rho
                        mma_commit_warp(&str_empty[(g - 1) % NSTAGE]);
                        mma_commit_warp(out_done);
                    }
                }
                prev_first = t == 0;
            }
            ++nres;
        }
        // the output GEMMs of the last step
        if (ok && g > 0 && !ST) {
            if (DQ) {
                ok = out_gemms(g - 1, prev_first);
            } else if (!out_ready(g - 1)) {
                ok = false;
            } else {
                const uint32_t pbase = sStrA + ((g - 1) % NSTAGE) * Cfg::STAGE_BYTES;
                gemm_out(tmem + Cfg::TM_ACC0, tmem + Cfg::TM_G, pbase + (Cfg::N_STR - 1) * Cfg::STR_TILE, prev_first,
                         true);
                gemm_out(tmem + Cfg::TM_ACC1, tmem + Cfg::TM_DS, pbase, prev_first, false);
                if (PLX) gemm_out(tmem + Cfg::TM_ACC1, tmem + Cfg::TM_DR, pbase + Cfg::STR_TILE, false, false);
                mma_commit_warp(&str_empty[(g - 1) % NSTAGE]);
                mma_commit_warp(out_done);
            }
        }
        if (!ok) fail();
        mma_commit_warp(drain);
        if (!wait_warp(drain, 0)) fail();
    } else if (warp >= 2 + Cfg::EW_WARPS) {
        // ===================================================== fp16 re-encode (warps 10..11)
        // After the S/R/G GEMMs of a step have read its streamed tiles (bf16),
        // the tiles the output GEMMs read are turned into fp16 in place
        // (element-wise, so the 128-byte swizzle is unchanged): the output
        // GEMMs take fp16 ds, dr, wv, and both operands of a kind::f16 MMA have
        // one type.  Per-stage barriers: this warp can never trail a stage by
        // more than one use, since the stage is reloaded only after its output
        // GEMMs, which wait for this warp.
        const int tcv = (warp - 2 - Cfg::EW_WARPS) * 32 + lane;
        auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity));
        };
        int g = 0;
        bool ok = !ST;          // the statistics pass has no output GEMMs: nothing to re-encode
        for (int r = 0; ok; ++r) {
            const int u = snake_item(r, c, G);
            if (u >= p.n_items || __shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            int bh, r0, n_steps, s0;
            item(u, bh, r0, n_steps, s0);
            for (int t = 0; t < n_steps; ++t, ++g) {
                const int st = g % NSTAGE;
                const uint32_t par = (g / NSTAGE) & 1;
                // the TMA data of the stage is visible to this warp, and the GEMMs
                // that read it as bf16 have completed
                if (!wait_warp(&str_full[st], par) || !wait_warp(&srg_stage[st], par)) { ok = false; break; }
                tc_fence_after();
                uint4* tile = reinterpret_cast<uint4*>(sStr + st * Cfg::STAGE_BYTES);
#pragma unroll 4
                for (int k = 0; k < Cfg::CONV_BYTES / 16 / Cfg::CV_THREADS; ++k) {
                    uint4 w = tile[tcv + Cfg::CV_THREADS * k];
                    w.x = bf16x2_to_f16x2(w.x);
                    w.y = bf16x2_to_f16x2(w.y);
                    w.z = bf16x2_to_f16x2(w.z);
                    w.w = bf16x2_to_f16x2(w.w);
                    tile[tcv + Cfg::CV_THREADS * k] = w;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&conv_done[st]);
            }
        }
        if (!ok && !ST) fail();
    } else if (ST) {
        // ===================================================== statistics (warps 2..9)
        // Per query row, with the weights the other passes use, w_ij = 2^(scale
        // log2e s_ij - log2e lse_i):  c_i = sum_j w_ij r_ij,  a_i = sum_j w_ij G_ij
        // (= dO_i . vbar_i),  e_i = sum_j w_ij r_ij G_ij,  and
        // D_i = sum_j w_ij ((1 + c_i - r_ij) G_ij + a_i r_ij) = (1 + 2 c_i) a_i - e_i.
        // Each warp keeps an online state (m, l, C, A, E) over its 32 keys of every
        // tile in fp32.  No rounded weights: the statistics must match the weights
        // of the dq and dkv passes, or D_i - sum_j w_ij (...) no longer cancels.
        // The pair merges its two states once per item.
        const int ew = warp - 2;
        const int quad = warp & 3;
        const int half = ew >> 2;
        const int row = quad * 32 + lane;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        float* xs = reinterpret_cast<float*>(smem + Cfg::OFF_STG);   // [2 items][2 halves][5][ROWS]
        auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity));
        };
        int g = 0, items = 0;
        bool ok = true;
        for (int r = 0; ok; ++r) {
            const int u = snake_item(r, c, G);
            if (u >= p.n_items || __shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            int bh, r0, n_steps, s0;
            item(u, bh, r0, n_steps, s0);
            const int rw = r0 + row;
            float m = -INFINITY, l = 0.f, C = 0.f, A = 0.f, E = 0.f;
            for (int t = 0; t < n_steps; ++t, ++g) {
                if (!wait_warp(srg_full, g & 1)) { ok = false; break; }
                tc_fence_after();
                uint32_t sraw[HALF], rraw[HALF], graw[HALF];
                tmem_ld32x32b_x32_nowait(lane_addr + Cfg::TM_S + half * HALF, sraw);
                if constexpr (PLX) tmem_ld32x32b_x32_nowait(lane_addr + Cfg::TM_R + half * HALF, rraw);
                tmem_ld32x32b_x32_nowait(lane_addr + Cfg::TM_G + half * HALF, graw);
                tmem_ld_wait(sraw);
                if constexpr (PLX) tmem_ld_wait(rraw);
                tmem_ld_wait(graw);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(srg_free);
                const int cbase = s0 + t * COLS + half * HALF;
                float tl[HALF];
                float mloc = -INFINITY;
#pragma unroll
                for (int cc = 0; cc < HALF; ++cc) {
                    tl[cc] = cbase + cc <= rw ? __uint_as_float(sraw[cc]) * p.scale_log2 : -INFINITY;
                    mloc = fmaxf(mloc, tl[cc]);
                }
                if (mloc == -INFINITY) continue;          // every key of this warp masked
                if (mloc > m) {
                    const float f = fast_exp2(m - mloc);  // 0 while m is still -inf
                    l *= f;
                    C *= f;
                    A *= f;
                    E *= f;
                    m = mloc;
                }
#pragma unroll
                for (int cc = 0; cc < HALF; ++cc) {
                    const float pw = fast_exp2(tl[cc] - m);     // 0 where masked
                    const float gg = __uint_as_float(graw[cc]);
                    l += pw;
                    A = fmaf(pw, gg, A);
                    if constexpr (PLX) {
                        const float pr = pw * __uint_as_float(rraw[cc]);
                        C += pr;
                        E = fmaf(pr, gg, E);
                    }
                }
            }
            if (!ok) break;
            // merge the pair's states through shared memory (slots alternate by item,
            // so a slot is rewritten only after the partner passed the next merge)
            float* xe = xs + (items & 1) * (2 * 5 * ROWS);
            float* mine = xe + half * 5 * ROWS;
            mine[0 * ROWS + row] = m;
            mine[1 * ROWS + row] = l;
            mine[2 * ROWS + row] = C;
            mine[3 * ROWS + row] = A;
            mine[4 * ROWS + row] = E;
            __syncwarp();
            if (lane == 0) mbar_arrive(&pair_bar[quad]);
            if (!wait_warp(&pair_bar[quad], items & 1)) { ok = false; break; }
            const float* other = xe + (1 - half) * 5 * ROWS;
            const float mo = other[row];
            const float M = fmaxf(m, mo);
            const float f0 = m == -INFINITY ? 0.f : fast_exp2(m - M);
            const float f1 = mo == -INFINITY ? 0.f : fast_exp2(mo - M);
            const float L = l * f0 + other[1 * ROWS + row] * f1;
            const float ci = (C * f0 + other[2 * ROWS + row] * f1) / L;
            const float ai = (A * f0 + other[3 * ROWS + row] * f1) / L;
            const float ei = (E * f0 + other[4 * ROWS + row] * f1) / L;
            if (half == 0 && rw < p.N && in_bounds(bh < p.BH))
                p.stats_out[static_cast<size_t>(bh) * p.N + rw] =
                    make_float4(M + __log2f(L), ci, ai, fmaf(2.f * ci, ai, ai) - ei);
            ++items;
        }
        if (!ok) fail();
    } else {
        // ===================================================== elementwise + epilogue (warps 2..9)
        const int ew = warp - 2;                // 0..7
        const int quad = warp & 3;              // TMEM lane quadrant
        const int half = ew >> 2;               // streamed columns [32 half, 32 half + 32)
        const int row = quad * 32 + lane;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        uint8_t* stg = smem + Cfg::OFF_STG + ew * Cfg::STG_SLOT_BYTES;
        auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity));
        };
        // one 32 x 32 fp32 block of an accumulator to global memory (through this
        // warp's staging slot in the output map's 128-byte swizzle, and a TMA store)
        auto store_block = [&](const CUtensorMap* map, uint32_t acc_col, int x, int y, int z, float mul) {
            uint32_t v32[32];
            tmem_ld32x32b_x32(lane_addr + acc_col, v32);
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
#pragma unroll
            for (int u4 = 0; u4 < 8; ++u4)
                *reinterpret_cast<uint4*>(stg + lane * 128 + ((u4 ^ (lane & 7)) << 4)) =
                    make_uint4(__float_as_uint(__uint_as_float(v32[4 * u4]) * mul),
                               __float_as_uint(__uint_as_float(v32[4 * u4 + 1]) * mul),
                               __float_as_uint(__uint_as_float(v32[4 * u4 + 2]) * mul),
                               __float_as_uint(__uint_as_float(v32[4 * u4 + 3]) * mul));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_3d(map, stg, x, y, z);
                bulk_commit_group();
            }
        };
        int g = 0;
        bool ok = true;
        for (int r = 0; ok; ++r) {
            const int u = snake_item(r, c, G);
            if (u >= p.n_items || __shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            int bh, r0, n_steps, s0;
            item(u, bh, r0, n_steps, s0);
            const int rw = r0 + row;                     // this thread's row: query (dq) or key (dkv)
            // dq pass: this row's statistics (rows past N take none: every weight is masked)
            float4 rs = make_float4(0.f, 0.f, 0.f, 0.f);
            if (DQ && rw < p.N) rs = p.stats[static_cast<size_t>(bh) * p.N + rw];
            for (int t = 0; t < n_steps; ++t, ++g) {
                if (!wait_warp(srg_full, g & 1)) { ok = false; break; }
                tc_fence_after();
                uint32_t sraw[HALF], rraw[HALF], graw[HALF];
                tmem_ld32x32b_x32_nowait(lane_addr + Cfg::TM_S + half * HALF, sraw);
                if constexpr (PLX) tmem_ld32x32b_x32_nowait(lane_addr + Cfg::TM_R + half * HALF, rraw);
                tmem_ld32x32b_x32_nowait(lane_addr + Cfg::TM_G + half * HALF, graw);
                tmem_ld_wait(sraw);
                if constexpr (PLX) tmem_ld_wait(rraw);
                tmem_ld_wait(graw);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(srg_free);
                const int cbase = s0 + t * COLS + half * HALF;   // first streamed index of this warp
                const float4* cst = nullptr;
                if (!DQ) {
                    // the queries' statistics of this step, landed with the stage
                    const int st = g % NSTAGE;
                    if (!wait_warp(&str_full[st], (g / NSTAGE) & 1)) { ok = false; break; }
                    cst = reinterpret_cast<const float4*>(sStr + st * Cfg::STAGE_BYTES + Cfg::N_STR * Cfg::STR_TILE) +
                          half * HALF;
                }
                uint32_t pds[HALF / 2], pdr[HALF / 2], pwv[HALF / 2];
#pragma unroll
                for (int cc = 0; cc < HALF; cc += 2) {
                    float ds2[2], dr2[2], wv2[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int col = cbase + cc + e;
                        // (log2e lse, c, a, D) of the query in this pair
                        const float4 qs = DQ ? rs : cst[cc + e];
                        const bool live = DQ ? (col <= rw && rw < p.N) : (col >= rw && col < p.N);
                        const float s = __uint_as_float(sraw[cc + e]);
                        const float rr = PLX ? __uint_as_float(rraw[cc + e]) : 0.f;
                        const float gg = __uint_as_float(graw[cc + e]);
                        const float w = live ? fast_exp2(fmaf(s, p.scale_log2, -qs.x)) : 0.f;
                        const float t1 = PLX ? (1.f + qs.y - rr) : 1.f;
                        ds2[e] = w * (PLX ? fmaf(t1, gg, fmaf(qs.z, rr, -qs.w)) : (gg - qs.w)) * p.scale;
                        dr2[e] = w * (qs.z - gg);
                        wv2[e] = w * t1;
                    }
                    pds[cc / 2] = pack_f16x2(ds2[0], ds2[1]);
                    pdr[cc / 2] = pack_f16x2(dr2[0], dr2[1]);
                    pwv[cc / 2] = pack_f16x2(wv2[0], wv2[1]);
                }
                // ds/dr of the previous step have been read by its output GEMMs
                if (g > 0 && !wait_warp(out_done, (g - 1) & 1)) { ok = false; break; }
                tc_fence_after();
                tmem_st32x32b_x16(lane_addr + Cfg::TM_DS + half * (HALF / 2), pds);
                if constexpr (PLX) tmem_st32x32b_x16(lane_addr + Cfg::TM_DR + half * (HALF / 2), pdr);
                // dkv: wv over the first half of the G columns this warp read itself
                // (G of this step is in its registers; dV of the previous step ran
                // before this step's G GEMM), so it never writes what its partner reads
                if (!DQ) tmem_st32x32b_x16(lane_addr + Cfg::TM_G + half * HALF, pwv);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(ab_full);
            }
            if (!ok) break;
            // ---- epilogue: the item's accumulators, once its last output GEMMs are done
            if (!wait_warp(out_done, (g - 1) & 1)) { ok = false; break; }
            tc_fence_after();
            if (r0 + quad * 32 < p.N) {
                const int y = r0 + quad * 32;
#pragma unroll 1
                for (int cb = half * (D / 2); cb < (half + 1) * (D / 2); cb += 32) {
                    if (DQ) {
                        store_block(&mapOut0, Cfg::TM_ACC0 + cb, cb, y, bh, 1.f);                 // dq (scale in ds)
                        if (PLX) store_block(&mapOut1, Cfg::TM_ACC1 + cb, cb, y, bh, 1.f);        // drho
                    } else {
                        store_block(&mapOut0, Cfg::TM_ACC0 + cb, cb, y, bh, 1.f);                 // dv
                        store_block(&mapOut1, Cfg::TM_ACC1 + cb, cb, y, bh, 1.f);                 // dk
                    }
                }
            }
            tc_fence_before();
        }
        if (!ok) fail();
        // no TMEM store of this warp is still pending, and the output stores have finished
        tmem_st_wait();
        if (lane == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::TM_COLS);
    }
}

// ---------------------------------------------------------------------------
// The row statistics from the training forward's saved values (plx_bwd_saved),
// instead of the statistics pass: with vbar_i = O_i / l_i and c_i from the
// forward, a_i = dO_i.vbar_i and D_i = dO_i.o_i + c_i a_i (the same identities
// as the header above: e_i = dO_i.u_i with u_i = (1 + c_i) vbar_i - o_i).  For
// softmax attention (no rho) vbar_i = o_i and c_i = 0.  Each warp takes two
// rows and issues both rows' loads before either reduction; each lane holds D/32
// consecutive elements of a row (coalesced 16- and 8-byte loads).
struct BwdPrepParams {
    const float* lse;      // natural-log lse per row, [rows]
    const float* c;        // c_i per row, or nullptr (softmax attention)
    const float* vbar;     // fp32 [rows][D], or nullptr (softmax attention: vbar = o)
    const void* out;       // the forward's o, fp32 or bf16 [rows][D]
    const uint16_t* dout;  // bf16 [rows][D]
    float4* stats;         // (log2e lse, c, a, D) per row
    long long rows;
    int out_f32;
};
constexpr int BWD_PREP_WARPS = 8;
constexpr int BWD_PREP_ROWS_PER_WARP = 2;   // both rows' loads in flight before either reduction
constexpr int BWD_PREP_ROWS_PER_BLOCK = BWD_PREP_WARPS * BWD_PREP_ROWS_PER_WARP;

template <int D>
__device__ __forceinline__ void load_bf16_vec(const uint16_t* src, float (&x)[D / 32]) {
    if constexpr (D == 128) {
        const uint2 w = *reinterpret_cast<const uint2*>(src);
        x[0] = bf16x2_lo(w.x); x[1] = bf16x2_hi(w.x); x[2] = bf16x2_lo(w.y); x[3] = bf16x2_hi(w.y);
    } else {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(src);
        x[0] = bf16x2_lo(w); x[1] = bf16x2_hi(w);
    }
}
template <int D>
__device__ __forceinline__ void load_f32_vec(const float* src, float (&x)[D / 32]) {
    if constexpr (D == 128) {
        const float4 w = *reinterpret_cast<const float4*>(src);
        x[0] = w.x; x[1] = w.y; x[2] = w.z; x[3] = w.w;
    } else {
        const float2 w = *reinterpret_cast<const float2*>(src);
        x[0] = w.x; x[1] = w.y;
    }
}

template <int D>
__global__ void __launch_bounds__(BWD_PREP_WARPS * 32)
plx_bwd_prep_kernel(const BwdPrepParams p) {
    constexpr int E = D / 32, R = BWD_PREP_ROWS_PER_WARP;
    const int lane = threadIdx.x & 31;
    const long long row0 = (static_cast<long long>(blockIdx.x) * BWD_PREP_WARPS + (threadIdx.x >> 5)) * R;
    float g[R][E], o[R][E], vb[R][E];
#pragma unroll
    for (int i = 0; i < R; ++i) {
        if (row0 + i >= p.rows) continue;
        const size_t base = static_cast<size_t>(row0 + i) * D + lane * E;
        load_bf16_vec<D>(p.dout + base, g[i]);
        if (p.out_f32)
            load_f32_vec<D>(static_cast<const float*>(p.out) + base, o[i]);
        else
            load_bf16_vec<D>(static_cast<const uint16_t*>(p.out) + base, o[i]);
        if (p.vbar) {
            load_f32_vec<D>(p.vbar + base, vb[i]);
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) vb[i][e] = o[i][e];
        }
    }
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const long long row = row0 + i;
        if (row >= p.rows) break;
        float a = 0.f, od = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            a = fmaf(g[i][e], vb[i][e], a);
            od = fmaf(g[i][e], o[i][e], od);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            a += __shfl_xor_sync(0xffffffffu, a, off);
            od += __shfl_xor_sync(0xffffffffu, od, off);
        }
        if (lane == 0) {
            const float ci = p.c ? p.c[row] : 0.f;
            p.stats[row] = make_float4(p.lse[row] * 1.4426950408889634f, ci, a, fmaf(ci, a, od));
        }
    }
}

}  // namespace plx
