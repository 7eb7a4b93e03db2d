// lla_f32.cuh -- plx_lla_f32: local linear attention with the solved probe,
// in fp32 on the CUDA cores.
//
// "Parallax: Parameterized Local Linear Attention for Language Modeling"
// introduces Parallax as a learned replacement for local linear attention
// (LLA), whose probe is the solution of a per-token linear system found by
// conjugate gradients (zhichai.net section 1.2; gist.science, "Enunciato del
// Problema").  For query i of one head (causal prefix j <= i):
//
//   w_ij = softmax_j(scale q_i . k_j),  kbar_i = sum_j w_ij k_j
//   (Sigma_KK^(i) + lambda I) rho_i = mu_i,   mu_i = kbar_i - q_i
//   Sigma_KK^(i) p = sum_j w_ij ((k_j - kbar_i) . p) (k_j - kbar_i)
//                  = sum_j w_ij ((k_j . p) - (kbar_i . p)) k_j      (since sum_j w_ij = 1)
//   o_i = vbar_i - Sigma_KV^(i) rho_i           (Parallax's output formula)
//
// The library runs it as a sequence of launches on one stream:
//   1. plx_fwd_f32_kernel<., false> with v := k: kbar_i and lse_i;
//   2. plx_lla_init_kernel: x = 0, r = p = mu, rs = rs0 = mu . mu;
//   3. max_iters conjugate-gradient steps, one launch each: Sigma_KK p formed
//      by streaming the keys once per block of rows (weights from the stored
//      lse, no online rescaling), the update done in registers; a row stops
//      once r . r <= tol^2 rs0 (or when p . Ap <= 0).  d = 64, 128:
//      plx_lla_cg_gemm_kernel (two block-level GEMMs per key tile, 64 rows a
//      block); other d: plx_lla_cg_step_kernel (4 rows a warp);
//   4. plx_lla_out_kernel: o from Parallax's output formula with rho := x,
//      in centred form.
// The pages warn that the solve is unstable in low precision; every step
// here is fp32.  With the weights kept (d = 64, 128, N % 4 == 0), the steps
// after the first run on the tensor cores instead (lla_tc.cuh), each product
// split in tf32 to stay at fp32-level rounding.
#pragma once
#include <type_traits>
#include "bwd_f32.cuh"   // warp_sum
#include "status.cuh"

namespace plx {

struct LlaParams {
    const float* q;      // [BH][N][d]
    const float* k;      // [BH][N][d]
    const float* kbar;   // [BH][N][d]
    const float* lse;    // [BH][N] (natural log)
    float* x;            // [BH][N][d] the probe iterate
    float* r;            // [BH][N][d] residual
    float* p;            // [BH][N][d] search direction
    float* rs;           // [BH][N] r . r (0 once the row has stopped)
    float* rs0;          // [BH][N] mu . mu
    int* steps;          // [BH][N] steps taken
    int N;
    float scale;
    float lambda;
    float tol2;          // tol^2
    // [BH][N][N] fp32: the CG steps' softmax weights w_ij = exp(s_ij - lse_i),
    // j <= i, kept from the first step, which forms them from the scores the
    // kbar pass stored there (nullptr: every step recomputes them)
    float* wts;
};

constexpr int LLA_WARPS = 4;
constexpr int LLA_ROWS_PER_BLOCK = 16;

template <int DPL>
__global__ void __launch_bounds__(LLA_WARPS * 32) plx_lla_init_kernel(const LlaParams p) {
    constexpr int D = DPL * 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t bh = blockIdx.y;
    for (int rr = warp; rr < LLA_ROWS_PER_BLOCK; rr += LLA_WARPS) {
        const int i = blockIdx.x * LLA_ROWS_PER_BLOCK + rr;
        if (i >= p.N) break;
        const size_t row = bh * p.N + i;
        const size_t o = row * D;
        float part = 0.f;
#pragma unroll
        for (int t = 0; t < DPL; ++t) {
            const float mu = p.kbar[o + lane + 32 * t] - p.q[o + lane + 32 * t];
            p.x[o + lane + 32 * t] = 0.f;
            p.r[o + lane + 32 * t] = mu;
            p.p[o + lane + 32 * t] = mu;
            part = fmaf(mu, mu, part);
        }
        const float rs = warp_sum(part);
        if (lane == 0) {
            p.rs[row] = rs;
            p.rs0[row] = rs;
            p.steps[row] = 0;
        }
    }
}

// lane L of a warp owns the DPL contiguous dims L*DPL .. L*DPL + DPL - 1 of
// every vector, so one key row is one 16-byte load per lane when DPL = 4
template <int DPL>
__device__ __forceinline__ void load_own(const float* row, int lane, float (&f)[DPL]) {
    const float* src = row + lane * DPL;
    if constexpr (DPL % 4 == 0) {
#pragma unroll
        for (int t = 0; t < DPL; t += 4) {
            const float4 x = *reinterpret_cast<const float4*>(src + t);
            f[t] = x.x;
            f[t + 1] = x.y;
            f[t + 2] = x.z;
            f[t + 3] = x.w;
        }
    } else if constexpr (DPL % 2 == 0) {
#pragma unroll
        for (int t = 0; t < DPL; t += 2) {
            const float2 x = *reinterpret_cast<const float2*>(src + t);
            f[t] = x.x;
            f[t + 1] = x.y;
        }
    } else {
#pragma unroll
        for (int t = 0; t < DPL; ++t) f[t] = src[t];
    }
}

// Sums 8 values over the warp and leaves the full sum of value (lane >> 2) & 7
// in each lane: lane masks 16, 8, 4 each halve the values a lane carries
// (it keeps one half and adds its partner's copy of that half), masks 2 and 1
// finish the single remaining sum.  9 shuffles instead of 40.
__device__ __forceinline__ float reduce_scatter8(const float (&a)[8], int lane) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float b[4], c[2];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        const float send = b4 ? a[x] : a[x + 4];
        const float keep = b4 ? a[x + 4] : a[x];
        b[x] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int x = 0; x < 2; ++x) {
        const float send = b3 ? b[x] : b[x + 2];
        const float keep = b3 ? b[x + 2] : b[x];
        c[x] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    const float send = b2 ? c[0] : c[1];
    const float keep = b2 ? c[1] : c[0];
    float val = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    val += __shfl_xor_sync(0xffffffffu, val, 2);
    val += __shfl_xor_sync(0xffffffffu, val, 1);
    return val;
}

// Keys per shared-memory tile of the CG step (16 KB per tile at d <= 128).
template <int DPL>
struct LlaTile {
    static constexpr int TK = DPL <= 4 ? 32 : 16;
    static constexpr int FLOATS = TK * DPL * 32;
    static constexpr int SMEM = 2 * FLOATS * 4 + 64;     // two tiles + 2 mbarriers + flag
};

// One conjugate-gradient step for 4 consecutive rows per warp, 16 rows per
// block.  The block's keys 0 .. i_b + 15 stream through two shared-memory
// tiles of TK keys: thread 0 issues one 1-D bulk copy per tile (the keys of a
// head are contiguous), the copy of tile t + 1 overlapping the work on tile
// t, and every wait on a copy is bounded.  Per key j the warp needs 8 dot
// products (q_r . k_j and p_r . k_j of its 4 rows): reduce_scatter8 leaves s
// of row (L >> 3) & 3 in the lanes L with bit 2 clear and its p . k in the
// lanes with bit 2 set; one exchange pairs them, those lanes form
// g = w (p.k - kbar.p), and four broadcasts hand every lane the 4 rows' g.
template <int DPL>
__global__ void __launch_bounds__(LLA_WARPS * 32) plx_lla_cg_step_kernel(const LlaParams p) {
    constexpr int D = DPL * 32;
    constexpr int RW = LLA_ROWS_PER_BLOCK / LLA_WARPS;   // rows per warp
    constexpr int TK = LlaTile<DPL>::TK;
    static_assert(RW == 4, "the butterfly is written for 4 rows per warp");
    extern __shared__ __align__(128) float lla_smem[];
    float* tile0 = lla_smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(lla_smem + 2 * LlaTile<DPL>::FLOATS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(full + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t bh = blockIdx.y;
    const float* K = p.k + bh * p.N * D;
    const int ib = blockIdx.x * LLA_ROWS_PER_BLOCK;
    const int i0 = ib + warp * RW;

    bool act[RW];
    float rs[RW], qv[RW][DPL], pv[RW][DPL], U[RW][DPL], kp[RW], lse[RW];
    bool any = false;
#pragma unroll
    for (int r = 0; r < RW; ++r) {
        const int i = i0 + r;
        const size_t row = bh * p.N + (i < p.N ? i : ib);
        rs[r] = p.rs[row];
        act[r] = i < p.N && rs[r] > p.tol2 * p.rs0[row];
        any |= act[r];
    }
    // a block whose rows have all stopped returns before it reads anything else
    if (!__syncthreads_or(any)) return;
#pragma unroll
    for (int r = 0; r < RW; ++r) {
        const int i = i0 + r;
        const size_t row = bh * p.N + (i < p.N ? i : ib);
        lse[r] = p.lse[row];
        float kb[DPL];
        load_own<DPL>(p.q + row * D, lane, qv[r]);
        load_own<DPL>(p.p + row * D, lane, pv[r]);
        load_own<DPL>(p.kbar + row * D, lane, kb);
        float part = 0.f;
#pragma unroll
        for (int t = 0; t < DPL; ++t) {
            qv[r][t] *= p.scale;
            part = fmaf(kb[t], pv[r][t], part);
            U[r][t] = 0.f;
        }
        kp[r] = warp_sum(part);
    }
    if (threadIdx.x == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const int kmax = min(ib + LLA_ROWS_PER_BLOCK, p.N) - 1;   // last key the block needs
    const int n_tiles = kmax / TK + 1;
    auto issue = [&](int t) {
        const int j0 = t * TK;
        const int nk = min(TK, kmax + 1 - j0);
        const uint32_t bytes = static_cast<uint32_t>(nk) * D * 4;
        if (in_bounds(nk > 0 && j0 + nk <= p.N)) {
            mbar_arrive_expect_tx(&full[t & 1], bytes);
            bulk_g2s(tile0 + (t & 1) * LlaTile<DPL>::FLOATS, K + static_cast<size_t>(j0) * D, bytes, &full[t & 1]);
        } else {
            mbar_arrive(&full[t & 1]);         // debug build: the copy is skipped, the phase still completes
        }
    };
    if (threadIdx.x == 0) issue(0);

    // this lane's row in the butterfly (the row whose s / p.k it ends up holding)
    const int my = (lane >> 3) & 3;
    float my_lse = lse[0], my_kp = kp[0];
    bool my_act = act[0];
#pragma unroll
    for (int r = 1; r < RW; ++r)
        if (my == r) {
            my_lse = lse[r];
            my_kp = kp[r];
            my_act = act[r];
        }
    const bool b2 = lane & 4;
    const bool warp_any = __any_sync(0xffffffffu, any);
    int last_issued = 0;

    for (int t = 0; t < n_tiles; ++t) {
        if (threadIdx.x == 0 && t + 1 < n_tiles) {        // the other tile was released at the last barrier
            issue(t + 1);
            last_issued = t + 1;
        }
        if (!mbar_wait(&full[t & 1], (t >> 1) & 1)) {
            atomicOr(&g_plx_status, PLX_DEV_ERR_TIMEOUT);
            *abort_flag = 1;
        }
        const float* tk = tile0 + (t & 1) * LlaTile<DPL>::FLOATS;
        // keys past the warp's last row are not needed, and keys past kmax were not copied
        const int j_end = min(min(t * TK + TK, i0 + RW), kmax + 1);
        if (warp_any && !*abort_flag) {
#pragma unroll 2
            for (int j = t * TK; j < j_end; ++j) {
                float kf[DPL];
                load_own<DPL>(tk + (j - t * TK) * D, lane, kf);
                float a[2 * RW];                            // a[2r] = s part of row r, a[2r+1] = p.k part
#pragma unroll
                for (int r = 0; r < RW; ++r) {
                    float sd = 0.f, rd = 0.f;
#pragma unroll
                    for (int x = 0; x < DPL; ++x) {
                        sd = fmaf(qv[r][x], kf[x], sd);
                        rd = fmaf(pv[r][x], kf[x], rd);
                    }
                    a[2 * r] = sd;
                    a[2 * r + 1] = rd;
                }
                const float val = reduce_scatter8(a, lane);
                // lanes with bit 2 clear hold s of row `my`, their partner (lane ^ 4) its p . k
                const float other = __shfl_xor_sync(0xffffffffu, val, 4);
                float g = 0.f;
                if (!b2 && my_act && j <= i0 + my) g = expf(val - my_lse) * (other - my_kp);
                float gr[RW];
#pragma unroll
                for (int r = 0; r < RW; ++r) gr[r] = __shfl_sync(0xffffffffu, g, 8 * r);
#pragma unroll
                for (int r = 0; r < RW; ++r)
#pragma unroll
                    for (int x = 0; x < DPL; ++x) U[r][x] = fmaf(gr[r], kf[x], U[r][x]);
            }
        }
        __syncthreads();                                  // tile t is free for the copy of tile t + 2
        if (*abort_flag) break;
    }
    // no copy may still be in flight when the block exits (only after an abort)
    if (threadIdx.x == 0 && *abort_flag) mbar_wait(&full[last_issued & 1], (last_issued >> 1) & 1);
    if (*abort_flag) return;

    // Ap = Sigma_KK p + lambda p, then one conjugate-gradient step per active row
#pragma unroll
    for (int r = 0; r < RW; ++r) {
        if (!act[r]) continue;                              // warp-uniform
        const size_t row = bh * p.N + i0 + r;
        float pap = 0.f;
#pragma unroll
        for (int t = 0; t < DPL; ++t) {
            U[r][t] = fmaf(p.lambda, pv[r][t], U[r][t]);
            pap = fmaf(pv[r][t], U[r][t], pap);
        }
        pap = warp_sum(pap);
        if (!(pap > 0.f)) {                                 // breakdown: stop the row
            if (lane == 0) p.rs[row] = 0.f;
            continue;
        }
        const float alpha = rs[r] / pap;
        float xv[DPL], rv[DPL];
        load_own<DPL>(p.x + row * D, lane, xv);
        load_own<DPL>(p.r + row * D, lane, rv);
        float rn = 0.f;
#pragma unroll
        for (int t = 0; t < DPL; ++t) {
            xv[t] = fmaf(alpha, pv[r][t], xv[t]);
            rv[t] = fmaf(-alpha, U[r][t], rv[t]);
            rn = fmaf(rv[t], rv[t], rn);
        }
        rn = warp_sum(rn);
        const float beta = rn / rs[r];
        float* xo = p.x + row * D + lane * DPL;
        float* ro = p.r + row * D + lane * DPL;
        float* po = p.p + row * D + lane * DPL;
#pragma unroll
        for (int t = 0; t < DPL; ++t) {
            xo[t] = xv[t];
            ro[t] = rv[t];
            po[t] = fmaf(beta, pv[r][t], rv[t]);
        }
        if (lane == 0) {
            p.rs[row] = rn;
            p.steps[row] += 1;
        }
    }
}

// ---------------------------------------------------------------------------
// The CG step as two block-level SIMT GEMMs per key tile (d = 64 or 128).
// A block owns BM = 64 query rows i_b .. i_b + 63 and streams keys
// 0 .. i_b + 63 in tiles of BK = 32:
//   phase 1   [S; R] = [scale q; p] K^T   (128 stacked rows x 32 keys, K = d)
//             thread (rg, kg) holds rows {rg, rg + 32} of q and the same two
//             rows of p (stacked rows rg + 64, rg + 96) against keys
//             {kg, kg + 8, kg + 16, kg + 24}, so it forms
//             G = exp(s - lse) ((p.k) - (kbar.p)) for 2 rows x 4 keys in
//             registers and writes it to shared memory;
//   phase 2   U += G K                    (64 rows x d, K = 32 keys)
//             thread (rgrp, dgrp) accumulates rows {rgrp + 16 i} x dims
//             {dgrp * 4 + 64 h + e} in registers across all tiles.
// The key rows of a tile arrive by one 1-D bulk copy each into a row-padded
// buffer (row stride d + 4 floats), so 8 consecutive keys read at the same
// dims fall in 8 different bank groups.  Two tile buffers: the copy of tile
// t + 1 overlaps the work on tile t.  The CG update of a row reduces over the
// 16 threads (a half-warp) that hold its dims.
template <int D>
struct LlaGemmCfg {
    static constexpr int BM = 64, BK = 32, THREADS = 256;
    static constexpr int LD = D + 4;                      // padded row stride (floats)
    static constexpr int DG = D / 16;                     // phase-2 dims per thread
    static constexpr int OFF_STAGE = 0;                   // 2 x [BK][LD]
    static constexpr int OFF_QP = OFF_STAGE + 2 * BK * LD;   // [2 BM][LD]: scale q rows, then p rows
    static constexpr int GLD = BM + 4;                    // G row stride: key kk, row a at (a % 16) * 4 + a / 16
    static constexpr int OFF_G = OFF_QP + 2 * BM * LD;    // [BK][GLD]
    static constexpr int OFF_ROW = OFF_G + BK * GLD;      // lse, kp, rs [BM] each, act [BM] (int)
    static constexpr int OFF_BAR = OFF_ROW + 4 * BM;      // 2 mbarriers + abort flag
    static constexpr int SMEM = OFF_BAR * 4 + 32;
    static_assert(D == 64 || D == 128, "the block GEMM step is built for d in {64, 128}");
};

// WMODE 0: the step computes the weights w_ij from s_ij = scale q_i.k_j and
// lse_i; 3 (the first step with the weights kept): it reads the scores s_ij
// the kbar pass stored in p.wts, forms the weights and stores them over the
// scores (active rows), and computes only p.k_j, half of phase 1; 2 (the
// later steps): it reads the weights.  The weights do not depend on the
// iterate, and the kbar pass forms s_ij with the same products in the same
// order, so the three modes give the same bits.
template <int D, int WMODE = 0>
__global__ void __launch_bounds__(256) plx_lla_cg_gemm_kernel(const LlaParams p) {
    using Cfg = LlaGemmCfg<D>;
    constexpr int BM = Cfg::BM, BK = Cfg::BK, LD = Cfg::LD, DG = Cfg::DG, GLD = Cfg::GLD;
    extern __shared__ __align__(128) float lla_gsmem[];
    float* stage = lla_gsmem + Cfg::OFF_STAGE;
    float* QP = lla_gsmem + Cfg::OFF_QP;
    float* Gs = lla_gsmem + Cfg::OFF_G;
    float* s_lse = lla_gsmem + Cfg::OFF_ROW;
    float* s_kp = s_lse + BM;
    float* s_rs = s_kp + BM;
    int* s_act = reinterpret_cast<int*>(s_rs + BM);
    uint64_t* full = reinterpret_cast<uint64_t*>(lla_gsmem + Cfg::OFF_BAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(full + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t bh = blockIdx.y;
    const int ib = blockIdx.x * BM;
    const float* K = p.k + bh * p.N * D;

    // ---- prologue: row scalars first; a block whose rows have all stopped
    // returns before it reads anything else (late steps launch every block, and
    // most of them have nothing left to do)
    int any_local = 0;
    if (tid < BM) {
        const int i = ib + tid;
        int a = 0;
        float lse = 0.f, rs = 0.f;
        if (i < p.N) {
            const size_t row = bh * p.N + i;
            rs = p.rs[row];
            lse = p.lse[row];
            a = rs > p.tol2 * p.rs0[row] ? 1 : 0;
        }
        s_act[tid] = a;
        s_lse[tid] = lse;
        s_rs[tid] = rs;
        any_local = a;
    }
    if (!__syncthreads_or(any_local)) return;             // every row of the block has stopped
    // q (scaled) and p rows into shared memory
    for (int idx = tid; idx < 2 * BM * (D / 4); idx += Cfg::THREADS) {
        const int r = idx / (D / 4), c = idx % (D / 4);
        const int i = ib + (r & (BM - 1));
        if (WMODE >= 2 && r < BM) continue;              // q rows: the weights (or scores) are stored
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < p.N) {
            const size_t off = (bh * p.N + i) * D + c * 4;
            v = *reinterpret_cast<const float4*>((r < BM ? p.q : p.p) + off);
            if (r < BM) {
                v.x *= p.scale;
                v.y *= p.scale;
                v.z *= p.scale;
                v.w *= p.scale;
            }
        }
        *reinterpret_cast<float4*>(QP + r * LD + c * 4) = v;
    }
    // kbar . p per row: warp w takes rows w, w + 8, ...
    for (int r = warp; r < BM; r += Cfg::THREADS / 32) {
        const int i = ib + r;
        float part = 0.f;
        if (i < p.N) {
            const size_t off = (bh * p.N + i) * D;
            for (int x = lane; x < D; x += 32) part = fmaf(p.kbar[off + x], p.p[off + x], part);
        }
        part = warp_sum(part);
        if (lane == 0) s_kp[r] = part;
    }
    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const int kmax = min(ib + BM, p.N) - 1;
    const int n_tiles = kmax / BK + 1;
    auto issue = [&](int t) {                             // warp 0, all lanes
        const int j0 = t * BK;
        const int nk = min(BK, kmax + 1 - j0);
        if (!in_bounds(nk > 0 && j0 + nk <= p.N)) {      // nk, j0: the same in every lane
            if (lane == 0) mbar_arrive(&full[t & 1]);   // debug build: the copies are skipped
            return;
        }
        if (lane == 0) mbar_arrive_expect_tx(&full[t & 1], static_cast<uint32_t>(nk) * D * 4);
        __syncwarp();
        if (lane < nk)
            bulk_g2s(stage + (t & 1) * BK * LD + lane * LD, K + static_cast<size_t>(j0 + lane) * D, D * 4,
                     &full[t & 1]);
    };
    if (warp == 0) issue(0);

    // phase-1 and phase-2 thread coordinates
    const int rg = tid >> 3, kg = tid & 7;               // rows {rg, rg+32} (+ their p rows), keys kg + 8 jj
    // rows rgrp + 16 i; dims dgrp * 4 + 64 h + e: the 8 lanes of a quarter-warp read
    // 128 contiguous bytes of a key row, so phase 2's loads are free of bank conflicts
    const int rgrp = tid >> 4, dgrp = tid & 15;
    float U[4][DG];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int x = 0; x < DG; ++x) U[i][x] = 0.f;
    const float lse0 = s_lse[rg], lse1 = s_lse[rg + 32];
    const float kp0 = s_kp[rg], kp1 = s_kp[rg + 32];
    const bool act0 = s_act[rg] != 0, act1 = s_act[rg + 32] != 0;
    int last_issued = 0;

    for (int t = 0; t < n_tiles; ++t) {
        if (warp == 0 && t + 1 < n_tiles) {              // that buffer was released at the last barrier
            issue(t + 1);
            last_issued = t + 1;
        }
        if (!mbar_wait(&full[t & 1], (t >> 1) & 1)) {
            atomicOr(&g_plx_status, PLX_DEV_ERR_TIMEOUT);
            *abort_flag = 1;
        }
        const float* kt = stage + (t & 1) * BK * LD;
        const int j0 = t * BK;
        const int nk = min(BK, kmax + 1 - j0);
        // rows rg, rg + 32 of the block and their weight rows (WMODE 2, 3)
        const size_t wrow0 = (bh * p.N + ib + rg) * static_cast<size_t>(p.N);
        const size_t wrow1 = wrow0 + 32 * static_cast<size_t>(p.N);
        float wv[2][4];
        if constexpr (WMODE >= 2) {
            // the stored weights (or scores) of this tile, loaded ahead of phase 1's FMAs
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int kk = kg + 8 * jj, j = j0 + kk;
                wv[0][jj] = (kk < nk && act0 && j <= ib + rg) ? p.wts[wrow0 + j] : 0.f;
                wv[1][jj] = (kk < nk && act1 && j <= ib + rg + 32) ? p.wts[wrow1 + j] : 0.f;
            }
        }
        // phase 1: acc[m][jj], m = 0, 1: s of rows rg, rg+32; m = 2, 3: p.k of the same rows
        // (WMODE 2, 3: only m = 2, 3)
        constexpr int M0 = WMODE >= 2 ? 2 : 0;
        float acc[4][4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) acc[m][jj] = 0.f;
#pragma unroll 4
        for (int c = 0; c < D; c += 4) {
            float4 a[4], b[4];
#pragma unroll
            for (int m = M0; m < 4; ++m) a[m] = *reinterpret_cast<const float4*>(QP + (rg + 32 * m) * LD + c);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) b[jj] = *reinterpret_cast<const float4*>(kt + (kg + 8 * jj) * LD + c);
#pragma unroll
            for (int m = M0; m < 4; ++m)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    acc[m][jj] = fmaf(a[m].x, b[jj].x, acc[m][jj]);
                    acc[m][jj] = fmaf(a[m].y, b[jj].y, acc[m][jj]);
                    acc[m][jj] = fmaf(a[m].z, b[jj].z, acc[m][jj]);
                    acc[m][jj] = fmaf(a[m].w, b[jj].w, acc[m][jj]);
                }
        }
        // G for rows rg, rg + 32 and keys kg + 8 jj (0 for stopped rows, keys past the row or the tile)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int kk = kg + 8 * jj, j = j0 + kk;
            const bool in = kk < nk;
            const bool live0 = in && act0 && j <= ib + rg, live1 = in && act1 && j <= ib + rg + 32;
            float w0, w1;
            if constexpr (WMODE == 2) {
                w0 = wv[0][jj];
                w1 = wv[1][jj];
            } else if constexpr (WMODE == 3) {
                w0 = live0 ? expf(wv[0][jj] - lse0) : 0.f;
                w1 = live1 ? expf(wv[1][jj] - lse1) : 0.f;
                if (live0) p.wts[wrow0 + j] = w0;
                if (live1) p.wts[wrow1 + j] = w1;
            } else {
                w0 = live0 ? expf(acc[0][jj] - lse0) : 0.f;
                w1 = live1 ? expf(acc[1][jj] - lse1) : 0.f;
            }
            const float g0 = live0 ? w0 * (acc[2][jj] - kp0) : 0.f;
            const float g1 = live1 ? w1 * (acc[3][jj] - kp1) : 0.f;
            Gs[kk * GLD + (rg & 15) * 4 + (rg >> 4)] = g0;
            Gs[kk * GLD + (rg & 15) * 4 + ((rg + 32) >> 4)] = g1;
        }
        __syncthreads();
        // phase 2: U[rows rgrp + 16 i][dims dgrp * 4 + 64 h + e] += G K
        if (!*abort_flag) {
#pragma unroll 2
            for (int kk = 0; kk < nk; ++kk) {
                const float4 g = *reinterpret_cast<const float4*>(Gs + kk * GLD + rgrp * 4);
                float kv[DG];
#pragma unroll
                for (int x = 0; x < DG; x += 4) {
                    const float4 k4 = *reinterpret_cast<const float4*>(kt + kk * LD + dgrp * 4 + 16 * x);
                    kv[x] = k4.x;
                    kv[x + 1] = k4.y;
                    kv[x + 2] = k4.z;
                    kv[x + 3] = k4.w;
                }
#pragma unroll
                for (int x = 0; x < DG; ++x) {
                    U[0][x] = fmaf(g.x, kv[x], U[0][x]);
                    U[1][x] = fmaf(g.y, kv[x], U[1][x]);
                    U[2][x] = fmaf(g.z, kv[x], U[2][x]);
                    U[3][x] = fmaf(g.w, kv[x], U[3][x]);
                }
            }
        }
        __syncthreads();                                  // G and this tile buffer may be reused
        if (*abort_flag) break;
    }
    // no copy may still be in flight when the block exits (only after an abort)
    if (warp == 0 && lane == 0 && *abort_flag) mbar_wait(&full[last_issued & 1], (last_issued >> 1) & 1);
    if (*abort_flag) return;

    // ---- Ap = U + lambda p and one conjugate-gradient step per active row.  A
    // row's 16 threads are one half-warp and the two half-warps of a warp may
    // hold rows in different states, so every lane runs the shuffles and only
    // the loads and stores depend on the row's state.
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int a = rgrp + 16 * i;
        const bool act = s_act[a] != 0;                   // implies ib + a < N
        const size_t row = bh * p.N + ib + a;
        const float* prow = QP + (BM + a) * LD + dgrp * 4;
        float pv[DG], pap = 0.f;
#pragma unroll
        for (int x = 0; x < DG; x += 4) {
            const float4 p4 = *reinterpret_cast<const float4*>(prow + 16 * x);
            pv[x] = p4.x;
            pv[x + 1] = p4.y;
            pv[x + 2] = p4.z;
            pv[x + 3] = p4.w;
        }
#pragma unroll
        for (int x = 0; x < DG; ++x) {
            U[i][x] = fmaf(p.lambda, pv[x], U[i][x]);
            pap = fmaf(pv[x], U[i][x], pap);
        }
#pragma unroll
        for (int m = 8; m >= 1; m >>= 1) pap += __shfl_xor_sync(0xffffffffu, pap, m);
        const bool ok = act && pap > 0.f;
        if (act && !ok && dgrp == 0) p.rs[row] = 0.f;      // breakdown: stop the row
        const float rs = s_rs[a];
        const float alpha = ok ? rs / pap : 0.f;
        float xv[DG], rv[DG], rn = 0.f;
#pragma unroll
        for (int x = 0; x < DG; ++x) {
            xv[x] = 0.f;
            rv[x] = 0.f;
        }
        if (ok) {
            const float* xo = p.x + row * D + dgrp * 4;
            const float* ro = p.r + row * D + dgrp * 4;
#pragma unroll
            for (int x = 0; x < DG; x += 4) {
                const float4 x4 = *reinterpret_cast<const float4*>(xo + 16 * x);
                const float4 r4 = *reinterpret_cast<const float4*>(ro + 16 * x);
                xv[x] = x4.x; xv[x + 1] = x4.y; xv[x + 2] = x4.z; xv[x + 3] = x4.w;
                rv[x] = r4.x; rv[x + 1] = r4.y; rv[x + 2] = r4.z; rv[x + 3] = r4.w;
            }
        }
#pragma unroll
        for (int x = 0; x < DG; ++x) {
            xv[x] = fmaf(alpha, pv[x], xv[x]);
            rv[x] = fmaf(-alpha, U[i][x], rv[x]);
            rn = fmaf(rv[x], rv[x], rn);
        }
#pragma unroll
        for (int m = 8; m >= 1; m >>= 1) rn += __shfl_xor_sync(0xffffffffu, rn, m);
        if (ok) {
            const float beta = rn / rs;
            float* xo = p.x + row * D + dgrp * 4;
            float* ro = p.r + row * D + dgrp * 4;
            float* po = p.p + row * D + dgrp * 4;
#pragma unroll
            for (int x = 0; x < DG; x += 4) {
                *reinterpret_cast<float4*>(xo + 16 * x) = make_float4(xv[x], xv[x + 1], xv[x + 2], xv[x + 3]);
                *reinterpret_cast<float4*>(ro + 16 * x) = make_float4(rv[x], rv[x + 1], rv[x + 2], rv[x + 3]);
                *reinterpret_cast<float4*>(po + 16 * x) =
                    make_float4(fmaf(beta, pv[x], rv[x]), fmaf(beta, pv[x + 1], rv[x + 1]),
                                fmaf(beta, pv[x + 2], rv[x + 2]), fmaf(beta, pv[x + 3], rv[x + 3]));
            }
            if (dgrp == 0) {
                p.rs[row] = rn;
                p.steps[row] += 1;
            }
        }
    }
}

// Parallax's output with the solved probe, in centred form (4 rows per warp,
// the same butterfly): with r'_j = k_j . rho - kbar . rho = (k_j - kbar) . rho,
//   o = vbar - Sigma_KV rho = sum_j w_j (1 - r'_j) v_j + vbar sum_j w_j r'_j,
// weights w_j = exp(s_j - lse) / L, L = sum_j exp(s_j - lse) (1 up to
// rounding).  The uncentred (1 + c) vbar - u cancels two terms of size
// |k| |rho| |v|, which is large on short prefixes where rho ~ mu / lambda;
// here r'_j is 0 on a one-key prefix and small elsewhere.
template <int DPL>
__global__ void __launch_bounds__(LLA_WARPS * 32) plx_lla_out_kernel(const LlaParams p, const float* v, float* out,
                                                                  float* lse_out) {
    constexpr int D = DPL * 32;
    constexpr int RW = LLA_ROWS_PER_BLOCK / LLA_WARPS;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t bh = blockIdx.y;
    const float* K = p.k + bh * p.N * D;
    const float* V = v + bh * p.N * D;
    const int i0 = blockIdx.x * LLA_ROWS_PER_BLOCK + warp * RW;
    if (i0 >= p.N) return;

    float qv[RW][DPL], xv[RW][DPL], O[RW][DPL], A[RW][DPL], kx[RW], lse[RW];
#pragma unroll
    for (int r = 0; r < RW; ++r) {
        const int i = i0 + r < p.N ? i0 + r : i0;
        const size_t row = bh * p.N + i;
        lse[r] = p.lse[row];
        float kb[DPL];
        load_own<DPL>(p.q + row * D, lane, qv[r]);
        load_own<DPL>(p.x + row * D, lane, xv[r]);
        load_own<DPL>(p.kbar + row * D, lane, kb);
        float part = 0.f;
#pragma unroll
        for (int t = 0; t < DPL; ++t) {
            qv[r][t] *= p.scale;
            part = fmaf(kb[t], xv[r][t], part);
            O[r][t] = 0.f;
            A[r][t] = 0.f;
        }
        kx[r] = warp_sum(part);
    }
    const int my = (lane >> 3) & 3;
    float my_lse = lse[0], my_kx = kx[0];
#pragma unroll
    for (int r = 1; r < RW; ++r)
        if (my == r) {
            my_lse = lse[r];
            my_kx = kx[r];
        }
    const bool b2 = lane & 4;
    const int jmax = min(i0 + RW - 1, p.N - 1);
    float wsum = 0.f, wr = 0.f;        // lanes 8 r: sum_j w_j and sum_j w_j r'_j of row r

#pragma unroll 2
    for (int j = 0; j <= jmax; ++j) {
        float kf[DPL], vf[DPL];
        load_own<DPL>(K + static_cast<size_t>(j) * D, lane, kf);
        load_own<DPL>(V + static_cast<size_t>(j) * D, lane, vf);
        float a[2 * RW];
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            float sd = 0.f, rd = 0.f;
#pragma unroll
            for (int t = 0; t < DPL; ++t) {
                sd = fmaf(qv[r][t], kf[t], sd);
                rd = fmaf(xv[r][t], kf[t], rd);
            }
            a[2 * r] = sd;
            a[2 * r + 1] = rd;
        }
        const float val = reduce_scatter8(a, lane);
        const float other = __shfl_xor_sync(0xffffffffu, val, 4);
        float w = 0.f, rc = 0.f;
        if (!b2 && j <= i0 + my) {
            w = expf(val - my_lse);
            rc = other - my_kx;
        }
        wsum += w;
        wr = fmaf(w, rc, wr);
        const float g = w - w * rc;                         // w (1 - r')
        float gr[RW], wv[RW];
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            gr[r] = __shfl_sync(0xffffffffu, g, 8 * r);
            wv[r] = __shfl_sync(0xffffffffu, w, 8 * r);
        }
#pragma unroll
        for (int r = 0; r < RW; ++r)
#pragma unroll
            for (int t = 0; t < DPL; ++t) {
                O[r][t] = fmaf(gr[r], vf[t], O[r][t]);
                A[r][t] = fmaf(wv[r], vf[t], A[r][t]);
            }
    }
#pragma unroll
    for (int r = 0; r < RW; ++r) {
        const float L = __shfl_sync(0xffffffffu, wsum, 8 * r);
        const float C = __shfl_sync(0xffffffffu, wr, 8 * r);
        if (i0 + r >= p.N) continue;                        // warp-uniform
        const size_t row = bh * p.N + i0 + r;
        const float inv = 1.f / L;
        const float cn = C * inv;
        float* dst = out + row * D + lane * DPL;
#pragma unroll
        for (int t = 0; t < DPL; ++t) dst[t] = fmaf(cn, A[r][t] * inv, O[r][t] * inv);
        if (lane == 0 && lse_out) lse_out[row] = lse[r];
    }
}

// The output pass in the block-GEMM form of the CG step (d = 64, 128): a
// block owns BM = 64 rows and streams the K and V rows of keys 0 .. i_b + 63
// in tiles of BK = 32, both through one bulk copy per row into two buffers.
//   phase 1   [S; R] = [scale q; rho] K^T    (128 stacked rows x 32 keys)
//             w = exp(s - lse), r' = (rho.k) - (kbar.rho); thread (rg, kg)
//             writes G1 = w (1 - r') and G2 = w for rows {rg, rg + 32} and
//             keys {kg + 8 jj} to shared memory and keeps its part of the row
//             sums L = sum w and C = sum w r';
//   phase 2   O += G1 V, A += G2 V           (64 rows x d, K = 32 keys)
// then o = (C/L) A/L + O/L, the centred form of plx_lla_out_kernel above.
template <int D>
struct LlaOutCfg {
    static constexpr int BM = 64, BK = 32, THREADS = 256;
    static constexpr int LD = D + 4;
    static constexpr int DG = D / 16;
    static constexpr int OFF_K = 0;                          // 2 x [BK][LD]
    static constexpr int OFF_V = OFF_K + 2 * BK * LD;        // 2 x [BK][LD]
    static constexpr int OFF_QP = OFF_V + 2 * BK * LD;       // [2 BM][LD]: scale q rows, then rho rows
    static constexpr int GLD = BM + 4;
    static constexpr int OFF_G = OFF_QP + 2 * BM * LD;       // 2 x [BK][GLD]: w (1 - r'), w
    static constexpr int OFF_ROW = OFF_G + 2 * BK * GLD;     // lse, kbar.rho, L, C [BM] each
    static constexpr int OFF_BAR = OFF_ROW + 4 * BM;         // 2 mbarriers + abort flag
    static constexpr int SMEM = OFF_BAR * 4 + 32;
    static_assert(D == 64 || D == 128, "the block output pass is built for d in {64, 128}");
};

// KEPT: p.wts holds the weights the first CG step kept (those of every row that
// took a step); a block whose rows all took one reads them instead of forming
// S = scale q K^T.  The first step formed them with this kernel's arithmetic
// (the same products in the same order, then exp(s - lse)), so the output is
// the same bit for bit; a block with a row that took no step forms S.
template <int D, bool KEPT = false>
__global__ void __launch_bounds__(256) plx_lla_out_gemm_kernel(const LlaParams p, const float* v, float* out,
                                                               float* lse_out) {
    using Cfg = LlaOutCfg<D>;
    constexpr int BM = Cfg::BM, BK = Cfg::BK, LD = Cfg::LD, DG = Cfg::DG, GLD = Cfg::GLD;
    extern __shared__ __align__(128) float lla_osmem[];
    float* kstage = lla_osmem + Cfg::OFF_K;
    float* vstage = lla_osmem + Cfg::OFF_V;
    float* QP = lla_osmem + Cfg::OFF_QP;
    float* G1s = lla_osmem + Cfg::OFF_G;
    float* G2s = G1s + BK * GLD;
    float* s_lse = lla_osmem + Cfg::OFF_ROW;
    float* s_kx = s_lse + BM;
    float* s_L = s_kx + BM;
    float* s_C = s_L + BM;
    uint64_t* full = reinterpret_cast<uint64_t*>(lla_osmem + Cfg::OFF_BAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(full + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t bh = blockIdx.y;
    const int ib = blockIdx.x * BM;
    if (ib >= p.N) return;
    const float* K = p.k + bh * p.N * D;
    const float* V = v + bh * p.N * D;

    // the kept weights serve this block if every row of it took a CG step
    int no_step = 0;
    if (KEPT && tid < BM && ib + tid < p.N) no_step = p.steps[bh * p.N + ib + tid] == 0;
    const bool use_w = KEPT && !__syncthreads_or(no_step);
    if (tid < BM) s_lse[tid] = ib + tid < p.N ? p.lse[bh * p.N + ib + tid] : 0.f;
    for (int idx = tid; idx < 2 * BM * (D / 4); idx += Cfg::THREADS) {
        const int r = idx / (D / 4), c = idx % (D / 4);
        if (use_w && r < BM) continue;                   // q rows: the weights are kept
        const int i = ib + (r & (BM - 1));
        float4 x4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < p.N) {
            const size_t off = (bh * p.N + i) * D + c * 4;
            x4 = *reinterpret_cast<const float4*>((r < BM ? p.q : p.x) + off);
            if (r < BM) {
                x4.x *= p.scale;
                x4.y *= p.scale;
                x4.z *= p.scale;
                x4.w *= p.scale;
            }
        }
        *reinterpret_cast<float4*>(QP + r * LD + c * 4) = x4;
    }
    // kbar . rho per row: warp w takes rows w, w + 8, ...
    for (int r = warp; r < BM; r += Cfg::THREADS / 32) {
        const int i = ib + r;
        float part = 0.f;
        if (i < p.N) {
            const size_t off = (bh * p.N + i) * D;
            for (int x = lane; x < D; x += 32) part = fmaf(p.kbar[off + x], p.x[off + x], part);
        }
        part = warp_sum(part);
        if (lane == 0) s_kx[r] = part;
    }
    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const int kmax = min(ib + BM, p.N) - 1;
    const int n_tiles = kmax / BK + 1;
    auto issue = [&](int t) {                             // warp 0, all lanes
        const int j0 = t * BK;
        const int nk = min(BK, kmax + 1 - j0);
        if (!in_bounds(nk > 0 && j0 + nk <= p.N)) {
            if (lane == 0) mbar_arrive(&full[t & 1]);
            return;
        }
        if (lane == 0) mbar_arrive_expect_tx(&full[t & 1], static_cast<uint32_t>(2 * nk) * D * 4);
        __syncwarp();
        if (lane < nk) {
            bulk_g2s(kstage + (t & 1) * BK * LD + lane * LD, K + static_cast<size_t>(j0 + lane) * D, D * 4,
                     &full[t & 1]);
            bulk_g2s(vstage + (t & 1) * BK * LD + lane * LD, V + static_cast<size_t>(j0 + lane) * D, D * 4,
                     &full[t & 1]);
        }
    };
    if (warp == 0) issue(0);

    const int rg = tid >> 3, kg = tid & 7;
    const int rgrp = tid >> 4, dgrp = tid & 15;
    float O[4][DG], A[4][DG];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int x = 0; x < DG; ++x) {
            O[i][x] = 0.f;
            A[i][x] = 0.f;
        }
    const float lse0 = s_lse[rg], lse1 = s_lse[rg + 32];
    const float kx0 = s_kx[rg], kx1 = s_kx[rg + 32];
    const bool in0 = ib + rg < p.N, in1 = ib + rg + 32 < p.N;
    float L0 = 0.f, L1 = 0.f, C0 = 0.f, C1 = 0.f;
    int last_issued = 0;

    for (int t = 0; t < n_tiles; ++t) {
        if (warp == 0 && t + 1 < n_tiles) {
            issue(t + 1);
            last_issued = t + 1;
        }
        if (!mbar_wait(&full[t & 1], (t >> 1) & 1)) {
            atomicOr(&g_plx_status, PLX_DEV_ERR_TIMEOUT);
            *abort_flag = 1;
        }
        const float* kt = kstage + (t & 1) * BK * LD;
        const float* vt = vstage + (t & 1) * BK * LD;
        const int j0 = t * BK;
        const int nk = min(BK, kmax + 1 - j0);
        // the kept weights of this tile (use_w), loaded ahead of phase 1's FMAs
        float wk[2][4];
        if (use_w) {
            const size_t wrow0 = (bh * p.N + ib + rg) * static_cast<size_t>(p.N);
            const size_t wrow1 = wrow0 + 32 * static_cast<size_t>(p.N);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int kk = kg + 8 * jj, j = j0 + kk;
                wk[0][jj] = (kk < nk && in0 && j <= ib + rg) ? p.wts[wrow0 + j] : 0.f;
                wk[1][jj] = (kk < nk && in1 && j <= ib + rg + 32) ? p.wts[wrow1 + j] : 0.f;
            }
        }
        // phase 1: acc[m][jj], m = 0, 1: s of rows rg, rg + 32; m = 2, 3: rho.k of
        // the same rows (with the kept weights only m = 2, 3)
        float acc[4][4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) acc[m][jj] = 0.f;
        auto phase1 = [&](auto m0c) {
            constexpr int M0 = decltype(m0c)::value;
#pragma unroll 4
            for (int c = 0; c < D; c += 4) {
                float4 a[4], b[4];
#pragma unroll
                for (int m = M0; m < 4; ++m) a[m] = *reinterpret_cast<const float4*>(QP + (rg + 32 * m) * LD + c);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) b[jj] = *reinterpret_cast<const float4*>(kt + (kg + 8 * jj) * LD + c);
#pragma unroll
                for (int m = M0; m < 4; ++m)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        acc[m][jj] = fmaf(a[m].x, b[jj].x, acc[m][jj]);
                        acc[m][jj] = fmaf(a[m].y, b[jj].y, acc[m][jj]);
                        acc[m][jj] = fmaf(a[m].z, b[jj].z, acc[m][jj]);
                        acc[m][jj] = fmaf(a[m].w, b[jj].w, acc[m][jj]);
                    }
            }
        };
        if (use_w)
            phase1(std::integral_constant<int, 2>{});
        else
            phase1(std::integral_constant<int, 0>{});
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int kk = kg + 8 * jj, j = j0 + kk;
            // keys past the tile's rows read unfilled shared memory: their r' is not
            // formed at all (0 x NaN would still be NaN)
            const bool v0 = kk < nk && in0 && j <= ib + rg, v1 = kk < nk && in1 && j <= ib + rg + 32;
            const float w0 = use_w ? wk[0][jj] : (v0 ? expf(acc[0][jj] - lse0) : 0.f);
            const float w1 = use_w ? wk[1][jj] : (v1 ? expf(acc[1][jj] - lse1) : 0.f);
            const float rc0 = v0 ? acc[2][jj] - kx0 : 0.f, rc1 = v1 ? acc[3][jj] - kx1 : 0.f;
            L0 += w0;
            L1 += w1;
            C0 = fmaf(w0, rc0, C0);
            C1 = fmaf(w1, rc1, C1);
            const int a0 = kk * GLD + (rg & 15) * 4 + (rg >> 4), a1 = kk * GLD + (rg & 15) * 4 + ((rg + 32) >> 4);
            G1s[a0] = w0 - w0 * rc0;
            G1s[a1] = w1 - w1 * rc1;
            G2s[a0] = w0;
            G2s[a1] = w1;
        }
        __syncthreads();
        if (!*abort_flag) {
#pragma unroll 2
            for (int kk = 0; kk < nk; ++kk) {
                const float4 g1 = *reinterpret_cast<const float4*>(G1s + kk * GLD + rgrp * 4);
                const float4 g2 = *reinterpret_cast<const float4*>(G2s + kk * GLD + rgrp * 4);
                float vv[DG];
#pragma unroll
                for (int x = 0; x < DG; x += 4) {
                    const float4 v4 = *reinterpret_cast<const float4*>(vt + kk * LD + dgrp * 4 + 16 * x);
                    vv[x] = v4.x;
                    vv[x + 1] = v4.y;
                    vv[x + 2] = v4.z;
                    vv[x + 3] = v4.w;
                }
#pragma unroll
                for (int x = 0; x < DG; ++x) {
                    O[0][x] = fmaf(g1.x, vv[x], O[0][x]);
                    O[1][x] = fmaf(g1.y, vv[x], O[1][x]);
                    O[2][x] = fmaf(g1.z, vv[x], O[2][x]);
                    O[3][x] = fmaf(g1.w, vv[x], O[3][x]);
                    A[0][x] = fmaf(g2.x, vv[x], A[0][x]);
                    A[1][x] = fmaf(g2.y, vv[x], A[1][x]);
                    A[2][x] = fmaf(g2.z, vv[x], A[2][x]);
                    A[3][x] = fmaf(g2.w, vv[x], A[3][x]);
                }
            }
        }
        __syncthreads();
        if (*abort_flag) break;
    }
    if (warp == 0 && lane == 0 && *abort_flag) mbar_wait(&full[last_issued & 1], (last_issued >> 1) & 1);
    if (*abort_flag) return;
    // row sums over the 8 threads of a row (consecutive lanes)
#pragma unroll
    for (int m = 4; m >= 1; m >>= 1) {
        L0 += __shfl_xor_sync(0xffffffffu, L0, m);
        L1 += __shfl_xor_sync(0xffffffffu, L1, m);
        C0 += __shfl_xor_sync(0xffffffffu, C0, m);
        C1 += __shfl_xor_sync(0xffffffffu, C1, m);
    }
    if (kg == 0) {
        s_L[rg] = L0;
        s_L[rg + 32] = L1;
        s_C[rg] = C0;
        s_C[rg + 32] = C1;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int a = rgrp + 16 * i;
        if (ib + a >= p.N) continue;
        const size_t row = bh * p.N + ib + a;
        const float inv = 1.f / s_L[a];
        const float cn = s_C[a] * inv;
        float* dst = out + row * D + dgrp * 4;
#pragma unroll
        for (int x = 0; x < DG; x += 4)
            *reinterpret_cast<float4*>(dst + 16 * x) =
                make_float4(fmaf(cn, A[i][x] * inv, O[i][x] * inv), fmaf(cn, A[i][x + 1] * inv, O[i][x + 1] * inv),
                            fmaf(cn, A[i][x + 2] * inv, O[i][x + 2] * inv),
                            fmaf(cn, A[i][x + 3] * inv, O[i][x + 3] * inv));
        if (dgrp == 0 && lse_out) lse_out[row] = s_lse[a];
    }
}

// kbar and lse (the softmax attention of the keys themselves) in the same
// block form (d = 64, 128): a block owns BM = 64 rows and streams key tiles
// of BK = 32 through two buffers, with an online softmax over the tiles.
//   phase 1   S = scale q K^T (64 rows x 32 keys); per row the tile max over
//             its 8 threads, m' = max(m, tile max), alpha = e^(m - m'),
//             P = e^(s - m') to shared memory, l = alpha l + sum P;
//   phase 2   U = alpha U + P K                 (64 rows x d, K = 32 keys)
// then kbar = U / l, lse = m + ln l.
template <int D>
struct LlaKbarCfg {
    static constexpr int BM = 64, BK = 32, THREADS = 256;
    static constexpr int LD = D + 4;
    static constexpr int DG = D / 16;
    static constexpr int OFF_K = 0;                          // 2 x [BK][LD]
    static constexpr int OFF_Q = OFF_K + 2 * BK * LD;        // [BM][LD]: scale q rows
    static constexpr int GLD = BM + 4;
    static constexpr int OFF_P = OFF_Q + BM * LD;            // [BK][GLD]
    static constexpr int OFF_ROW = OFF_P + BK * GLD;         // alpha, l, m [BM] each
    static constexpr int OFF_BAR = OFF_ROW + 3 * BM;         // 2 mbarriers + abort flag
    static constexpr int SMEM = OFF_BAR * 4 + 32;
    static_assert(D == 64 || D == 128, "the block kbar pass is built for d in {64, 128}");
};

// KEEP: also store each causal pair's score s_ij = scale q_i . k_j in p.wts
// (the first CG step turns those of its active rows into the weights).
template <int D, bool KEEP = false>
__global__ void __launch_bounds__(256) plx_lla_kbar_gemm_kernel(const LlaParams p, float* kbar, float* lse) {
    using Cfg = LlaKbarCfg<D>;
    constexpr int BM = Cfg::BM, BK = Cfg::BK, LD = Cfg::LD, DG = Cfg::DG, GLD = Cfg::GLD;
    extern __shared__ __align__(128) float lla_ksmem[];
    float* kstage = lla_ksmem + Cfg::OFF_K;
    float* Qs = lla_ksmem + Cfg::OFF_Q;
    float* Ps = lla_ksmem + Cfg::OFF_P;
    float* s_alpha = lla_ksmem + Cfg::OFF_ROW;
    float* s_l = s_alpha + BM;
    float* s_m = s_l + BM;
    uint64_t* full = reinterpret_cast<uint64_t*>(lla_ksmem + Cfg::OFF_BAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(full + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t bh = blockIdx.y;
    const int ib = blockIdx.x * BM;
    if (ib >= p.N) return;
    const float* K = p.k + bh * p.N * D;

    for (int idx = tid; idx < BM * (D / 4); idx += Cfg::THREADS) {
        const int r = idx / (D / 4), c = idx % (D / 4);
        const int i = ib + r;
        float4 x4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < p.N) {
            x4 = *reinterpret_cast<const float4*>(p.q + (bh * p.N + i) * D + c * 4);
            x4.x *= p.scale;
            x4.y *= p.scale;
            x4.z *= p.scale;
            x4.w *= p.scale;
        }
        *reinterpret_cast<float4*>(Qs + r * LD + c * 4) = x4;
    }
    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const int kmax = min(ib + BM, p.N) - 1;
    const int n_tiles = kmax / BK + 1;
    auto issue = [&](int t) {                             // warp 0, all lanes
        const int j0 = t * BK;
        const int nk = min(BK, kmax + 1 - j0);
        if (!in_bounds(nk > 0 && j0 + nk <= p.N)) {
            if (lane == 0) mbar_arrive(&full[t & 1]);
            return;
        }
        if (lane == 0) mbar_arrive_expect_tx(&full[t & 1], static_cast<uint32_t>(nk) * D * 4);
        __syncwarp();
        if (lane < nk)
            bulk_g2s(kstage + (t & 1) * BK * LD + lane * LD, K + static_cast<size_t>(j0 + lane) * D, D * 4,
                     &full[t & 1]);
    };
    if (warp == 0) issue(0);

    const int rg = tid >> 3, kg = tid & 7;               // phase 1: rows {rg, rg + 32}, keys kg + 8 jj
    const int rgrp = tid >> 4, dgrp = tid & 15;          // phase 2: rows rgrp + 16 i, dims dgrp * 4 + 64 h + e
    float U[4][DG];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int x = 0; x < DG; ++x) U[i][x] = 0.f;
    const bool in0 = ib + rg < p.N, in1 = ib + rg + 32 < p.N;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // per thread: its keys' part of l
    int last_issued = 0;

    for (int t = 0; t < n_tiles; ++t) {
        if (warp == 0 && t + 1 < n_tiles) {
            issue(t + 1);
            last_issued = t + 1;
        }
        if (!mbar_wait(&full[t & 1], (t >> 1) & 1)) {
            atomicOr(&g_plx_status, PLX_DEV_ERR_TIMEOUT);
            *abort_flag = 1;
        }
        const float* kt = kstage + (t & 1) * BK * LD;
        const int j0 = t * BK;
        const int nk = min(BK, kmax + 1 - j0);
        float acc[2][4];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) acc[m][jj] = 0.f;
#pragma unroll 4
        for (int c = 0; c < D; c += 4) {
            float4 a[2], b[4];
#pragma unroll
            for (int m = 0; m < 2; ++m) a[m] = *reinterpret_cast<const float4*>(Qs + (rg + 32 * m) * LD + c);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) b[jj] = *reinterpret_cast<const float4*>(kt + (kg + 8 * jj) * LD + c);
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    acc[m][jj] = fmaf(a[m].x, b[jj].x, acc[m][jj]);
                    acc[m][jj] = fmaf(a[m].y, b[jj].y, acc[m][jj]);
                    acc[m][jj] = fmaf(a[m].z, b[jj].z, acc[m][jj]);
                    acc[m][jj] = fmaf(a[m].w, b[jj].w, acc[m][jj]);
                }
        }
        // masked scores (keys past the row, past the tile's rows, rows past N) are -inf
        float t0 = -INFINITY, t1 = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int kk = kg + 8 * jj, j = j0 + kk;
            if constexpr (KEEP) {
                if (kk < nk && in0 && j <= ib + rg) p.wts[(bh * p.N + ib + rg) * static_cast<size_t>(p.N) + j] = acc[0][jj];
                if (kk < nk && in1 && j <= ib + rg + 32)
                    p.wts[(bh * p.N + ib + rg + 32) * static_cast<size_t>(p.N) + j] = acc[1][jj];
            }
            if (!(kk < nk && in0 && j <= ib + rg)) acc[0][jj] = -INFINITY;
            if (!(kk < nk && in1 && j <= ib + rg + 32)) acc[1][jj] = -INFINITY;
            t0 = fmaxf(t0, acc[0][jj]);
            t1 = fmaxf(t1, acc[1][jj]);
        }
#pragma unroll
        for (int off = 4; off >= 1; off >>= 1) {
            t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, off));
            t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, off));
        }
        const float n0 = fmaxf(m0, t0), n1 = fmaxf(m1, t1);
        // a row with no valid key so far keeps alpha = 1 and P = 0
        const float a0 = n0 == -INFINITY ? 1.f : expf(m0 - n0), a1 = n1 == -INFINITY ? 1.f : expf(m1 - n1);
        m0 = n0;
        m1 = n1;
        l0 *= a0;
        l1 *= a1;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int kk = kg + 8 * jj;
            const float p0 = acc[0][jj] == -INFINITY ? 0.f : expf(acc[0][jj] - n0);
            const float p1 = acc[1][jj] == -INFINITY ? 0.f : expf(acc[1][jj] - n1);
            l0 += p0;
            l1 += p1;
            Ps[kk * GLD + (rg & 15) * 4 + (rg >> 4)] = p0;
            Ps[kk * GLD + (rg & 15) * 4 + ((rg + 32) >> 4)] = p1;
        }
        if (kg == 0) {
            s_alpha[rg] = a0;
            s_alpha[rg + 32] = a1;
        }
        __syncthreads();
        if (!*abort_flag) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float al = s_alpha[rgrp + 16 * i];
#pragma unroll
                for (int x = 0; x < DG; ++x) U[i][x] *= al;
            }
#pragma unroll 2
            for (int kk = 0; kk < nk; ++kk) {
                const float4 g = *reinterpret_cast<const float4*>(Ps + kk * GLD + rgrp * 4);
                float kv[DG];
#pragma unroll
                for (int x = 0; x < DG; x += 4) {
                    const float4 k4 = *reinterpret_cast<const float4*>(kt + kk * LD + dgrp * 4 + 16 * x);
                    kv[x] = k4.x;
                    kv[x + 1] = k4.y;
                    kv[x + 2] = k4.z;
                    kv[x + 3] = k4.w;
                }
#pragma unroll
                for (int x = 0; x < DG; ++x) {
                    U[0][x] = fmaf(g.x, kv[x], U[0][x]);
                    U[1][x] = fmaf(g.y, kv[x], U[1][x]);
                    U[2][x] = fmaf(g.z, kv[x], U[2][x]);
                    U[3][x] = fmaf(g.w, kv[x], U[3][x]);
                }
            }
        }
        __syncthreads();
        if (*abort_flag) break;
    }
    if (warp == 0 && lane == 0 && *abort_flag) mbar_wait(&full[last_issued & 1], (last_issued >> 1) & 1);
    if (*abort_flag) return;
#pragma unroll
    for (int off = 4; off >= 1; off >>= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    if (kg == 0) {
        s_l[rg] = l0;
        s_l[rg + 32] = l1;
        s_m[rg] = m0;
        s_m[rg + 32] = m1;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int a = rgrp + 16 * i;
        if (ib + a >= p.N) continue;
        const size_t row = bh * p.N + ib + a;
        const float inv = 1.f / s_l[a];
        float* dst = kbar + row * D + dgrp * 4;
#pragma unroll
        for (int x = 0; x < DG; x += 4)
            *reinterpret_cast<float4*>(dst + 16 * x) =
                make_float4(U[i][x] * inv, U[i][x + 1] * inv, U[i][x + 2] * inv, U[i][x + 3] * inv);
        if (dgrp == 0) lse[row] = s_m[a] + logf(s_l[a]);
    }
}

}  // namespace plx
