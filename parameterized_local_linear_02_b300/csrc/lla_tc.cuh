// lla_tc.cuh -- the conjugate-gradient step of plx_lla_f32 on the tensor
// cores, for the steps that read the kept softmax weights (d = 64, 128).
//
// Local linear attention solves (Sigma_KK^(i) + lambda I) rho_i = mu_i per
// token by conjugate gradients (zhichai.net section 1.2; gist.science,
// "Enunciato del Problema").  One step needs, for every active row i and its
// search direction p_i,
//
//   Sigma_KK^(i) p_i = sum_{j<=i} w_ij ((k_j . p_i) - (kbar_i . p_i)) k_j,
//
// two contractions over the key tile: R = P K^T (p_i . k_j) and U += G K with
// G_ij = w_ij (R_ij - kbar_i . p_i).  The pages warn that the solve is unstable
// in low precision, so each operand x is split as x = hi + lo with hi = x
// rounded to tf32 and lo = x - hi (exact in fp32), and every product is
// formed as hi.hi + hi.lo + lo.hi on kind::tf32 MMAs with fp32 accumulation:
// the dropped lo.lo term and the tf32 rounding of lo are below 2^-21 of each
// product, near fp32's own rounding.
//
// One CTA owns 128 rows of one head (TMEM lane = row) and streams keys
// 0 .. its last row in tiles of 32.  TMEM (512 columns): P_hi, P_lo (d each,
// A of the first GEMM), U_tile (d), R (two partial sums of 32), G_hi, G_lo
// (32 each, A of the second GEMM).  The tensor core's fp32 accumulation rounds
// toward zero, so over hundreds of MMAs into one accumulator the error grows
// as a bias; each tile's G K goes into a fresh U_tile (12 MMAs, the small
// products first) that the row warps add to an fp32 register sum.  Warps:
//   0-3  row warps (warp w holds TMEM lanes 32w..32w+31, thread = row): split
//        p into TMEM, then per tile read R from TMEM (releasing it for the
//        next tile's GEMM), add the previous tile's U_tile to the row's sum,
//        read the row's 32 weights from shared memory, form G and split it
//        into TMEM; at the end the CG update of the row from the sum, its
//        rows of p, x and r moved by 1-D bulk copies through the freed ring
//        buffers;
//   4    weight producer: one TMA load per tile of the [BH][N][N] weights
//        (box 32 keys x 128 rows, 128-byte swizzle), a 4-stage ring;
//   5    MMA issuer (one elected lane; one asm block per GEMM of a tile);
//   6-7  converters: read the key tile from global memory, split it and
//        store K_hi, K_lo twice, as [32 keys][d] (B of R = P K^T) and as
//        [d][32 keys] (B of U += G K), both K-major with 128-byte swizzle;
//        keys past the block's last row are stored as 0.
// Every wait is bounded; a role whose wait gives up records
// PLX_DEV_ERR_TIMEOUT, and TMEM is freed only after the MMAs and the TMA
// loads issued have completed.
#pragma once
#include "lla_f32.cuh"
#include "ptx.cuh"
#include "status.cuh"

namespace plx {

template <int D>
struct LlaTcCfg {
    static_assert(D == 64 || D == 128, "the tensor-core CG step is built for d in {64, 128}");
    static constexpr int BM = 128, BK = 32;
    static constexpr int NCV = 2;                          // converted key-tile stages
    static constexpr int NW = 4;                           // weight-tile stages
    // 8 warps, two per SM sub-partition: up to 255 registers a thread (the row
    // warps keep their row's fp32 sum of U in registers)
    static constexpr int ROW_WARPS = 4, CV_WARPS = 2;
    static constexpr int W_PROD = ROW_WARPS, W_MMA = ROW_WARPS + 1, W_CV0 = ROW_WARPS + 2;
    static constexpr int THREADS = (ROW_WARPS + 2 + CV_WARPS) * 32;
    static constexpr int PANEL = BK * 128;                 // one 32-dim panel of a [32 keys][d] tile
    static constexpr int KA_BYTES = BK * D * 4;            // [D/32 panels][BK rows][128 B]
    static constexpr int KB_BYTES = D * BK * 4;            // [D rows][128 B]
    static constexpr int CV_STAGE = 2 * KA_BYTES + 2 * KB_BYTES;   // KA_hi, KA_lo, KB_hi, KB_lo
    static constexpr int W_STAGE = BM * BK * 4;            // [128 rows][128 B], swizzled by the TMA
    static constexpr int OFF_CV = 0;
    static constexpr int OFF_W = OFF_CV + NCV * CV_STAGE;
    // the epilogue: p, x, r rows of each row warp, rows padded to D + 4 floats,
    // over the converter and weight buffers (free by then)
    static constexpr int LDE = D + 4;
    static constexpr int EPI_BYTES = ROW_WARPS * 3 * 32 * LDE * 4;
    static constexpr int OFF_BAR = (OFF_W + NW * W_STAGE) > EPI_BYTES ? (OFF_W + NW * W_STAGE) : EPI_BYTES;
    // cv_full, cv_empty [NCV]; w_full, w_empty [NW]; r_full, r_free, g_full, g_free, p_ready, drain; epi [ROW_WARPS]
    static constexpr int N_BARS = 2 * NCV + 2 * NW + 6 + ROW_WARPS;
    static constexpr int SMEM = OFF_BAR + N_BARS * 8 + 16 + 1024;   // + TMEM slot and abort flag, + alignment
    // TMEM columns
    // R: two partial sums (dims 0 .. d/2 - 1 and d/2 .. d - 1), 32 columns each
    static constexpr uint32_t TM_PHI = 0, TM_PLO = D, TM_U = 2 * D, TM_R = 3 * D, TM_GHI = 3 * D + 2 * BK,
                              TM_GLO = TM_GHI + BK, TM_COLS = 512;
    static_assert(TM_GLO + BK <= TM_COLS, "TMEM columns");
    // the column and byte offsets lla_mma_r and lla_mma_u are written for
    static_assert(BK == 32 && TM_PLO == TM_PHI + D && TM_GLO == TM_GHI + 32 && PANEL == 4096, "MMA batch layout");
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

// ------------------------------------------------- batched tf32 MMA issue
// One warp-wide asm block per GEMM of a key tile, one elected lane issuing;
// the descriptors are the stage's base descriptors plus a compile-time offset
// in their low word (start address in 16-byte units; the offsets keep the
// address below 256 KB, so no carry into the next field).
//
// lla_mma_r<D>: R = P K^T of a 32-key tile as two partial sums, over dims
// [0, d/2) into t_d and [d/2, d) into t_d + 32; k-step s (8 dims) reads
// P_hi / P_lo at TMEM columns t_a + 8 s / t_a + d + 8 s and the K tile's
// panel s / 4 (32 rows x 128 B, 256 x 16 bytes apart) at (s % 4) x 32 bytes.
// In each partial the hi.lo and lo.hi products come first, the hi.hi ones
// last; the first MMA of a partial overwrites it.
template <int D>
__device__ __forceinline__ void lla_mma_r(uint32_t t_d, uint32_t t_a, uint64_t b_hi, uint64_t b_lo, uint32_t idesc);

template <>
__device__ __forceinline__ void lla_mma_r<64>(uint32_t t_d, uint32_t t_a, uint64_t b_hi, uint64_t b_lo, uint32_t idesc) {
    asm volatile("{\n\t.reg .pred e, pf, pt;\n\t.reg .b32 lo, ta, td;\n\t.reg .b64 db;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 pf, %0, %0;\n\tsetp.eq.b32 pt, %0, %0;\n\tadd.u32 td, %0, 0;\n\tadd.u32 ta, %1, 0; add.u32 lo, %4, 0; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pf;\n\tadd.u32 ta, %1, 64; add.u32 lo, %2, 0; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 8; add.u32 lo, %4, 2; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 72; add.u32 lo, %2, 2; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 16; add.u32 lo, %4, 4; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 80; add.u32 lo, %2, 4; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 24; add.u32 lo, %4, 6; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 88; add.u32 lo, %2, 6; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 0; add.u32 lo, %2, 0; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 8; add.u32 lo, %2, 2; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 16; add.u32 lo, %2, 4; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 24; add.u32 lo, %2, 6; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 td, %0, 32;\n\tadd.u32 ta, %1, 32; add.u32 lo, %4, 256; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pf;\n\tadd.u32 ta, %1, 96; add.u32 lo, %2, 256; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 40; add.u32 lo, %4, 258; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 104; add.u32 lo, %2, 258; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 48; add.u32 lo, %4, 260; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 112; add.u32 lo, %2, 260; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 56; add.u32 lo, %4, 262; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 120; add.u32 lo, %2, 262; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 32; add.u32 lo, %2, 256; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 40; add.u32 lo, %2, 258; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 48; add.u32 lo, %2, 260; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 56; add.u32 lo, %2, 262; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\t}"
                 ::"r"(t_d), "r"(t_a), "r"(static_cast<uint32_t>(b_hi)), "r"(static_cast<uint32_t>(b_hi >> 32)),
                   "r"(static_cast<uint32_t>(b_lo)), "r"(static_cast<uint32_t>(b_lo >> 32)), "r"(idesc)
                 : "memory");
}

template <>
__device__ __forceinline__ void lla_mma_r<128>(uint32_t t_d, uint32_t t_a, uint64_t b_hi, uint64_t b_lo, uint32_t idesc) {
    asm volatile("{\n\t.reg .pred e, pf, pt;\n\t.reg .b32 lo, ta, td;\n\t.reg .b64 db;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 pf, %0, %0;\n\tsetp.eq.b32 pt, %0, %0;\n\tadd.u32 td, %0, 0;\n\tadd.u32 ta, %1, 0; add.u32 lo, %4, 0; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pf;\n\tadd.u32 ta, %1, 128; add.u32 lo, %2, 0; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 8; add.u32 lo, %4, 2; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 136; add.u32 lo, %2, 2; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 16; add.u32 lo, %4, 4; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 144; add.u32 lo, %2, 4; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 24; add.u32 lo, %4, 6; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 152; add.u32 lo, %2, 6; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 32; add.u32 lo, %4, 256; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 160; add.u32 lo, %2, 256; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 40; add.u32 lo, %4, 258; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 168; add.u32 lo, %2, 258; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 48; add.u32 lo, %4, 260; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 176; add.u32 lo, %2, 260; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 56; add.u32 lo, %4, 262; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 184; add.u32 lo, %2, 262; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 0; add.u32 lo, %2, 0; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 8; add.u32 lo, %2, 2; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 16; add.u32 lo, %2, 4; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 24; add.u32 lo, %2, 6; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 32; add.u32 lo, %2, 256; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 40; add.u32 lo, %2, 258; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 48; add.u32 lo, %2, 260; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 56; add.u32 lo, %2, 262; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 td, %0, 32;\n\tadd.u32 ta, %1, 64; add.u32 lo, %4, 512; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pf;\n\tadd.u32 ta, %1, 192; add.u32 lo, %2, 512; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 72; add.u32 lo, %4, 514; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 200; add.u32 lo, %2, 514; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 80; add.u32 lo, %4, 516; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 208; add.u32 lo, %2, 516; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 88; add.u32 lo, %4, 518; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 216; add.u32 lo, %2, 518; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 96; add.u32 lo, %4, 768; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 224; add.u32 lo, %2, 768; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 104; add.u32 lo, %4, 770; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 232; add.u32 lo, %2, 770; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 112; add.u32 lo, %4, 772; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 240; add.u32 lo, %2, 772; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 120; add.u32 lo, %4, 774; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 248; add.u32 lo, %2, 774; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 64; add.u32 lo, %2, 512; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 72; add.u32 lo, %2, 514; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 80; add.u32 lo, %2, 516; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 88; add.u32 lo, %2, 518; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 96; add.u32 lo, %2, 768; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 104; add.u32 lo, %2, 770; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 112; add.u32 lo, %2, 772; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 120; add.u32 lo, %2, 774; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\t}"
                 ::"r"(t_d), "r"(t_a), "r"(static_cast<uint32_t>(b_hi)), "r"(static_cast<uint32_t>(b_hi >> 32)),
                   "r"(static_cast<uint32_t>(b_lo)), "r"(static_cast<uint32_t>(b_lo >> 32)), "r"(idesc)
                 : "memory");
}
// lla_mma_u: U_tile = G K of a 32-key tile (fresh): G_hi / G_lo at TMEM
// columns t_a + 8 s / t_a + 32 + 8 s, K^T [d][32 keys] at s x 32 bytes.
__device__ __forceinline__ void lla_mma_u(uint32_t t_d, uint32_t t_a, uint64_t b_hi, uint64_t b_lo, uint32_t idesc) {
    asm volatile("{\n\t.reg .pred e, pf, pt;\n\t.reg .b32 lo, ta, td;\n\t.reg .b64 db;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 pf, %0, %0;\n\tsetp.eq.b32 pt, %0, %0;\n\tmov.b32 td, %0;\n\tadd.u32 ta, %1, 0; add.u32 lo, %4, 0; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pf;\n\tadd.u32 ta, %1, 32; add.u32 lo, %2, 0; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 8; add.u32 lo, %4, 2; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 40; add.u32 lo, %2, 2; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 16; add.u32 lo, %4, 4; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 48; add.u32 lo, %2, 4; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 24; add.u32 lo, %4, 6; mov.b64 db, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 56; add.u32 lo, %2, 6; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 0; add.u32 lo, %2, 0; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 8; add.u32 lo, %2, 2; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 16; add.u32 lo, %2, 4; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\tadd.u32 ta, %1, 24; add.u32 lo, %2, 6; mov.b64 db, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::tf32 [td], [ta], db, %6, pt;\n\t}"
                 ::"r"(t_d), "r"(t_a), "r"(static_cast<uint32_t>(b_hi)), "r"(static_cast<uint32_t>(b_hi >> 32)),
                   "r"(static_cast<uint32_t>(b_lo)), "r"(static_cast<uint32_t>(b_lo >> 32)), "r"(idesc)
                 : "memory");
}

// One CG step over every row that is still active, reading the weights kept
// by the first step (p.wts, through mapW: dims {N, N, BH}, box {32, 128, 1}).
// The grid is n_blk * BH CTAs, the longest key ranges first.
template <int D>
__global__ void __launch_bounds__(LlaTcCfg<D>::THREADS, 1)
    plx_lla_cg_tc_kernel(const __grid_constant__ CUtensorMap mapW, const LlaParams p, int n_blk) {
    using Cfg = LlaTcCfg<D>;
    constexpr int BM = Cfg::BM, BK = Cfg::BK, NCV = Cfg::NCV, NW = Cfg::NW;
    extern __shared__ uint8_t lla_tc_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(lla_tc_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sCV = smem + Cfg::OFF_CV;
    uint8_t* sW = smem + Cfg::OFF_W;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    uint64_t* cv_full = bars;
    uint64_t* cv_empty = cv_full + NCV;
    uint64_t* w_full = cv_empty + NCV;
    uint64_t* w_empty = w_full + NW;
    uint64_t* r_full = w_empty + NW;
    uint64_t* r_free = r_full + 1;
    uint64_t* g_full = r_free + 1;
    uint64_t* g_free = g_full + 1;
    uint64_t* p_ready = g_free + 1;
    uint64_t* drain = p_ready + 1;
    uint64_t* epi = drain + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(epi + Cfg::ROW_WARPS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int BH = static_cast<int>(gridDim.x) / n_blk;
    const int xb = static_cast<int>(blockIdx.x) / BH;
    const int bh = static_cast<int>(blockIdx.x) - xb * BH;
    const int ib = (n_blk - 1 - xb) * BM;                  // the longest key ranges are launched first
    const int N = p.N;
    const int kend = min(ib + BM, N);                      // keys 0 .. kend - 1
    const int n_tiles = (kend + BK - 1) / BK;

    // ---- row scalars; a CTA whose rows have all stopped returns at once
    int act = 0;
    float rs = 0.f;
    const int i = ib + tid;                                // row warps: this thread's row
    const size_t grow = static_cast<size_t>(bh) * N + i;
    if (warp < Cfg::ROW_WARPS && i < N) {
        rs = p.rs[grow];
        act = rs > p.tol2 * p.rs0[grow] ? 1 : 0;
    }
    if (!__syncthreads_or(act)) return;

    if (warp == Cfg::W_MMA) {
        tmem_alloc(tmem_slot, Cfg::TM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < NCV; ++s) {
            mbar_init(&cv_full[s], Cfg::CV_WARPS);
            mbar_init(&cv_empty[s], 1);
        }
        for (int s = 0; s < NW; ++s) {
            mbar_init(&w_full[s], 1);
            mbar_init(&w_empty[s], Cfg::ROW_WARPS);
        }
        mbar_init(r_full, 1);
        mbar_init(r_free, Cfg::ROW_WARPS);
        mbar_init(g_full, Cfg::ROW_WARPS);
        mbar_init(g_free, 1);
        mbar_init(p_ready, Cfg::ROW_WARPS);
        mbar_init(drain, 1);
        for (int w = 0; w < Cfg::ROW_WARPS; ++w) mbar_init(&epi[w], 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&mapW);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto fail = [&]() {
        atomicOr(&g_plx_status, PLX_DEV_ERR_TIMEOUT);
        *abort_flag = 1;
    };
    auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity));
    };

    if (warp < Cfg::ROW_WARPS) {
        // ===================================================== row warps
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const float* prow = p.p + grow * D;
        const float* kbrow = p.kbar + grow * D;
        // p split into TMEM (0 for rows past N), and kbar . p
        float kbp = 0.f;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
            uint32_t hi[32], lo[32];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float4 pv = make_float4(0.f, 0.f, 0.f, 0.f), kv = pv;
                if (i < N) {
                    pv = *reinterpret_cast<const float4*>(prow + c * 32 + 4 * e);
                    kv = *reinterpret_cast<const float4*>(kbrow + c * 32 + 4 * e);
                }
                const float v4[4] = {pv.x, pv.y, pv.z, pv.w}, k4[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    kbp = fmaf(k4[m], v4[m], kbp);
                    const float h = tf32_hi(v4[m]);
                    hi[4 * e + m] = __float_as_uint(h);
                    lo[4 * e + m] = __float_as_uint(v4[m] - h);
                }
            }
            tmem_st32x32b_x32(lane_base + Cfg::TM_PHI + 32 * c, hi);
            tmem_st32x32b_x32(lane_base + Cfg::TM_PLO + 32 * c, lo);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_ready);

        // Sigma p of this row, summed tile by tile in fp32 with round-to-nearest:
        // each tile's G K is accumulated in TMEM by 12 MMAs only (the tensor
        // core's accumulation rounds toward zero, which over hundreds of MMAs
        // would bias the sum)
        float acc[D];
#pragma unroll
        for (int x = 0; x < D; ++x) acc[x] = 0.f;
        auto add_tile = [&]() {
#pragma unroll
            for (int c = 0; c < D / 16; ++c) {
                uint32_t u[16];
                tmem_ld32x32b_x16(lane_base + Cfg::TM_U + 16 * c, u);
#pragma unroll
                for (int x = 0; x < 16; ++x) acc[16 * c + x] += __uint_as_float(u[x]);
            }
        };
        bool ok = true;
        const uint8_t* wbase = sW + tid * 128;
        for (int t = 0; t < n_tiles; ++t) {
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) { ok = false; break; }   // one read for the warp
            // R of this tile first (its two partial sums, added in fp32), so the
            // next tile's R GEMM can start
            if (!wait_warp(r_full, t & 1)) { ok = false; break; }
            tc_fence_after();
            float rsum[BK];
            {
                uint32_t ra[32], rb2[32];
                tmem_ld32x32b_x32(lane_base + Cfg::TM_R, ra);
                tmem_ld32x32b_x32(lane_base + Cfg::TM_R + BK, rb2);
#pragma unroll
                for (int x = 0; x < BK; ++x) rsum[x] = __uint_as_float(ra[x]) + __uint_as_float(rb2[x]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(r_free);
            // the previous tile's G K is complete: add it, which also frees G
            if (t > 0) {
                if (!wait_warp(g_free, (t - 1) & 1)) { ok = false; break; }
                tc_fence_after();
                add_tile();
            }
            const int ws = t % NW;
            if (!wait_warp(&w_full[ws], (t / NW) & 1)) { ok = false; break; }
            const int j0 = t * BK;
            // G = w (R - kbar . p) in chunks of 8 keys, split into TMEM
#pragma unroll
            for (int c = 0; c < BK / 8; ++c) {
                uint32_t gh[8], gl[8];
                const uint8_t* wrow = wbase + ws * Cfg::W_STAGE;
                const float4 w0 = *reinterpret_cast<const float4*>(wrow + (((2 * c) ^ (tid & 7)) << 4));
                const float4 w1 = *reinterpret_cast<const float4*>(wrow + (((2 * c + 1) ^ (tid & 7)) << 4));
                const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    const int j = j0 + 8 * c + x;
                    const bool live = act && j <= i;       // act implies i < N
                    const float g = live ? wv[x] * (rsum[8 * c + x] - kbp) : 0.f;
                    const float h = tf32_hi(g);
                    gh[x] = __float_as_uint(h);
                    gl[x] = __float_as_uint(g - h);
                }
                asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                             ::"r"(lane_base + Cfg::TM_GHI + 8 * c), "r"(gh[0]), "r"(gh[1]), "r"(gh[2]),
                               "r"(gh[3]), "r"(gh[4]), "r"(gh[5]), "r"(gh[6]), "r"(gh[7])
                             : "memory");
                asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                             ::"r"(lane_base + Cfg::TM_GLO + 8 * c), "r"(gl[0]), "r"(gl[1]), "r"(gl[2]),
                               "r"(gl[3]), "r"(gl[4]), "r"(gl[5]), "r"(gl[6]), "r"(gl[7])
                             : "memory");
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&w_empty[ws]);
                mbar_arrive(g_full);
            }
        }
        // the epilogue's rows (below) in shared memory: p, x, r of each row warp,
        // padded to D + 4 floats, over the converter and weight buffers
        constexpr int LDE = Cfg::LDE;
        float* pr = reinterpret_cast<float*>(smem) + (warp * 3 * 32 + lane) * LDE;
        float* xr = pr + 32 * LDE;
        float* rr = xr + 32 * LDE;
        if (ok) {
            if (wait_warp(g_free, (n_tiles - 1) & 1)) {
                // every MMA has finished and every tile has been consumed, so those
                // buffers are free: each lane fetches its row of p, x and r by 1-D bulk
                // copies (all in flight at once) while the last tile is added
                const int nrow = max(0, min(32, N - (ib + warp * 32)));   // the warp's rows inside the head
                if (lane == 0) mbar_arrive_expect_tx(&epi[warp], static_cast<uint32_t>(nrow) * 3 * D * 4);
                __syncwarp();
                if (i < N) {
                    bulk_g2s(pr, p.p + grow * D, D * 4, &epi[warp]);
                    bulk_g2s(xr, p.x + grow * D, D * 4, &epi[warp]);
                    bulk_g2s(rr, p.r + grow * D, D * 4, &epi[warp]);
                }
                tc_fence_after();
                add_tile();
                if (!wait_warp(&epi[warp], 0)) ok = false;   // (the copies complete on their own)
            } else {
                ok = false;
            }
        }
        if (!ok) {
            fail();
        } else {
            // ---- Ap = U + lambda p and one conjugate-gradient step per active row,
            // on the row in shared memory (the lanes' padded rows fall on different
            // banks); the updated rows go back by 1-D bulk copies
            {
                float pap = 0.f;
                if (act) {
#pragma unroll
                    for (int o = 0; o < D; o += 4) {
                        const float4 pv = *reinterpret_cast<const float4*>(pr + o);
                        const float v4[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            acc[o + m] = fmaf(p.lambda, v4[m], acc[o + m]);   // acc := Ap
                            pap = fmaf(v4[m], acc[o + m], pap);
                        }
                        asm volatile("" ::: "memory");
                    }
                }
                const bool okr = act && pap > 0.f;
                if (act && !okr) p.rs[grow] = 0.f;         // breakdown: stop the row
                if (okr) {
                    const float alpha = rs / pap;
                    float rn = 0.f;
#pragma unroll
                    for (int o = 0; o < D; o += 4) {
                        const float4 pv = *reinterpret_cast<const float4*>(pr + o);
                        const float4 xv = *reinterpret_cast<const float4*>(xr + o);
                        const float4 rv = *reinterpret_cast<const float4*>(rr + o);
                        const float v4[4] = {pv.x, pv.y, pv.z, pv.w};
                        float x4[4] = {xv.x, xv.y, xv.z, xv.w}, r4[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            x4[m] = fmaf(alpha, v4[m], x4[m]);
                            r4[m] = fmaf(-alpha, acc[o + m], r4[m]);
                            rn = fmaf(r4[m], r4[m], rn);
                        }
                        *reinterpret_cast<float4*>(xr + o) = make_float4(x4[0], x4[1], x4[2], x4[3]);
                        *reinterpret_cast<float4*>(rr + o) = make_float4(r4[0], r4[1], r4[2], r4[3]);
                        asm volatile("" ::: "memory");     // keep the loads of later dims from being hoisted
                    }
                    const float beta = rn / rs;
#pragma unroll
                    for (int o = 0; o < D; o += 4) {
                        const float4 pv = *reinterpret_cast<const float4*>(pr + o);
                        const float4 rv = *reinterpret_cast<const float4*>(rr + o);
                        *reinterpret_cast<float4*>(pr + o) = make_float4(fmaf(beta, pv.x, rv.x), fmaf(beta, pv.y, rv.y),
                                                                         fmaf(beta, pv.z, rv.z), fmaf(beta, pv.w, rv.w));
                    }
                    p.rs[grow] = rn;
                    p.steps[grow] += 1;
                    // the rows back to global memory; the CTA leaves only once they are written
                    fence_proxy_async_smem();
                    bulk_s2g(p.x + grow * D, xr, D * 4);
                    bulk_s2g(p.r + grow * D, rr, D * 4);
                    bulk_s2g(p.p + grow * D, pr, D * 4);
                    bulk_commit_group();
                    bulk_wait_all();
                }
            }
        }
    } else if (warp == Cfg::W_PROD) {
        // ===================================================== weight producer
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            for (int t = 0; t < n_tiles; ++t) {
                if (*abort_flag) break;
                const int ws = t % NW;
                if (t >= NW && !mbar_wait(&w_empty[ws], ((t / NW) - 1) & 1)) { ok = false; break; }
                mbar_arrive_expect_tx(&w_full[ws], Cfg::W_STAGE);
                tma_load_3d(sW + ws * Cfg::W_STAGE, &mapW, &w_full[ws], t * BK, ib, bh);
                ++issued;
            }
            if (!ok) fail();
            // never leave with loads in flight into this CTA's shared memory
            for (int t = max(0, issued - NW); t < issued; ++t)
                if (!mbar_wait(&w_full[t % NW], (t / NW) & 1)) fail();
        }
    } else if (warp == Cfg::W_MMA) {
        // ===================================================== MMA issuer
        constexpr uint32_t ID_R = idesc_tf32_f32(128, BK), ID_U = idesc_tf32_f32(128, D);
        const uint32_t cv0 = smem_u32(sCV);
        bool ok = wait_warp(p_ready, 0);
        int issued_any = 0;
        // U_tile = G K for tile tp (G in TMEM, K^T of its stage), a fresh
        // accumulator per tile; the small hi.lo and lo.hi products first, so
        // only the 4 hi.hi MMAs add to a sum of full size
        auto gemm_u = [&](int tp) -> bool {
            if (!wait_warp(g_full, tp & 1)) return false;
            tc_fence_after();
            const uint32_t kb_hi = cv0 + (tp % NCV) * Cfg::CV_STAGE + 2 * Cfg::KA_BYTES;
            lla_mma_u(tmem + Cfg::TM_U, tmem + Cfg::TM_GHI, sdesc_sw128(kb_hi, 16, 1024),
                      sdesc_sw128(kb_hi + Cfg::KB_BYTES, 16, 1024), ID_U);
            mma_commit_warp(g_free);                     // U_tile complete, G free
            mma_commit_warp(&cv_empty[tp % NCV]);
            return true;
        };
        for (int t = 0; ok && t < n_tiles; ++t) {
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) { ok = false; break; }   // one read for the warp
            const int cs = t % NCV;
            if (!wait_warp(&cv_full[cs], (t / NCV) & 1)) { ok = false; break; }
            // R of the previous tile has been read by the row warps
            if (t >= 1 && !wait_warp(r_free, (t - 1) & 1)) { ok = false; break; }
            tc_fence_after();
            {
                // two partial sums over halves of the dims (the small products first)
                const uint32_t ka_hi = cv0 + cs * Cfg::CV_STAGE;
                lla_mma_r<D>(tmem + Cfg::TM_R, tmem + Cfg::TM_PHI, sdesc_sw128(ka_hi, 16, 1024),
                             sdesc_sw128(ka_hi + Cfg::KA_BYTES, 16, 1024), ID_R);
                mma_commit_warp(r_full);
            }
            issued_any = 1;
            // the previous tile's U GEMM after this tile's R GEMM, so the row warps
            // form G of tile t - 1 while R of tile t runs
            if (t > 0 && !gemm_u(t - 1)) { ok = false; break; }
        }
        if (ok && n_tiles > 0 && !gemm_u(n_tiles - 1)) ok = false;
        if (!ok) fail();
        // drain: every MMA issued by this warp has finished before TMEM is freed
        if (issued_any) {
            mma_commit_warp(drain);
            if (!wait_warp(drain, 0)) fail();
        }
    } else {
        // ===================================================== converters
        // Thread ct handles 4 x 4 blocks: keys 4l .. 4l+3 and dims 32c + 4u .. +3
        // with l = ct % 8, u = l ^ x, (c, x) = combo z = ct / 8 + 8 h.  In a
        // quarter-warp (l = 0..7, one z) the 16-byte units written to both layouts
        // fall on 8 different bank groups.
        constexpr int QW = Cfg::CV_WARPS * 4;              // quarter-warps of the converters
        constexpr int Z = D / 4;                           // combos (c, x): D/32 panels x 8
        constexpr int NB = Z / QW;                         // blocks per thread
        static_assert(Z % QW == 0, "converter blocks");
        const int ct = tid - Cfg::W_CV0 * 32;
        const int l = ct & 7, qw = ct >> 3;
        const float* K = p.k + static_cast<size_t>(bh) * N * D;
        float4 cur[NB][4];
        auto load_tile = [&](int t, float4 (&v)[NB][4]) {
            const int j0 = t * BK;
#pragma unroll
            for (int h = 0; h < NB; ++h) {
                const int z = qw + QW * h, c = z >> 3, u = l ^ (z & 7);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = j0 + 4 * l + e;
                    v[h][e] = j < kend ? *reinterpret_cast<const float4*>(K + static_cast<size_t>(j) * D + 32 * c + 4 * u)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
        };
        bool ok = true;
        for (int t = 0; t < n_tiles; ++t) {
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) { ok = false; break; }   // one read for the warp
            // the tile's loads go out before the wait for a free stage (the ring of
            // NCV converted stages keeps the converters ahead of the MMAs)
            load_tile(t, cur);
            const int cs = t % NCV;
            if (t >= NCV && !wait_warp(&cv_empty[cs], ((t / NCV) - 1) & 1)) { ok = false; break; }
            uint8_t* ka_hi = sCV + cs * Cfg::CV_STAGE;
            uint8_t* ka_lo = ka_hi + Cfg::KA_BYTES;
            uint8_t* kb_hi = ka_hi + 2 * Cfg::KA_BYTES;
            uint8_t* kb_lo = kb_hi + Cfg::KB_BYTES;
#pragma unroll
            for (int h = 0; h < NB; ++h) {
                const int z = qw + QW * h, c = z >> 3, u = l ^ (z & 7);
                float hv[4][4], lv[4][4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float x4[4] = {cur[h][e].x, cur[h][e].y, cur[h][e].z, cur[h][e].w};
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        hv[e][m] = tf32_hi(x4[m]);
                        lv[e][m] = x4[m] - hv[e][m];
                    }
                }
                // [32 keys][d]: key n = 4l + e, 16-byte unit u of panel c
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int n = 4 * l + e;
                    const int off = c * Cfg::PANEL + n * 128 + ((u ^ (n & 7)) << 4);
                    *reinterpret_cast<float4*>(ka_hi + off) = make_float4(hv[e][0], hv[e][1], hv[e][2], hv[e][3]);
                    *reinterpret_cast<float4*>(ka_lo + off) = make_float4(lv[e][0], lv[e][1], lv[e][2], lv[e][3]);
                }
                // [d][32 keys]: dim dd = 32c + 4u + m, 16-byte unit l (keys 4l .. 4l+3)
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int dd = 32 * c + 4 * u + m;
                    const int off = dd * 128 + ((l ^ (dd & 7)) << 4);
                    *reinterpret_cast<float4*>(kb_hi + off) = make_float4(hv[0][m], hv[1][m], hv[2][m], hv[3][m]);
                    *reinterpret_cast<float4*>(kb_lo + off) = make_float4(lv[0][m], lv[1][m], lv[2][m], lv[3][m]);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&cv_full[cs]);
        }
        if (!ok) fail();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == Cfg::W_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::TM_COLS);
    }
}

}  // namespace plx
