// bwd_f32.cuh -- plx_bwd_f32: gradients of causal PLX attention in fp32 on
// the CUDA cores.
//
// Forward ("Parallax: Parameterized Local Linear Attention for Language
// Modeling", zhichai.net section 1.3; gist.science "Meccanismo Principale"):
//   s_ij = scale q_i.k_j,  w_ij = softmax_{j<=i} s_ij,  r_ij = rho_i.k_j,
//   vbar_i = sum_j w_ij v_j,  c_i = sum_j w_ij r_ij,  u_i = sum_j w_ij r_ij v_j,
//   o_i = (1 + c_i) vbar_i - u_i.
// The pages give no backward pass; differentiating the forward with
// dO_i = dL/do_i, G_ij = dO_i.v_j and a_i = dO_i.vbar_i gives
//   dL/dw_ij = (1 + c_i - r_ij) G_ij + a_i r_ij
//   dL/ds_ij = w_ij (dL/dw_ij - D_i),  D_i = sum_j w_ij dL/dw_ij = dO_i.o_i + c_i a_i
//   dL/dr_ij = w_ij (a_i - G_ij)
//   dq_i = scale sum_j ds_ij k_j          drho_i = sum_j dr_ij k_j
//   dk_j = scale sum_i ds_ij q_i + sum_i dr_ij rho_i
//   dv_j = sum_i w_ij (1 + c_i - r_ij) dO_i
// with w_ij = e^{s_ij - lse_i} from the forward's log-sum-exp.
//
// Three passes, each one warp per row with lane t owning dims t, t+32, ...:
//   pre:  per query row, vbar_i and c_i again from lse, then (c_i, a_i, D_i)
//         into the workspace;
//   dq:   per query row, over keys j <= i: dq_i, drho_i;
//   dkv:  per key row, over queries i >= j: dk_j, dv_j.
// Every (i, j) pair is recomputed in each pass, so no pass needs atomics and
// the result does not depend on the order of the blocks.
#pragma once
#include "status.cuh"

namespace plx {

struct BwdF32Params {
    const float* q;
    const float* k;
    const float* v;
    const float* rho;     // nullptr: softmax attention (rho = 0)
    const float* out;
    const float* lse;
    const float* dout;
    float* dq;
    float* dk;
    float* dv;
    float* drho;          // unused when rho is nullptr
    float* ws;            // per query row: c, a, D, (pad)
    int N;
    float scale;
};

constexpr int BWD_WARPS = 4;
constexpr int BWD_ROWS_PER_BLOCK = 16;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    return x;
}

template <int DPL>
__device__ __forceinline__ void load_row_f32(const float* row, int lane, float (&f)[DPL]) {
#pragma unroll
    for (int t = 0; t < DPL; ++t) f[t] = row[lane + 32 * t];
}

// pre-pass: (c_i, a_i, D_i) for every query row
template <int DPL, bool PLX>
__global__ void __launch_bounds__(BWD_WARPS * 32) plx_bwd_pre_kernel(const BwdF32Params p) {
    constexpr int D = DPL * 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.y;
    const size_t head = static_cast<size_t>(bh) * p.N * D;
    for (int rr = warp; rr < BWD_ROWS_PER_BLOCK; rr += BWD_WARPS) {
        const int i = blockIdx.x * BWD_ROWS_PER_BLOCK + rr;
        if (i >= p.N) break;
        const size_t ri = head + static_cast<size_t>(i) * D;
        float qv[DPL], rv[DPL], vbar[DPL];
        load_row_f32<DPL>(p.q + ri, lane, qv);
        if constexpr (PLX) load_row_f32<DPL>(p.rho + ri, lane, rv);
#pragma unroll
        for (int t = 0; t < DPL; ++t) vbar[t] = 0.f;
        const float lse = p.lse[static_cast<size_t>(bh) * p.N + i];
        float c = 0.f;
        for (int j = 0; j <= i; ++j) {
            float kf[DPL], vf[DPL];
            load_row_f32<DPL>(p.k + head + static_cast<size_t>(j) * D, lane, kf);
            load_row_f32<DPL>(p.v + head + static_cast<size_t>(j) * D, lane, vf);
            float sd = 0.f, rd = 0.f;
#pragma unroll
            for (int t = 0; t < DPL; ++t) {
                sd = fmaf(qv[t], kf[t], sd);
                if constexpr (PLX) rd = fmaf(rv[t], kf[t], rd);
            }
            sd = warp_sum(sd);
            if constexpr (PLX) rd = warp_sum(rd);
            const float w = expf(sd * p.scale - lse);
#pragma unroll
            for (int t = 0; t < DPL; ++t) vbar[t] = fmaf(w, vf[t], vbar[t]);
            if constexpr (PLX) c = fmaf(w, rd, c);
        }
        float go[DPL], of[DPL];
        load_row_f32<DPL>(p.dout + ri, lane, go);
        load_row_f32<DPL>(p.out + ri, lane, of);
        float a = 0.f, dodo = 0.f;
#pragma unroll
        for (int t = 0; t < DPL; ++t) {
            a = fmaf(go[t], vbar[t], a);
            dodo = fmaf(go[t], of[t], dodo);
        }
        a = warp_sum(a);
        dodo = warp_sum(dodo);
        if (lane == 0) {
            float4* w4 = reinterpret_cast<float4*>(p.ws) + static_cast<size_t>(bh) * p.N + i;
            *w4 = make_float4(c, a, fmaf(c, a, dodo), 0.f);
        }
    }
}

// dq, drho: one warp per query row, keys j <= i
template <int DPL, bool PLX>
__global__ void __launch_bounds__(BWD_WARPS * 32) plx_bwd_dq_kernel(const BwdF32Params p) {
    constexpr int D = DPL * 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.y;
    const size_t head = static_cast<size_t>(bh) * p.N * D;
    for (int rr = warp; rr < BWD_ROWS_PER_BLOCK; rr += BWD_WARPS) {
        const int i = blockIdx.x * BWD_ROWS_PER_BLOCK + rr;
        if (i >= p.N) break;
        const size_t ri = head + static_cast<size_t>(i) * D;
        float qv[DPL], rv[DPL], go[DPL], dq[DPL], dr[DPL];
        load_row_f32<DPL>(p.q + ri, lane, qv);
        load_row_f32<DPL>(p.dout + ri, lane, go);
        if constexpr (PLX) load_row_f32<DPL>(p.rho + ri, lane, rv);
#pragma unroll
        for (int t = 0; t < DPL; ++t) {
            dq[t] = 0.f;
            dr[t] = 0.f;
        }
        const float lse = p.lse[static_cast<size_t>(bh) * p.N + i];
        const float4 cad = reinterpret_cast<const float4*>(p.ws)[static_cast<size_t>(bh) * p.N + i];
        for (int j = 0; j <= i; ++j) {
            float kf[DPL], vf[DPL];
            load_row_f32<DPL>(p.k + head + static_cast<size_t>(j) * D, lane, kf);
            load_row_f32<DPL>(p.v + head + static_cast<size_t>(j) * D, lane, vf);
            float sd = 0.f, rd = 0.f, gd = 0.f;
#pragma unroll
            for (int t = 0; t < DPL; ++t) {
                sd = fmaf(qv[t], kf[t], sd);
                gd = fmaf(go[t], vf[t], gd);
                if constexpr (PLX) rd = fmaf(rv[t], kf[t], rd);
            }
            sd = warp_sum(sd);
            gd = warp_sum(gd);
            if constexpr (PLX) rd = warp_sum(rd);
            const float w = expf(sd * p.scale - lse);
            // dL/dw = (1 + c - r) G + a r;  ds = w (dL/dw - D);  dr = w (a - G)
            const float gw = fmaf(1.f + cad.x - rd, gd, cad.y * rd);
            const float ds = w * (gw - cad.z);
            const float drr = w * (cad.y - gd);
#pragma unroll
            for (int t = 0; t < DPL; ++t) {
                dq[t] = fmaf(ds, kf[t], dq[t]);
                if constexpr (PLX) dr[t] = fmaf(drr, kf[t], dr[t]);
            }
        }
#pragma unroll
        for (int t = 0; t < DPL; ++t) {
            p.dq[ri + lane + 32 * t] = dq[t] * p.scale;
            if constexpr (PLX) p.drho[ri + lane + 32 * t] = dr[t];
        }
    }
}

// dk, dv: one warp per key row j, queries i >= j
template <int DPL, bool PLX>
__global__ void __launch_bounds__(BWD_WARPS * 32) plx_bwd_dkv_kernel(const BwdF32Params p) {
    constexpr int D = DPL * 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.y;
    const size_t head = static_cast<size_t>(bh) * p.N * D;
    for (int rr = warp; rr < BWD_ROWS_PER_BLOCK; rr += BWD_WARPS) {
        const int j = blockIdx.x * BWD_ROWS_PER_BLOCK + rr;
        if (j >= p.N) break;
        const size_t rj = head + static_cast<size_t>(j) * D;
        float kf[DPL], vf[DPL], dk[DPL], dv[DPL];
        load_row_f32<DPL>(p.k + rj, lane, kf);
        load_row_f32<DPL>(p.v + rj, lane, vf);
#pragma unroll
        for (int t = 0; t < DPL; ++t) {
            dk[t] = 0.f;
            dv[t] = 0.f;
        }
        for (int i = j; i < p.N; ++i) {
            const size_t ri = head + static_cast<size_t>(i) * D;
            float qv[DPL], rv[DPL], go[DPL];
            load_row_f32<DPL>(p.q + ri, lane, qv);
            load_row_f32<DPL>(p.dout + ri, lane, go);
            if constexpr (PLX) load_row_f32<DPL>(p.rho + ri, lane, rv);
            float sd = 0.f, rd = 0.f, gd = 0.f;
#pragma unroll
            for (int t = 0; t < DPL; ++t) {
                sd = fmaf(qv[t], kf[t], sd);
                gd = fmaf(go[t], vf[t], gd);
                if constexpr (PLX) rd = fmaf(rv[t], kf[t], rd);
            }
            sd = warp_sum(sd);
            gd = warp_sum(gd);
            if constexpr (PLX) rd = warp_sum(rd);
            const float lse = p.lse[static_cast<size_t>(bh) * p.N + i];
            const float4 cad = reinterpret_cast<const float4*>(p.ws)[static_cast<size_t>(bh) * p.N + i];
            const float w = expf(sd * p.scale - lse);
            const float gw = fmaf(1.f + cad.x - rd, gd, cad.y * rd);
            const float ds = w * (gw - cad.z) * p.scale;
            const float drr = w * (cad.y - gd);
            const float wv = w * (1.f + cad.x - rd);
#pragma unroll
            for (int t = 0; t < DPL; ++t) {
                dk[t] = fmaf(ds, qv[t], dk[t]);
                if constexpr (PLX) dk[t] = fmaf(drr, rv[t], dk[t]);
                dv[t] = fmaf(wv, go[t], dv[t]);
            }
        }
#pragma unroll
        for (int t = 0; t < DPL; ++t) {
            p.dk[rj + lane + 32 * t] = dk[t];
            p.dv[rj + lane + 32 * t] = dv[t];
        }
    }
}

}  // namespace plx
