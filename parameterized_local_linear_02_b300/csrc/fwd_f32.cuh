// fwd_f32.cuh -- plx_fwd_f32: causal PLX forward in fp32 on the CUDA cores.
//
// The high-precision path (fp32 inputs, fp32 arithmetic, no tensor cores).
// One warp owns one query row i at a time and streams keys j = 0..i with an
// exact (non-lazy) online softmax in natural-log units:
//   s = scale q.k_j, r = rho.k_j,  m' = max(m, s),  a = e^{m-m'},  p = e^{s-m'}
//   l = a l + p,  C = a C + p r,  A = a A + p v_j,  U = a U + p r v_j
// and finishes o = (1 + C/l) A/l - U/l, lse = m + ln l ("Parallax:
// Parameterized Local Linear Attention for Language Modeling", zhichai.net
// section 1.3, with the streaming identity of gist.science "Algoritmo
// Consapevole dell'Hardware").  Lane t owns dims t, t+32, ... so every key
// row is read with coalesced 128-byte accesses.
#pragma once
#include "status.cuh"

namespace plx {

struct FwdF32Params {
    const float* q;
    const float* k;
    const float* v;
    const float* rho;
    float* out;
    float* lse;
    int N;
    float scale;
};

constexpr int F32_WARPS = 4;
constexpr int F32_ROWS_PER_BLOCK = 16;

template <int DPL, bool PLX>
__global__ void __launch_bounds__(F32_WARPS * 32) plx_fwd_f32_kernel(const FwdF32Params p) {
    constexpr int D = DPL * 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.y;
    const size_t head = static_cast<size_t>(bh) * p.N * D;
    const float* K = p.k + head;
    const float* V = p.v + head;
    for (int rr = warp; rr < F32_ROWS_PER_BLOCK; rr += F32_WARPS) {
        const int i = blockIdx.x * F32_ROWS_PER_BLOCK + rr;
        if (i >= p.N) break;
        float qv[DPL], rv[DPL], A[DPL], U[DPL];
#pragma unroll
        for (int t = 0; t < DPL; ++t) {
            qv[t] = p.q[head + static_cast<size_t>(i) * D + lane + 32 * t];
            rv[t] = PLX ? p.rho[head + static_cast<size_t>(i) * D + lane + 32 * t] : 0.f;
            A[t] = 0.f;
            U[t] = 0.f;
        }
        float m = -INFINITY, l = 0.f, C = 0.f;
        for (int j = 0; j <= i; ++j) {
            const float* kj = K + static_cast<size_t>(j) * D;
            const float* vj = V + static_cast<size_t>(j) * D;
            float kf[DPL], vf[DPL];
            float sd = 0.f, rd = 0.f;
#pragma unroll
            for (int t = 0; t < DPL; ++t) {
                kf[t] = kj[lane + 32 * t];
                vf[t] = vj[lane + 32 * t];
                sd = fmaf(qv[t], kf[t], sd);
                if constexpr (PLX) rd = fmaf(rv[t], kf[t], rd);
            }
#pragma unroll
            for (int msk = 16; msk >= 1; msk >>= 1) {
                sd += __shfl_xor_sync(0xffffffffu, sd, msk);
                if constexpr (PLX) rd += __shfl_xor_sync(0xffffffffu, rd, msk);
            }
            const float s = sd * p.scale;
            const float m_new = fmaxf(m, s);
            const float a = expf(m - m_new);
            const float pe = expf(s - m_new);
            l = fmaf(a, l, pe);
#pragma unroll
            for (int t = 0; t < DPL; ++t) A[t] = fmaf(a, A[t], pe * vf[t]);
            if constexpr (PLX) {
                const float pr = pe * rd;
                C = fmaf(a, C, pr);
#pragma unroll
                for (int t = 0; t < DPL; ++t) U[t] = fmaf(a, U[t], pr * vf[t]);
            }
            m = m_new;
        }
        const float inv = 1.f / l;
        const float c = C * inv;
#pragma unroll
        for (int t = 0; t < DPL; ++t) {
            const float vbar = A[t] * inv;
            const float o = PLX ? fmaf(c, vbar, vbar) - U[t] * inv : vbar;
            p.out[head + static_cast<size_t>(i) * D + lane + 32 * t] = o;
        }
        if (lane == 0 && p.lse) p.lse[static_cast<size_t>(bh) * p.N + i] = m + logf(l);
    }
}

}  // namespace plx
