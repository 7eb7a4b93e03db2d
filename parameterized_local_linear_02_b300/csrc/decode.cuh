// decode.cuh -- plx_decode: one query token per (b, h) against a bf16 KV
// cache, split over thread blocks, merged by a log-sum-exp weighted combine.
//
// Streaming decode of "Parallax: Parameterized Local Linear Attention for
// Language Modeling" (gist.science, "Algoritmo Consapevole dell'Hardware":
// the softmax and covariance branches share one K/V stream).  Per cache row
// j of a split the kernel forms
//   s_j = scale * q.k_j  (kept in log2 units),  r_j = rho.k_j,
// and keeps the online-softmax state
//   m = max s,  l = sum e^{s-m},  C = sum e^{s-m} r,
//   A = sum e^{s-m} v_j,  U = sum e^{s-m} r_j v_j,
// from which o = (1 + C/l) A/l - U/l (zhichai.net section 1.3 with the
// streaming identity Sigma_KV rho = sum w r v - vbar (kbar.rho)).
//
// Memory path: one producer thread streams T-row K and V tiles of the split
// into an NSTAGE ring in shared memory with 1-D bulk copies (TMA engine,
// L2 evict-first); four consumer warps each take T/4 rows of every tile.  A
// warp computes the two dot products of its rows with lanes owning D/32
// dims, reduces all of them at once with a transposed butterfly (one shuffle
// per dot product), and updates its own online state.  The four warp states
// are merged in shared memory at the end of the split.
#pragma once
#include "status.cuh"

namespace plx {

// the largest split count whose combine runs inside one thread-block cluster
// (clusters of more than 8 CTAs are the non-portable, opt-in sizes)
constexpr int DECODE_MAX_CLUSTER_SPLITS = 16;

template <int D>
struct DecodeCfg {
    static constexpr int T = 32;                    // cache rows per stage
    static constexpr int NSTAGE = 4;
    static constexpr int CWARPS = 4;                // consumer warps
    static constexpr int THREADS = (CWARPS + 1) * 32;
    static constexpr int ROWS_PER_WARP = T / CWARPS;
    static constexpr int DPL = D / 32;              // dims per lane
    static constexpr int TILE_BYTES = T * D * 2;    // one tensor, one stage
    static constexpr int PART = 2 * D + 4;          // floats per partial: m, l, C, pad, A[D], U[D]
    // smem: K ring, V ring, merge area, barriers
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = NSTAGE * TILE_BYTES;
    static constexpr int OFF_MERGE = 2 * NSTAGE * TILE_BYTES;
    static constexpr int MERGE_FLOATS = CWARPS * PART;
    // the block's own state, read by the cluster's rank 0 in the fused combine
    static constexpr int OFF_CPART = OFF_MERGE + MERGE_FLOATS * 4;
    static constexpr int OFF_BAR = OFF_CPART + PART * 4;
    static constexpr int SMEM = OFF_BAR + 2 * NSTAGE * 8 + 16;
    static_assert(D == 64 || D == 128, "decode supports d in {64, 128}");
    static_assert(ROWS_PER_WARP == 8, "transposed reduction assumes 8 rows per warp");
};

struct DecodeParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* rho;
    const __nv_bfloat16* kc;
    const __nv_bfloat16* vc;
    const int* seqlens;
    void* out;
    float* lse;
    float* ws;          // partials [B*H][splits][PART] (unused when splits == 1)
    int H;
    int S_cap;
    int splits;
    float scale_log2;   // scale * log2(e)
    int out_f32;
    int no_intercept;   // the family's no-intercept member: o = -u
    // paged cache (block_table != nullptr): kc, vc are [num_blocks][H][page][D]
    // and row r of sequence b lives in block block_table[b][r / page] at row
    // r % page; S_cap is max_blocks * page.  page is a multiple of T, so a
    // tile never straddles two blocks.
    const int* block_table;
    int max_blocks;
    int page;
    int num_blocks;
    // A shard of the key range (plx_decode_partials): the cache holds the
    // positions key_begin .. key_begin + S_cap - 1, so sequence b has
    // clamp(seqlens[b] - key_begin, 0, S_cap) of its keys here; the split
    // partials are always written (never the output), and a length past this
    // shard is not an error (those keys live in a later shard).
    int key_begin = 0;
    int partials_only = 0;
    // the combine merges groups x splits partials per (b, h), laid out
    // [groups][B*H][splits][PART] (groups = 1: the split kernel's own layout)
    int groups = 1;
};

__device__ __forceinline__ float bf16lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

// Load this lane's DPL dims of one bf16 row from shared memory as floats.
template <int DPL>
__device__ __forceinline__ void load_row(const __nv_bfloat16* row, int lane, float (&f)[DPL]) {
    if constexpr (DPL == 4) {
        uint2 u = *reinterpret_cast<const uint2*>(row + lane * 4);
        f[0] = bf16lo(u.x); f[1] = bf16hi(u.x); f[2] = bf16lo(u.y); f[3] = bf16hi(u.y);
    } else {
        uint32_t u = *reinterpret_cast<const uint32_t*>(row + lane * 2);
        f[0] = bf16lo(u); f[1] = bf16hi(u);
    }
}

// Finalise: o = (1 + C/L) A/L - U/L, written as out_dtype.
__device__ __forceinline__ void store_out(void* out, int out_f32, size_t idx, float v) {
    if (out_f32) reinterpret_cast<float*>(out)[idx] = v;
    else reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
}

// The cluster combine: every split of one (b, h) is a CTA of one thread-block
// cluster (splits <= 16), each CTA leaves its state in its shared memory,
// and the cluster's rank 0 reads them through distributed shared memory and
// writes the output.  One launch instead of split kernel + combine kernel.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ float ld_cluster_f32(const float* local, uint32_t rank) {
    uint32_t remote;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

template <int D, bool PLX, bool FUSED = false>
__global__ void __launch_bounds__(DecodeCfg<D>::THREADS)
plx_decode_split_kernel(const DecodeParams p) {
    using Cfg = DecodeCfg<D>;
    constexpr int T = Cfg::T, NSTAGE = Cfg::NSTAGE, DPL = Cfg::DPL;
    extern __shared__ __align__(128) uint8_t smem[];
    __nv_bfloat16* kbuf = reinterpret_cast<__nv_bfloat16*>(smem + Cfg::OFF_K);
    __nv_bfloat16* vbuf = reinterpret_cast<__nv_bfloat16*>(smem + Cfg::OFF_V);
    float* merge = reinterpret_cast<float*>(smem + Cfg::OFF_MERGE);
    float* cpart = reinterpret_cast<float*>(smem + Cfg::OFF_CPART);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    uint64_t* empty = full + NSTAGE;
    int* abort_flag = reinterpret_cast<int*>(empty + NSTAGE);

    const int bh = blockIdx.x;          // grid: x = b*h (up to 2^31-1), y = split
    const int split = blockIdx.y;
    const int b = bh / p.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    int L = p.seqlens[b];
    if (p.partials_only) {
        L -= p.key_begin;
        L = L > p.S_cap ? p.S_cap : L;
    } else if (L > p.S_cap) {
        if (threadIdx.x == 0 && split == 0 && (bh % p.H) == 0) atomicOr(&g_plx_status, PLX_DEV_ERR_SEQLEN);
        L = p.S_cap;
    }
    if (L < 0) L = 0;
    const int ntiles = (L + T - 1) / T;
    const int tps = (ntiles + p.splits - 1) / p.splits;
    const int t_begin = min(split * tps, ntiles);
    const int t_end = min(t_begin + tps, ntiles);
    const int my_tiles = t_end - t_begin;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], Cfg::CWARPS);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const size_t head_row0 = static_cast<size_t>(bh) * p.S_cap;

    if (warp == Cfg::CWARPS) {
        // ---------------- producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int issued = 0;
            for (int i = 0; i < my_tiles; ++i) {
                const int s = i % NSTAGE;
                if (i >= NSTAGE) {
                    if (!mbar_wait(&empty[s], ((i / NSTAGE) - 1) & 1)) {
                        atomicOr(&g_plx_status, PLX_DEV_ERR_TIMEOUT);
                        atomicExch(abort_flag, 1);
                        break;
                    }
                }
                if (*reinterpret_cast<volatile int*>(abort_flag)) break;
                const int t = t_begin + i;
                const int rows = min(T, L - t * T);
                const uint32_t bytes = static_cast<uint32_t>(rows) * D * 2;
                size_t g = (head_row0 + static_cast<size_t>(t) * T) * D;
                if (p.block_table) {
                    const int r0 = t * T;
                    const int pg = r0 / p.page;
                    int blk = p.block_table[static_cast<size_t>(b) * p.max_blocks + pg];
                    if (blk < 0 || blk >= p.num_blocks) {
                        // an invalid block id: flag it and read block 0 instead, so
                        // the copy stays inside the cache
                        atomicOr(&g_plx_status, PLX_DEV_ERR_SEQLEN);
                        blk = 0;
                    }
                    g = ((static_cast<size_t>(blk) * p.H + (bh % p.H)) * p.page + (r0 - pg * p.page)) * D;
                }
                const size_t cache_elems = p.block_table
                                               ? static_cast<size_t>(p.num_blocks) * p.H * p.page * D
                                               : static_cast<size_t>(gridDim.x) * p.S_cap * D;
                if (in_bounds(rows > 0 && g + static_cast<size_t>(rows) * D <= cache_elems)) {
                    mbar_arrive_expect_tx(&full[s], 2 * bytes);
                    bulk_g2s_hint(kbuf + s * T * D, p.kc + g, bytes, &full[s], pol);
                    bulk_g2s_hint(vbuf + s * T * D, p.vc + g, bytes, &full[s], pol);
                } else {
                    mbar_arrive(&full[s]);   // debug build: the copies are skipped, the phase still completes
                }
                ++issued;
            }
            // never leave with copies in flight into this block's shared memory
            for (int i = max(0, issued - NSTAGE); i < issued; ++i)
                if (!mbar_wait(&full[i % NSTAGE], (i / NSTAGE) & 1)) atomicOr(&g_plx_status, PLX_DEV_ERR_TIMEOUT);
        }
        if constexpr (!FUSED) return;
    } else {

    // ---------------- consumers (warps 0..3)
    float qr[DPL], rr[DPL];
    {
        const size_t base = static_cast<size_t>(bh) * D + lane * DPL;
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
            qr[i] = __bfloat162float(p.q[base + i]) * p.scale_log2;
            rr[i] = PLX ? __bfloat162float(p.rho[base + i]) : 0.f;
        }
    }
    float m = -INFINITY, l = 0.f, C = 0.f;
    float A[DPL], U[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) { A[i] = 0.f; U[i] = 0.f; }

    constexpr int NV = PLX ? 16 : 8;     // dot products per warp per stage
    for (int i = 0; i < my_tiles; ++i) {
        const int s = i % NSTAGE;
        if (!mbar_wait(&full[s], (i / NSTAGE) & 1)) {
            atomicOr(&g_plx_status, PLX_DEV_ERR_TIMEOUT);
            atomicExch(abort_flag, 1);
        }
        if (*reinterpret_cast<volatile int*>(abort_flag)) break;
        const int t = t_begin + i;
        const int rows = min(T, L - t * T);
        const int r0 = warp * Cfg::ROWS_PER_WARP;
        const __nv_bfloat16* kt = kbuf + s * T * D;
        const __nv_bfloat16* vt = vbuf + s * T * D;

        float v[NV];
#pragma unroll
        for (int tt = 0; tt < 8; ++tt) {
            float kf[DPL];
            load_row<DPL>(kt + (r0 + tt) * D, lane, kf);
            float sd = 0.f, rd = 0.f;
#pragma unroll
            for (int k = 0; k < DPL; ++k) {
                sd = fmaf(qr[k], kf[k], sd);
                if constexpr (PLX) rd = fmaf(rr[k], kf[k], rd);
            }
            if constexpr (PLX) { v[2 * tt] = sd; v[2 * tt + 1] = rd; }
            else v[tt] = sd;
        }
        // transposed butterfly: after it lane l holds value (l >> 1) & 15
        // (PLX) or (l >> 2) (SA), summed over all 32 lanes
#pragma unroll
        for (int msk = 16, n = NV; n > 1; msk >>= 1, n >>= 1) {
            const bool upper = (lane & msk) != 0;
#pragma unroll
            for (int k = 0; k < n / 2; ++k) {
                const float send = upper ? v[k] : v[k + n / 2];
                const float keep = upper ? v[k + n / 2] : v[k];
                v[k] = keep + __shfl_xor_sync(0xffffffffu, send, msk);
            }
        }
#pragma unroll
        for (int msk = (32 / NV) / 2; msk >= 1; msk >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], msk);

        // every lane gathers the 8 scores and probe terms: s_tt in lane 4tt, r_tt in lane 4tt+2
        float sv[8], rv[8];
        float mt = -INFINITY;
#pragma unroll
        for (int tt = 0; tt < 8; ++tt) {
            sv[tt] = __shfl_sync(0xffffffffu, v[0], 4 * tt);
            rv[tt] = PLX ? __shfl_sync(0xffffffffu, v[0], 4 * tt + 2) : 0.f;
            if (r0 + tt < rows) mt = fmaxf(mt, sv[tt]);
        }
        if (mt != -INFINITY) {
            const float m_new = fmaxf(m, mt);
            const float alpha = exp2f(m - m_new);   // m = -inf -> 0
            l *= alpha;
            C *= alpha;
#pragma unroll
            for (int k = 0; k < DPL; ++k) { A[k] *= alpha; if constexpr (PLX) U[k] *= alpha; }
#pragma unroll
            for (int tt = 0; tt < 8; ++tt) {
                if (r0 + tt < rows) {
                    const float pe = exp2f(sv[tt] - m_new);
                    float vf[DPL];
                    load_row<DPL>(vt + (r0 + tt) * D, lane, vf);
                    l += pe;
#pragma unroll
                    for (int k = 0; k < DPL; ++k) A[k] = fmaf(pe, vf[k], A[k]);
                    if constexpr (PLX) {
                        const float pr = pe * rv[tt];
                        C += pr;
#pragma unroll
                        for (int k = 0; k < DPL; ++k) U[k] = fmaf(pr, vf[k], U[k]);
                    }
                }
            }
            m = m_new;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }

    // ---------------- merge the four warp states
    {
        float* mine = merge + warp * Cfg::PART;
        if (lane == 0) { mine[0] = m; mine[1] = l; mine[2] = C; mine[3] = 0.f; }
#pragma unroll
        for (int k = 0; k < DPL; ++k) {
            mine[4 + lane * DPL + k] = A[k];
            mine[4 + D + lane * DPL + k] = U[k];
        }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(Cfg::CWARPS * 32) : "memory");
    if (threadIdx.x < D) {
        const int t = threadIdx.x;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < Cfg::CWARPS; ++w) M = fmaxf(M, merge[w * Cfg::PART]);
        float Lsum = 0.f, Cs = 0.f, As = 0.f, Us = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < Cfg::CWARPS; ++w) {
                const float* pw = merge + w * Cfg::PART;
                const float sc = exp2f(pw[0] - M);
                Lsum = fmaf(sc, pw[1], Lsum);
                Cs = fmaf(sc, pw[2], Cs);
                As = fmaf(sc, pw[4 + t], As);
                Us = fmaf(sc, pw[4 + D + t], Us);
            }
        }
        if (p.splits == 1 && !p.partials_only) {
            float o = 0.f;
            if (Lsum > 0.f) {
                const float inv = 1.f / Lsum;
                const float vbar = As * inv;
                o = PLX ? (p.no_intercept ? -Us * inv : fmaf(Cs * inv, vbar, vbar) - Us * inv) : vbar;
            }
            store_out(p.out, p.out_f32, static_cast<size_t>(bh) * D + t, o);
            if (t == 0 && p.lse)
                p.lse[bh] = Lsum > 0.f ? (M + log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
        } else if (FUSED) {
            if (t == 0) { cpart[0] = M; cpart[1] = Lsum; cpart[2] = Cs; cpart[3] = 0.f; }
            cpart[4 + t] = As;
            cpart[4 + D + t] = Us;
        } else {
            float* part = p.ws + (static_cast<size_t>(bh) * p.splits + split) * Cfg::PART;
            if (t == 0) { part[0] = M; part[1] = Lsum; part[2] = Cs; part[3] = 0.f; }
            part[4 + t] = As;
            part[4 + D + t] = Us;
        }
    }
    }   // consumers
    if constexpr (FUSED) {
        // every thread of every CTA of the cluster reaches both barriers: the
        // first publishes the CTAs' states, the second keeps them alive until
        // rank 0 has read them.  The merge is the combine kernel's, in rank order.
        cluster_sync_all();
        if (cluster_rank() == 0 && threadIdx.x < D) {
            // The remote reads go four ranks at a time, all of a group's loads in
            // flight before any is used: a loop that used each value before the
            // next load waited out the distributed-shared-memory latency once per
            // load (three or four times per rank).  Same operations, same order.
            constexpr int G4 = 4;
            static_assert(DECODE_MAX_CLUSTER_SPLITS % G4 == 0, "groups of four ranks");
            const int t = threadIdx.x;
            float M = -INFINITY;
#pragma unroll
            for (int r0 = 0; r0 < DECODE_MAX_CLUSTER_SPLITS; r0 += G4) {
                if (r0 >= p.splits) break;
                float mv[G4];
#pragma unroll
                for (int k = 0; k < G4; ++k) mv[k] = r0 + k < p.splits ? ld_cluster_f32(cpart, r0 + k) : -INFINITY;
#pragma unroll
                for (int k = 0; k < G4; ++k) M = fmaxf(M, mv[k]);
            }
            float Lsum = 0.f, Cs = 0.f, As = 0.f, Us = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int r0 = 0; r0 < DECODE_MAX_CLUSTER_SPLITS; r0 += G4) {
                    if (r0 >= p.splits) break;
                    float mv[G4], lv[G4], cv[G4], av[G4], uv[G4];
#pragma unroll
                    for (int k = 0; k < G4; ++k) {
                        const int r = r0 + k;
                        mv[k] = -INFINITY;
                        lv[k] = cv[k] = av[k] = uv[k] = 0.f;
                        if (r < p.splits) {
                            mv[k] = ld_cluster_f32(cpart, r);
                            lv[k] = ld_cluster_f32(cpart + 1, r);
                            cv[k] = ld_cluster_f32(cpart + 2, r);
                            av[k] = ld_cluster_f32(cpart + 4 + t, r);
                            if constexpr (PLX) uv[k] = ld_cluster_f32(cpart + 4 + D + t, r);
                        }
                    }
#pragma unroll
                    for (int k = 0; k < G4; ++k) {
                        if (mv[k] == -INFINITY) continue;
                        const float sc = exp2f(mv[k] - M);
                        Lsum = fmaf(sc, lv[k], Lsum);
                        Cs = fmaf(sc, cv[k], Cs);
                        As = fmaf(sc, av[k], As);
                        if constexpr (PLX) Us = fmaf(sc, uv[k], Us);
                    }
                }
            }
            float o = 0.f;
            if (Lsum > 0.f) {
                const float inv = 1.f / Lsum;
                const float vbar = As * inv;
                o = PLX ? (p.no_intercept ? -Us * inv : fmaf(Cs * inv, vbar, vbar) - Us * inv) : vbar;
            }
            store_out(p.out, p.out_f32, static_cast<size_t>(bh) * D + t, o);
            if (t == 0 && p.lse) p.lse[bh] = Lsum > 0.f ? (M + log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
        }
        cluster_sync_all();
    }
}

// Merge the partials of one (b, h) -- every split of every group (shard of
// the key range), in group-major order: M = max m_s, w_s = 2^(m_s - M),
// L = sum w_s l_s, then the weighted sums of C, A, U, and the PLX output.
template <int D, bool PLX>
__global__ void __launch_bounds__(D) plx_decode_combine_kernel(const DecodeParams p) {
    constexpr int PART = DecodeCfg<D>::PART;
    const int bh = blockIdx.x, t = threadIdx.x;
    const size_t group_stride = static_cast<size_t>(gridDim.x) * p.splits * PART;
    float M = -INFINITY;
    for (int g = 0; g < p.groups; ++g) {
        const float* base = p.ws + g * group_stride + static_cast<size_t>(bh) * p.splits * PART;
        for (int s = 0; s < p.splits; ++s) M = fmaxf(M, base[s * PART]);
    }
    float Lsum = 0.f, Cs = 0.f, As = 0.f, Us = 0.f;
    if (M != -INFINITY) {
        // four splits' values loaded before any is used (one memory latency per
        // four splits rather than two per split); same operations, same order
        constexpr int G4 = 4;
        for (int g = 0; g < p.groups; ++g) {
            const float* base = p.ws + g * group_stride + static_cast<size_t>(bh) * p.splits * PART;
            for (int s0 = 0; s0 < p.splits; s0 += G4) {
                float mv[G4], lv[G4], cv[G4], av[G4], uv[G4];
#pragma unroll
                for (int k = 0; k < G4; ++k) {
                    const float* ps = base + (s0 + k) * PART;
                    const bool in = s0 + k < p.splits;
                    mv[k] = in ? ps[0] : -INFINITY;
                    lv[k] = in ? ps[1] : 0.f;
                    cv[k] = in ? ps[2] : 0.f;
                    av[k] = in ? ps[4 + t] : 0.f;
                    uv[k] = (PLX && in) ? ps[4 + D + t] : 0.f;
                }
#pragma unroll
                for (int k = 0; k < G4; ++k) {
                    if (mv[k] == -INFINITY) continue;
                    const float sc = exp2f(mv[k] - M);
                    Lsum = fmaf(sc, lv[k], Lsum);
                    Cs = fmaf(sc, cv[k], Cs);
                    As = fmaf(sc, av[k], As);
                    if constexpr (PLX) Us = fmaf(sc, uv[k], Us);
                }
            }
        }
    }
    float o = 0.f;
    if (Lsum > 0.f) {
        const float inv = 1.f / Lsum;
        const float vbar = As * inv;
        o = PLX ? (p.no_intercept ? -Us * inv : fmaf(Cs * inv, vbar, vbar) - Us * inv) : vbar;
    }
    store_out(p.out, p.out_f32, static_cast<size_t>(bh) * D + t, o);
    if (t == 0 && p.lse) p.lse[bh] = Lsum > 0.f ? (M + log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace plx
