// ptx.cuh -- inline-PTX wrappers for sm_103a: mbarrier, bulk/TMA copies,
// tcgen05 (TMEM allocation, MMA, loads/stores) and the shared-memory and
// instruction descriptors the tcgen05 MMAs take.
//
// Every wait on an mbarrier is bounded (iteration count and wall time); on
// expiry the wait returns false and the caller records PLX_DEV_ERR_TIMEOUT in
// the device status word instead of spinning forever.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

namespace plx {

// device status word bits (read back by plx_last_device_error)
constexpr unsigned PLX_DEV_ERR_TIMEOUT = 1u;
constexpr unsigned PLX_DEV_ERR_SEQLEN = 2u;
constexpr unsigned PLX_DEV_ERR_NONFINITE = 4u;
constexpr unsigned PLX_DEV_ERR_BOUNDS = 8u;       // debug builds: an index outside its buffer

// a wait gives up after this much wall time (ns) or this many polls
constexpr unsigned long long PLX_WAIT_TIMEOUT_NS = 4000000000ull;
constexpr unsigned PLX_WAIT_MAX_POLLS = 1u << 30;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// The same test, but the thread may be suspended (issuing nothing) until the
// phase completes or about ns nanoseconds have passed.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}
constexpr uint32_t PLX_WAIT_SUSPEND_NS = 1000;
// Wait until the phase with the given parity has completed.  Waiting threads
// are suspended between polls, so they leave the issue slots to the warps that
// work.  Bounded: returns false after PLX_WAIT_TIMEOUT_NS of wall time or
// PLX_WAIT_MAX_POLLS polls.
// The same wait with the wall-time limit given in nanoseconds.
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t polls = 0; polls < PLX_WAIT_MAX_POLLS; ++polls) {
        if (mbar_try_wait_suspend(bar, parity, PLX_WAIT_SUSPEND_NS)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return false;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    return mbar_wait_for(bar, parity, PLX_WAIT_TIMEOUT_NS);
}

// ------------------------------------------------------------- bulk copies
// 1-D bulk copy global -> shared (TMA engine), completes tx bytes on bar.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// same with an L2 eviction-priority policy (streamed data read once)
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 3-D tiled TMA load; x (innermost) must be a multiple of 8 bf16 elements.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, "
        "%5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}
// 3-D tiled TMA store shared -> global, tracked by this thread's bulk groups.
// Box elements outside the tensor are not written.  x * element size must be
// a multiple of 16 bytes and x, y, z non-negative.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}
// 1-D bulk copy shared -> global (TMA engine) in this thread's bulk group;
// both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// until at most N of this thread's bulk groups are still reading shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// until every bulk group of this thread has completed (global writes done)
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Prefetch one 3-D tile of a tensor map into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_slot)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T   (kind::f16, operands by descriptor)
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive once on bar when every tcgen05.mma issued so far by this thread is done
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// Warp-wide tcgen05 issue: every lane of the warp executes these (so their
// operands stay warp-uniform), one lane chosen by elect.sync issues.
__device__ __forceinline__ void mma_ss_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit_warp(uint64_t* bar) {
    asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (tiles 1024-byte aligned).
//   bits  0-13 start address >> 4      bits 16-29 leading byte offset >> 4
//   bits 32-45 stride byte offset >> 4 bits 46-47 version (1)
//   bits 49-51 base offset (0)         bits 61-63 layout (2 = 128B swizzle)
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format,
//   bit 15 A major (0 = K-major), bit 16 B major (1 = MN-major),
//   bits 17-22 N >> 3, bits 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
// same with fp16 A/B (A and B formats 0)
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// kind::tf32 with fp32 D: A and B formats 2 (tf32, read from 32-bit
// containers), both K-major.
__host__ __device__ constexpr uint32_t idesc_tf32_f32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}
// x rounded to the nearest tf32 value (ties away from zero), as fp32: the
// high part of the split x = hi + lo, with lo = x - hi exact in fp32
__device__ __forceinline__ float tf32_hi(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// the two bf16 halves of a packed pair, widened exactly to fp32
__device__ __forceinline__ float bf16x2_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16x2_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

// fp16 pair: pack with round-to-nearest-even, and widen back (exact)
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ void unpack_f16x2(uint32_t x, float& lo, float& hi) {
    asm("{\n\t.reg .f16 a, b;\n\t"
        "mov.b32 {a, b}, %2;\n\t"
        "cvt.f32.f16 %0, a;\n\t"
        "cvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(x));
}
// a packed bf16 pair re-encoded as a packed fp16 pair (round-to-nearest-even)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x) {
    return pack_f16x2(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u));
}
// order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA / tensor core) accesses
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ------------------------------------------------- sm_100+ packed / mixed fp32 ops
// max of three (one instruction on sm_100+)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
// (a.x*b.x + c.x, a.y*b.y + c.y) as one packed instruction
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 r;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return r;
}
// (a.x + b.x, a.y + b.y) as one packed instruction
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 r;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}
// (a.x*b.x, a.y*b.y) as one packed instruction
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    float2 r;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}
// acc + lo + hi of a packed fp16 pair, each half widened exactly (mixed-precision adds)
__device__ __forceinline__ float add_f16x2(float acc, uint32_t x) {
    float r;
    asm("{\n\t.reg .f16 lo, hi;\n\t.reg .f32 t;\n\t"
        "mov.b32 {lo, hi}, %1;\n\t"
        "add.rn.f32.f16 t, lo, %2;\n\t"
        "add.rn.f32.f16 %0, hi, t;\n\t}"
        : "=f"(r)
        : "r"(x), "f"(acc));
    return r;
}

// generated: tcgen05.ld (fused with wait::ld) and tcgen05.st, 32x32b shape
__device__ __forceinline__ void tmem_ld32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr) : "memory");
}
__device__ __forceinline__ void tmem_ld32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr) : "memory");
}
__device__ __forceinline__ void tmem_ld32x32b_x64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
                 : "r"(taddr) : "memory");
}
__device__ __forceinline__ void tmem_ld32x32b_x32_nowait(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr) : "memory");
}
// Complete this thread's outstanding tcgen05.ld.  The destination registers
// of the loads are in/out operands here, so no use of them can be scheduled
// before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;\n\t// %0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :: "memory");
}
__device__ __forceinline__ void tmem_st32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
                 :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]) : "memory");
}
__device__ __forceinline__ void tmem_st32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
                 :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]) : "memory");
}

// ------------------------------------------------- batched tcgen05 issue
// One warp-wide asm block per batch of MMAs: a single elect.sync picks the
// issuing lane, and each MMA's shared-memory descriptors are the batch's base
// descriptors plus a compile-time offset added to their low word (the start
// address field, bits 0-13, in 16-byte units: adding an offset that keeps the
// address below 256 KB cannot carry into the next field).  So a batch costs
// about three instructions per MMA.
//
// The S/R batch of the prefill: D(S) (+)= Q K^T and, for PLX, D(R) (+)= rho K^T
// over D/16 k-steps of 16; Q, rho and K tiles are K-major, 128B-swizzled
// 64-column panels (the k-step's 32 bytes at (k % 4) * 32 within a panel),
// Q/rho panels A16 x 16 bytes apart (BM rows of 128 bytes) and K panels
// 512 x 16 bytes apart (64 rows).  The first k-step overwrites D.
template <int D, bool PLX, int A16>
__device__ __forceinline__ void mma_sr_batch(uint32_t t_s, uint32_t t_r, uint64_t a_q, uint64_t a_r, uint64_t b_k,
                                             uint32_t idesc);
template <>
__device__ __forceinline__ void mma_sr_batch<64, true, 1024>(uint32_t t_s, uint32_t t_r, uint64_t a_q,
                                                              uint64_t a_r, uint64_t b_k, uint32_t idesc) {
    asm volatile("{\n\t.reg .pred e, pf, pt;\n\t.reg .b32 lo;\n\t.reg .b64 da, db;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 pf, %0, %0;\n\tsetp.eq.b32 pt, %0, %0;\n\tadd.u32 lo, %6, 0; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 0; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pf;\n\tadd.u32 lo, %4, 0; mov.b64 da, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %8, pf;\n\tadd.u32 lo, %6, 2; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 2; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pt;\n\tadd.u32 lo, %4, 2; mov.b64 da, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %8, pt;\n\tadd.u32 lo, %6, 4; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 4; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pt;\n\tadd.u32 lo, %4, 4; mov.b64 da, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %8, pt;\n\tadd.u32 lo, %6, 6; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 6; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pt;\n\tadd.u32 lo, %4, 6; mov.b64 da, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %8, pt;\n\t}"
                 ::"r"(t_s), "r"(t_r), "r"(static_cast<uint32_t>(a_q)), "r"(static_cast<uint32_t>(a_q >> 32)),
                   "r"(static_cast<uint32_t>(a_r)), "r"(static_cast<uint32_t>(a_r >> 32)),
                   "r"(static_cast<uint32_t>(b_k)), "r"(static_cast<uint32_t>(b_k >> 32)), "r"(idesc)
                 : "memory");
}
template <>
__device__ __forceinline__ void mma_sr_batch<64, false, 1024>(uint32_t t_s, uint32_t t_r, uint64_t a_q,
                                                              uint64_t a_r, uint64_t b_k, uint32_t idesc) {
    asm volatile("{\n\t.reg .pred e, pf, pt;\n\t.reg .b32 lo;\n\t.reg .b64 da, db;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 pf, %0, %0;\n\tsetp.eq.b32 pt, %0, %0;\n\tadd.u32 lo, %6, 0; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 0; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pf;\n\tadd.u32 lo, %6, 2; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 2; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pt;\n\tadd.u32 lo, %6, 4; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 4; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pt;\n\tadd.u32 lo, %6, 6; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 6; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pt;\n\t}"
                 ::"r"(t_s), "r"(t_r), "r"(static_cast<uint32_t>(a_q)), "r"(static_cast<uint32_t>(a_q >> 32)),
                   "r"(static_cast<uint32_t>(a_r)), "r"(static_cast<uint32_t>(a_r >> 32)),
                   "r"(static_cast<uint32_t>(b_k)), "r"(static_cast<uint32_t>(b_k >> 32)), "r"(idesc)
                 : "memory");
}
template <>
__device__ __forceinline__ void mma_sr_batch<128, true, 1024>(uint32_t t_s, uint32_t t_r, uint64_t a_q,
                                                              uint64_t a_r, uint64_t b_k, uint32_t idesc) {
    asm volatile("{\n\t.reg .pred e, pf, pt;\n\t.reg .b32 lo;\n\t.reg .b64 da, db;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 pf, %0, %0;\n\tsetp.eq.b32 pt, %0, %0;\n\tadd.u32 lo, %6, 0; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 0; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pf;\n\tadd.u32 lo, %4, 0; mov.b64 da, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %8, pf;\n\tadd.u32 lo, %6, 2; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 2; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pt;\n\tadd.u32 lo, %4, 2; mov.b64 da, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %8, pt;\n\tadd.u32 lo, %6, 4; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 4; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pt;\n\tadd.u32 lo, %4, 4; mov.b64 da, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %8, pt;\n\tadd.u32 lo, %6, 6; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 6; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pt;\n\tadd.u32 lo, %4, 6; mov.b64 da, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %8, pt;\n\tadd.u32 lo, %6, 512; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 1024; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pt;\n\tadd.u32 lo, %4, 1024; mov.b64 da, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %8, pt;\n\tadd.u32 lo, %6, 514; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 1026; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pt;\n\tadd.u32 lo, %4, 1026; mov.b64 da, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %8, pt;\n\tadd.u32 lo, %6, 516; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 1028; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pt;\n\tadd.u32 lo, %4, 1028; mov.b64 da, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %8, pt;\n\tadd.u32 lo, %6, 518; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 1030; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pt;\n\tadd.u32 lo, %4, 1030; mov.b64 da, {lo, %5};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%1], da, db, %8, pt;\n\t}"
                 ::"r"(t_s), "r"(t_r), "r"(static_cast<uint32_t>(a_q)), "r"(static_cast<uint32_t>(a_q >> 32)),
                   "r"(static_cast<uint32_t>(a_r)), "r"(static_cast<uint32_t>(a_r >> 32)),
                   "r"(static_cast<uint32_t>(b_k)), "r"(static_cast<uint32_t>(b_k >> 32)), "r"(idesc)
                 : "memory");
}
template <>
__device__ __forceinline__ void mma_sr_batch<128, false, 1024>(uint32_t t_s, uint32_t t_r, uint64_t a_q,
                                                              uint64_t a_r, uint64_t b_k, uint32_t idesc) {
    asm volatile("{\n\t.reg .pred e, pf, pt;\n\t.reg .b32 lo;\n\t.reg .b64 da, db;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 pf, %0, %0;\n\tsetp.eq.b32 pt, %0, %0;\n\tadd.u32 lo, %6, 0; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 0; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pf;\n\tadd.u32 lo, %6, 2; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 2; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pt;\n\tadd.u32 lo, %6, 4; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 4; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pt;\n\tadd.u32 lo, %6, 6; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 6; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pt;\n\tadd.u32 lo, %6, 512; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 1024; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pt;\n\tadd.u32 lo, %6, 514; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 1026; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pt;\n\tadd.u32 lo, %6, 516; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 1028; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pt;\n\tadd.u32 lo, %6, 518; mov.b64 db, {lo, %7};\n\tadd.u32 lo, %2, 1030; mov.b64 da, {lo, %3};\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %8, pt;\n\t}"
                 ::"r"(t_s), "r"(t_r), "r"(static_cast<uint32_t>(a_q)), "r"(static_cast<uint32_t>(a_q >> 32)),
                   "r"(static_cast<uint32_t>(a_r)), "r"(static_cast<uint32_t>(a_r >> 32)),
                   "r"(static_cast<uint32_t>(b_k)), "r"(static_cast<uint32_t>(b_k >> 32)), "r"(idesc)
                 : "memory");
}

// The PV batch of the prefill: O (+)= P V and, for PLX, U (+)= (P o R) V over
// the tile's 64 keys in 4 k-steps of 16.  P and PR are fp16 pairs in TMEM:
// keys [32h, 32h + 32) at columns [32h, 32h + 16) of the buffer t_p + P_OFF
// (P) and t_p + PR_OFF (PR); V is the MN-major B operand, k-step kk at
// kk * 2048 bytes (b_v its base descriptor).  acc0 = 0: the first k-step
// overwrites O and U.
template <bool PLX, int P_OFF, int PR_OFF>
__device__ __forceinline__ void mma_pv_batch(uint32_t t_o, uint32_t t_u, uint32_t t_p, uint64_t b_v, uint32_t idesc,
                                             uint32_t acc0);
template <>
__device__ __forceinline__ void mma_pv_batch<true, 0, 64>(uint32_t t_o, uint32_t t_u, uint32_t t_p, uint64_t b_v,
                                                        uint32_t idesc, uint32_t acc0) {
    asm volatile("{\n\t.reg .pred e, pa, pt;\n\t.reg .b32 lo, ta;\n\t.reg .b64 db;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 pa, %6, 0;\n\tsetp.eq.b32 pt, %6, %6;\n\tadd.u32 lo, %3, 0; mov.b64 db, {lo, %4};\n\tadd.u32 ta, %2, 0;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %5, pa;\n\tadd.u32 ta, %2, 64;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%1], [ta], db, %5, pa;\n\tadd.u32 lo, %3, 128; mov.b64 db, {lo, %4};\n\tadd.u32 ta, %2, 8;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %5, pt;\n\tadd.u32 ta, %2, 72;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%1], [ta], db, %5, pt;\n\tadd.u32 lo, %3, 256; mov.b64 db, {lo, %4};\n\tadd.u32 ta, %2, 32;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %5, pt;\n\tadd.u32 ta, %2, 96;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%1], [ta], db, %5, pt;\n\tadd.u32 lo, %3, 384; mov.b64 db, {lo, %4};\n\tadd.u32 ta, %2, 40;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %5, pt;\n\tadd.u32 ta, %2, 104;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%1], [ta], db, %5, pt;\n\t}"
                 ::"r"(t_o), "r"(t_u), "r"(t_p), "r"(static_cast<uint32_t>(b_v)), "r"(static_cast<uint32_t>(b_v >> 32)),
                   "r"(idesc), "r"(acc0)
                 : "memory");
}
template <>
__device__ __forceinline__ void mma_pv_batch<false, 0, 0>(uint32_t t_o, uint32_t t_u, uint32_t t_p, uint64_t b_v,
                                                        uint32_t idesc, uint32_t acc0) {
    asm volatile("{\n\t.reg .pred e, pa, pt;\n\t.reg .b32 lo, ta;\n\t.reg .b64 db;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 pa, %6, 0;\n\tsetp.eq.b32 pt, %6, %6;\n\tadd.u32 lo, %3, 0; mov.b64 db, {lo, %4};\n\tadd.u32 ta, %2, 0;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %5, pa;\n\tadd.u32 lo, %3, 128; mov.b64 db, {lo, %4};\n\tadd.u32 ta, %2, 8;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %5, pt;\n\tadd.u32 lo, %3, 256; mov.b64 db, {lo, %4};\n\tadd.u32 ta, %2, 32;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %5, pt;\n\tadd.u32 lo, %3, 384; mov.b64 db, {lo, %4};\n\tadd.u32 ta, %2, 40;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %5, pt;\n\t}"
                 ::"r"(t_o), "r"(t_u), "r"(t_p), "r"(static_cast<uint32_t>(b_v)), "r"(static_cast<uint32_t>(b_v >> 32)),
                   "r"(idesc), "r"(acc0)
                 : "memory");
}

}  // namespace plx
