/*
 * plx.h -- C ABI of the Parallax (PLX) attention hot path on B300 (sm_103a).
 *
 * PLX is causal softmax attention with a covariance correction driven by a
 * per-token probe ("Parallax: Parameterized Local Linear Attention for
 * Language Modeling", arXiv:2605.29157; zhichai.net section 1.3 and
 * gist.science "Meccanismo Principale"):
 *
 *   o_i = o_i^SA - Sigma_KV^(i) rho_i
 *   o_i^SA = sum_{j<=i} w_ij v_j,  w_ij = softmax_{j<=i}(scale * q_i . k_j)
 *   Sigma_KV^(i) = sum_{j<=i} w_ij (v_j - vbar_i)(k_j - kbar_i)^T   (d_v x d_k)
 *   vbar_i = o_i^SA,  kbar_i = sum_j w_ij k_j
 *
 * The probe rho_i = W_R x_i is an input (its projection is computed before
 * this call).  The boundary term eta_i is zero and there is no solve
 * (gist.science, "Meccanismo Principale").  The kernels never form Sigma_KV:
 * they stream K/V once and use
 *
 *   Sigma_KV rho = sum_j w_j (k_j . rho) v_j - vbar (kbar . rho),
 *   so o = (1 + c) vbar - u,  c = sum_j w_j (k_j . rho),  u = sum_j w_j (k_j . rho) v_j,
 *
 * the FlashAttention-compatible streaming algorithm that reuses the K/V
 * stream (gist.science, "Algoritmo Consapevole dell'Hardware").
 *
 * Conventions for every entry point:
 *   - Tensors are row-major and contiguous: q, k, v, rho, out are [B][H][N][d]
 *     (d fastest); the decode cache is [B][H][S_cap][d].
 *   - All pointers are DEVICE pointers owned by the caller; the library keeps
 *     no reference after the call returns and allocates no device memory
 *     (the decode workspace is passed in).  The library holds one device
 *     status word per GPU (a static __device__ variable).
 *   - stream is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Every call is asynchronous on that stream and never synchronises,
 *     except plx_last_device_error.
 *   - Arguments are validated before any launch; on a failed check the call
 *     returns a status and launches nothing.  A launch error maps to
 *     PLX_ERR_CUDA.  No C++ exception crosses this boundary.
 *   - Passing rho == NULL selects the softmax-attention instantiation of the
 *     same kernel (the zero probe of the attention family, zhichai.net
 *     section 2.1): it skips the probe GEMMs, so it is the baseline for
 *     timing, and its output equals PLX with rho = 0.
 *   - scale multiplies q.k only; rho.k is not scaled.  lse is the natural
 *     log of sum_j exp(scale * q_i . k_j), fp32.
 */
#ifndef PLX_H
#define PLX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PLX_OK = 0,
    PLX_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, bad dtype */
    PLX_ERR_UNSUPPORTED = 2, /* head dim or size this build has no kernel for */
    PLX_ERR_MISALIGNED = 3,  /* pointer not 16-byte aligned (lse: 4-byte) */
    PLX_ERR_CUDA = 4,        /* a CUDA call or kernel launch failed */
    PLX_ERR_TIMEOUT = 5,     /* a device-side wait gave up (see plx_last_device_error) */
    PLX_ERR_WORKSPACE = 6,   /* workspace missing or too small (any entry point that takes one) */
    PLX_ERR_RANGE = 7,       /* plx_fwd produced a non-finite output (see plx_last_device_error) */
    PLX_ERR_BOUNDS = 8       /* the debug build (PLX_DEBUG) caught an index outside its buffer and skipped
                                the access (see plx_last_device_error) */
} plx_status;

typedef enum { PLX_BF16 = 0, PLX_F32 = 1 } plx_dtype;

/* Library version, e.g. 100 for 0.1.0. */
int plx_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* plx_strerror(plx_status status);

/*
 * plx_fwd -- causal prefill / training forward, bf16 inputs, fp32 accumulate.
 * Streaming algorithm of gist.science "Algoritmo Consapevole dell'Hardware":
 * per K/V tile, S = scale Q K^T and R = rho K^T on the tensor cores, online
 * softmax, then O += P V and U += (P o R) V, finally o = (1 + c) vbar - u.
 *
 *   q, k, v, rho : bf16 [B][H][N][d], 16-byte aligned; rho may be NULL (SA).
 *   out          : [B][H][N][d] of out_dtype (PLX_BF16 or PLX_F32), 16-byte aligned.
 *   lse          : fp32 [B][H][N], 4-byte aligned, or NULL.
 *   B, H, N >= 1; d in {64, 128}.  scale >= 0 finite (usually 1/sqrt(d)).
 * Numerics: S = QK^T and R = rho K^T take the bf16 inputs exactly with fp32
 * accumulation; P, P o R and V enter the PV GEMMs as fp16 (V is re-encoded
 * from bf16 in shared memory), with fp32 accumulation.  Supported range:
 * |v| < 65504 and |rho . k| < 4094 (P o R stays inside fp16 because the
 * lazily updated softmax keeps P <= 16).  Outside it the output may be
 * non-finite; the kernel then sets a device flag that plx_last_device_error
 * reports as PLX_ERR_RANGE.
 * Errors: PLX_ERR_INVALID_ARG, PLX_ERR_UNSUPPORTED (other d, or more than
 * 2^31 - 1 work items), PLX_ERR_MISALIGNED, PLX_ERR_CUDA.
 */
plx_status plx_fwd(const void* q, const void* k, const void* v, const void* rho, void* out, float* lse,
                   int B, int H, int N, int d, float scale, plx_dtype out_dtype, void* stream);

/*
 * plx_fwd_cached -- several new query tokens per sequence against a bf16 KV
 * cache, on the tensor cores: the T newest positions of each sequence attend
 * causally to its cache (speculative verification, chunked prefill).  Query
 * row i of sequence b sits at position seqlens[b] - T + i and attends to
 * cache rows 0 .. seqlens[b] - T + i.  The same kernel as plx_fwd (plx_fwd is
 * this with T = N and seqlens[b] = N).
 *
 *   q, rho       : bf16 [B][H][T][d], 16-byte aligned; rho may be NULL (SA).
 *   k_cache, v_cache : bf16 [B][H][S_cap][d], 16-byte aligned, already holding
 *                  the T new tokens at positions seqlens[b] - T .. seqlens[b] - 1.
 *   seqlens      : int32 [B] on the device, T <= seqlens[b] <= S_cap; a length
 *                  outside that range is clamped into it and reported by
 *                  plx_last_device_error as PLX_ERR_INVALID_ARG.
 *   out          : [B][H][T][d] of out_dtype;  lse : fp32 [B][H][T] or NULL.
 *   B, H >= 1, 1 <= T <= S_cap; d in {64, 128}.  Cache rows past seqlens[b]
 *   are never used (they may hold anything, including non-finite values).
 * Errors: as plx_fwd.
 */
plx_status plx_fwd_cached(const void* q, const void* rho, const void* k_cache, const void* v_cache,
                          const int32_t* seqlens, void* out, float* lse, int B, int H, int T, int S_cap, int d,
                          float scale, plx_dtype out_dtype, void* stream);

/*
 * Family switches (zhichai.net section 2.1: the attention family is spanned
 * by the kernel bandwidth, the probe and the affine term; gist.science
 * "Significato e Affermazioni"):
 *   PLX_FAMILY_UNIFORM_WEIGHTS  w_ij = 1/(i+1) over the causal prefix, the
 *                               bandwidth -> infinity limit (scale is taken
 *                               as 0; lse is then ln(i+1)).
 *   PLX_FAMILY_NO_INTERCEPT     no affine term: vbar = kbar = 0 inside
 *                               Sigma_KV, so o_i = -sum_j w_ij (rho_i.k_j) v_j
 *                               (needs rho).  With uniform weights this is
 *                               linear attention with probe -rho.
 */
#define PLX_FAMILY_UNIFORM_WEIGHTS 0x1u
#define PLX_FAMILY_NO_INTERCEPT 0x2u

/*
 * plx_fwd_family -- plx_fwd with family switches (flags: a bitwise OR of the
 * PLX_FAMILY_* values; 0 is plx_fwd itself).  Same kernels, same arguments.
 * Errors: as plx_fwd, plus PLX_ERR_INVALID_ARG for unknown flag bits and for
 * PLX_FAMILY_NO_INTERCEPT without rho.
 */
plx_status plx_fwd_family(const void* q, const void* k, const void* v, const void* rho, void* out, float* lse,
                          int B, int H, int N, int d, float scale, unsigned flags, plx_dtype out_dtype,
                          void* stream);

/*
 * plx_fwd_f32 -- the same causal forward with fp32 inputs, fp32 arithmetic on
 * the CUDA cores (the high-precision path; no tensor cores).
 *
 *   q, k, v, rho : fp32 [B][H][N][d], 16-byte aligned; rho may be NULL (SA).
 *   out          : fp32 [B][H][N][d];  lse : fp32 [B][H][N] or NULL.
 *   B, H, N >= 1; d a multiple of 32 in [32, 256].
 * Errors: as plx_fwd.
 */
plx_status plx_fwd_f32(const float* q, const float* k, const float* v, const float* rho, float* out,
                       float* lse, int B, int H, int N, int d, float scale, void* stream);

/*
 * plx_bwd_f32 -- gradients of the causal PLX forward with respect to q, k, v
 * and rho, fp32 inputs and arithmetic on the CUDA cores.  The pages define
 * the forward only (zhichai.net section 1.3; gist.science "Meccanismo
 * Principale"); this is that forward differentiated.  With dO = dL/do,
 * G_ij = dO_i.v_j, a_i = dO_i.vbar_i and w_ij = exp(scale q_i.k_j - lse_i):
 *   dL/ds_ij = w_ij ((1 + c_i - r_ij) G_ij + a_i r_ij - D_i),  D_i = dO_i.o_i + c_i a_i
 *   dL/dr_ij = w_ij (a_i - G_ij),  dv_j = sum_i w_ij (1 + c_i - r_ij) dO_i
 *   dq = scale dS K,  drho = dR K,  dk = scale dS^T Q + dR^T rho.
 *
 *   q, k, v, rho : fp32 [B][H][N][d], 16-byte aligned; rho may be NULL
 *                  (softmax attention; drho is then ignored).
 *   out, lse     : the forward's o (fp32 [B][H][N][d]) and lse (fp32 [B][H][N],
 *                  natural log), e.g. from plx_fwd_f32.
 *   dout         : dL/do, fp32 [B][H][N][d].
 *   dq, dk, dv, drho : fp32 [B][H][N][d] outputs (written, not accumulated).
 *   workspace    : device scratch of plx_bwd_workspace_size(B, H, N, d) bytes,
 *                  16-byte aligned; no initialisation needed.
 *   B, H, N >= 1, B*H <= 65535; d a multiple of 32 in [32, 256].
 * Three launches on `stream`: a per-row pre-pass, a pass over query rows
 * (dq, drho) and a pass over key rows (dk, dv); no atomics, deterministic.
 * Errors: PLX_ERR_INVALID_ARG, PLX_ERR_UNSUPPORTED, PLX_ERR_MISALIGNED,
 * PLX_ERR_WORKSPACE, PLX_ERR_CUDA.
 */
plx_status plx_bwd_f32(const float* q, const float* k, const float* v, const float* rho, const float* out,
                       const float* lse, const float* dout, float* dq, float* dk, float* dv, float* drho,
                       void* workspace, size_t workspace_bytes, int B, int H, int N, int d, float scale,
                       void* stream);

/* Workspace bytes plx_bwd_f32 needs: B*H*N*16 (0 for invalid sizes). */
size_t plx_bwd_workspace_size(int B, int H, int N, int d);

/*
 * plx_bwd -- the same gradients for the bf16 forward, on the tensor cores
 * (tcgen05, fp32 accumulation; ds, dr and the dv weights enter their GEMMs as
 * fp16, the streamed bf16 tiles they multiply re-encoded to fp16).  Same
 * formulas as plx_bwd_f32.  The forward's o and lse are not inputs: a
 * statistics pass recomputes, per row and with the weights the gradient
 * passes use, log2e lse_i, c_i, a_i = dO_i.vbar_i = sum_j w_ij G_ij and
 * D_i = dO_i.o_i + c_i a_i = (1 + 2 c_i) a_i - sum_j w_ij r_ij G_ij.
 *
 *   q, k, v, rho : bf16 [B][H][N][d], 16-byte aligned; rho may be NULL
 *                  (softmax attention; drho is then ignored).
 *   dout         : dL/do, bf16 [B][H][N][d], 16-byte aligned.
 *   dq, dk, dv, drho : fp32 [B][H][N][d] outputs (written, not accumulated),
 *                  16-byte aligned.
 *   workspace    : device scratch of plx_bwd_bf16_workspace_size(B, H, N, d)
 *                  bytes (16 per row), 16-byte aligned, no initialisation.
 *   B, H, N >= 1; d in {64, 128}.  Inputs and the values ds, dr, wv must lie
 *   within the fp16 range.
 * Three launches on `stream`: the statistics pass and a pass over 128-query
 * tiles (dq, drho), both over query tiles, then a pass over 128-key tiles
 * (dk, dv).  No atomics: the result is
 * deterministic.
 * Errors: PLX_ERR_INVALID_ARG, PLX_ERR_UNSUPPORTED, PLX_ERR_MISALIGNED,
 * PLX_ERR_WORKSPACE, PLX_ERR_CUDA; device-side wait timeouts are reported by
 * plx_last_device_error.
 */
plx_status plx_bwd(const void* q, const void* k, const void* v, const void* rho, const void* dout, float* dq,
                   float* dk, float* dv, float* drho, void* workspace, size_t workspace_bytes, int B, int H, int N,
                   int d, float scale, void* stream);

/* Workspace bytes plx_bwd needs (0 for invalid sizes). */
size_t plx_bwd_bf16_workspace_size(int B, int H, int N, int d);

/*
 * plx_fwd_host -- plx_fwd on HOST buffers (the paper has no counterpart: this
 * is the transfer path around the forward of "Parallax: Parameterized Local
 * Linear Attention for Language Modeling", gist.science, "Algoritmo
 * Consapevole dell'Hardware").  q, k, v, rho, out and lse live in host memory
 * (page-locked, for the copies to run asynchronously and to overlap; pageable
 * memory works, with the copies staged by the driver).  The heads go through
 * the device workspace in up to 8 chunks: while chunk c is computed, chunk
 * c + 1 is copied in and chunk c - 1 copied out, on the GPU's copy engines
 * (two streams of the library, one cudaMemcpyAsync per array and chunk).  The
 * results are those of plx_fwd on the same values, bit for bit.
 *
 *   q, k, v, rho : host bf16 [B][H][N][d]; rho may be NULL (softmax attention).
 *   out          : host [B][H][N][d], fp32 or bf16 as out_dtype.
 *   lse          : host fp32 [B][H][N], or NULL.
 *   workspace    : device scratch of plx_fwd_host_workspace_size(B, H, N, d,
 *                  out_dtype) bytes, 256-byte aligned, no initialisation.
 *   B, H, N >= 1; d in {64, 128}; scale finite and >= 0.
 * Asynchronous: the copies start after the work already on `stream`, the
 * kernels run on `stream`, and `stream` waits for the last copy back, so a
 * synchronisation of `stream` returns with out and lse in host memory.  Calls
 * that share a workspace must be ordered (the same stream orders them).  The
 * host buffers must stay valid, and out/lse unread, until then.
 * Errors: PLX_ERR_INVALID_ARG, PLX_ERR_UNSUPPORTED, PLX_ERR_MISALIGNED (the
 * workspace), PLX_ERR_WORKSPACE, PLX_ERR_CUDA.
 */
plx_status plx_fwd_host(const void* q, const void* k, const void* v, const void* rho, void* out, float* lse,
                        void* workspace, size_t workspace_bytes, int B, int H, int N, int d, float scale,
                        plx_dtype out_dtype, void* stream);

/* Workspace bytes plx_fwd_host needs (0 for invalid sizes). */
size_t plx_fwd_host_workspace_size(int B, int H, int N, int d, plx_dtype out_dtype);

/*
 * plx_fwd_train -- plx_fwd for training: the same o and lse (bit for bit), and
 * also vbar_i = sum_j w_ij v_j (the softmax-attention output o_i^SA of the
 * same weights) and c_i = sum_j w_ij (rho_i.k_j), the two per-row values the
 * gradients' row statistics are formed from (plx_bwd_saved).  The pages give
 * no backward pass; the split follows the streaming identity of
 * zhichai.net section 1.3 (o = (1 + c) vbar - u).
 *
 *   q, k, v, rho : bf16 [B][H][N][d], 16-byte aligned; rho is required.
 *   out, lse     : as plx_fwd (lse is required here).
 *   vbar         : fp32 [B][H][N][d] output, 16-byte aligned.
 *   c            : fp32 [B][H][N] output, 4-byte aligned.
 *   B, H, N >= 1; d in {64, 128}; scale finite and >= 0.
 * One launch on `stream`; vbar leaves through the same shared-memory staging
 * and TMA store as o, so the epilogue of every 128-row tile stores twice.
 * Errors: PLX_ERR_INVALID_ARG, PLX_ERR_UNSUPPORTED, PLX_ERR_MISALIGNED,
 * PLX_ERR_CUDA; device-side conditions as plx_fwd.
 */
plx_status plx_fwd_train(const void* q, const void* k, const void* v, const void* rho, void* out, float* lse,
                         float* vbar, float* c, int B, int H, int N, int d, float scale, plx_dtype out_dtype,
                         void* stream);

/*
 * plx_bwd_saved -- plx_bwd's gradients from the training forward's saved
 * values instead of a statistics pass: a bandwidth-bound kernel forms each
 * row's (log2e lse_i, c_i, a_i = dO_i.vbar_i, D_i = dO_i.o_i + c_i a_i), then
 * the same dq/drho and dk/dv passes as plx_bwd run.  Inputs as plx_bwd, plus:
 *
 *   out, out_dtype : the forward's o (PLX_F32 or PLX_BF16), 16-byte aligned.
 *   lse            : the forward's lse, fp32 [B][H][N] (natural log).
 *   vbar, c        : plx_fwd_train's outputs; required with rho, ignored (may
 *                    be NULL) for softmax attention (rho = NULL), where
 *                    vbar = o and c = 0.
 *   workspace      : plx_bwd_bf16_workspace_size(B, H, N, d) bytes.
 * Three launches on `stream` (the row statistics, the query-tile pass, the
 * key-tile pass); deterministic.  The gradient passes take the weights from
 * the forward's lse, whose sum l was formed from the fp16-rounded P, so the
 * gradients differ from plx_bwd's in the last bits of that rounding.
 * Errors: PLX_ERR_INVALID_ARG, PLX_ERR_UNSUPPORTED, PLX_ERR_MISALIGNED,
 * PLX_ERR_WORKSPACE, PLX_ERR_CUDA; device-side wait timeouts are reported by
 * plx_last_device_error.
 */
plx_status plx_bwd_saved(const void* q, const void* k, const void* v, const void* rho, const void* dout,
                         const void* out, plx_dtype out_dtype, const float* lse, const float* vbar, const float* c,
                         float* dq, float* dk, float* dv, float* drho, void* workspace, size_t workspace_bytes, int B,
                         int H, int N, int d, float scale, void* stream);

/*
 * plx_decode -- one query token per sequence against a bf16 KV cache
 * (the streaming decode of gist.science "Algoritmo Consapevole
 * dell'Hardware").  The cache already holds the current token at position
 * seqlens[b]-1; the query attends to positions 0..seqlens[b]-1.  The cache
 * of each (b, h) is split into num_splits ranges processed by separate
 * thread blocks; their partial states (max, sum, sum of probe terms and the
 * two weighted value sums) are merged with a log-sum-exp weighted combine.
 *
 *   q, rho            : bf16 [B][H][d], 16-byte aligned; rho may be NULL (SA).
 *   k_cache, v_cache  : bf16 [B][H][S_cap][d], 16-byte aligned.
 *   seqlens           : int32 [B] on the device.  A length <= 0 gives o = 0
 *                       and lse = -inf; a length > S_cap is clamped to S_cap
 *                       and flags PLX_ERR_INVALID_ARG in the device status word.
 *   out               : [B][H][d] of out_dtype;  lse : fp32 [B][H] or NULL.
 *   d in {64, 128};  S_cap >= 1.
 *   num_splits        : 0 picks a split count for this GPU; else 1..1024.
 *   workspace         : device scratch of at least
 *                       plx_decode_workspace_size(B, H, d, S_cap, num_splits)
 *                       bytes, 16-byte aligned (may be NULL when that size is 0).
 *                       Its contents need no initialisation.
 * Errors: PLX_ERR_INVALID_ARG, PLX_ERR_UNSUPPORTED, PLX_ERR_MISALIGNED,
 * PLX_ERR_WORKSPACE, PLX_ERR_CUDA.
 */
plx_status plx_decode(const void* q, const void* rho, const void* k_cache, const void* v_cache,
                      const int32_t* seqlens, void* out, float* lse, int B, int H, int d, int S_cap,
                      float scale, int num_splits, void* workspace, size_t workspace_bytes,
                      plx_dtype out_dtype, void* stream);

/* The split count plx_decode uses for these sizes when num_splits == 0, on
 * the current device (queries the SM count once per device). */
int plx_decode_num_splits(int B, int H, int d, int S_cap);

/* Workspace bytes plx_decode needs (0 when one split suffices). */
size_t plx_decode_workspace_size(int B, int H, int d, int S_cap, int num_splits);

/*
 * plx_decode_paged -- plx_decode over a paged KV cache.
 *
 *   k_pages, v_pages : bf16 [num_blocks][H][page_size][d], 16-byte aligned.
 *   block_table      : int32 [B][max_blocks_per_seq] on the device, 4-byte
 *                      aligned: row r (0 <= r < seqlens[b]) of sequence b is
 *                      row r % page_size of block block_table[b][r / page_size].
 *   page_size        : a multiple of 32 (a decode tile never straddles blocks).
 *   The cache capacity per sequence is max_blocks_per_seq * page_size; it plays
 *   the part of S_cap (lengths above it are clamped and flagged, as in
 *   plx_decode), also for plx_decode_workspace_size.  A block id outside
 *   [0, num_blocks) is never dereferenced: block 0 is read in its place and the
 *   device status word reports PLX_ERR_INVALID_ARG through
 *   plx_last_device_error.
 * Other arguments, the result and the errors are those of plx_decode.
 */
plx_status plx_decode_paged(const void* q, const void* rho, const void* k_pages, const void* v_pages,
                            const int32_t* block_table, const int32_t* seqlens, void* out, float* lse, int B, int H,
                            int d, int page_size, int max_blocks_per_seq, int num_blocks, float scale, int num_splits,
                            void* workspace, size_t workspace_bytes, plx_dtype out_dtype, void* stream);

/*
 * plx_decode_family -- plx_decode with the family switches above (flags 0 is
 * plx_decode itself).  Same kernels, same arguments and errors, plus
 * PLX_ERR_INVALID_ARG for unknown flag bits and for PLX_FAMILY_NO_INTERCEPT
 * without rho.
 */
plx_status plx_decode_family(const void* q, const void* rho, const void* k_cache, const void* v_cache,
                             const int32_t* seqlens, void* out, float* lse, int B, int H, int d, int S_cap,
                             float scale, int num_splits, void* workspace, size_t workspace_bytes, unsigned flags,
                             plx_dtype out_dtype, void* stream);

/*
 * plx_decode_noalloc -- plx_decode for callers that cannot allocate device
 * memory: code running where cudaMalloc is off limits (under an allocator
 * that owns all device memory, or in a process that must not grow its
 * footprint after start-up) cannot provide the workspace that plx_decode
 * asks for.  This entry point takes no workspace
 * and allocates nothing; the split partials go to a scratch array that the
 * library holds in static device memory, PLX_DECODE_NOALLOC_SCRATCH_BYTES
 * (4 MiB) on every GPU that loads the library, until the process exits.
 * The paper has no counterpart: this is an interface convenience only.
 *
 * Arguments, layouts, numerics and results are those of plx_decode, which
 * it calls with the scratch array as the workspace.
 *   num_splits : 0 picks plx_decode's split count, lowered if needed to the
 *                largest count whose partials fit in the scratch
 *                (B * H * splits * (2 d + 4) * 4 bytes <= 4 MiB); two or
 *                more splits need B * H <= 2016 at d = 128 (B * H <= 3971 at
 *                d = 64), and above that one split runs, which needs no
 *                scratch.  An explicit count whose partials do not fit is
 *                rejected with PLX_ERR_UNSUPPORTED before anything is
 *                launched.
 * The first call on a device looks up the scratch array's device address
 * (cudaGetSymbolAddress, once per device and context, with that device
 * current); make that first call before any stream capture.  After
 * cudaDeviceReset the next call looks the address up again.  Every call on a device shares
 * the one array, so calls that may overlap on the GPU (on different streams,
 * or from several host threads) race with each other: order them on one
 * stream.  The array keeps the previous call's partials; nothing in it needs
 * to start at zero because every split writes its whole partial before the
 * combine reads it.
 * Errors: as plx_decode, and PLX_ERR_UNSUPPORTED for the case above.
 */
#define PLX_DECODE_NOALLOC_SCRATCH_BYTES (4u << 20)
plx_status plx_decode_noalloc(const void* q, const void* rho, const void* k_cache, const void* v_cache,
                              const int32_t* seqlens, void* out, float* lse, int B, int H, int d, int S_cap,
                              float scale, int num_splits, plx_dtype out_dtype, void* stream);

/*
 * plx_decode_partials / plx_decode_combine -- plx_decode with its key range
 * split over several caches (for instance over GPUs, each holding a slice of
 * every sequence's positions), merged afterwards.  The decode streams K and V
 * once with an online softmax ("Parallax: Parameterized Local Linear
 * Attention for Language Modeling", gist.science, "Algoritmo Consapevole
 * dell'Hardware"); over any set of disjoint key ranges it keeps the state
 *   m = max s_j,  l = sum e^{s_j - m},  C = sum e^{s_j - m} r_j,
 *   A = sum e^{s_j - m} v_j,  U = sum e^{s_j - m} r_j v_j
 * (s_j = scale q.k_j in log2 units, r_j = rho.k_j), and states of disjoint
 * ranges merge exactly by the log-sum-exp weighting the split combine of
 * plx_decode uses: M = max m_g, w_g = 2^(m_g - M), L = sum w_g l_g, C, A, U
 * likewise, then o = (1 + C/L) A/L - U/L and lse = (M + log2 L) ln 2.
 *
 * plx_decode_partials: the states of one shard.
 *   k_shard, v_shard : bf16 [B][H][S_shard][d]; row r of sequence b is
 *                      position key_begin + r.  Sequence b has
 *                      clamp(seqlens[b] - key_begin, 0, S_shard) keys here
 *                      (its query at position seqlens[b] - 1 sees every
 *                      position below seqlens[b]); a shard with none of a
 *                      sequence's keys writes the empty state (m = -inf,
 *                      l = 0).  A length past the shard is not an error.
 *   q, rho, seqlens  : as plx_decode (rho NULL: softmax attention).
 *   partials         : fp32 [B*H][num_splits][2 d + 4] = (m, l, C, 0, A[d],
 *                      U[d]) per split of the shard's range, m in log2 units;
 *                      plx_decode_partials_size(B, H, d, num_splits) bytes,
 *                      16-byte aligned.
 *   key_begin >= 0, S_shard >= 1, num_splits in [1, 1024] (explicit: every
 *   shard must use the count the combine is told).
 * plx_decode_combine: merges `groups` such buffers, concatenated in shard
 * order ([groups][B*H][num_splits][2 d + 4], e.g. an all-gather of every
 * shard's partials), into out (bf16 or fp32 [B][H][d]) and lse (fp32 [B][H],
 * natural log, may be NULL).  with_rho: the shards ran with rho (PLX) or
 * without (softmax attention); flags: 0 or PLX_FAMILY_NO_INTERCEPT (needs
 * with_rho).  The result equals plx_decode over the whole range up to fp32
 * rounding of the merge order.  One launch each on `stream`.
 * Errors: PLX_ERR_INVALID_ARG, PLX_ERR_UNSUPPORTED (d), PLX_ERR_MISALIGNED,
 * PLX_ERR_WORKSPACE (partials buffer too small), PLX_ERR_CUDA.
 */
size_t plx_decode_partials_size(int B, int H, int d, int num_splits);
plx_status plx_decode_partials(const void* q, const void* rho, const void* k_shard, const void* v_shard,
                               const int32_t* seqlens, int key_begin, void* partials, size_t partials_bytes, int B,
                               int H, int d, int S_shard, float scale, int num_splits, void* stream);
plx_status plx_decode_combine(const void* partials, int groups, int num_splits, void* out, float* lse, int B, int H,
                              int d, int with_rho, unsigned flags, plx_dtype out_dtype, void* stream);

/*
 * plx_lla_f32 -- local linear attention (LLA) with the solved probe, the
 * method Parallax replaces ("Parallax: Parameterized Local Linear Attention
 * for Language Modeling", zhichai.net section 1.2; gist.science "Enunciato
 * del Problema"): each token's probe solves a ridge-regularised linear system
 * by conjugate gradients, then Parallax's output formula uses it.  For query
 * i of one head (causal prefix j <= i), with w_ij = softmax_j(scale q_i.k_j):
 *
 *   (Sigma_KK^(i) + lambda I) rho_i = mu_i,   mu_i = kbar_i - q_i
 *   Sigma_KK^(i) = sum_j w_ij (k_j - kbar_i)(k_j - kbar_i)^T,  kbar_i = sum_j w_ij k_j
 *   o_i = vbar_i - Sigma_KV^(i) rho_i
 *
 * (the intercept at k = q_i of the weighted ridge fit of v on k - q_i).
 * Conjugate gradients start from rho = 0.  Each row runs at most max_iters
 * steps and stops once |r|^2 <= tol^2 |mu|^2 (tol = 0 runs every step), or
 * when p . Ap <= 0.  The arithmetic is fp32 on the CUDA cores, except the
 * CG steps after the first of the kept-weights path with N % 4 == 0 (see
 * plx_lla_kept_weights_workspace_size), which run on the tensor cores with
 * every product split in tf32 (fp32 accumulation).
 *
 *   q, k, v  : fp32 [B][H][N][d], 16-byte aligned.
 *   out      : fp32 [B][H][N][d] output, 16-byte aligned.
 *   rho_out  : fp32 [B][H][N][d], the solved probe, or NULL; 16-byte aligned.
 *   lse      : fp32 [B][H][N] natural-log softmax normaliser, or NULL.
 *   steps_out: int32 [B][H][N] conjugate-gradient steps taken per row, or NULL.
 *   workspace: device scratch of plx_lla_workspace_size(B, H, N, d) bytes,
 *              256-byte aligned, no initialisation; with at least
 *              plx_lla_kept_weights_workspace_size(B, H, N, d) bytes the
 *              softmax weights are kept across the CG steps (see there).
 *   B, H, N >= 1, B * H <= 65535; d a multiple of 32 in [32, 256];
 *   lambda >= 0 (finite); max_iters >= 0; tol >= 0 (finite).
 *   lambda = 0 needs every row's Sigma_KK to be non-singular (a prefix of at
 *   least d + 1 keys in general position); a row with p . Ap <= 0 stops.
 * max_iters + 3 launches on `stream`, plus a device-to-device copy for each
 * of rho_out and steps_out that is given.
 * Errors: PLX_ERR_INVALID_ARG, PLX_ERR_UNSUPPORTED, PLX_ERR_MISALIGNED,
 * PLX_ERR_WORKSPACE, PLX_ERR_CUDA.
 */
plx_status plx_lla_f32(const float* q, const float* k, const float* v, float* out, float* rho_out, float* lse,
                       int32_t* steps_out, void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                       float scale, float lambda, int max_iters, float tol, void* stream);

/* Workspace bytes plx_lla_f32 needs: about B*H*N*(4d + 4)*4 (0 for invalid sizes). */
size_t plx_lla_workspace_size(int B, int H, int N, int d);

/*
 * Workspace bytes with which plx_lla_f32 keeps the CG steps' softmax weights
 * w_ij = exp(s_ij - lse_i) from the first step instead of recomputing them in
 * every step (they do not depend on the iterate): plx_lla_workspace_size plus
 * B*H*N*N*4 bytes (rounded up to 256), for d in {64, 128} (for other d the
 * same as plx_lla_workspace_size).  A call given at least this many bytes
 * takes that path: the kbar pass stores the scores s_ij, the first step
 * (CUDA cores, fp32) turns them into the weights, the output pass reads them
 * (for blocks of rows that all took a step), and
 *   - N % 4 == 0: the later steps read them by TMA and run on the tensor
 *     cores with every product split in tf32 (x = hi + lo, hi.hi + hi.lo +
 *     lo.hi, fp32 sums): results within fp32 rounding of the recomputing
 *     path's, not bit for bit;
 *   - N % 4 != 0: the later steps read them on the CUDA cores: the
 *     recomputing path's results, bit for bit (the scores and weights are
 *     formed with the recomputing path's products, in the same order).
 * The extra space grows as N^2 (1.07 GB at B = 4, H = 16, N = 2048; 275 GB
 * at N = 32768), so it is for short contexts.
 */
size_t plx_lla_kept_weights_workspace_size(int B, int H, int N, int d);

/*
 * plx_probe_proj -- the probe projection rho_i = W_R x_i that feeds every
 * PLX entry point (zhichai.net section 1.3: the probe is a learned linear
 * map of the token's hidden state), on the tensor cores (tcgen05, bf16
 * operands, fp32 accumulation, bf16 result):
 *
 *   rho[b][h][n][:] = W_R[h d : (h + 1) d][:] . x[b][n][:]
 *
 *   x    : bf16 [B][N][Dx] hidden states, 16-byte aligned.
 *   w_r  : bf16 [H * d][Dx], head h's d x Dx block in rows h d .. h d + d - 1,
 *          16-byte aligned.
 *   rho  : bf16 [B][H][N][d] output (the layout plx_fwd, plx_bwd and
 *          plx_fwd_cached read), written, 16-byte aligned; must not overlap
 *          x or w_r.
 *   B, N, H, Dx >= 1; d in {64, 128}; Dx a multiple of 8 (16-byte rows).
 * One persistent launch on `stream`; each output element is one fp32 dot
 * product of length Dx rounded once to bf16, and the result does not depend
 * on the launch configuration.
 * Errors: PLX_ERR_INVALID_ARG (null pointer, non-positive size),
 * PLX_ERR_UNSUPPORTED (d, or Dx not a multiple of 8), PLX_ERR_MISALIGNED,
 * PLX_ERR_CUDA; device-side wait timeouts are reported by
 * plx_last_device_error.
 */
plx_status plx_probe_proj(const void* x, const void* w_r, void* rho, int B, int N, int H, int d, int Dx,
                          void* stream);

/*
 * plx_last_device_error -- synchronises `stream`, then reads and clears the
 * current device's status word.  Returns PLX_ERR_TIMEOUT if a kernel gave up
 * a bounded wait, PLX_ERR_INVALID_ARG if a decode length exceeded S_cap,
 * PLX_ERR_RANGE if plx_fwd wrote a non-finite output, PLX_ERR_BOUNDS if a
 * library built with PLX_DEBUG caught an index outside its buffer, PLX_ERR_CUDA if
 * synchronisation failed, else PLX_OK.
 */
plx_status plx_last_device_error(void* stream);

/*
 * plx_selftest_wait -- a diagnostic of the device-side failure detection.
 * Every kernel of the library waits on shared-memory barriers with a bounded
 * wait: after a wall-time limit (4 s in the kernels) it gives up, records
 * PLX_ERR_TIMEOUT in the device status word and returns instead of hanging.
 * This call runs that same wait once, in a one-thread kernel, on a barrier
 * with nothing asynchronous in flight, with the limit given here.
 *   limit_us : 1 .. 1000000 (microseconds).
 *   arrive   : nonzero arrives on the barrier first, so the wait completes
 *              and the status word is left alone; zero leaves the barrier
 *              alone, so the wait gives up after limit_us and the next
 *              plx_last_device_error returns PLX_ERR_TIMEOUT.
 * The device stays usable afterwards.  The pages have no counterpart: this
 * checks the library's own bounded waits.
 * Errors: PLX_ERR_INVALID_ARG (limit out of range), PLX_ERR_CUDA.
 */
plx_status plx_selftest_wait(unsigned int limit_us, int arrive, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PLX_H */
