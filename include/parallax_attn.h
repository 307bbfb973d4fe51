/*
 * parallax_attn.h -- C ABI of the Parallax attention forward hot path (sm_103a).
 *
 * Parallax attention ("Parallax mantem softmax, correcao de covariancia
 * aprendida", zubnet.ai news page, paragraph 2; the French twin of that page,
 * paragraph 2) keeps softmax attention and subtracts a learned correction: the
 * key/value covariance under the softmax weights, multiplied by a probe
 * rho_i = W_R x_i computed from the layer input.  For query row i over its key
 * set J(i):
 *
 *   p_ij  = softmax_j(scale * q_i . k_j)
 *   mu_v  = sum_j p_ij v_j,   mu_k = sum_j p_ij k_j
 *   C_i   = sum_j p_ij (k_j - mu_k)(v_j - mu_v)^T          (d x d)
 *   o_i   = mu_v - C_i^T rho_i
 *
 * The kernels evaluate the same quantity in one pass over K and V, with
 * r_ij = rho_i . k_j (unscaled):
 *   o_i = mu_v - ( sum_j p_ij r_ij v_j - (sum_j p_ij r_ij) mu_v ),
 * so each key/value tile feeds both the softmax branch and the correction
 * branch (the pages' "same KV stream reused for both branches").
 * Passing rho == NULL selects the W_R = 0 path, which is exactly softmax
 * attention (the pages' retrofit property).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never frees or retains them.  Every tensor is dense row-major.
 *   - Every pointer must be 16-byte aligned.
 *   - Every pointer and `stream` belong to the calling thread's current CUDA
 *     device (cudaSetDevice): the library launches there and keeps its
 *     workspaces per device.  The library does not check where a pointer lives;
 *     the Python binding refuses tensors on another device.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream) and never
 *     synchronise, except parallax_check_device_error().
 *   - Return value: PARALLAX_OK or a negative parallax_status.  Argument errors
 *     are detected on the host before anything is launched; the message is
 *     available from parallax_last_error() on the calling thread.
 *   - Head dimension d must be 64 or 128 (PARALLAX_ERR_UNSUPPORTED otherwise).
 *   - Attention outputs o are always fp32 (the projection writes bf16).
 *   - The library keeps per-device state (workspaces, the no-allocation array's
 *     address, kernel attributes) for the life of the process: do not use it
 *     across a cudaDeviceReset() of a device it has run on.
 */
#ifndef PARALLAX_ATTN_H
#define PARALLAX_ATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PARALLAX_OK = 0,
    PARALLAX_ERR_INVALID = -1,     /* bad pointer, size, flag or scale           */
    PARALLAX_ERR_UNSUPPORTED = -2, /* valid but not implemented (e.g. d = 96)    */
    PARALLAX_ERR_CUDA = -3,        /* a CUDA runtime call or launch failed       */
    PARALLAX_ERR_DEVICE = -4       /* a kernel reported an error (see below)     */
} parallax_status;

/* Bits of the device error word returned by parallax_check_device_error(). */
#define PARALLAX_DEVERR_SEQLEN_CLAMPED 0x1u /* a seqlens[b] lay outside [0, Lmax] */
#define PARALLAX_DEVERR_WAIT_TIMEOUT 0x2u   /* a pipeline wait gave up (bug)      */
#define PARALLAX_DEVERR_PAGE_OUT_OF_RANGE 0x4u /* a block-table entry lay outside
                                                  [0, num_pages); page 0 was read */
#define PARALLAX_DEVERR_SMEM_MISALIGNED 0x8u /* a kernel's dynamic shared memory was not
                                                1024-byte aligned; it did no work (bug) */
#define PARALLAX_DEVERR_BOUNDS 0x10u /* debug builds only: a global write or copy would have
                                        left its tensor; it was skipped or redirected (bug) */

/*
 * Causal or full prefill, bf16 inputs, fp32 output.
 *   q, rho, k, v : bf16 [B, H, L, d]   (rho may be NULL: W_R = 0 fast path)
 *   o            : fp32 [B, H, L, d]   written in full
 *   causal       : 1 -> query i sees keys 0..i (diagonal included); 0 -> all L keys
 *   scale        : multiplies q . k only (typically 1/sqrt(d)); must be finite
 * Uses the tcgen05 tensor-core kernel (TMA-fed, TMEM accumulators).
 * B, H, L >= 1.  No workspace.
 */
int parallax_attn_prefill(const void* q, const void* rho, const void* k, const void* v, void* o,
                          int B, int H, int L, int d, int causal, float scale,
                          cudaStream_t stream);

/*
 * Chunked causal prefill that continues cached sequences (bf16 in, fp32 out):
 * a serving engine prefills a long prompt, or appends a turn, a chunk at a time
 * against the KV cache that the pages' decode setting keeps.
 *   q, rho, k_new, v_new : bf16 [B, H, Lq, d]    the chunk (rho may be NULL)
 *   k_cache, v_cache     : bf16 [B, H, Lmax, d]  sequence b holds cache_lens[b] tokens
 *   cache_lens           : int32 [B] on the device (not modified)
 *   o                    : fp32 [B, H, Lq, d]
 * The call first writes the chunk's k_new / v_new rows into the caches at rows
 * cache_lens[b] .. cache_lens[b] + Lq - 1, then chunk token i (position
 * p = cache_lens[b] + i) attends causally to cache rows 0 .. p -- the earlier
 * tokens and the chunk's own tokens up to itself.  Rows of o equal the rows
 * p of one causal parallax_attn_prefill over the whole sequence.  A
 * cache_lens[b] outside [0, Lmax - Lq] is clamped into it and raises
 * PARALLAX_DEVERR_SEQLEN_CLAMPED.  The caller advances cache_lens by Lq.
 * Lmax >= Lq >= 1.  No workspace.
 */
int parallax_attn_prefill_chunk(const void* q, const void* rho, const void* k_new,
                                const void* v_new, void* k_cache, void* v_cache,
                                const int32_t* cache_lens, void* o, int B, int H, int Lq,
                                int Lmax, int d, float scale, cudaStream_t stream);

/*
 * Training forward: parallax_attn_prefill (bf16, tensor cores) that also keeps
 * the per-row quantities the backward pass needs.
 *   lse   : fp32 [B, H, L]     log sum_j exp(scale q_i.k_j) over the row's keys
 *   rbar  : fp32 [B, H, L]     sum_j p_ij r_ij (the p-weighted mean of rho_i.k_j; 0 if rho == NULL)
 *   mu_v  : fp32 [B, H, L, d]  sum_j p_ij v_j (the softmax branch alone)
 * Other arguments as parallax_attn_prefill.  No workspace.
 */
int parallax_attn_prefill_train(const void* q, const void* rho, const void* k, const void* v,
                                void* o, float* lse, float* rbar, float* mu_v, int B, int H, int L,
                                int d, int causal, float scale, cudaStream_t stream);

/*
 * Backward pass of the prefill (the pages' results all come from pretraining;
 * this is the gradient of the forward above).  Writing o_i = sum_j w_ij v_j with
 * w_ij = p_ij (1 + rbar_i - r_ij), r_ij = rho_i.k_j, and given dout = dL/do:
 *   dv_j = sum_i w_ij dout_i
 *   dq_i = scale sum_j ds_ij k_j,    drho_i = sum_j dr_ij k_j
 *   dk_j = scale sum_i ds_ij q_i + sum_i dr_ij rho_i
 *   dr_ij = p_ij (abar_i - D_ij),    ds_ij = p_ij ((D_ij - abar_i)(rbar_i - r_ij) + D_ij - delta_i)
 * with D_ij = dout_i.v_j, abar_i = dout_i.mu_v,i, delta_i = dout_i.o_i.
 *   q, rho, k, v      : bf16 [B, H, L, d] (the forward's inputs; rho may be NULL)
 *   o, mu_v, lse, rbar: fp32, from parallax_attn_prefill_train on the same inputs
 *   dout              : bf16 [B, H, L, d]
 *   dq, drho, dk, dv  : fp32 [B, H, L, d], written in full (drho unused if rho == NULL)
 * The contractions run on the tcgen05 tensor cores with bf16 operands (p-weighted
 * terms rounded to bf16) and fp32 accumulation.  Uses a library-owned per-device
 * workspace of 16 B per query row, grown in stream order like the decode
 * workspace (same concurrency rules).
 */
int parallax_attn_prefill_backward(const void* q, const void* rho, const void* k, const void* v,
                                   const float* o, const float* mu_v, const float* lse,
                                   const float* rbar, const void* dout, float* dq, float* drho,
                                   float* dk, float* dv, int B, int H, int L, int d, int causal,
                                   float scale, cudaStream_t stream);

/* Same as parallax_attn_prefill with fp32 q, rho, k, v (fp32 SIMT arithmetic). */
int parallax_attn_prefill_f32(const void* q, const void* rho, const void* k, const void* v,
                              void* o, int B, int H, int L, int d, int causal, float scale,
                              cudaStream_t stream);

/*
 * Single-token decode against a KV cache, bf16 inputs, fp32 output.
 *   q, rho            : bf16 [B, H, d]          (rho may be NULL: W_R = 0)
 *   k_cache, v_cache  : bf16 [B, H, Lmax, d]    sequence b uses rows 0..seqlens[b]-1
 *   seqlens           : int32 [B] on the device
 *   o                 : fp32 [B, H, d]
 * The softmax scale is 1/sqrt(d).  A seqlens[b] outside [0, Lmax] is clamped
 * into range and PARALLAX_DEVERR_SEQLEN_CLAMPED is raised on the device; a
 * sequence of length 0 yields o = 0.
 * Long caches are split into fixed-size key chunks processed in parallel
 * (split-KV); the per-chunk partial states are merged by a log-sum-exp combine
 * kernel.  The partials live in a library-owned device workspace, one per
 * device, grown on demand in stream order: a call that needs more space frees
 * the old buffer with cudaFreeAsync and allocates the new one with
 * cudaMallocAsync on `stream`, after making `stream` wait for the last call
 * that used the old buffer (whatever its stream), so growing never
 * synchronises the device.  The workspace is shared by all calls on a device:
 * calls issued concurrently from several host threads, or on several streams
 * that may overlap, race on its contents.
 */
int parallax_attn_decode(const void* q, const void* rho, const void* k_cache,
                         const void* v_cache, const int32_t* seqlens, void* o, int B, int H,
                         int Lmax, int d, cudaStream_t stream);

/* Same as parallax_attn_decode with fp32 q, rho, k_cache, v_cache. */
int parallax_attn_decode_f32(const void* q, const void* rho, const void* k_cache,
                             const void* v_cache, const int32_t* seqlens, void* o, int B, int H,
                             int Lmax, int d, cudaStream_t stream);

/*
 * Decode with key/value heads shared by groups of query heads (grouped-query
 * attention), bf16 inputs, fp32 output.
 *   q, rho            : bf16 [B, H, d]            (rho may be NULL: W_R = 0)
 *   k_cache, v_cache  : bf16 [B, H_kv, Lmax, d]   query head h reads head h / (H / H_kv)
 *   seqlens, o        : as in parallax_attn_decode
 * H / H_kv must be 1, 2, 4 or 8 (PARALLAX_ERR_UNSUPPORTED otherwise); each key
 * and value row is read from HBM once for the whole group.  Workspace and
 * concurrency rules of parallax_attn_decode; the split plan depends on the group
 * size (parallax_attn_decode_plan_keys).
 * The Parallax pages do not discuss head sharing; the result is, per query
 * head, exactly parallax_attn_decode against that head's key/value head.
 */
int parallax_attn_decode_gqa(const void* q, const void* rho, const void* k_cache,
                             const void* v_cache, const int32_t* seqlens, void* o, int B, int H,
                             int H_kv, int Lmax, int d, cudaStream_t stream);

/*
 * Decode against a paged key/value cache (the pages' decode setting keeps a KV
 * cache; a serving engine keeps it in fixed-size pages), bf16 inputs, fp32 out.
 *   q, rho            : bf16 [B, H, d]            (rho may be NULL: W_R = 0)
 *   k_pages, v_pages  : bf16 [num_pages, H_kv, page_size, d]  the page pool
 *   block_table       : int32 [B, max_pages] on the device; key t of sequence b
 *                       is row t % page_size of page block_table[b, t / page_size]
 *   seqlens           : int32 [B] on the device, clamped to [0, max_pages * page_size]
 *   o                 : fp32 [B, H, d]
 * page_size must be a multiple of 16; H / H_kv must be 1, 2, 4 or 8.  Only the
 * table entries of a sequence's first ceil(seqlens[b] / page_size) pages are
 * read; an entry outside [0, num_pages) is replaced by page 0 and raises
 * PARALLAX_DEVERR_PAGE_OUT_OF_RANGE (no read leaves the pool).  Workspace and
 * concurrency rules of parallax_attn_decode.
 */
int parallax_attn_decode_paged(const void* q, const void* rho, const void* k_pages,
                               const void* v_pages, const int32_t* block_table,
                               const int32_t* seqlens, void* o, int B, int H, int H_kv,
                               int page_size, int max_pages, int num_pages, int d,
                               cudaStream_t stream);

/*
 * Exact local linear attention (LLA) decode, the method whose per-query solve the
 * Parallax probe replaces (the pages: Parallax keeps LLA's covariance correction
 * and swaps the solve for rho = W_R x).  For one query token per (b, h):
 *   p_j = softmax_j(q.k_j / sqrt(d)),  mu_k = sum p k,
 *   Sigma_kk = sum_j p_j (k_j - mu_k)(k_j - mu_k)^T,
 *   rho = Sigma_kk^-1 (mu_k - q)  by conjugate gradient from rho = 0 (cg_iters
 *         steps, 0 = d; it also stops at a relative residual of 1e-6),
 *   o   = mu_v - C^T rho,  mu_v = sum p v,  C = sum_j p_j (k_j - mu_k)(v_j - mu_v)^T
 *         (the Parallax output with that probe, in fp32).
 *   q                 : bf16 [B, H, d]
 *   k_cache, v_cache  : bf16 [B, H, Lmax, d];  seqlens: int32 [B] on the device
 *   o                 : fp32 [B, H, d];  rho: fp32 [B, H, d] (the solved probes)
 * One CTA per (b, h) reads K and V once, accumulates the p-weighted key/key and
 * key/value second moments on the tensor cores (bf16 keys times p k and p v split
 * into a bf16 high part and residual, fp32 accumulators), and runs the CG in shared
 * memory.  A sequence with no keys gives o = 0 and rho = 0.  Allocates nothing.
 */
int parallax_lla_decode(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* seqlens, void* o, float* rho, int B, int H, int Lmax,
                        int d, int cg_iters, cudaStream_t stream);

/*
 * parallax_attn_decode without any device allocation (bf16 inputs, fp32 o).
 * This entry point has no counterpart in the Parallax paper; it exists for
 * callers that cannot let a library call cudaMalloc -- serving engines that
 * reserve nearly all device memory for their own KV-cache pool up front, and
 * latency-critical decode loops where an allocation's implicit device
 * synchronisation would stall every other stream.
 * Arguments, layout, result and split plan are those of parallax_attn_decode;
 * only the split-KV partial states live in a fixed array inside the library:
 * 8 MiB per device (2 * 4 B * d + 16 B per head per key chunk), held by every
 * GPU that loads the library until the process exits.  A shape whose split
 * needs more returns PARALLAX_ERR_UNSUPPORTED before anything is launched
 * (parallax_attn_decode handles it).  The first call on a device looks up
 * the array's device address (no allocation); make that first call before
 * any stream capture.  The array, like the decode kernels' code, is placed in
 * device memory when the library's decode module is first loaded on a device:
 * under CUDA's default lazy module loading that can be this entry point's first
 * call (or the first decode of any kind), so make one call -- or run one decode
 * -- on each device before reserving the rest of its memory for a cache pool.
 * All calls on a device share the array, so calls that may overlap on the GPU
 * (other streams, other host threads) race on it.
 */
int parallax_attn_decode_noalloc(const void* q, const void* rho, const void* k_cache,
                                 const void* v_cache, const int32_t* seqlens, void* o, int B,
                                 int H, int Lmax, int d, cudaStream_t stream);

/*
 * The layer's input projections in one tensor-core product: q, k, v and the
 * probe rho_i = W_R x_i (the probe is a learned linear map of the layer input:
 * "Parallax mantem softmax ...", zubnet.ai news page, paragraph 2).
 *   x      : bf16 [B, L, width]                one row per token
 *   w      : bf16 [n_out * H * d, width]       stacked weight W_q; W_k; W_v; W_R,
 *                                              rows = output features (n_out = 4,
 *                                              or 3 when rho == NULL: W_R = 0)
 *   q, k, v, rho : bf16 [B, H, L, d]           written in full; rho may be NULL
 *   out[t][b, h, l, c] = sum_a x[b, l, a] * w[t*H*d + h*d + c, a]
 * fp32 accumulation on the tcgen05 tensor cores, rounded to bf16 (nearest even).
 * The outputs are exactly the tensors parallax_attn_prefill reads.
 * Requirements: B, L, H >= 1; d = 64 or 128; H*d a multiple of 128 and width a
 * multiple of 8 (PARALLAX_ERR_UNSUPPORTED otherwise).  No workspace.
 */
int parallax_attn_qkvr_projection(const void* x, const void* w, void* q, void* k, void* v,
                                  void* rho, int B, int L, int width, int H, int d,
                                  cudaStream_t stream);

/*
 * Keys per split-KV chunk that parallax_attn_decode{,_f32} would use for this
 * shape (elem_bytes = 2 for bf16, 4 for fp32; one query head per key/value
 * head).  Returns a negative
 * parallax_status for invalid arguments.  A result >= Lmax means no split.
 */
int parallax_attn_decode_chunk_keys(int B, int H, int Lmax, int d, int elem_bytes);

/*
 * Keys per work item that parallax_attn_decode, parallax_attn_decode_gqa
 * (page_size = 0) or parallax_attn_decode_paged (page_size > 0, Lmax =
 * page_size * max_pages) would use for this shape.  The plan depends on the
 * group size H / H_kv: one query head per key/value head aims at about 16
 * items per SM, groups of 2 at about 8, groups of 4 and 8 take the longest
 * chunk that leaves at least 1.7 items per SM; chunks are 256..4096 keys, and
 * grouped heads on a paged cache take at most 2048.  A forced chunk
 * (parallax_attn_set_decode_chunk_keys) takes precedence.  Host-only: no
 * device work; without a device the SM count is taken as 148.
 * Errors: PARALLAX_ERR_INVALID for B, H, Lmax < 1, H not a multiple of H_kv
 * or page_size < 0; PARALLAX_ERR_UNSUPPORTED for d not 64 or 128, group sizes
 * other than 1, 2, 4, 8, or page_size not a multiple of 16.
 * A result >= Lmax means no split.
 */
int parallax_attn_decode_plan_keys(int B, int H, int H_kv, int Lmax, int d, int page_size);

/*
 * Which kernel the bf16 decode entry points run for this shape (same arguments and
 * errors as parallax_attn_decode_plan_keys): 1 for the tensor-core kernel (warp-level
 * MMAs on the stacked [q; rho] operand of a head group; grouped heads, and one head per
 * key/value head when every CTA gets at least two work items of 512 keys or more), 0 for
 * the SIMT kernel.  fp32 inputs always take the SIMT kernel.  Host-only.
 */
int parallax_attn_decode_plan_kernel(int B, int H, int H_kv, int Lmax, int d, int page_size);

/*
 * Force the decode chunk size (keys, a positive multiple of 256) for later
 * calls in this process, or restore the automatic choice with 0.  Meant for
 * tests that exercise the combine path at small sizes.
 */
int parallax_attn_set_decode_chunk_keys(int keys);

/* Bytes currently held by the calling device's decode workspace. */
size_t parallax_attn_workspace_bytes(void);

/*
 * Free the calling device's decode and backward workspaces.  Synchronises the
 * device first, so no call in flight still uses them.
 */
int parallax_attn_release_workspace(void);

/*
 * Thread-local description of the last error returned on this host thread
 * (empty string if none).  The pointer stays valid until the thread's next call.
 */
const char* parallax_last_error(void);

/*
 * Synchronise `stream`, then read and clear the device error word of the
 * current device.  Returns PARALLAX_OK if it was zero, PARALLAX_ERR_DEVICE if
 * not, or PARALLAX_ERR_CUDA if the synchronisation failed.  The bits that were
 * set (PARALLAX_DEVERR_*) stay available on the calling host thread through
 * parallax_last_device_error_bits() until its next check.
 */
int parallax_check_device_error(cudaStream_t stream);

/*
 * PARALLAX_DEVERR_* bits read by the calling thread's last
 * parallax_check_device_error() (0 if none were set, or if that check failed
 * before reading them).  Host-only.
 */
unsigned int parallax_last_device_error_bits(void);

/*
 * Overrun check of the library-owned workspaces (decode split-KV partials,
 * backward row statistics) of the current device.  Each workspace sits between
 * two 4 KB guard bands filled with 0xA5 when it is allocated; this call
 * synchronises the device and returns 1 if every band of every workspace still
 * holds that pattern, 0 if one was overwritten, or a negative parallax_status.
 * A debugging and test aid; it copies 8 KB per workspace to the host.
 */
int parallax_workspace_guards_intact(void);

/*
 * Test hook for the failure path of the bounded pipeline waits.  Every wait in
 * the library's kernels gives up after a time limit instead of spinning forever;
 * it then raises PARALLAX_DEVERR_WAIT_TIMEOUT in its kernel family's device
 * error word, and CTAs launched later in that family see the bit and return
 * without work until parallax_check_device_error() clears it.  This call launches
 * one thread that waits, with a limit of limit_us microseconds (1 .. 1000000), on
 * an mbarrier nothing arrives on, in the error word of `family`:
 *   PARALLAX_SELFTEST_DECODE  (0): the decode kernels (plain, grouped, paged)
 *   PARALLAX_SELFTEST_PREFILL (1): the tensor-core prefill kernels
 * Nothing faults and nothing hangs: the kernel ends after about limit_us.
 * Asynchronous on `stream`; read the result with parallax_check_device_error().
 */
#define PARALLAX_SELFTEST_DECODE 0
#define PARALLAX_SELFTEST_PREFILL 1
int parallax_selftest_wait_timeout(int family, unsigned int limit_us, cudaStream_t stream);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int parallax_version(void);

/*
 * 1 if this library was built with device-side bounds checks (the debug build,
 * libparallax_attn_debug.so: a global write or copy that would leave its tensor is
 * skipped or redirected and raises PARALLAX_DEVERR_BOUNDS), 0 for the release build.
 */
int parallax_debug_checks(void);

#ifdef __cplusplus
}
#endif

#endif /* PARALLAX_ATTN_H */
