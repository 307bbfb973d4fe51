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
 *   - Calls are asynchronous on `stream` (0 = legacy default stream) and never
 *     synchronise, except parallax_check_device_error().
 *   - Return value: PARALLAX_OK or a negative parallax_status.  Argument errors
 *     are detected on the host before anything is launched; the message is
 *     available from parallax_last_error() on the calling thread.
 *   - Head dimension d must be 64 or 128 (PARALLAX_ERR_UNSUPPORTED otherwise).
 *   - Output o is always fp32.
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
 * device, grown on demand (cudaMalloc; growing synchronises the device).  The
 * workspace is shared by all calls on a device: calls issued concurrently from
 * several host threads, or on several streams that may overlap, race on it.
 */
int parallax_attn_decode(const void* q, const void* rho, const void* k_cache,
                         const void* v_cache, const int32_t* seqlens, void* o, int B, int H,
                         int Lmax, int d, cudaStream_t stream);

/* Same as parallax_attn_decode with fp32 q, rho, k_cache, v_cache. */
int parallax_attn_decode_f32(const void* q, const void* rho, const void* k_cache,
                             const void* v_cache, const int32_t* seqlens, void* o, int B, int H,
                             int Lmax, int d, cudaStream_t stream);

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
 * any stream capture.  All calls on a device share the array, so calls that
 * may overlap on the GPU (other streams, other host threads) race on it.
 */
int parallax_attn_decode_noalloc(const void* q, const void* rho, const void* k_cache,
                                 const void* v_cache, const int32_t* seqlens, void* o, int B,
                                 int H, int Lmax, int d, cudaStream_t stream);

/*
 * Keys per split-KV chunk that parallax_attn_decode{,_f32} would use for this
 * shape (elem_bytes = 2 for bf16, 4 for fp32).  Returns a negative
 * parallax_status for invalid arguments.  A result >= Lmax means no split.
 */
int parallax_attn_decode_chunk_keys(int B, int H, int Lmax, int d, int elem_bytes);

/*
 * Force the decode chunk size (keys, a positive multiple of 256) for later
 * calls in this process, or restore the automatic choice with 0.  Meant for
 * tests that exercise the combine path at small sizes.
 */
int parallax_attn_set_decode_chunk_keys(int keys);

/* Bytes currently held by the calling device's decode workspace. */
size_t parallax_attn_workspace_bytes(void);

/* Free the calling device's decode workspace (synchronises the device). */
int parallax_attn_release_workspace(void);

/*
 * Thread-local description of the last error returned on this host thread
 * (empty string if none).  The pointer stays valid until the thread's next call.
 */
const char* parallax_last_error(void);

/*
 * Synchronise `stream`, then read and clear the device error word of the
 * current device.  Returns PARALLAX_OK if it was zero, PARALLAX_ERR_DEVICE if
 * not (the bits, PARALLAX_DEVERR_*, are stored to *bits when bits != NULL), or
 * PARALLAX_ERR_CUDA if the synchronisation failed.
 */
int parallax_check_device_error(cudaStream_t stream, unsigned int* bits);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int parallax_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PARALLAX_ATTN_H */
