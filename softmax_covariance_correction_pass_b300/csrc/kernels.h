// Internal interface between the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace parallax {

// ---------------------------------------------------------------- decode
struct DecodePlan {
    int B, H, Lmax, d;
    int Hkv;  // key/value heads (H for plain attention; H / group size with shared heads)
    // paged cache: page_size > 0; key t of sequence b is row t % page_size of page
    // block_table[b * max_pages + t / page_size]; Lmax = max_pages * page_size
    int page_size, max_pages, num_pages;
    int chunk;   // keys per split-KV chunk (a multiple of the stage size)
    int nsplit;  // ceil(Lmax / chunk); 1 = no split, no combine kernel
    int grid;    // persistent CTAs
    float scale;
    // bf16, one query head per key/value head: run the tensor-core decode kernel (the
    // grouped kernels always do when their cache layout allows it)
    bool mma;
};

size_t decode_workspace_bytes(const DecodePlan& plan);
// Whether a decode with this plan runs the tensor-core kernel (decode_mma_kernel) rather than
// the SIMT kernel (decode_kernel); every launch decides with this function.
bool decode_uses_mma(const DecodePlan& plan, bool bf16);
int decode_stage_keys(int d, int elem_bytes);
int decode_threads();
int decode_ctas_per_sm();  // resident decode CTAs per SM the kernel is built for
cudaError_t decode_launch(const DecodePlan& plan, bool bf16, const void* q, const void* rho,
                          const void* kc, const void* vc, const int32_t* seqlens, float* o,
                          void* ws, cudaStream_t stream, const int32_t* block_table = nullptr);
// Largest chunk (keys) whose page ids fit the per-item table of the paged decode.
int decode_paged_max_chunk(int page_size);
unsigned decode_take_error();
// One thread waits, with the given limit, on an mbarrier nothing arrives on (test hook).
cudaError_t decode_wait_selftest(uint64_t limit_ns, cudaStream_t stream);
// Same as decode_launch with the split-KV partials in a fixed device array
// (no allocation).  Fails with cudaErrorInvalidValue if the plan needs more
// than decode_noalloc_capacity() bytes.
size_t decode_noalloc_capacity();
cudaError_t decode_launch_noalloc(const DecodePlan& plan, bool bf16, const void* q,
                                  const void* rho, const void* kc, const void* vc,
                                  const int32_t* seqlens, float* o, cudaStream_t stream);

// ---------------------------------------------------------------- prefill
struct PrefillShape {
    int B, H, L, d;
    int causal;
    float scale;
};

// fp32 (or bf16, for cross-checks inside the library) SIMT prefill
cudaError_t prefill_simt_launch(const PrefillShape& s, bool bf16, const void* q, const void* rho,
                                const void* k, const void* v, float* o, cudaStream_t stream);
unsigned prefill_simt_take_error();

// Per-row quantities a training forward keeps for the backward pass (all null: none).
struct TrainStats {
    float* lse = nullptr;   // [B, H, L] log-sum-exp of the scaled scores (natural log)
    float* rbar = nullptr;  // [B, H, L] sum_j p_j r_j (0 without the probe)
    float* mu = nullptr;    // [B, H, L, d] mu_v = sum_j p_j v_j
};

// bf16 tcgen05 / TMEM / TMA prefill
cudaError_t prefill_tc_launch(const PrefillShape& s, const void* q, const void* rho,
                              const void* k, const void* v, float* o, int num_sms,
                              cudaStream_t stream, const TrainStats& ts = TrainStats{});
unsigned prefill_tc_take_error();
cudaError_t prefill_tc_wait_selftest(uint64_t limit_ns, cudaStream_t stream);
// Chunked prefill: append k_new / v_new [B, H, L, d] to the caches [B, H, Lmax, d] at
// rows cache_lens[b].., then causal attention of the chunk's queries over the cache.
cudaError_t prefill_tc_chunk_launch(const PrefillShape& s, const void* q, const void* rho,
                                    const void* k_new, const void* v_new, void* k_cache,
                                    void* v_cache, const int32_t* cache_lens, int Lmax, float* o,
                                    int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------- prefill backward
// Row-stats workspace (float4 per query row) the backward needs.
size_t prefill_backward_workspace_bytes(int B, int H, int L);
cudaError_t prefill_backward_launch(const PrefillShape& s, const void* q, const void* rho,
                                    const void* k, const void* v, const float* o,
                                    const float* mu, const float* lse, const float* rbar,
                                    const void* dout, float* dq, float* drho, float* dk,
                                    float* dv, void* ws, cudaStream_t stream);
unsigned prefill_backward_take_error();

// ---------------------------------------------------------------- exact LLA decode
// Per (b, h), one pass over K and V: rho = Sigma_kk^-1 (mu_k - q) by conjugate gradient and
// o = mu_v - C^T rho (both fp32 [B*H, d]).
cudaError_t lla_launch(const void* q, const void* kc, const void* vc, const int32_t* seqlens,
                       float* rho, float* o, int B, int H, int Lmax, int d, int iters,
                       cudaStream_t stream);
unsigned lla_take_error();

// ---------------------------------------------------------------- tensor maps
// bf16 tensor of `rank` dims (innermost first; strides in bytes of dims 1..rank-1),
// box `box`, 128-byte swizzle, out-of-range elements read as zero.
bool make_tmap_bf16(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box);
// The same for an fp32 tensor (box[0] * 4 bytes must be 128: one swizzle row).
bool make_tmap_f32(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                   const uint64_t* strides_bytes, const uint32_t* box);

// ---------------------------------------------------------------- q/k/v/probe projection
struct ProjShape {
    int B, L, width, H, d;
    int n_out;  // 4 (q, k, v, rho) or 3 (no probe)
};

// out[t] = bf16 [B, H, L, d] slices of x [B, L, width] times w[t*H*d .. (t+1)*H*d - 1, :]^T
cudaError_t proj_tc_launch(const ProjShape& s, const void* x, const void* w, void* const out[4],
                           int num_sms, cudaStream_t stream);
unsigned proj_tc_take_error();

}  // namespace parallax
