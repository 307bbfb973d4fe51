// Internal interface between the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace parallax {

// ---------------------------------------------------------------- decode
struct DecodePlan {
    int B, H, Lmax, d;
    int chunk;   // keys per split-KV chunk (a multiple of the stage size)
    int nsplit;  // ceil(Lmax / chunk); 1 = no split, no combine kernel
    int grid;    // persistent CTAs
    float scale;
};

size_t decode_workspace_bytes(const DecodePlan& plan);
int decode_stage_keys(int d, int elem_bytes);
int decode_threads();
cudaError_t decode_launch(const DecodePlan& plan, bool bf16, const void* q, const void* rho,
                          const void* kc, const void* vc, const int32_t* seqlens, float* o,
                          void* ws, cudaStream_t stream);
unsigned decode_take_error();
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

// bf16 tcgen05 / TMEM / TMA prefill
cudaError_t prefill_tc_launch(const PrefillShape& s, const void* q, const void* rho,
                              const void* k, const void* v, float* o, int num_sms,
                              cudaStream_t stream);
unsigned prefill_tc_take_error();

}  // namespace parallax
