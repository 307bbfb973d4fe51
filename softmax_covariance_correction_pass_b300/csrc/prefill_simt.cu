// Parallax prefill on the CUDA cores (fp32 path; also instantiated for bf16).
//
// A CTA owns QROWS = 8 consecutive query rows of one head (one warp per row)
// and streams that head's key/value rows through shared memory in tiles; all
// eight warps reuse each tile, and every warp updates both Parallax branches
// (softmax and covariance correction) from the same bytes.  Arithmetic is
// fp32 FMA throughout -- no tensor cores -- so the fp32 entry point keeps the
// full fp32 accuracy the tests ask of it.
#include "warp_stream.cuh"
#include "kernels.h"

namespace parallax {
namespace {

__device__ unsigned g_simt_err = 0;

constexpr int kRows = 8;  // query rows (= warps) per CTA
constexpr int kThreads = kRows * 32;
constexpr int kTileBytes = 16384;  // bytes of K (and of V) per tile

struct SimtArgs {
    const void* q;
    const void* rho;
    const void* k;
    const void* v;
    float* o;
    int L;
    float qscale;
    size_t o_elems;  // B * H * L * D (debug bounds checks)
};

template <typename T, int D, bool RHO, bool CAUSAL>
__global__ void __launch_bounds__(kThreads) prefill_simt_kernel(const SimtArgs a) {
    using KL = KeyLayout<T, D>;
    constexpr int VEC = KL::VEC;
    constexpr int TILE_KEYS = kTileBytes / KL::ROW_BYTES;
    __shared__ __align__(16) T sK[TILE_KEYS * D];
    __shared__ __align__(16) T sV[TILE_KEYS * D];

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int row_blocks = (a.L + kRows - 1) / kRows;
    const int bh = blockIdx.x / row_blocks;
    const int rb = blockIdx.x - bh * row_blocks;
    const int i = rb * kRows + warp;  // this warp's query row
    const int L = a.L;
    const size_t head = (size_t)bh * L * D;
    const T* Kh = static_cast<const T*>(a.k) + head;
    const T* Vh = static_cast<const T*>(a.v) + head;

    // keys any row of this CTA can see
    const int key_end = CAUSAL ? min(L, (rb + 1) * kRows) : L;
    const int my_end = (i < L) ? (CAUSAL ? i + 1 : L) : 0;  // keys this row sees

    const int e = lane % KL::LPK;
    float qf[VEC], rf[VEC];
    const int iq = min(i, L - 1);
    load_row_slice<T, D>(static_cast<const T*>(a.q) + head + (size_t)iq * D, e, a.qscale, qf);
    if (RHO) load_row_slice<T, D>(static_cast<const T*>(a.rho) + head + (size_t)iq * D, e, 1.f, rf);
    else
#pragma unroll
        for (int x = 0; x < VEC; ++x) rf[x] = 0.f;

    RowState<T, D> st;
    st.reset();
    constexpr int VECS_PER_TILE = TILE_KEYS * D / (16 / (int)sizeof(T));
    for (int t0 = 0; t0 < key_end; t0 += TILE_KEYS) {
        const int nk = min(TILE_KEYS, key_end - t0);
        __syncthreads();  // previous tile fully consumed
        const uint4* gK = reinterpret_cast<const uint4*>(Kh + (size_t)t0 * D);
        const uint4* gV = reinterpret_cast<const uint4*>(Vh + (size_t)t0 * D);
        const int nvec = nk * D / (16 / (int)sizeof(T));
        for (int x = threadIdx.x; x < VECS_PER_TILE; x += kThreads) {
            const uint4 zero = make_uint4(0, 0, 0, 0);
            reinterpret_cast<uint4*>(sK)[x] = x < nvec ? __ldg(gK + x) : zero;
            reinterpret_cast<uint4*>(sV)[x] = x < nvec ? __ldg(gV + x) : zero;
        }
        __syncthreads();
        const int nvalid = min(nk, my_end - t0);  // may be <= 0: the row sees none of this tile
        for (int kb = 0; kb < nvalid; kb += KL::BLOCK_KEYS)
            warp_block<T, D, RHO>(st, qf, rf, sK, sV, kb, nvalid, lane);
    }
    warp_merge_groups<T, D, RHO>(st);
    if (i < L && lane < KL::LPK &&
        in_bounds(&g_simt_err, head + (size_t)i * D + (e + 1) * VEC, a.o_elems))
        finish_slice<T, D, RHO>(st, a.o + head + (size_t)i * D + e * VEC);
}

template <typename T, int D, bool RHO>
cudaError_t run(const PrefillShape& s, const SimtArgs& a, cudaStream_t stream) {
    const unsigned grid = (unsigned)(((s.L + kRows - 1) / kRows) * (size_t)s.B * s.H);
    if (s.causal) prefill_simt_kernel<T, D, RHO, true><<<grid, kThreads, 0, stream>>>(a);
    else prefill_simt_kernel<T, D, RHO, false><<<grid, kThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t prefill_simt_launch(const PrefillShape& s, bool bf16, const void* q, const void* rho,
                                const void* k, const void* v, float* o, cudaStream_t stream) {
    SimtArgs a{q, rho, k, v, o, s.L, s.scale * kLog2e, (size_t)s.B * s.H * s.L * s.d};
    const bool r = rho != nullptr;
#define PARALLAX_SIMT_CASE(T, DD)                                           \
    if (s.d == DD) return r ? run<T, DD, true>(s, a, stream) : run<T, DD, false>(s, a, stream);
    if (bf16) {
        PARALLAX_SIMT_CASE(__nv_bfloat16, 64)
        PARALLAX_SIMT_CASE(__nv_bfloat16, 128)
    } else {
        PARALLAX_SIMT_CASE(float, 64)
        PARALLAX_SIMT_CASE(float, 128)
    }
#undef PARALLAX_SIMT_CASE
    return cudaErrorInvalidValue;
}

unsigned prefill_simt_take_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_simt_err, sizeof(v)) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_simt_err, &zero, sizeof(zero));
    return v;
}

}  // namespace parallax
