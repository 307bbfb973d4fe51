// Exact local linear attention (LLA) decode: the per-query solve that the
// Parallax probe replaces.  The Parallax pages describe their method as LLA's
// covariance correction with the per-query probe Sigma_kk^-1 (mu_k - q) swapped
// for the learned rho = W_R x ("Parallax mantem softmax ...", paragraphs 1-2);
// this computes the original, for comparison, for one query token per head:
//
//   p_j = softmax_j(scale q.k_j),  mu_k = sum p k,  Sigma_kk = sum_j p_j (k_j - mu_k)(k_j - mu_k)^T
//   rho = Sigma_kk^-1 (mu_k - q)    by conjugate gradient from rho = 0
//   o   = mu_v - C^T rho            (the Parallax decode with that rho)
//
// lla_probe_kernel: one CTA per (b, h).  Pass 1 streams the head's keys through
// shared memory in tiles of 32 (bf16 -> fp32), keeps an online-softmax max,
// and accumulates l = sum p, sum p k and the p-weighted second moment
// sum p k k^T (each of the 256 threads owns a (D/16) x (D/16) block of it, in
// registers).  The centred covariance then goes to shared memory and the CG
// iterations run there (matrix-vector products split over 256 threads, dot
// products by block reduction), stopping after `iters` steps or at a relative
// residual of 1e-6.  The probe is written in fp32 (returned) and bf16 (for the
// decode pass); o comes from the Parallax decode kernel with that probe.
#include "kernels.h"
#include "common.cuh"

namespace parallax {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 32;  // keys per tile
constexpr float kCgTol = 1e-6f;

struct LlaArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* kc;
    const int32_t* seqlens;
    float* rho;                 // [B*H, D]
    __nv_bfloat16* rho_bf16;    // [B*H, D]
    int H, Lmax, iters;
    float qscale;               // scale * log2(e)
};

__device__ unsigned g_lla_err = 0;

// Sum over the block; every thread gets the result.  `red` holds 8 floats.
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(kFullMask, v, off);
    __syncthreads();  // red is free
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) s += red[w];
    return s;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) lla_probe_kernel(const LlaArgs a) {
    constexpr int BS = D / 16;          // this thread's block of the second moment: BS x BS
    constexpr int TPR = kThreads / D;   // threads per matrix row in the CG products
    constexpr int LD = D + 1;           // padded row stride of the covariance (bank spread)
    extern __shared__ __align__(16) float sm[];
    float* kt = sm;                     // [kTile][D] key tile (fp32)
    float* sig = kt + kTile * D;        // [D][LD] covariance
    float* qv = sig + D * LD;           // [D] query
    float* mu = qv + D;                 // [D] mu_k
    float* xv = mu + D;                 // [D] CG iterate
    float* rv = xv + D;                 // [D] residual
    float* pv = rv + D;                 // [D] search direction
    float* ap = pv + D;                 // [D] Sigma p
    float* s2 = ap + D;                 // [kTile] scaled scores of the tile
    float* red = s2 + kTile;            // [8] reduction scratch

    const int t = threadIdx.x, warp = t / 32, lane = t % 32;
    const int bh = blockIdx.x, b = bh / a.H;
    int n = a.seqlens[b];
    if (n < 0 || n > a.Lmax) {
        if (t == 0) raise_error(&g_lla_err, PARALLAX_DEVERR_SEQLEN_CLAMPED);
        n = n < 0 ? 0 : a.Lmax;
    }
    if (t < D) qv[t] = __bfloat162float(a.q[(size_t)bh * D + t]);
    __syncthreads();

    // ---------------------------------------------------------------- pass 1
    const int ra = BS * (t >> 4), cb = BS * (t & 15);
    float acc[BS][BS];
#pragma unroll
    for (int x = 0; x < BS; ++x)
#pragma unroll
        for (int y = 0; y < BS; ++y) acc[x][y] = 0.f;
    float muacc = 0.f, l = 0.f, m = -INFINITY;
    const __nv_bfloat16* kh = a.kc + (size_t)bh * a.Lmax * D;
    constexpr int VPR = D / 8;  // 16-byte vectors per key row
    for (int j0 = 0; j0 < n; j0 += kTile) {
        const int nk = min(kTile, n - j0);
        __syncthreads();  // the previous tile is consumed
        for (int vi = t; vi < kTile * VPR; vi += kThreads) {
            const int row = vi / VPR, c8 = (vi - row * VPR) * 8;
            float f[8];
            if (row < nk) {
                Vec16<__nv_bfloat16>::unpack(ld_global_16(kh + (size_t)(j0 + row) * D + c8), f);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) kt[row * D + c8 + e] = f[e];
        }
        __syncthreads();
        // scores: warp w takes keys 4w .. 4w + 3
#pragma unroll
        for (int e = 0; e < kTile / (kThreads / 32); ++e) {
            const int j = warp * (kTile / (kThreads / 32)) + e;
            float dot = 0.f;
#pragma unroll
            for (int c = lane; c < D; c += 32) dot = fmaf(qv[c], kt[j * D + c], dot);
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) dot += __shfl_xor_sync(kFullMask, dot, off);
            if (lane == 0) s2[j] = j < nk ? dot * a.qscale : -INFINITY;
        }
        __syncthreads();
        float bm = -INFINITY;
#pragma unroll
        for (int j = 0; j < kTile; ++j) bm = fmaxf(bm, s2[j]);
        const float m_new = fmaxf(m, bm);
        if (m_new > m) {  // uniform: every thread sees the same scores
            const float alpha = m == -INFINITY ? 0.f : fast_exp2(m - m_new);
            l *= alpha;
            muacc *= alpha;
#pragma unroll
            for (int x = 0; x < BS; ++x)
#pragma unroll
                for (int y = 0; y < BS; ++y) acc[x][y] *= alpha;
            m = m_new;
        }
        for (int j = 0; j < nk; ++j) {
            const float p = fast_exp2(s2[j] - m);
            l += p;
            float ka[BS], kb[BS];
#pragma unroll
            for (int x = 0; x < BS; ++x) {
                ka[x] = p * kt[j * D + ra + x];
                kb[x] = kt[j * D + cb + x];
            }
#pragma unroll
            for (int x = 0; x < BS; ++x)
#pragma unroll
                for (int y = 0; y < BS; ++y) acc[x][y] = fmaf(ka[x], kb[y], acc[x][y]);
            if (t < D) muacc = fmaf(p, kt[j * D + t], muacc);
        }
    }

    // ---------------------------------------------------------------- covariance
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    if (t < D) mu[t] = muacc * inv_l;
    __syncthreads();
#pragma unroll
    for (int x = 0; x < BS; ++x)
#pragma unroll
        for (int y = 0; y < BS; ++y)
            sig[(ra + x) * LD + cb + y] = acc[x][y] * inv_l - mu[ra + x] * mu[cb + y];
    if (t < D) {
        const float bt = n > 0 ? mu[t] - qv[t] : 0.f;
        xv[t] = 0.f;
        rv[t] = bt;
        pv[t] = bt;
    }
    __syncthreads();

    // ---------------------------------------------------------------- conjugate gradient
    const int row = t / TPR, part = t % TPR;
    float rs = block_sum(t < D ? rv[t] * rv[t] : 0.f, red);
    const float stop = kCgTol * kCgTol * rs;
    for (int it = 0; it < a.iters && rs > stop && rs > 0.f; ++it) {
        float partial = 0.f;
#pragma unroll 8
        for (int c = part; c < D; c += TPR) partial = fmaf(sig[row * LD + c], pv[c], partial);
#pragma unroll
        for (int off = TPR / 2; off >= 1; off >>= 1)
            partial += __shfl_xor_sync(kFullMask, partial, off);
        if (part == 0) ap[row] = partial;
        __syncthreads();
        const float pap = block_sum(t < D ? pv[t] * ap[t] : 0.f, red);
        if (!(pap > 0.f)) break;  // uniform; Sigma is only semi-definite
        const float alpha = rs / pap;
        float rn = 0.f;
        if (t < D) {
            xv[t] = fmaf(alpha, pv[t], xv[t]);
            rn = fmaf(-alpha, ap[t], rv[t]);
            rv[t] = rn;
        }
        const float rs_new = block_sum(rn * rn, red);
        if (t < D) pv[t] = fmaf(rs_new / rs, pv[t], rn);
        __syncthreads();
        rs = rs_new;
    }
    if (t < D) {
        a.rho[(size_t)bh * D + t] = xv[t];
        a.rho_bf16[(size_t)bh * D + t] = __float2bfloat16_rn(xv[t]);
    }
}

template <int D>
size_t smem_bytes() {
    return sizeof(float) * ((size_t)kTile * D + (size_t)D * (D + 1) + 6 * D + kTile + 8);
}

template <int D>
cudaError_t launch(const LlaArgs& a, int BH, cudaStream_t stream) {
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(lla_probe_kernel<D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem_bytes<D>());
        if (e != cudaSuccess) return e;
        configured = true;
    }
    lla_probe_kernel<D><<<BH, kThreads, smem_bytes<D>(), stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t lla_probe_launch(const void* q, const void* kc, const int32_t* seqlens, float* rho,
                             void* rho_bf16, int B, int H, int Lmax, int d, int iters,
                             cudaStream_t stream) {
    LlaArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.kc = static_cast<const __nv_bfloat16*>(kc);
    a.seqlens = seqlens;
    a.rho = rho;
    a.rho_bf16 = static_cast<__nv_bfloat16*>(rho_bf16);
    a.H = H;
    a.Lmax = Lmax;
    a.iters = iters;
    a.qscale = kLog2e / sqrtf((float)d);
    if (d == 64) return launch<64>(a, B * H, stream);
    if (d == 128) return launch<128>(a, B * H, stream);
    return cudaErrorInvalidValue;
}

unsigned lla_take_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_lla_err, sizeof(v)) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_lla_err, &zero, sizeof(zero));
    return v;
}

}  // namespace parallax
