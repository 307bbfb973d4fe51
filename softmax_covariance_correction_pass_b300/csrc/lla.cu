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
// lla_probe_kernel: one CTA per (b, h), 8 warps.  Pass 1 streams the head's keys
// through shared memory in tiles of 32, keeps an online-softmax max, and
// accumulates l = sum p and sum p k on the FMA pipes and the p-weighted second
// moment G = sum_j k_j (p_j k_j)^T on the tensor cores: warp w owns rows
// 16w .. 16w + 15 of G as warp-level mma.sync m16n8k16 accumulators (fp32), with
// A = the keys (exact bf16) and B = p_j k_j split into a bf16 high part and a
// bf16 residual (two MMAs, so the product keeps ~16 bits).  The centred
// covariance then goes to shared memory (over the dead key tiles) and the CG
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

__device__ __forceinline__ uint32_t smem_u32_lla(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t smem_u32_lla(uint32_t a) { return a; }

// Two fp32 -> packed bf16x2 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16_lla(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

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

__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32_lla(addr)));
}

template <int D>
struct LlaLayout {
    static constexpr int PITCH = D * 2 + 16;  // bytes per bf16 key row: conflict-free ldmatrix
    static constexpr int KT_F32 = 0;                                 // [kTile][D] fp32 keys
    static constexpr int KT_B16 = KT_F32 + kTile * D * 4;            // [kTile][PITCH] bf16 keys
    static constexpr int PK_HI = KT_B16 + kTile * PITCH;             // bf16(p k)
    static constexpr int PK_LO = PK_HI + kTile * PITCH;              // bf16(p k - hi)
    static constexpr int TILES_END = PK_LO + kTile * PITCH;
    static constexpr int SIG_BYTES = D * (D + 1) * 4;                // covariance (aliases tiles)
    static constexpr int VEC_OFF = (TILES_END > SIG_BYTES ? TILES_END : SIG_BYTES);
    static constexpr size_t SMEM_BYTES = VEC_OFF + sizeof(float) * (6 * D + 2 * kTile + 8);
};

template <int D>
__global__ void __launch_bounds__(kThreads, 2) lla_probe_kernel(const LlaArgs a) {
    using LY = LlaLayout<D>;
    constexpr int TPR = kThreads / D;   // threads per matrix row in the CG products
    constexpr int LD = D + 1;           // padded row stride of the covariance (bank spread)
    // warp -> a 16-row stripe and a column group of the Gram matrix
    constexpr int STRIPES = D / 16, CGS = (kThreads / 32) / STRIPES, COLS = D / CGS, NT = COLS / 8;
    static_assert(STRIPES * CGS == kThreads / 32 && NT % 2 == 0, "Gram matrix tiling");
    extern __shared__ __align__(16) unsigned char smb[];
    float* kt = reinterpret_cast<float*>(smb + LY::KT_F32);   // [kTile][D] key tile (fp32)
    unsigned char* kb16 = smb + LY::KT_B16;
    unsigned char* pkh = smb + LY::PK_HI;
    unsigned char* pkl = smb + LY::PK_LO;
    float* sig = reinterpret_cast<float*>(smb);               // [D][LD], after pass 1
    float* qv = reinterpret_cast<float*>(smb + LY::VEC_OFF);  // [D] query
    float* mu = qv + D;                 // [D] mu_k
    float* xv = mu + D;                 // [D] CG iterate
    float* rv = xv + D;                 // [D] residual
    float* pv = rv + D;                 // [D] search direction
    float* ap = pv + D;                 // [D] Sigma p
    float* s2 = ap + D;                 // [kTile] scaled scores of the tile
    float* pw = s2 + kTile;             // [kTile] their weights p = 2^(s - m)
    float* red = pw + kTile;            // [8] reduction scratch

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
    const int stripe = warp % STRIPES, col0 = (warp / STRIPES) * COLS;
    float acc[NT][4];  // rows 16 stripe + g (and + 8) of G, columns col0 + 8 nt + 2 (lane & 3) (+1)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    float muacc = 0.f, l = 0.f, m = -INFINITY;
    const __nv_bfloat16* kh = a.kc + (size_t)bh * a.Lmax * D;
    constexpr int VPR = D / 8;  // 16-byte vectors per key row
    const int mi = lane >> 3, r8 = lane & 7;
    for (int j0 = 0; j0 < n; j0 += kTile) {
        const int nk = min(kTile, n - j0);
        __syncthreads();  // the previous tile is consumed
        for (int vi = t; vi < kTile * VPR; vi += kThreads) {
            const int row = vi / VPR, c8 = (vi - row * VPR) * 8;
            uint4 raw = make_uint4(0, 0, 0, 0);
            if (row < nk) raw = ld_global_16(kh + (size_t)(j0 + row) * D + c8);
            *reinterpret_cast<uint4*>(kb16 + row * LY::PITCH + c8 * 2) = raw;
            float f[8];
            Vec16<__nv_bfloat16>::unpack(raw, f);
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
            for (int nt = 0; nt < NT; ++nt) {
                acc[nt][0] *= alpha;
                acc[nt][1] *= alpha;
                acc[nt][2] *= alpha;
                acc[nt][3] *= alpha;
            }
            m = m_new;
        }
        if (t < kTile) pw[t] = fast_exp2(s2[t] - m);  // 0 for keys past the sequence
        __syncthreads();
        // p_j k_j as a bf16 pair (high part, residual): the B operand of the Gram MMAs
        for (int e = t; e < kTile * D / 2; e += kThreads) {
            const int row = e / (D / 2), c2 = 2 * (e - row * (D / 2));
            const float p = pw[row];
            const float v0 = p * kt[row * D + c2], v1 = p * kt[row * D + c2 + 1];
            const uint32_t hi = pack_bf16_lla(v0, v1);
            const float h0 = __uint_as_float(hi << 16), h1 = __uint_as_float(hi & 0xffff0000u);
            *reinterpret_cast<uint32_t*>(pkh + row * LY::PITCH + c2 * 2) = hi;
            *reinterpret_cast<uint32_t*>(pkl + row * LY::PITCH + c2 * 2) = pack_bf16_lla(v0 - h0, v1 - h1);
        }
        for (int j = 0; j < nk; ++j) {
            const float p = pw[j];
            l += p;
            if (t < D) muacc = fmaf(p, kt[j * D + t], muacc);
        }
        __syncthreads();
        // G[stripe rows][column group] += K[:, stripe]^T (p K)[:, group] over the tile's keys
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ++ks) {
            const int j0k = 16 * ks;
            uint32_t af[4];
            ldsm_x4_t(smem_u32_lla(kb16) + (j0k + (mi >> 1) * 8 + r8) * LY::PITCH +
                          (16 * stripe + (mi & 1) * 8) * 2,
                      af[0], af[1], af[2], af[3]);
            // ldmatrix.trans hands out A fragments in the order (rows g, g+8) x (keys lo, hi)
            const uint32_t a4[4] = {af[0], af[1], af[2], af[3]};
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
                const uint32_t off =
                    (j0k + (mi & 1) * 8 + r8) * LY::PITCH + (col0 + 16 * np + (mi >> 1) * 8) * 2;
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(smem_u32_lla(pkh) + off, b0, b1, b2, b3);
                mma_16816(acc[2 * np], a4, b0, b1);
                mma_16816(acc[2 * np + 1], a4, b2, b3);
                ldsm_x4_t(smem_u32_lla(pkl) + off, b0, b1, b2, b3);
                mma_16816(acc[2 * np], a4, b0, b1);
                mma_16816(acc[2 * np + 1], a4, b2, b3);
            }
        }
    }

    // ---------------------------------------------------------------- covariance
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    if (t < D) mu[t] = muacc * inv_l;
    __syncthreads();  // the key tiles are dead: sig takes their place
    {
        const int g = lane >> 2, c = 2 * (lane & 3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int row = 16 * stripe + g + 8 * (e >> 1), col = col0 + 8 * nt + c + (e & 1);
                sig[row * LD + col] = acc[nt][e] * inv_l - mu[row] * mu[col];
            }
    }
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
    return LlaLayout<D>::SMEM_BYTES;
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
