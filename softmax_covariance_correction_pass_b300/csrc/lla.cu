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
// through shared memory in tiles of 64 (cp.async, double-buffered, so the next
// tile loads while this one is used).  Per tile: the scores (each warp 8 keys,
// the query held in registers), the online-softmax max, then p_j k_j written as
// a bf16 pair (high part, residual) with p_j itself in the row's spare columns.
// The p-weighted second moment G = sum_j k_j (p_j k_j)^T and the weighted mean
// l mu_k = sum_j p_j k_j run on the tensor cores: warp w owns a 16-row stripe of
// G (and of l mu_k) as warp-level mma.sync m16n8k16 accumulators (fp32), with
// A = the keys (exact bf16) and B = the high part and the residual (two MMAs, so
// the product keeps ~16 bits).  The centred covariance then goes to shared
// memory (over the dead key tiles) and the CG iterations run there
// (matrix-vector products split over 256 threads, dot products by block
// reduction), stopping after `iters` steps or at a relative residual of 1e-6.
// The probe is written in fp32 (returned) and bf16 (for the decode pass); o
// comes from the Parallax decode kernel with that probe.
#include "kernels.h"
#include "common.cuh"

namespace parallax {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = 64;  // keys per tile
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
    for (int w = 0; w < kWarps; ++w) s += red[w];
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
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}

// 16-byte global -> shared copy; src_bytes = 0 fills the destination with zeros.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

template <int D>
struct LlaLayout {
    // bytes per key row: the D bf16 values, then 8 spare bf16 columns.  The
    // 16-byte pad also spreads 8 consecutive rows over the 8 bank groups, so the
    // transposing ldmatrix loads are conflict-free.
    static constexpr int PITCH = D * 2 + 16;
    static constexpr int TILE_BYTES = kTile * PITCH;
    static constexpr int KB = 0;                          // 2 x [kTile][PITCH] keys (double buffer)
    static constexpr int PK_HI = 2 * TILE_BYTES;          // bf16(p k); spare column 0 = bf16(p)
    static constexpr int PK_LO = 3 * TILE_BYTES;          // the residuals p k - hi, p - hi
    static constexpr int TILES_END = 4 * TILE_BYTES;
    static constexpr int SIG_BYTES = D * (D + 1) * 4;     // covariance (aliases the tiles)
    static constexpr int VEC_OFF = (TILES_END > SIG_BYTES ? TILES_END : SIG_BYTES);
    static constexpr size_t SMEM_BYTES = VEC_OFF + sizeof(float) * (6 * D + kTile + 2 * kWarps);
};

template <int D>
__global__ void __launch_bounds__(kThreads, 2) lla_probe_kernel(const LlaArgs a) {
    using LY = LlaLayout<D>;
    constexpr int TPR = kThreads / D;   // threads per matrix row in the CG products
    constexpr int LD = D + 1;           // padded row stride of the covariance (bank spread)
    // warp -> a 16-row stripe and a column group of the Gram matrix
    constexpr int STRIPES = D / 16, CGS = kWarps / STRIPES, COLS = D / CGS, NT = COLS / 8;
    static_assert(STRIPES * CGS == kWarps && NT % 2 == 0, "Gram matrix tiling");
    constexpr int QPL = D / 32;          // query elements per lane in the score dot products
    constexpr int VPR = D / 8;           // 16-byte vectors per key row
    constexpr int KPW = kTile / kWarps;  // keys per warp in the score pass
    constexpr int RPP = kThreads / 8;    // rows per pass of the p k pass (8 threads per row)
    static_assert(KPW <= 32 && kTile % RPP == 0 && VPR % 8 == 0, "tile shape");
    extern __shared__ __align__(16) unsigned char smb[];
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
    float* wmax = s2 + kTile;           // [kWarps] per-warp maxima of the tile
    float* red = wmax + kWarps;         // [kWarps] reduction scratch

    const int t = threadIdx.x, warp = t / 32, lane = t % 32;
    const int bh = blockIdx.x, b = bh / a.H;
    int n = a.seqlens[b];
    if (n < 0 || n > a.Lmax) {
        if (t == 0) raise_error(&g_lla_err, PARALLAX_DEVERR_SEQLEN_CLAMPED);
        n = n < 0 ? 0 : a.Lmax;
    }
    const __nv_bfloat16* qh = a.q + (size_t)bh * D;
    if (t < D) qv[t] = __bfloat162float(qh[t]);
    __syncthreads();

    // ---------------------------------------------------------------- pass 1
    const int stripe = warp % STRIPES, col0 = (warp / STRIPES) * COLS;
    const bool mean_warp = col0 + COLS == D;  // also accumulates l mu_k for its stripe
    float acc[NT][4];  // rows 16 stripe + g (and + 8) of G, columns col0 + 8 nt + 2 (lane & 3) (+1)
    float accx[4] = {0.f, 0.f, 0.f, 0.f};  // column 0: l mu_k for the same rows
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    float lpart = 0.f, m = -INFINITY;
    const __nv_bfloat16* kh = a.kc + (size_t)bh * a.Lmax * D;
    const uint32_t kb_s = smem_u32(smb + LY::KB);
    const uint32_t pkh_s = smem_u32(pkh), pkl_s = smem_u32(pkl);
    const int mi = lane >> 3, r8 = lane & 7;
    const int ntiles = (n + kTile - 1) / kTile;
    auto issue = [&](int tile, int buf) {
        const int j0 = tile * kTile;
#pragma unroll
        for (int vi = t; vi < kTile * VPR; vi += kThreads) {
            const int row = vi / VPR, c8 = (vi - row * VPR) * 8;
            const bool in = j0 + row < n;  // rows past the sequence are zero-filled
            cp_async_16(kb_s + buf * LY::TILE_BYTES + row * LY::PITCH + c8 * 2,
                        kh + (size_t)(in ? j0 + row : 0) * D + c8, in ? 16u : 0u);
        }
        cp_async_commit();
    };
    if (ntiles > 0) issue(0, 0);
    for (int it = 0; it < ntiles; ++it) {
        const int buf = it & 1, nk = min(kTile, n - it * kTile);
        cp_async_wait_all();
        __syncthreads();  // tile `it` is in for every thread; tile it - 1 is consumed
        if (it + 1 < ntiles) issue(it + 1, buf ^ 1);
        const unsigned char* kb = smb + LY::KB + buf * LY::TILE_BYTES;
        // scores: warp w takes keys KPW w .. KPW w + KPW - 1
        float mine = -INFINITY, wm = -INFINITY;
#pragma unroll
        for (int e = 0; e < KPW; ++e) {
            const int j = warp * KPW + e;
            float dot = 0.f;
            if constexpr (QPL == 4) {
                const uint2 raw = *reinterpret_cast<const uint2*>(kb + j * LY::PITCH + lane * 8);
                const float4 qq = *reinterpret_cast<const float4*>(qv + 4 * lane);
                dot = qq.x * __uint_as_float(raw.x << 16);
                dot = fmaf(qq.y, __uint_as_float(raw.x & 0xffff0000u), dot);
                dot = fmaf(qq.z, __uint_as_float(raw.y << 16), dot);
                dot = fmaf(qq.w, __uint_as_float(raw.y & 0xffff0000u), dot);
            } else {
                const uint32_t raw = *reinterpret_cast<const uint32_t*>(kb + j * LY::PITCH + lane * 4);
                const float2 qq = *reinterpret_cast<const float2*>(qv + 2 * lane);
                dot = qq.x * __uint_as_float(raw << 16);
                dot = fmaf(qq.y, __uint_as_float(raw & 0xffff0000u), dot);
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) dot += __shfl_xor_sync(kFullMask, dot, off);
            const float s = j < nk ? dot * a.qscale : -INFINITY;
            wm = fmaxf(wm, s);
            if (lane == e) mine = s;
        }
        if (lane < KPW) s2[warp * KPW + lane] = mine;
        if (lane == 0) wmax[warp] = wm;
        __syncthreads();
        float bm = wmax[0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) bm = fmaxf(bm, wmax[w]);
        const float m_new = fmaxf(m, bm);
        if (m_new > m) {  // uniform: every thread sees the same maxima
            const float alpha = m == -INFINITY ? 0.f : fast_exp2(m - m_new);
            lpart *= alpha;
#pragma unroll
            for (int e = 0; e < 4; ++e) accx[e] *= alpha;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                acc[nt][0] *= alpha;
                acc[nt][1] *= alpha;
                acc[nt][2] *= alpha;
                acc[nt][3] *= alpha;
            }
            m = m_new;
        }
        // p_j k_j (and p_j) as a bf16 pair (high part, residual): the B operand of the MMAs.
        // 8 threads per key row, each taking 16-byte vectors e8, e8 + 8, ...
        {
            const int e8 = t & 7;
#pragma unroll
            for (int pass = 0; pass < kTile / RPP; ++pass) {
                const int row = (t >> 3) + pass * RPP;
                const float p = fast_exp2(s2[row] - m);  // 0 past the sequence
                if (e8 == 0) {
                    lpart += p;
                    const uint32_t ph = pack_bf16_lla(p, 0.f);
                    const uint32_t pl = pack_bf16_lla(p - __uint_as_float(ph << 16), 0.f);
                    *reinterpret_cast<uint4*>(pkh + row * LY::PITCH + D * 2) = make_uint4(ph, 0, 0, 0);
                    *reinterpret_cast<uint4*>(pkl + row * LY::PITCH + D * 2) = make_uint4(pl, 0, 0, 0);
                }
#pragma unroll
                for (int cc = 0; cc < VPR / 8; ++cc) {
                    const int off = row * LY::PITCH + (e8 + 8 * cc) * 16;
                    float f[8];
                    Vec16<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4*>(kb + off), f);
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const float v0 = p * f[2 * h], v1 = p * f[2 * h + 1];
                        hi[h] = pack_bf16_lla(v0, v1);
                        lo[h] = pack_bf16_lla(v0 - __uint_as_float(hi[h] << 16),
                                              v1 - __uint_as_float(hi[h] & 0xffff0000u));
                    }
                    *reinterpret_cast<uint4*>(pkh + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4*>(pkl + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
            }
        }
        __syncthreads();
        // G[stripe rows][column group] += K[:, stripe]^T (p K)[:, group] over the tile's keys
        const uint32_t kb_a = kb_s + buf * LY::TILE_BYTES;
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ++ks) {
            const int j0k = 16 * ks;
            uint32_t af[4];
            // ldmatrix.trans hands out A fragments in the order (rows g, g+8) x (keys lo, hi)
            ldsm_x4_t(kb_a + (j0k + (mi >> 1) * 8 + r8) * LY::PITCH + (16 * stripe + (mi & 1) * 8) * 2,
                      af[0], af[1], af[2], af[3]);
            const uint32_t brow = (j0k + (mi & 1) * 8 + r8) * LY::PITCH;
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
                const uint32_t off = brow + (col0 + 16 * np + (mi >> 1) * 8) * 2;
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(pkh_s + off, b0, b1, b2, b3);
                mma_16816(acc[2 * np], af, b0, b1);
                mma_16816(acc[2 * np + 1], af, b2, b3);
                ldsm_x4_t(pkl_s + off, b0, b1, b2, b3);
                mma_16816(acc[2 * np], af, b0, b1);
                mma_16816(acc[2 * np + 1], af, b2, b3);
            }
            if (mean_warp) {  // the n8 tile of the spare columns: p, then zeros
                uint32_t b0, b1;
                ldsm_x2_t(pkh_s + brow + D * 2, b0, b1);
                mma_16816(accx, af, b0, b1);
                ldsm_x2_t(pkl_s + brow + D * 2, b0, b1);
                mma_16816(accx, af, b0, b1);
            }
        }
    }

    // ---------------------------------------------------------------- covariance
    const float l = block_sum(lpart, red);  // every warp is past its last MMA
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    if (mean_warp && (lane & 3) == 0) {
        mu[16 * stripe + (lane >> 2)] = accx[0] * inv_l;
        mu[16 * stripe + (lane >> 2) + 8] = accx[2] * inv_l;
    }
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
