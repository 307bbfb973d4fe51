// Exact local linear attention (LLA) decode: the per-query solve that the
// Parallax probe replaces.  The Parallax pages describe their method as LLA's
// covariance correction with the per-query probe Sigma_kk^-1 (mu_k - q) swapped
// for the learned rho = W_R x ("Parallax mantem softmax ...", paragraphs 1-2);
// this computes the original, for comparison, for one query token per head:
//
//   p_j = softmax_j(scale q.k_j),  mu_k = sum p k,  mu_v = sum p v
//   Sigma_kk = sum_j p_j (k_j - mu_k)(k_j - mu_k)^T,  C = sum_j p_j (k_j - mu_k)(v_j - mu_v)^T
//   rho = Sigma_kk^-1 (mu_k - q)    by conjugate gradient from rho = 0
//   o   = mu_v - C^T rho            (the Parallax output with that probe)
//
// lla_kernel: one CTA per (b, h), one pass over the head's keys and values.
// Warp 0 streams 64-key tiles of K and V by TMA (3-deep ring, 128-byte
// swizzle); warps 2-17 own one 16-byte chunk (8 features) of every key row they
// touch: they compute the scores (a row's partial dot products summed over the
// row's lanes), the online-softmax max (moved only when a score exceeds it by
// more than 2^8; the accumulators are then rescaled), the weights p~_j, the
// weighted sums l = sum p~, l mu_k, l mu_v (fp32), and write p~_j k_j and
// p~_j v_j as bf16 pairs (high part, residual) into shared memory; warp 1
// issues the tcgen05 MMAs
//   G_kk += K^T (p~ K),   G_kv += K^T (p~ V)      (fp32 accumulators in TMEM)
// with the key tile itself as the (MN-major) A operand and the two parts of
// each product as B (so the products keep ~16 significant bits); even and odd
// key tiles accumulate into two TMEM sets (the accumulation error grows with
// the number of MMAs added into one accumulator).  After the
// stream: Sigma_kk = G_kk / l - mu_k mu_k^T and C = G_kv / l - mu_k mu_v^T go
// to shared memory, conjugate gradient runs there (matrix-vector products over
// 512 threads, dot products by group reduction), stopping after `iters` steps or
// at a relative residual of 1e-6, and o = mu_v - C^T rho is formed in fp32.
#include "tcgen05.cuh"
#include "kernels.h"

namespace parallax {
namespace {

constexpr int kThreads = 576;   // warp 0 TMA, warp 1 MMA + TMEM, warps 2-17 compute
constexpr int kCompute = 512;
constexpr int kComputeWarps = kCompute / 32;
constexpr int kTile = 64;       // keys per tile
constexpr int kStages = 3;
constexpr float kCgTol = 1e-6f;
constexpr float kRescale = 8.f;  // log2 units

struct LlaArgs {
    const __nv_bfloat16* q;
    const int32_t* seqlens;
    float* rho;  // [B*H, D]
    float* o;    // [B*H, D]
    int H, Lmax, iters;
    float qscale;  // scale * log2(e)
    size_t out_elems;  // B * H * D (debug bounds checks)
};

__device__ unsigned g_lla_err = 0;

// Two fp32 -> packed bf16x2 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16_lla(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Plain 16-byte shared-memory accesses (the compiler may schedule them freely).
__device__ __forceinline__ void st16(unsigned char* p, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
    *reinterpret_cast<uint4*>(p) = make_uint4(x, y, z, w);
}
__device__ __forceinline__ uint4 ld16(const unsigned char* p) { return *reinterpret_cast<const uint4*>(p); }

__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier 1 over the compute threads, returning the AND of `p` over all of them
// (so that a failed wait takes every compute warp down the same path).
__device__ __forceinline__ bool named_bar_and(int nthreads, bool p) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.and.pred po, 1, %2, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)p), "r"(nthreads)
        : "memory");
    return r != 0;
}

// Named barrier 1 over the compute threads, returning the OR of `p` over all of them.
__device__ __forceinline__ bool named_bar_or(int nthreads, bool p) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, 1, %2, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)p), "r"(nthreads)
        : "memory");
    return r != 0;
}

// Sum over the compute threads (named barrier 1); every one gets the result.
__device__ __forceinline__ float grp_sum(float v, float* red, int cw, int lane) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(kFullMask, v, off);
    named_bar_sync(1, kCompute);  // red is free
    if (lane == 0) red[cw] = v;
    named_bar_sync(1, kCompute);
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kComputeWarps; ++w) s += red[w];
    return s;
}

// kind::f16 instruction descriptor with both operands MN-major (A: M contiguous,
// B: N contiguous), bf16 in, fp32 accumulate.
constexpr uint32_t idesc_mn_mn(int M, int N) { return tc::idesc_bf16_f32(M, N, true) | (1u << 15); }

template <int D>
struct LlaLayout {
    static constexpr int NCB = D / 64;                 // 64-feature column blocks
    static constexpr int SUBT = kTile * 128;           // [64 keys x 64 features] bf16, swizzled
    static constexpr int TILE = NCB * SUBT;            // a 64-key tile of K or V
    static constexpr int STAGE = 2 * TILE;             // K, then V
    // 2 buffers of {p~K hi, p~V hi, p~K lo, p~V lo}: each half is one N = 2d MN-major operand
    static constexpr int B_OFF = kStages * STAGE;
    static constexpr int BBUF = 4 * TILE;
    // d = 64: a zero block stands in for features 64..127 of the M = 128 A operand
    static constexpr int ZERO_OFF = B_OFF + 2 * BBUF;
    static constexpr int STREAM_END = ZERO_OFF + (D == 64 ? SUBT : 0);
    // after the stream the same bytes hold Sigma_kk, C^T (rows padded to LD), the
    // per-thread partial means and the CG vectors
    static constexpr int LD = D + 1;
    static constexpr int SIG_OFF = 0;
    static constexpr int CT_OFF = D * LD * 4;
    static constexpr int CPR = D / 8;                  // 16-byte chunks per key row
    static constexpr int RGRP = kCompute / CPR;        // rows handled in parallel
    static constexpr int MUP_OFF = 2 * D * LD * 4;     // [RGRP][2][D] partial sums
    static constexpr int CGV_OFF = MUP_OFF + RGRP * 2 * D * 4;  // 6 x [D]
    static constexpr int POST_END = CGV_OFF + 6 * D * 4;
    static constexpr int VEC_OFF = (STREAM_END > POST_END ? STREAM_END : POST_END);
    // red[kComputeWarps]: reduction scratch
    static constexpr int BAR_OFF = VEC_OFF + 4 * kComputeWarps;
    // kv_full[S], kv_empty[S], b_full[2], b_empty[2], acc_full
    static constexpr int NBARS = 2 * kStages + 5;
    static constexpr int SMEM_BYTES = BAR_OFF + NBARS * 8 + 16 + 1024;
    // two accumulator sets [G_kk | G_kv] (even / odd key tiles) at 0 and 2D: each takes half
    // of a head's MMAs, and the two are added at the end
    static constexpr uint32_t TMEM_COLS = 4 * D;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    lla_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const LlaArgs a) {
    using LY = LlaLayout<D>;
    constexpr int S = kStages;
    constexpr int ROWS_PER_T = kTile * LY::CPR / kCompute;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* red = reinterpret_cast<float*>(smem + LY::VEC_OFF);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LY::BAR_OFF);
    uint64_t* kv_full = bars;
    uint64_t* kv_empty = bars + S;
    uint64_t* b_full = bars + 2 * S;   // [2] kCompute arrivals
    uint64_t* b_empty = bars + 2 * S + 2;
    uint64_t* acc_full = bars + 2 * S + 4;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + LY::NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    const int bh = blockIdx.x, b = bh / a.H;
    int n = a.seqlens[b];
    if (n < 0 || n > a.Lmax) {
        if (threadIdx.x == 0) raise_error(&g_lla_err, PARALLAX_DEVERR_SEQLEN_CLAMPED);
        n = n < 0 ? 0 : a.Lmax;
    }
    const int ntiles = (n + kTile - 1) / kTile;

    if (threadIdx.x == 0) {
        for (int i = 0; i < LY::NBARS; ++i)
            mbar_init(&bars[i], (i == 2 * S || i == 2 * S + 1) ? kCompute : 1);
        *abort_flag = (*(volatile unsigned*)&g_lla_err & PARALLAX_DEVERR_WAIT_TIMEOUT) ? 1 : 0;
        fence_mbar_init();
    }
    if (D == 64 && warp >= 2) {  // the zero block of the padded A operand
        for (int i = threadIdx.x - 64; i < LY::SUBT / 16; i += kCompute)
            reinterpret_cast<uint4*>(smem + LY::ZERO_OFF)[i] = make_uint4(0, 0, 0, 0);
        fence_async_smem();
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tmap(&tmK);
        tc::prefetch_tmap(&tmV);
    }
    if (warp == 1) tc::tmem_alloc(tmem_slot, LY::TMEM_COLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const bool skip = *abort_flag != 0;
    const uint32_t sbase = smem_u32(smem);

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0 && !skip) {
            int issued = 0;
            bool ok = true;
            for (int t = 0; t < ntiles; ++t) {
                const int s = t % S;
                if (t >= S && !mbar_wait(&kv_empty[s], ((t / S) - 1) & 1, &g_lla_err)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&kv_full[s], LY::STAGE);
                unsigned char* st = smem + s * LY::STAGE;
                for (int cb = 0; cb < LY::NCB; ++cb) {
                    tc::tma_load_3d(st + cb * LY::SUBT, &tmK, cb * 64, t * kTile, bh, &kv_full[s]);
                    tc::tma_load_3d(st + LY::TILE + cb * LY::SUBT, &tmV, cb * 64, t * kTile, bh,
                                    &kv_full[s]);
                }
                issued = t + 1;
            }
            if (!ok) {
                *abort_flag = 1;
                for (int t = issued >= S ? issued - S : 0; t < issued; ++t)
                    mbar_wait(&kv_full[t % S], (t / S) & 1, &g_lla_err);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (!skip) {
            constexpr uint32_t kIdesc = idesc_mn_mn(128, 2 * D);  // [G_kk | G_kv] in one MMA
            bool ok = true;
            for (int t = 0; t < ntiles && ok; ++t) {
                const int s = t % S, buf = t & 1;
                if (*abort_flag || !mbar_wait_warp(&b_full[buf], (t >> 1) & 1, &g_lla_err)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                // A = the key tile, M = features (MN-major: 64-feature atoms LBO apart; for
                // d = 64 the second atom is the zero block), K = keys
                const uint32_t abase = sbase + s * LY::STAGE;
                const uint32_t lbo = D == 64 ? (uint32_t)(LY::ZERO_OFF - s * LY::STAGE) : LY::SUBT;
                const uint64_t dA = tc::opaque(tc::smem_desc_sw128(abase, lbo, 1024));
                const uint64_t dB =
                    tc::opaque(tc::smem_desc_sw128(sbase + LY::B_OFF + buf * LY::BBUF, LY::SUBT, 1024));
                constexpr uint32_t kTileStep = LY::TILE >> 4;
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk) {
                    const uint32_t off = (kk * 16 * 128) >> 4;
                    const uint32_t acc = (t > 1 || kk > 0) ? 1u : 0u;
                    const uint32_t dacc = tmem + (uint32_t)(t & 1) * 2 * D;
                    tc::mma_ss(dacc, dA + off, dB + off, kIdesc, acc);                 // high parts
                    tc::mma_ss(dacc, dA + off, dB + 2 * kTileStep + off, kIdesc, 1u);  // residuals
                }
                tc::commit(&b_empty[buf]);
                tc::commit(&kv_empty[s]);
            }
            tc::commit(acc_full);
            if (!ok) {
                *abort_flag = 1;
                mbar_wait_warp(acc_full, 0, &g_lla_err);
            }
        }
    } else {
        // ---------------------------------------------------------------- compute
        const int t = threadIdx.x - 64;  // 0 .. kCompute - 1
        const int cw = warp - 2;          // compute warp 0 .. kComputeWarps - 1
        const int q4 = warp & 3;          // TMEM lane quarter
        const int half = (cw >> 2) & 1;   // TMEM: G_kk (0) or G_kv (1)
        const int chalf = cw >> 3;        // which half of its D columns
        constexpr int CW = D / 2;         // columns per warp in TMEM passes
        bool ok = !skip;
        // this thread's 16-byte chunk of every key row (8 features) and its rows of each
        // tile; the CPR threads of a row are consecutive lanes of one warp
        const int c = t % LY::CPR, rg = t / LY::CPR;
        const uint32_t coff = (uint32_t)((c / 8) * LY::SUBT);
        const int cc = c % 8;
        float qc[8];  // the query's features 8c .. 8c + 7, pre-scaled
#pragma unroll
        for (int e = 0; e < 8; ++e) qc[e] = __bfloat162float(a.q[(size_t)bh * D + 8 * c + e]) * a.qscale;
        float2 mk[4], mv[4];  // partial sums of p~ k and p~ v over this thread's rows
#pragma unroll
        for (int e = 0; e < 4; ++e) mk[e] = mv[e] = make_float2(0.f, 0.f);
        float lpart = 0.f, m = -INFINITY;

        for (int it = 0; it < ntiles; ++it) {
            const int s = it % S, buf = it & 1;
            const int nk = min(kTile, n - it * kTile);
            const bool got = ok && !*abort_flag && mbar_wait(&kv_full[s], (it / S) & 1, &g_lla_err);
            ok = __all_sync(kFullMask, got);
            unsigned char* kst = smem + s * LY::STAGE;
            // scores of this thread's rows: 8 features here, summed over the row's CPR lanes
            float sj[ROWS_PER_T];
            float kf[ROWS_PER_T][8];  // this thread's key chunks as fp32, reused for p~ k
            bool need = false;
#pragma unroll
            for (int r = 0; r < ROWS_PER_T; ++r) {
                const int j = rg + r * LY::RGRP;
                float (&f)[8] = kf[r];
                Vec16<__nv_bfloat16>::unpack(ld16(kst + coff + j * 128 + ((cc ^ (j & 7)) * 16)), f);
                float d0 = qc[0] * f[0], d1 = qc[1] * f[1];
#pragma unroll
                for (int e = 2; e < 8; e += 2) {
                    d0 = fmaf(qc[e], f[e], d0);
                    d1 = fmaf(qc[e + 1], f[e + 1], d1);
                }
                float d = d0 + d1;
#pragma unroll
                for (int off = 1; off < LY::CPR; off <<= 1) d += __shfl_xor_sync(kFullMask, d, off);
                sj[r] = j < nk ? d : -INFINITY;
                need |= sj[r] > m + kRescale;  // true for every live row while m = -inf
            }
            // one barrier per tile in the common case: it also stops every compute warp at
            // the same tile when a wait failed
            if (named_bar_or(kCompute, need || !ok)) {
                if (!named_bar_and(kCompute, ok)) break;
                // the tile's max: the first one sets m, a later one rescales what is accumulated
                float wm = sj[0];
#pragma unroll
                for (int r = 1; r < ROWS_PER_T; ++r) wm = fmaxf(wm, sj[r]);
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) wm = fmaxf(wm, __shfl_xor_sync(kFullMask, wm, off));
                if (lane == 0) red[cw] = wm;
                named_bar_sync(1, kCompute);
                float tmax = red[0];
#pragma unroll
                for (int w = 1; w < kComputeWarps; ++w) tmax = fmaxf(tmax, red[w]);
                if (m != -INFINITY) {
                    const float alpha = fast_exp2(m - tmax);
                    lpart *= alpha;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        mk[e] = __fmul2_rn(mk[e], make_float2(alpha, alpha));
                        mv[e] = __fmul2_rn(mv[e], make_float2(alpha, alpha));
                    }
                    // after the MMAs of the previous tile, rescale the TMEM accumulators
                    const bool done = !*abort_flag &&
                                      mbar_wait(&b_empty[(it - 1) & 1], ((it - 1) >> 1) & 1, &g_lla_err);
                    if (__all_sync(kFullMask, done)) {
                        tc::fence_after_sync();
                        const uint32_t trow = tmem + ((uint32_t)(32 * q4) << 16) + half * D + chalf * CW;
#pragma unroll 1
                        for (int x = 0; x < 2 * (CW / 32); ++x) {  // both accumulator sets
                            const uint32_t col = (x / (CW / 32)) * 2 * D + 32 * (x % (CW / 32));
                            uint32_t u[32];
                            tc::tmem_ld32(trow + col, u);
                            tc::tmem_ld_wait();
#pragma unroll
                            for (int y = 0; y < 32; ++y)
                                u[y] = __float_as_uint(__uint_as_float(u[y]) * alpha);
                            tc::tmem_st32(trow + col, u);
                        }
                        tc::tmem_st_wait();
                        tc::fence_before_sync();
                    } else {
                        ok = false;  // every compute warp stops at the next tile's barrier
                        *abort_flag = 1;
                    }
                }
                m = tmax;
                // red is read by every compute thread before anyone writes it again
                named_bar_sync(1, kCompute);
            }
            if (!ok) continue;  // (no barrier is skipped: the next tile's first one stops all)
            // the B operands of this tile go into buffer `buf`, last read by the MMAs of it - 2
            if (it >= 2) {
                const bool freed = !*abort_flag &&
                                   mbar_wait(&b_empty[buf], ((it >> 1) - 1) & 1, &g_lla_err);
                if (!__all_sync(kFullMask, freed)) {
                    ok = false;
                    *abort_flag = 1;
                    continue;
                }
            }
            unsigned char* bb = smem + LY::B_OFF + buf * LY::BBUF;
            // p~ x as a bf16 pair: the high part and the residual x - hi, each rounded to
            // nearest (about 16 significant bits together)
            auto split_store = [&](const float2 (&v)[4], unsigned char* dst) {
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    hi[h] = pack_bf16_lla(v[h].x, v[h].y);
                    const float2 r = __fadd2_rn(v[h], make_float2(-__uint_as_float(hi[h] << 16),
                                                                  -__uint_as_float(hi[h] & 0xffff0000u)));
                    lo[h] = pack_bf16_lla(r.x, r.y);
                }
                st16(dst, hi[0], hi[1], hi[2], hi[3]);
                st16(dst + 2 * LY::TILE, lo[0], lo[1], lo[2], lo[3]);
            };
            const bool full = nk == kTile;  // uniform
#pragma unroll
            for (int r = 0; r < ROWS_PER_T; ++r) {
                const int j = rg + r * LY::RGRP;
                const uint32_t off = coff + j * 128 + ((cc ^ (j & 7)) * 16);
                if (full || j < nk) {
                    const float p = fast_exp2(sj[r] - m);
                    if (c == 0) lpart += p;
                    const float2 p2 = make_float2(p, p);
#pragma unroll
                    for (int kv = 0; kv < 2; ++kv) {
                        float f[8];
                        if (kv == 0) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) f[e] = kf[r][e];
                        } else {
                            Vec16<__nv_bfloat16>::unpack(ld16(kst + LY::TILE + off), f);
                        }
                        float2 v[4];
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            v[h] = __fmul2_rn(p2, make_float2(f[2 * h], f[2 * h + 1]));
                            if (kv == 0) mk[h] = __fadd2_rn(mk[h], v[h]);
                            else mv[h] = __fadd2_rn(mv[h], v[h]);
                        }
                        split_store(v, bb + kv * LY::TILE + off);
                    }
                } else {
                    // past the sequence (the rows may hold anything): zero B rows, and zero the
                    // key row, which is also the A operand
#pragma unroll
                    for (int x = 0; x < 4; ++x) st16(bb + x * LY::TILE + off, 0u, 0u, 0u, 0u);
                    st16(kst + off, 0u, 0u, 0u, 0u);
                }
            }
            fence_async_smem();  // visible to the tensor core's reads
            mbar_arrive(&b_full[buf]);
        }

        // ---------------------------------------------------------------- covariances
        const bool acc = ok && !*abort_flag && mbar_wait(acc_full, 0, &g_lla_err);
        if (!__all_sync(kFullMask, acc)) ok = false;
        // every compute warp is past the stream before its buffers are reused
        named_bar_sync(1, kCompute);
        tc::fence_after_sync();
        const float l = grp_sum(lpart, red, cw, lane);
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        float* sig = reinterpret_cast<float*>(smem + LY::SIG_OFF);
        float* ct = reinterpret_cast<float*>(smem + LY::CT_OFF);
        float* mup = reinterpret_cast<float*>(smem + LY::MUP_OFF);
        float* cgv = reinterpret_cast<float*>(smem + LY::CGV_OFF);
        float* muk = cgv;           // [D] mu_k
        float* muv = cgv + D;       // [D] mu_v
        float* xv = cgv + 2 * D;    // CG iterate
        float* rv = cgv + 3 * D;    // residual
        float* pv = cgv + 4 * D;    // search direction
        float* ap = cgv + 5 * D;    // Sigma p
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            mup[(rg * 2 + 0) * D + 8 * c + 2 * e] = mk[e].x;
            mup[(rg * 2 + 0) * D + 8 * c + 2 * e + 1] = mk[e].y;
            mup[(rg * 2 + 1) * D + 8 * c + 2 * e] = mv[e].x;
            mup[(rg * 2 + 1) * D + 8 * c + 2 * e + 1] = mv[e].y;
        }
        named_bar_sync(1, kCompute);
        if (t < 2 * D) {
            const int f = t % D, kind = t / D;
            float sum = 0.f;
            for (int r = 0; r < LY::RGRP; ++r) sum += mup[(r * 2 + kind) * D + f];
            (kind ? muv : muk)[f] = sum * inv_l;
        }
        named_bar_sync(1, kCompute);
        {
            // Sigma_kk (half 0) or C^T (half 1) from TMEM: lane = feature of k; each warp
            // takes half of the columns
            const int f1 = 32 * q4 + lane;
            const uint32_t trow = tmem + ((uint32_t)(32 * q4) << 16) + half * D + chalf * CW;
            const bool have = ntiles > 0 && ok;
            if (f1 < D) {
                const float mk1 = muk[f1];
#pragma unroll 1
                for (int x = 0; x < CW / 32; ++x) {
                    uint32_t u[32];
                    if (have) {
                        tc::tmem_ld32(trow + 32 * x, u);
                        if (ntiles > 1) {  // the odd tiles' set
                            uint32_t u2[32];
                            tc::tmem_ld32(trow + 2 * D + 32 * x, u2);
                            tc::tmem_ld_wait();
#pragma unroll
                            for (int y = 0; y < 32; ++y)
                                u[y] = __float_as_uint(__uint_as_float(u[y]) + __uint_as_float(u2[y]));
                        }
                        tc::tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int y = 0; y < 32; ++y) u[y] = 0u;
                    }
#pragma unroll
                    for (int y = 0; y < 32; ++y) {
                        const int f2 = chalf * CW + 32 * x + y;
                        const float g = __uint_as_float(u[y]) * inv_l;
                        if (half == 0)
                            sig[f1 * LY::LD + f2] = g - mk1 * muk[f2];
                        else
                            ct[f2 * LY::LD + f1] = g - mk1 * muv[f2];
                    }
                }
            }
        }
        if (t < D) {
            const float bt = n > 0 ? muk[t] - __bfloat162float(a.q[(size_t)bh * D + t]) : 0.f;
            xv[t] = 0.f;
            rv[t] = bt;
            pv[t] = bt;
        }
        named_bar_sync(1, kCompute);

        // ---------------------------------------------------------------- conjugate gradient
        constexpr int TPR = kCompute / D;  // threads per matrix row
        const int row = t / TPR, part = t % TPR;
        float rs = grp_sum(t < D ? rv[t] * rv[t] : 0.f, red, cw, lane);
        const float stop = kCgTol * kCgTol * rs;
        for (int i = 0; i < a.iters && rs > stop && rs > 0.f; ++i) {
            float partial = 0.f;
#pragma unroll 8
            for (int c2 = part; c2 < D; c2 += TPR) partial = fmaf(sig[row * LY::LD + c2], pv[c2], partial);
#pragma unroll
            for (int off = TPR / 2; off >= 1; off >>= 1) partial += __shfl_xor_sync(kFullMask, partial, off);
            if (part == 0) ap[row] = partial;
            named_bar_sync(1, kCompute);
            const float pap = grp_sum(t < D ? pv[t] * ap[t] : 0.f, red, cw, lane);
            if (!(pap > 0.f)) break;  // uniform; Sigma is only semi-definite
            const float alpha = rs / pap;
            float rn = 0.f;
            if (t < D) {
                xv[t] = fmaf(alpha, pv[t], xv[t]);
                rn = fmaf(-alpha, ap[t], rv[t]);
                rv[t] = rn;
            }
            const float rs_new = grp_sum(rn * rn, red, cw, lane);
            if (t < D) pv[t] = fmaf(rs_new / rs, pv[t], rn);
            named_bar_sync(1, kCompute);
            rs = rs_new;
        }
        // o = mu_v - C^T rho
        if (t < D) {
            float acc_o = 0.f;
#pragma unroll 8
            for (int f1 = 0; f1 < D; ++f1) acc_o = fmaf(ct[t * LY::LD + f1], xv[f1], acc_o);
            if (in_bounds(&g_lla_err, (size_t)bh * D + t + 1, a.out_elems)) {
                a.rho[(size_t)bh * D + t] = xv[t];
                a.o[(size_t)bh * D + t] = muv[t] - acc_o;
            }
        }
        if (!ok) *abort_flag = 1;
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, LY::TMEM_COLS);
    }
}

template <int D>
cudaError_t launch(const LlaArgs& a, const void* kc, const void* vc, int BH, cudaStream_t stream) {
    CUtensorMap mk, mv;
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)a.Lmax, (uint64_t)BH};
    const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)a.Lmax * D * 2};
    const uint32_t box[3] = {64, (uint32_t)kTile, 1};
    if (!make_tmap_bf16(&mk, kc, 3, dims, strides, box) ||
        !make_tmap_bf16(&mv, vc, 3, dims, strides, box))
        return cudaErrorInvalidValue;
    static std::atomic<uint64_t> smem_set{0};
    if (cudaError_t e = ensure_dynamic_smem(lla_kernel<D>, (int)LlaLayout<D>::SMEM_BYTES, smem_set))
        return e;
    lla_kernel<D><<<BH, kThreads, LlaLayout<D>::SMEM_BYTES, stream>>>(mk, mv, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t lla_launch(const void* q, const void* kc, const void* vc, const int32_t* seqlens,
                       float* rho, float* o, int B, int H, int Lmax, int d, int iters,
                       cudaStream_t stream) {
    LlaArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.seqlens = seqlens;
    a.rho = rho;
    a.o = o;
    a.H = H;
    a.Lmax = Lmax;
    a.iters = iters;
    a.qscale = kLog2e / sqrtf((float)d);
    a.out_elems = (size_t)B * H * d;
    if (d == 64) return launch<64>(a, kc, vc, B * H, stream);
    if (d == 128) return launch<128>(a, kc, vc, B * H, stream);
    return cudaErrorInvalidValue;
}

unsigned lla_take_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_lla_err, sizeof(v)) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_lla_err, &zero, sizeof(zero));
    return v;
}

}  // namespace parallax
