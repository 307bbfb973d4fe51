// Backward pass of the Parallax prefill on the tcgen05 tensor cores (sm_103a).
//
// Forward, per query row i over its keys j: p_ij = softmax_j(scale q_i.k_j),
// r_ij = rho_i.k_j, rbar_i = sum_j p_ij r_ij, and the output is one weighted sum
//   o_i = sum_j w_ij v_j,   w_ij = p_ij (1 + rbar_i - r_ij)
// (softmax attention minus the probe-projected key/value covariance, "Parallax
// mantem softmax ...", paragraph 2, since sum_j p_ij (r_ij - rbar_i) mu_v = 0).
// With dO the gradient of o, D_ij = dO_i.v_j, abar_i = dO_i.mu_v,i and
// delta_i = dO_i.o_i, the gradients are
//   dv_j  = sum_i w_ij dO_i
//   dr_ij = p_ij (abar_i - D_ij),   ds_ij = p_ij ((D_ij - abar_i)(rbar_i - r_ij) + D_ij - delta_i)
//   dq_i  = scale sum_j ds_ij k_j,  drho_i = sum_j dr_ij k_j
//   dk_j  = scale sum_i ds_ij q_i + sum_i dr_ij rho_i.
// p is recomputed from the forward's per-row log-sum-exp.
//
// Three kernels, in stream order:
//   bwd_pre_kernel  per row: (-lse2, 1 + rbar, abar, delta - abar) into a row-stats buffer;
//   bwd_kv_kernel   per 128-key tile: loops over 64-query tiles; MMAs
//                   [S^T | R^T] = K [Q; rho]^T and D^T = V dO^T, the compute
//                   warps form W, dS, dR (bf16, written back to TMEM), MMAs
//                   dV += W dO and dK += dS Q + dR rho (A from TMEM);
//   bwd_q_kernel    per 64-query tile, the forward's stacked layout (TMEM lane
//                   32g+i: query 16g+i's S row, lane 32g+16+i: its R row): MMAs
//                   [S; R] = [Q; rho] K^T and D = dO V^T (M = 64: D lands in the S lanes), the compute
//                   warps form dS, dR, MMA [dQ; drho] += [dS; dR] K.
// Every contraction is a tcgen05.mma with bf16 operands and fp32 TMEM
// accumulators; K, V and the query-side tiles arrive by TMA (128-byte swizzle).
#include <type_traits>

#include "tcgen05.cuh"
#include "kernels.h"

namespace parallax {
namespace {

__device__ unsigned g_bwd_err = 0;

// warp 0 TMA, warp 1 MMA, warps 2-3 set-up, warps 4-11 compute: two warps per TMEM
// lane quarter, each taking half of the columns of every tile
constexpr int kThreads = 384;
constexpr int kComputeThreads = 256;
constexpr int SUB = 128 * 128;  // [128 rows x 64 columns] bf16, 128-byte swizzled
constexpr int SUB64 = 64 * 128; // [64 rows x 64 columns]
constexpr int kBwdHeadGroup = 16;  // heads per CTA-scheduling group

struct BwdArgs {
    const float* o;               // [BH, L, D] forward output
    const float* mu;              // [BH, L, D] forward mu_v
    const __nv_bfloat16* dout;    // [BH, L, D] gradient of o
    const float* lse;             // [BH, L]
    const float* rbar;            // [BH, L]
    // [BH][4][Lp] per row (0 past L): -lse log2(e), 1 + rbar, abar, delta - abar -- the
    // forms the per-pair arithmetic uses directly
    float* rs;
    float* dq;
    float* drho;
    float* dk;
    float* dv;                    // [BH, L, D] fp32
    int L, BH;
    int Lp;                       // L rounded up to 64 (row-statistics stride)
    int n_kt, n_qt;               // 128-key tiles and 64-query tiles per head
    float scale, qscale;          // softmax scale, scale * log2(e)
};

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t x, uint32_t y, uint32_t z,
                                             uint32_t w) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(x), "r"(y), "r"(z),
                 "r"(w)
                 : "memory");
}

// ------------------------------------------------------------------------ row statistics
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdArgs a) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const size_t prow = (size_t)blockIdx.x * 8 + warp;  // padded row: (bh, i < Lp)
    if (prow >= (size_t)a.BH * a.Lp) return;
    const int bh = (int)(prow / a.Lp), i = (int)(prow - (size_t)bh * a.Lp);
    float* out = a.rs + (size_t)bh * 4 * a.Lp + i;
    if (!in_bounds(&g_bwd_err, (size_t)bh * 4 * a.Lp + 3 * (size_t)a.Lp + i + 1,
                   (size_t)a.BH * 4 * a.Lp))
        return;
    if (i >= a.L) {  // padding rows: zeros, so that tiles past L read finite values
        if (lane < 4) out[(size_t)lane * a.Lp] = 0.f;
        return;
    }
    const size_t row = (size_t)bh * a.L + i;
    constexpr int PER = D / 32;
    float ab = 0.f, de = 0.f;
#pragma unroll
    for (int x = 0; x < PER; ++x) {
        const size_t idx = row * D + lane + 32 * x;
        const float g = __bfloat162float(a.dout[idx]);
        ab = fmaf(g, a.mu[idx], ab);
        de = fmaf(g, a.o[idx], de);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        ab += __shfl_xor_sync(kFullMask, ab, off);
        de += __shfl_xor_sync(kFullMask, de, off);
    }
    if (lane == 0) {
        out[0] = -a.lse[row] * kLog2e;
        out[a.Lp] = 1.f + a.rbar[row];
        out[2 * (size_t)a.Lp] = ab;
        out[3 * (size_t)a.Lp] = de - ab;
    }
}


// The per-(query, key) gradient terms for two pairs at once (packed fp32x2).  In:
// the scores s, probe scores r and D = dO.v of the pairs; the rows' statistics
// nl = -lse log2(e), rb1 = 1 + rbar, ab = abar, ne = delta - abar; keep = which
// of the two pairs are visible.  With g = 1 + rbar - r and u = abar - D:
//   w = p g,   dr = p u,   ds scale = p (u g + ne) (-scale)
// (u g + ne = -((D - abar)(rbar - r) + D - delta)).
struct PairTerms {
    float2 w, ds, dr;
};
template <bool MASKED, bool WANT_W>
__device__ __forceinline__ PairTerms pair_terms(float2 s, float2 r, float2 d, float2 qs2, float2 nl,
                                                float2 rb1, float2 ab, float2 ne, float2 nsc2,
                                                bool keep0, bool keep1) {
    const float2 m1 = make_float2(-1.f, -1.f);
    const float2 t = __ffma2_rn(s, qs2, nl);
    float2 p = make_float2(fast_exp2(t.x), fast_exp2(t.y));
    if (MASKED) {
        p.x = keep0 ? p.x : 0.f;
        p.y = keep1 ? p.y : 0.f;
    }
    const float2 g = __ffma2_rn(r, m1, rb1);
    const float2 u = __ffma2_rn(d, m1, ab);
    PairTerms o;
    if (WANT_W) o.w = __fmul2_rn(p, g);
    o.dr = __fmul2_rn(p, u);
    o.ds = __fmul2_rn(__fmul2_rn(p, __ffma2_rn(u, g, ne)), nsc2);
    return o;
}

// ------------------------------------------------------------------------ dK, dV
// One 128-key tile per CTA (one key per TMEM lane), 64-query tiles of Q, rho and
// dO in a 3-deep TMA ring.  V sits in TMEM as the A operand of D^T = V dO^T, so
// shared memory holds K, the ring and the gradient operands W, dS, dR (bf16,
// [128 keys x 64 queries], written by the compute warps).  The compute warps
// release TMEM as soon as they have loaded S, R and D of a tile: the MMAs of
// the next tile then run while they work, and dV += W dO, dK += dS Q + dR rho
// (A from shared memory) follow once the operands are written.
// Warps: 0 TMA, 1 MMA (+ TMEM owner), 2-9 compute: warp w serves TMEM lane
// quarter w % 4, warps 2-5 queries 0-31 and warps 6-9 queries 32-63 of a tile.
// Ten warps leave each thread 200 registers.
constexpr int kKvThreads = 320;
constexpr int kKvStages = 3;

template <int D>
struct KvLayout {
    static constexpr int NCB = D / 64;
    static constexpr int OPB = NCB * SUB;                // [128 x D] operand
    static constexpr int K_OFF = 0;
    static constexpr int QR_BYTES = OPB;                 // [Q; rho] rows 0..63 / 64..127
    static constexpr int DO_BYTES = NCB * SUB64;         // dO [64 x D]
    static constexpr int STAGE = QR_BYTES + DO_BYTES;
    static constexpr int ST_OFF = OPB;
    // W, dS, dR: [128 keys x 64 queries] bf16 each, 128-byte swizzled (K-major A operands).
    // The V tile lands here first, on its way to TMEM.
    static constexpr int G_OFF = ST_OFF + kKvStages * STAGE;
    // row statistics of a query tile, [4][64] fp32, in two slots
    static constexpr int RS_OFF = G_OFF + 3 * SUB;
    static constexpr int BAR_OFF = RS_OFF + 2 * 1024;
    // kv_full, v_ready, qr_full[S], qr_empty[S], s_full, y_free, p_full, g_done, o_full,
    // rs_full[2], rs_free[2], staged
    static constexpr int B_STAGED = 2 + 2 * kKvStages + 9;
    static constexpr int NBARS = B_STAGED + 1;
    // Epilogue: once every MMA has completed, the query-side ring holds dV and dK as
    // [128 keys x 32 columns] fp32 boxes (128-byte swizzle) for TMA stores.
    static constexpr int OUT_BOX = 128 * 128;
    static_assert(2 * (D / 32) * OUT_BOX <= kKvStages * STAGE, "dK/dV staging fits the ring");
    // the buffers start at the (1024-byte aligned) base of dynamic shared memory
    static constexpr int SMEM_BYTES = BAR_OFF + NBARS * 8 + 16;
    static_assert(OPB <= 3 * SUB, "the V tile must fit in the gradient-operand area");
    // TMEM columns
    static constexpr uint32_t SR = 0, DT = 128, VA = 192, DV = 256, DK = 256 + D;
};

template <int D, bool CAUSAL, bool RHO>
__global__ void __launch_bounds__(kKvThreads, 1)
    bwd_kv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmR,
                  const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmDV,
                  const __grid_constant__ CUtensorMap tmDK, const BwdArgs a) {
    using LY = KvLayout<D>;
    constexpr int S = kKvStages;
    extern __shared__ __align__(1024) unsigned char smem[];
    // the 128-byte-swizzled tiles need 1024-byte alignment; the layout leaves no room to
    // realign, so a misaligned base is reported instead of used
    if (smem_u32(smem) & 1023u) {
        if (threadIdx.x == 0) raise_error(&g_bwd_err, PARALLAX_DEVERR_SMEM_MISALIGNED);
        return;
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LY::BAR_OFF);
    uint64_t* kv_full = bars;
    uint64_t* v_ready = bars + 1;        // V is in TMEM (128 arrivals)
    uint64_t* qr_full = bars + 2;
    uint64_t* qr_empty = bars + 2 + S;
    uint64_t* s_full = bars + 2 + 2 * S;
    uint64_t* y_free = bars + 3 + 2 * S;  // S, R, D of the tile loaded (256 arrivals)
    uint64_t* p_full = bars + 4 + 2 * S;  // W, dS, dR of the tile written (256 arrivals)
    uint64_t* g_done = bars + 5 + 2 * S;  // the gradient MMAs of the tile have read them
    uint64_t* o_full = bars + 6 + 2 * S;
    uint64_t* rs_full = bars + 7 + 2 * S;  // [2] statistics slot loaded
    uint64_t* rs_free = bars + 9 + 2 * S;  // [2] statistics slot read (256 arrivals)
    uint64_t* staged = bars + LY::B_STAGED;  // dV, dK staged for the TMA stores (256 arrivals)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + LY::NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    // CTA -> (head, key tile): heads in groups of kBwdHeadGroup, the key tiles that
    // see the most queries first within a group, so that the CTAs resident at any
    // time share the query-side tiles of a few heads in L2
    const int group = blockIdx.x / (kBwdHeadGroup * a.n_kt);
    const int gsize = min(kBwdHeadGroup, a.BH - group * kBwdHeadGroup);
    const int r_in = blockIdx.x - group * kBwdHeadGroup * a.n_kt;
    const int kt = r_in / gsize;
    const int bh = group * kBwdHeadGroup + r_in % gsize;
    const int k0 = kt * 128;
    const int qt0 = CAUSAL ? k0 / 64 : 0;
    const int n_t = a.n_qt - qt0;

    if (threadIdx.x == 0) {
        for (int b = 0; b < LY::NBARS; ++b) {
            uint32_t count = 1;
            if (b == 1) count = 128;
            if (b == 3 + 2 * S || b == 4 + 2 * S || b == 9 + 2 * S || b == 10 + 2 * S ||
                b == LY::B_STAGED)
                count = kComputeThreads;
            mbar_init(&bars[b], count);
        }
        const bool abort0 = (*(volatile unsigned*)&g_bwd_err & PARALLAX_DEVERR_WAIT_TIMEOUT) != 0;
        *abort_flag = abort0 ? 1 : 0;
        fence_mbar_init();
        tc::prefetch_tmap(&tmQ);
        if (RHO) tc::prefetch_tmap(&tmR);
        tc::prefetch_tmap(&tmK);
        tc::prefetch_tmap(&tmV);
        tc::prefetch_tmap(&tmO);
        tc::prefetch_tmap(&tmDV);
        tc::prefetch_tmap(&tmDK);
        // the key tile, V and the first query-side tiles go out before the CTA-wide set-up
        // (TMEM allocation and the barrier below); the producer loop continues after them
        if (!abort0) {
            mbar_arrive_expect_tx(kv_full, 2 * LY::OPB);
            for (int cb = 0; cb < LY::NCB; ++cb) {
                tc::tma_load_3d(smem + LY::K_OFF + cb * SUB, &tmK, cb * 64, k0, bh, kv_full);
                tc::tma_load_3d(smem + LY::G_OFF + cb * SUB, &tmV, cb * 64, k0, bh, kv_full);
            }
            for (int t = 0; t < min(n_t, S); ++t) {
                const int q0 = (qt0 + t) * 64;
                unsigned char* stage = smem + LY::ST_OFF + t * LY::STAGE;
                mbar_arrive_expect_tx(&qr_full[t], (RHO ? 2 : 1) * LY::NCB * SUB64 + LY::DO_BYTES);
                for (int cb = 0; cb < LY::NCB; ++cb) {
                    tc::tma_load_3d(stage + cb * SUB, &tmQ, cb * 64, q0, bh, &qr_full[t]);
                    if (RHO)
                        tc::tma_load_3d(stage + cb * SUB + SUB64, &tmR, cb * 64, q0, bh, &qr_full[t]);
                    tc::tma_load_3d(stage + LY::QR_BYTES + cb * SUB64, &tmO, cb * 64, q0, bh,
                                    &qr_full[t]);
                }
            }
        }
    }
    if (warp == 1) tc::tmem_alloc(tmem_slot, 512);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const bool skip = *abort_flag != 0;

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        // lane 0 streams the query-side tiles, lane 1 the row statistics: each waits only on
        // its own slots, so a statistics slot still in use never holds up a tile load
        // (the key tile, V and the first min(n_t, S) query-side tiles went out at set-up)
        if (lane == 0 && !skip) {
            int issued = min(n_t, S);
            bool ok = true;
            for (int t = issued; t < n_t; ++t) {
                const int st = t % S;
                if (t >= S && !mbar_wait(&qr_empty[st], ((t / S) - 1) & 1, &g_bwd_err)) {
                    ok = false;
                    break;
                }
                const int q0 = (qt0 + t) * 64;
                unsigned char* stage = smem + LY::ST_OFF + st * LY::STAGE;
                mbar_arrive_expect_tx(&qr_full[st], (RHO ? 2 : 1) * LY::NCB * SUB64 + LY::DO_BYTES);
                for (int cb = 0; cb < LY::NCB; ++cb) {
                    tc::tma_load_3d(stage + cb * SUB, &tmQ, cb * 64, q0, bh, &qr_full[st]);
                    if (RHO)
                        tc::tma_load_3d(stage + cb * SUB + SUB64, &tmR, cb * 64, q0, bh, &qr_full[st]);
                    tc::tma_load_3d(stage + LY::QR_BYTES + cb * SUB64, &tmO, cb * 64, q0, bh,
                                    &qr_full[st]);
                }
                issued = t + 1;
            }
            if (!ok) {
                *abort_flag = 1;
                mbar_wait(kv_full, 0, &g_bwd_err);
                for (int t = issued >= S ? issued - S : 0; t < issued; ++t)
                    mbar_wait(&qr_full[t % S], (t / S) & 1, &g_bwd_err);
            }
        } else if (lane == 1 && !skip) {
            int rs_issued = 0;
            bool ok = true;
            for (int t = 0; t < n_t; ++t) {
                // the 64 rows' statistics (one 256-byte copy per array) into slot t % 2, once
                // the compute warps are done with tile t - 2
                const int rsl = t & 1;
                if (t >= 2 && !mbar_wait(&rs_free[rsl], ((t >> 1) - 1) & 1, &g_bwd_err)) {
                    ok = false;
                    break;
                }
                const int q0 = (qt0 + t) * 64;
                mbar_arrive_expect_tx(&rs_full[rsl], 4 * 64 * 4);
                for (int k = 0; k < 4; ++k)
                    bulk_g2s(smem + LY::RS_OFF + rsl * 1024 + k * 256,
                             a.rs + ((size_t)bh * 4 + k) * a.Lp + q0, 256, &rs_full[rsl]);
                rs_issued = t + 1;
            }
            if (!ok) {
                *abort_flag = 1;
                for (int t = rs_issued >= 2 ? rs_issued - 2 : 0; t < rs_issued; ++t)
                    mbar_wait(&rs_full[t & 1], (t >> 1) & 1, &g_bwd_err);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (!skip) {
            constexpr uint32_t kIdescA = tc::idesc_bf16_f32(128, RHO ? 128 : 64, false);
            constexpr uint32_t kIdescB = tc::idesc_bf16_f32(128, 64, false);
            constexpr uint32_t kIdescMN = tc::idesc_bf16_f32(128, D, true);
            const uint32_t sbase = smem_u32(smem);
            const uint64_t dK = tc::smem_desc_sw128(sbase + LY::K_OFF, 16, 1024);
            const uint64_t dG = tc::smem_desc_sw128(sbase + LY::G_OFF, 16, 1024);
            const uint32_t stb = sbase + LY::ST_OFF;
            constexpr uint32_t kStStep = LY::STAGE >> 4;
            // [S^T | R^T] = K [Q; rho]^T (A and B from shared memory) and D^T = V dO^T
            // (A = V from TMEM) of query tile t
            auto issue_srd = [&](int t) -> bool {
                const int st = t % S;
                if (*abort_flag || !mbar_wait_warp(&qr_full[st], (t / S) & 1, &g_bwd_err))
                    return false;
                tc::fence_after_sync();
                const uint64_t dQR = tc::opaque(tc::smem_desc_sw128(stb, 16, 1024) + st * kStStep);
                const uint64_t dDO =
                    tc::opaque(tc::smem_desc_sw128(stb + LY::QR_BYTES, 16, 1024) + st * kStStep);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk / 4) * SUB + (kk % 4) * 32) >> 4;
                    tc::mma_ss(tmem + LY::SR, dK + off, dQR + off, kIdescA, kk > 0);
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t offB = ((kk / 4) * SUB64 + (kk % 4) * 32) >> 4;
                    tc::mma_ts(tmem + LY::DT, tmem + LY::VA + 8 * kk, dDO + offB, kIdescB, kk > 0);
                }
                tc::commit(s_full);
                return true;
            };
            bool ok = mbar_wait_warp(kv_full, 0, &g_bwd_err) && mbar_wait_warp(v_ready, 0, &g_bwd_err);
            if (ok) ok = issue_srd(0);
            for (int t = 0; t < n_t && ok; ++t) {
                if (t + 1 < n_t) {  // the next tile's S|R and D as soon as TMEM is free
                    if (!mbar_wait_warp(y_free, t & 1, &g_bwd_err)) {
                        ok = false;
                        break;
                    }
                    if (!(ok = issue_srd(t + 1))) break;
                }
                if (*abort_flag || !mbar_wait_warp(p_full, t & 1, &g_bwd_err)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const int st = t % S;
                // MN-major views of the query-side tiles: rows = queries (the K dimension)
                const uint64_t mQR = tc::opaque(tc::smem_desc_sw128(stb, SUB, 1024) + st * kStStep);
                const uint64_t mDO =
                    tc::opaque(tc::smem_desc_sw128(stb + LY::QR_BYTES, SUB64, 1024) + st * kStStep);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {  // queries 16kk .. 16kk + 15
                    const uint32_t acc = (t > 0 || kk > 0) ? 1u : 0u;
                    const uint32_t ka = (kk * 32) >> 4;
                    // dV += W dO
                    tc::mma_ss(tmem + LY::DV, dG + ka, mDO + ((kk * 16 * 128) >> 4), kIdescMN, acc);
                    // dK += dS Q  (scale folded into dS)
                    tc::mma_ss(tmem + LY::DK, dG + (SUB >> 4) + ka, mQR + ((kk * 16 * 128) >> 4),
                               kIdescMN, acc);
                    if (RHO)  // dK += dR rho
                        tc::mma_ss(tmem + LY::DK, dG + ((2 * SUB) >> 4) + ka,
                                   mQR + (((64 + kk * 16) * 128) >> 4), kIdescMN, 1u);
                }
                tc::commit(g_done);
                tc::commit(&qr_empty[st]);
            }
            tc::commit(o_full);
            if (!ok) {
                *abort_flag = 1;
                mbar_wait_warp(o_full, 0, &g_bwd_err);
            }
        }
    } else {
        // ---------------------------------------------------------------- compute + epilogue
        const int q4 = warp & 3;                // TMEM lane quarter
        const int c = (warp - 2) >> 2;          // queries 32c .. 32c + 31 of every tile
        const int row = 32 * q4 + lane;         // this thread's key within the tile
        const int j = k0 + row;
        const uint32_t trow = tmem + ((uint32_t)(32 * q4) << 16);
        const float qs = a.qscale, scale = a.scale;
        bool ok = !skip;
        if (c == 0) {
            // V -> TMEM: lane = key, column x holds elements 2x, 2x + 1 (the A-operand layout)
            const bool got = ok && mbar_wait(kv_full, 0, &g_bwd_err);
            if (__all_sync(kFullMask, got)) {
#pragma unroll 1
                for (int cb = 0; cb < LY::NCB; ++cb) {
                    uint32_t u[32];
                    const unsigned char* vrow = smem + LY::G_OFF + cb * SUB + row * 128;
#pragma unroll
                    for (int x = 0; x < 8; ++x) {
                        const uint4 q = *reinterpret_cast<const uint4*>(vrow + ((x ^ (row & 7)) * 16));
                        u[4 * x] = q.x;
                        u[4 * x + 1] = q.y;
                        u[4 * x + 2] = q.z;
                        u[4 * x + 3] = q.w;
                    }
                    tc::tmem_st32(trow + LY::VA + 32 * cb, u);
                }
                tc::tmem_st_wait();
            } else {
                ok = false;
                *abort_flag = 1;
            }
            tc::fence_before_sync();
            mbar_arrive(v_ready);
        }
        const uint32_t gbase = smem_u32(smem + LY::G_OFF) + row * 128;
        for (int t = 0; t < n_t && ok; ++t) {
            const bool got = !*abort_flag && mbar_wait(s_full, t & 1, &g_bwd_err);
            if (!__all_sync(kFullMask, got)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            const int qc = (qt0 + t) * 64 + 32 * c;
            // row statistics of the 32 queries (rows past L hold zeros): slot t % 2 holds
            // [4][64] for the tile
            const bool have = !*abort_flag && mbar_wait(&rs_full[t & 1], (t >> 1) & 1, &g_bwd_err);
            if (!__all_sync(kFullMask, have)) {
                ok = false;
                break;
            }
            const float* st0 = reinterpret_cast<const float*>(smem + LY::RS_OFF + (t & 1) * 1024) + 32 * c;
            const float2 qs2 = make_float2(qs, qs), nsc2 = make_float2(-scale, -scale);
            uint32_t wpk[16], spk[16], rpk[16];
            // S, R, D of the thread's 32 queries, all loaded before TMEM is released
            uint32_t sv[32], rv[32], dv[32];
            tc::tmem_ld32(trow + LY::SR + 32 * c, sv);
            if (RHO) tc::tmem_ld32(trow + LY::SR + 64 + 32 * c, rv);
            tc::tmem_ld32(trow + LY::DT + 32 * c, dv);
            tc::tmem_ld_wait();
            tc::fence_before_sync();
            mbar_arrive(y_free);  // the next tile's MMAs may overwrite S, R, D
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {  // 16 queries at a time
                // queries past L or (causal) before this key get no weight
                const int qb16 = qc + 16 * qq;
                const int nvalid = min(16, a.L - qb16);
                uint32_t vmask = nvalid >= 16 ? 0xffffu : nvalid <= 0 ? 0u : ((1u << nvalid) - 1u);
                if (CAUSAL && j > qb16) vmask &= j - qb16 >= 16 ? 0u : ~((1u << (j - qb16)) - 1u);
                const float* sq = st0 + 16 * qq;
                auto run = [&](auto masked) {
                    constexpr bool M = decltype(masked)::value;
#pragma unroll
                    for (int y4 = 0; y4 < 4; ++y4) {  // four queries per step: 128-bit stat loads
                        const int x4 = 4 * y4;
                        const float4 nl = *reinterpret_cast<const float4*>(sq + x4);
                        const float4 rb = *reinterpret_cast<const float4*>(sq + 64 + x4);
                        const float4 ab = *reinterpret_cast<const float4*>(sq + 128 + x4);
                        const float4 ne = *reinterpret_cast<const float4*>(sq + 192 + x4);
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int xl = x4 + 2 * hh, x = 16 * qq + xl, y = x / 2;
                            const float2 s2 = make_float2(__uint_as_float(sv[x]), __uint_as_float(sv[x + 1]));
                            const float2 r2 = RHO ? make_float2(__uint_as_float(rv[x]),
                                                                __uint_as_float(rv[x + 1]))
                                                  : make_float2(0.f, 0.f);
                            const float2 d2 = make_float2(__uint_as_float(dv[x]), __uint_as_float(dv[x + 1]));
                            const PairTerms pt = pair_terms<M, true>(
                                s2, r2, d2, qs2, hh ? make_float2(nl.z, nl.w) : make_float2(nl.x, nl.y),
                                hh ? make_float2(rb.z, rb.w) : make_float2(rb.x, rb.y),
                                hh ? make_float2(ab.z, ab.w) : make_float2(ab.x, ab.y),
                                hh ? make_float2(ne.z, ne.w) : make_float2(ne.x, ne.y), nsc2,
                                (vmask >> xl) & 1u, (vmask >> (xl + 1)) & 1u);
                            wpk[y] = tc::pack_bf16(pt.w.x, pt.w.y);
                            spk[y] = tc::pack_bf16(pt.ds.x, pt.ds.y);
                            rpk[y] = tc::pack_bf16(pt.dr.x, pt.dr.y);
                        }
                    }
                };
                // warp-uniform: every (key, query) pair of the warp's 16 queries is visible
                if (__all_sync(kFullMask, vmask == 0xffffu))
                    run(std::false_type{});
                else
                    run(std::true_type{});
            }
            mbar_arrive(&rs_free[t & 1]);  // this thread is done with the slot
            // the previous tile's gradient MMAs must have read the operand area
            const bool free_g = t == 0 || (!*abort_flag && mbar_wait(g_done, (t - 1) & 1, &g_bwd_err));
            if (!__all_sync(kFullMask, free_g)) {
                ok = false;
                break;
            }
            // row `row` of W, dS, dR: queries 32c .. 32c + 31 = 16-byte chunks 4c .. 4c + 3,
            // stored at chunk (index ^ row % 8) of the 128-byte row (128-byte swizzle)
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const uint32_t off = (uint32_t)(((4 * c + x) ^ (row & 7)) * 16);
                st_shared_v4(gbase + off, wpk[4 * x], wpk[4 * x + 1], wpk[4 * x + 2], wpk[4 * x + 3]);
                st_shared_v4(gbase + SUB + off, spk[4 * x], spk[4 * x + 1], spk[4 * x + 2], spk[4 * x + 3]);
                if (RHO)
                    st_shared_v4(gbase + 2 * SUB + off, rpk[4 * x], rpk[4 * x + 1], rpk[4 * x + 2],
                                 rpk[4 * x + 3]);
            }
            fence_proxy_async_smem();  // visible to the tensor core's reads
            mbar_arrive(p_full);
        }
        const bool done = ok && !*abort_flag && mbar_wait(o_full, 0, &g_bwd_err);
        // half 0 stages dV, half 1 dK, each row into [128 keys x 32 columns] boxes
        unsigned char* stage = smem + LY::ST_OFF + c * (D / 32) * LY::OUT_BOX;
        if (__all_sync(kFullMask, done)) {
            tc::fence_after_sync();
            const uint32_t base = trow + (c == 0 ? LY::DV : LY::DK);
            uint32_t uu[D / 32][32];  // the whole row behind one wait
#pragma unroll
            for (int b = 0; b < D / 32; ++b) tc::tmem_ld32(base + 32 * b, uu[b]);
            tc::tmem_ld_wait();
#pragma unroll
            for (int b = 0; b < D / 32; ++b) {
                const uint32_t(&u)[32] = uu[b];
                unsigned char* box = stage + b * LY::OUT_BOX + row * 128;
#pragma unroll
                for (int x = 0; x < 8; ++x)
                    st_shared_v4(smem_u32(box + ((x ^ (row & 7)) << 4)), u[4 * x], u[4 * x + 1],
                                 u[4 * x + 2], u[4 * x + 3]);
            }
        } else {
            *abort_flag = 1;
        }
        // every compute thread arrives, whichever way it went; one thread then stores the
        // tile's dV and dK rows (rows past L are clipped by the tensor maps)
        fence_proxy_async_smem();
        mbar_arrive(staged);
        if (warp == 2 && lane == 0 && mbar_wait(staged, 0, &g_bwd_err) && !*abort_flag) {
            unsigned char* st0 = smem + LY::ST_OFF;
#pragma unroll 1
            for (int b = 0; b < D / 32; ++b) {
                tc::tma_store_3d(&tmDV, 32 * b, k0, bh, st0 + b * LY::OUT_BOX);
                tc::tma_store_3d(&tmDK, 32 * b, k0, bh, st0 + (D / 32 + b) * LY::OUT_BOX);
            }
            tc::bulk_commit_group();
            tc::bulk_wait_group_read0();
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------------ dQ, drho
// One 64-query tile per CTA (the forward's stacked lane layout), 128-key tiles
// (K and V in 3-deep TMA rings).  TMEM: Y = [S; R] (128 columns)
// and D (128 columns, in the query lanes only: an M = 64 MMA) of the current key
// tile, the [dQ; drho] accumulator,
// the packed dS/dR operand slot, and the stacked [Q; rho] tile itself (the A
// operand of [S; R], copied in once, which leaves shared memory to the K ring).
// The compute warps release Y as soon as they have loaded it, so the MMAs of
// key tile t + 1 run while they work on tile t; [dQ; drho] += [dS; dR] K of
// tile t follows.  Every MMA has N = 128 (the tensor core's full rate; N = 64
// runs at ~60% of it).  Eight compute warps: two per TMEM lane quarter, each
// taking 64 of the 128 key columns.
constexpr int Q_KT = 128;     // keys per tile
constexpr int Q_KSTAGES = 3;  // K is read by two MMA groups (S|R of its tile, then dQ)
constexpr int Q_VSTAGES = 3;

template <int D>
struct QLayout {
    static constexpr int NCB = D / 64;
    static constexpr int OPB = NCB * SUB;             // [128 x D] operand, also one K or V tile
    static constexpr int DO_OFF = 0;                  // dO [64 x D] (the A operand of D, M = 64)
    static constexpr int K_OFF = NCB * SUB64;         // K ring
    static constexpr int V_OFF = K_OFF + Q_KSTAGES * OPB;  // V ring
    // the stacked [Q; rho] tile lands in the last K stage, on its way to TMEM
    static constexpr int QR_OFF = K_OFF + (Q_KSTAGES - 1) * OPB;
    static constexpr int BAR_OFF = V_OFF + Q_VSTAGES * OPB;
    // q_full, k_full[KS], k_empty[KS], v_full[VS], v_empty[VS], s_full, y_free, p_full,
    // pk_empty, o_full, qr_in, staged
    static constexpr int B_S = 1 + 2 * Q_KSTAGES + 2 * Q_VSTAGES;
    static constexpr int NBARS = B_S + 7;
    // Epilogue: once every MMA has completed, the K ring holds dQ and drho as
    // [64 queries x 32 columns] fp32 boxes (128-byte swizzle) for TMA stores.
    static constexpr int OUT_BOX = 64 * 128;
    static_assert(2 * (D / 32) * OUT_BOX <= (Q_KSTAGES + Q_VSTAGES) * OPB, "dQ staging fits the rings");
    static constexpr int SMEM_BYTES = BAR_OFF + NBARS * 8 + 16 + 1024;
    // TMEM columns: [S; R] at 0, D at YD, the accumulator at O, the packed slot at PK,
    // [Q; rho] (bf16 pairs) at QA
    static constexpr uint32_t YD = 128, O = 256, PK = 256 + D, QA = 256 + D + 64;
};

template <int D, bool CAUSAL, bool RHO>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_q_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmR,
                 const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmDQ,
                 const __grid_constant__ CUtensorMap tmDR, const BwdArgs a) {
    using LY = QLayout<D>;
    constexpr int KS = Q_KSTAGES, VS = Q_VSTAGES;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LY::BAR_OFF);
    uint64_t* q_full = bars;
    uint64_t* k_full = bars + 1;
    uint64_t* k_empty = bars + 1 + KS;
    uint64_t* v_full = bars + 1 + 2 * KS;
    uint64_t* v_empty = bars + 1 + 2 * KS + VS;
    uint64_t* s_full = bars + LY::B_S;
    uint64_t* y_free = bars + LY::B_S + 1;    // the compute warps have loaded Y
    uint64_t* p_full = bars + LY::B_S + 2;    // packed slot written
    uint64_t* pk_empty = bars + LY::B_S + 3;  // packed slot read by its dQ MMAs
    uint64_t* o_full = bars + LY::B_S + 4;
    uint64_t* qr_in = bars + LY::B_S + 5;     // [Q; rho] copied to TMEM (128 arrivals)
    uint64_t* staged = bars + LY::B_S + 6;    // dQ, drho staged for the TMA stores (256 arrivals)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + LY::NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    // CTA -> (head, query tile): heads in groups of kBwdHeadGroup, heaviest query
    // tile first within a group (their K/V tiles stay in L2 while the group runs)
    const int group = blockIdx.x / (kBwdHeadGroup * a.n_qt);
    const int gsize = min(kBwdHeadGroup, a.BH - group * kBwdHeadGroup);
    const int r_in = (blockIdx.x - group * kBwdHeadGroup * a.n_qt) / gsize;
    const int bh = group * kBwdHeadGroup + (blockIdx.x - group * kBwdHeadGroup * a.n_qt) % gsize;
    const int qb = CAUSAL ? a.n_qt - 1 - r_in : r_in;
    const int q0 = qb * 64;
    const int n_all = (a.L + Q_KT - 1) / Q_KT;
    const int n_t = CAUSAL ? min(n_all, (q0 + 63) / Q_KT + 1) : n_all;  // key tiles up to the diagonal

    if (threadIdx.x == 0) {
        for (int b = 0; b < LY::NBARS; ++b) {
            uint32_t count = 1;
            if (b == LY::B_S + 1 || b == LY::B_S + 2 || b == LY::B_S + 6) count = kComputeThreads;
            if (b == LY::B_S + 5) count = 128;
            mbar_init(&bars[b], count);
        }
        const bool abort0 = (*(volatile unsigned*)&g_bwd_err & PARALLAX_DEVERR_WAIT_TIMEOUT) != 0;
        *abort_flag = abort0 ? 1 : 0;
        fence_mbar_init();
        tc::prefetch_tmap(&tmQ);
        if (RHO) tc::prefetch_tmap(&tmR);
        tc::prefetch_tmap(&tmK);
        tc::prefetch_tmap(&tmV);
        tc::prefetch_tmap(&tmO);
        // Q (and rho), dO and the first key tiles go out before the CTA-wide set-up (TMEM
        // allocation and the barrier below); the producer loop continues after them
        if (!abort0) {
            // Q (and rho) once in 16-row boxes (the stacked layout), dO once as a 64-row box
            mbar_arrive_expect_tx(q_full, (RHO ? 2 : 1) * LY::NCB * (SUB / 2) + LY::NCB * SUB64);
            for (int cb = 0; cb < LY::NCB; ++cb) {
                unsigned char* qr = smem + LY::QR_OFF + cb * SUB;
                for (int g = 0; g < 4; ++g) {
                    const int row = q0 + 16 * g;
                    tc::tma_load_3d(qr + (32 * g) * 128, &tmQ, cb * 64, row, bh, q_full);
                    if (RHO) tc::tma_load_3d(qr + (32 * g + 16) * 128, &tmR, cb * 64, row, bh, q_full);
                }
                tc::tma_load_3d(smem + LY::DO_OFF + cb * SUB64, &tmO, cb * 64, q0, bh, q_full);
            }
            for (int j = 0; j < min(n_t, KS - 1); ++j) {
                mbar_arrive_expect_tx(&v_full[j], LY::OPB);
                for (int cb = 0; cb < LY::NCB; ++cb)
                    tc::tma_load_3d(smem + LY::V_OFF + j * LY::OPB + cb * SUB, &tmV, cb * 64,
                                    j * Q_KT, bh, &v_full[j]);
                mbar_arrive_expect_tx(&k_full[j], LY::OPB);
                for (int cb = 0; cb < LY::NCB; ++cb)
                    tc::tma_load_3d(smem + LY::K_OFF + j * LY::OPB + cb * SUB, &tmK, cb * 64,
                                    j * Q_KT, bh, &k_full[j]);
            }
        }
    }
    if (!RHO && (warp == 2 || warp == 3)) {
        // no probe: the rho rows of the stacked operand are zero (R = 0)
        for (int i = threadIdx.x - 64; i < LY::NCB * 64 * 8; i += 64) {
            const int cb = i / 512, rem = i % 512, g = rem / 128, w = rem % 128;
            reinterpret_cast<uint4*>(smem + LY::QR_OFF + cb * SUB + (32 * g + 16) * 128)[w] =
                make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    if (warp == 1) tc::tmem_alloc(tmem_slot, 512);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const bool skip = *abort_flag != 0;

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        // (Q, rho, dO and the key tiles before min(n_t, KS - 1) went out at set-up)
        if (lane == 0 && !skip) {
            bool ok = true;
            int kj = min(n_t, KS - 1), vj = kj;
            for (int j = kj; j < n_t && ok; ++j) {
                // V first: its slot frees (S|R MMAs of tile j - VS) before K's (dQ of tile j - KS)
                const int vs = j % VS, ks = j % KS;
                if (j >= VS && !mbar_wait(&v_empty[vs], ((j / VS) - 1) & 1, &g_bwd_err)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&v_full[vs], LY::OPB);
                for (int cb = 0; cb < LY::NCB; ++cb)
                    tc::tma_load_3d(smem + LY::V_OFF + vs * LY::OPB + cb * SUB, &tmV, cb * 64,
                                    j * Q_KT, bh, &v_full[vs]);
                vj = j + 1;
                if (j >= KS && !mbar_wait(&k_empty[ks], ((j / KS) - 1) & 1, &g_bwd_err)) {
                    ok = false;
                    break;
                }
                // the last stage first holds [Q; rho] until it is in TMEM
                if (j == KS - 1 && !mbar_wait(qr_in, 0, &g_bwd_err)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&k_full[ks], LY::OPB);
                for (int cb = 0; cb < LY::NCB; ++cb)
                    tc::tma_load_3d(smem + LY::K_OFF + ks * LY::OPB + cb * SUB, &tmK, cb * 64,
                                    j * Q_KT, bh, &k_full[ks]);
                kj = j + 1;
            }
            if (!ok) {
                *abort_flag = 1;
                mbar_wait(q_full, 0, &g_bwd_err);
                for (int k = (kj >= KS ? kj - KS : 0); k < kj; ++k)
                    mbar_wait(&k_full[k % KS], (k / KS) & 1, &g_bwd_err);
                for (int k = (vj >= VS ? vj - VS : 0); k < vj; ++k)
                    mbar_wait(&v_full[k % VS], (k / VS) & 1, &g_bwd_err);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (!skip) {
            constexpr uint32_t kIdesc1 = tc::idesc_bf16_f32(128, Q_KT, false);
            // M = 64: row r of D lands in TMEM lane 32 (r / 16) + r % 16, the lane of query r's
            // S row in the stacked layout
            constexpr uint32_t kIdescD = tc::idesc_bf16_f32(64, Q_KT, false);
            constexpr uint32_t kIdesc2 = tc::idesc_bf16_f32(128, D, true);
            const uint32_t sbase = smem_u32(smem);
            const uint64_t dDO = tc::smem_desc_sw128(sbase + LY::DO_OFF, 16, 1024);
            const uint64_t dK0 = tc::smem_desc_sw128(sbase + LY::K_OFF, 16, 1024);
            const uint64_t dV0 = tc::smem_desc_sw128(sbase + LY::V_OFF, 16, 1024);
            // MN-major view of a K tile: rows = keys (the K dimension of dQ += dS K)
            const uint64_t mK0 = tc::smem_desc_sw128(sbase + LY::K_OFF, SUB, 1024);
            constexpr uint32_t kStep = LY::OPB >> 4;
            auto issue_ab = [&](int j) -> bool {  // [S; R] and D of key tile j into Y
                const int ks = j % KS, vs = j % VS;
                if (*abort_flag || !mbar_wait_warp(&k_full[ks], (j / KS) & 1, &g_bwd_err) ||
                    !mbar_wait_warp(&v_full[vs], (j / VS) & 1, &g_bwd_err))
                    return false;
                tc::fence_after_sync();
                const uint64_t dK = tc::opaque(dK0 + ks * kStep);
                const uint64_t dV = tc::opaque(dV0 + vs * kStep);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {  // [S; R] = [Q; rho] K^T, A from TMEM
                    const uint32_t off = ((kk / 4) * SUB + (kk % 4) * 32) >> 4;
                    tc::mma_ts(tmem, tmem + LY::QA + 8 * kk, dK + off, kIdesc1, kk > 0);
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {  // D = dO V^T
                    const uint32_t offA = ((kk / 4) * SUB64 + (kk % 4) * 32) >> 4;
                    const uint32_t offB = ((kk / 4) * SUB + (kk % 4) * 32) >> 4;
                    tc::mma_ss(tmem + LY::YD, dDO + offA, dV + offB, kIdescD, kk > 0);
                }
                tc::commit(s_full);
                tc::commit(&v_empty[vs]);
                return true;
            };
            bool ok = mbar_wait_warp(q_full, 0, &g_bwd_err) && mbar_wait_warp(qr_in, 0, &g_bwd_err);
            if (ok) ok = issue_ab(0);
            for (int t = 0; t < n_t && ok; ++t) {
                if (t + 1 < n_t) {  // the next tile's S|R and D as soon as Y is free
                    if (!mbar_wait_warp(y_free, t & 1, &g_bwd_err)) {
                        ok = false;
                        break;
                    }
                    if (!(ok = issue_ab(t + 1))) break;
                }
                if (!mbar_wait_warp(p_full, t & 1, &g_bwd_err)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const uint64_t mK = tc::opaque(mK0 + (t % KS) * kStep);
                const uint32_t pk = LY::PK;
#pragma unroll
                for (int kk = 0; kk < Q_KT / 16; ++kk)  // [dQ; drho] += [dS; dR] K
                    tc::mma_ts(tmem + LY::O, tmem + pk + 8 * kk, mK + ((kk * 16 * 128) >> 4),
                               kIdesc2, (t > 0 || kk > 0) ? 1u : 0u);
                tc::commit(&k_empty[t % KS]);
                tc::commit(pk_empty);
            }
            tc::commit(o_full);
            if (!ok) {
                *abort_flag = 1;
                mbar_wait_warp(o_full, 0, &g_bwd_err);
            }
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------------- compute + epilogue
        const int g = warp & 3;
        const int set = (warp - 4) >> 2;               // key columns 64 set .. 64 set + 63
        const int h = lane >> 4;                       // which half of those
        const int i = q0 + 16 * g + (lane & 15);       // query row
        const uint32_t rowS = tmem + ((uint32_t)(32 * g) << 16);
        const uint32_t rowR = tmem + ((uint32_t)(32 * g + 16) << 16);
        const float qs = a.qscale, scale = a.scale;
        float4 z = make_float4(0.f, 0.f, 0.f, 0.f);  // (-lse2, 1 + rbar, abar, delta - abar)
        if (i < a.L) {
            const float* zr = a.rs + (size_t)bh * 4 * a.Lp + i;
            z = make_float4(zr[0], zr[a.Lp], zr[2 * (size_t)a.Lp], zr[3 * (size_t)a.Lp]);
        }
        bool ok = !skip;
        if (set == 0) {
            // [Q; rho] -> TMEM: lane = operand row, column x holds elements 2x, 2x + 1
            const int orow = 32 * g + lane;
            const bool got = ok && mbar_wait(q_full, 0, &g_bwd_err);
            if (__all_sync(kFullMask, got)) {
#pragma unroll 1
                for (int cb = 0; cb < LY::NCB; ++cb) {
                    uint32_t u[32];
                    const unsigned char* src = smem + LY::QR_OFF + cb * SUB + orow * 128;
#pragma unroll
                    for (int x = 0; x < 8; ++x) {
                        const uint4 q = *reinterpret_cast<const uint4*>(src + ((x ^ (orow & 7)) * 16));
                        u[4 * x] = q.x;
                        u[4 * x + 1] = q.y;
                        u[4 * x + 2] = q.z;
                        u[4 * x + 3] = q.w;
                    }
                    tc::tmem_st32(rowS + LY::QA + 32 * cb, u);
                }
                tc::tmem_st_wait();
            } else {
                ok = false;
                *abort_flag = 1;
            }
            tc::fence_before_sync();
            mbar_arrive(qr_in);
        }
        for (int t = 0; t < n_t && ok; ++t) {
            const bool got = !*abort_flag && mbar_wait(s_full, t & 1, &g_bwd_err);
            if (!__all_sync(kFullMask, got)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            uint32_t sv[32], rv[32], dv[32];
            tc::tmem_ld32_split<32>(rowS + 64 * set, sv);
            if (RHO) tc::tmem_ld32_split<32>(rowR + 64 * set, rv);
            tc::tmem_ld32_split<32>(rowS + LY::YD + 64 * set, dv);
            tc::tmem_ld_wait();
            tc::fence_before_sync();
            mbar_arrive(y_free);  // the next tile's MMAs may overwrite Y
            const int k0 = t * Q_KT + 64 * set + 32 * h;
            // keys past L or (causal) past this query get no weight
            const int lim = min(a.L - 1, CAUSAL ? i : a.L - 1) - k0;  // last valid x
            const uint32_t vmask = i >= a.L || lim < 0 ? 0u
                                   : lim >= 31     ? 0xffffffffu
                                                   : ((2u << lim) - 1u);
            const float2 qs2 = make_float2(qs, qs), nsc2 = make_float2(-scale, -scale);
            const float2 nl2 = make_float2(z.x, z.x), rb2 = make_float2(z.y, z.y);
            const float2 ab2 = make_float2(z.z, z.z), ne2 = make_float2(z.w, z.w);
            uint32_t spk[16], rpk[16];
            auto run = [&](auto masked) {
                constexpr bool M = decltype(masked)::value;
#pragma unroll
                for (int y = 0; y < 16; ++y) {
                    const int x = 2 * y;
                    const float2 s2 = make_float2(__uint_as_float(sv[x]), __uint_as_float(sv[x + 1]));
                    const float2 r2 = RHO ? make_float2(__uint_as_float(rv[x]), __uint_as_float(rv[x + 1]))
                                          : make_float2(0.f, 0.f);
                    const float2 d2 = make_float2(__uint_as_float(dv[x]), __uint_as_float(dv[x + 1]));
                    const PairTerms pt = pair_terms<M, false>(s2, r2, d2, qs2, nl2, rb2, ab2, ne2, nsc2,
                                                              (vmask >> x) & 1u, (vmask >> (x + 1)) & 1u);
                    spk[y] = tc::pack_bf16(pt.ds.x, pt.ds.y);
                    rpk[y] = tc::pack_bf16(pt.dr.x, pt.dr.y);
                }
            };
            // warp-uniform: every (query, key) pair of the warp's columns is visible
            if (__all_sync(kFullMask, vmask == 0xffffffffu))
                run(std::false_type{});
            else
                run(std::true_type{});
            // the packed slot was read by the dQ MMAs of tile t - 1
            const bool slot_free = t < 1 || (!*abort_flag && mbar_wait(pk_empty, (t - 1) & 1, &g_bwd_err));
            if (!__all_sync(kFullMask, slot_free)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            // packed slot (keys 2c, 2c+1 at column c): dS in the query lanes, dR in the probe lanes
            const uint32_t pk = LY::PK + 32 * set;
            tc::tmem_st16_split<16>(rowS + pk, spk);
            tc::tmem_st16_split<16>(rowR + pk, rpk);
            tc::tmem_st_wait();
            tc::fence_before_sync();
            mbar_arrive(p_full);
        }
        const bool done = ok && !*abort_flag && mbar_wait(o_full, 0, &g_bwd_err);
        // set 0 stages dQ (query lanes), set 1 drho (probe lanes): columns h D/2 + 32 b of
        // row rl go to the [64 queries x 32 columns] box h (D/64) + b of the set
        const int rl = 16 * g + (lane & 15);
        unsigned char* stage = smem + LY::K_OFF + set * (D / 32) * LY::OUT_BOX;
        if (__all_sync(kFullMask, done)) {
            tc::fence_after_sync();
            if (set == 0 || RHO) {
                const uint32_t base = (set == 0 ? rowS : rowR) + LY::O;
                uint32_t uu[D / 64][32];  // this thread's half row behind one wait
#pragma unroll
                for (int b = 0; b < D / 64; ++b) tc::tmem_ld32_split<D / 2>(base + 32 * b, uu[b]);
                tc::tmem_ld_wait();
#pragma unroll
                for (int b = 0; b < D / 64; ++b) {
                    const uint32_t(&u)[32] = uu[b];
                    unsigned char* box = stage + (h * (D / 64) + b) * LY::OUT_BOX + rl * 128;
#pragma unroll
                    for (int x = 0; x < 8; ++x)
                        st_shared_v4(smem_u32(box + ((x ^ (rl & 7)) << 4)), u[4 * x], u[4 * x + 1],
                                     u[4 * x + 2], u[4 * x + 3]);
                }
            }
        } else {
            *abort_flag = 1;
        }
        // every compute thread arrives, whichever way it went; one thread then stores the
        // tile's rows (rows past L are clipped by the tensor maps)
        fence_proxy_async_smem();
        mbar_arrive(staged);
        if (warp == 4 && lane == 0 && mbar_wait(staged, 0, &g_bwd_err) && !*abort_flag) {
            unsigned char* st0 = smem + LY::K_OFF;
#pragma unroll 1
            for (int b = 0; b < D / 32; ++b) {
                tc::tma_store_3d(&tmDQ, 32 * b, q0, bh, st0 + b * LY::OUT_BOX);
                if (RHO) tc::tma_store_3d(&tmDR, 32 * b, q0, bh, st0 + (D / 32 + b) * LY::OUT_BOX);
            }
            tc::bulk_commit_group();
            tc::bulk_wait_group_read0();
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------------ host side
bool make_map(CUtensorMap* m, const void* base, int BH, int L, int D, int box_rows) {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)L, (uint64_t)BH};
    const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)L * D * 2};
    const uint32_t box[3] = {64, (uint32_t)box_rows, 1};
    return make_tmap_bf16(m, base, 3, dims, strides, box);
}

template <int D, bool CAUSAL, bool RHO>
cudaError_t launch_all(const BwdArgs& a, const void* q, const void* rho, const void* k,
                       const void* v, cudaStream_t stream) {
    CUtensorMap q32, r32, k128, v128, o32, q16, r16;
    if (!make_map(&q32, q, a.BH, a.L, D, 64) || !make_map(&k128, k, a.BH, a.L, D, 128) ||
        !make_map(&v128, v, a.BH, a.L, D, 128) || !make_map(&o32, a.dout, a.BH, a.L, D, 64) ||
        !make_map(&q16, q, a.BH, a.L, D, 16))
        return cudaErrorInvalidValue;
    if (RHO) {
        if (!make_map(&r32, rho, a.BH, a.L, D, 64) || !make_map(&r16, rho, a.BH, a.L, D, 16))
            return cudaErrorInvalidValue;
    } else {
        r32 = q32;
        r16 = q16;
    }
    // the fp32 gradients [BH, L, D] for the epilogues' TMA stores: boxes of 32 columns x 128
    // keys (dK, dV) or x 64 queries (dQ, drho)
    CUtensorMap dk128, dv128, dq64, dr64;
    auto grad_map = [&](CUtensorMap* m, const float* base, int rows) {
        const uint64_t dims[3] = {(uint64_t)D, (uint64_t)a.L, (uint64_t)a.BH};
        const uint64_t strides[2] = {(uint64_t)D * 4, (uint64_t)a.L * D * 4};
        const uint32_t box[3] = {32, (uint32_t)rows, 1};
        return make_tmap_f32(m, base, 3, dims, strides, box);
    };
    if (!grad_map(&dk128, a.dk, 128) || !grad_map(&dv128, a.dv, 128) ||
        !grad_map(&dq64, a.dq, 64) || !grad_map(&dr64, RHO ? a.drho : a.dq, 64))
        return cudaErrorInvalidValue;
    static std::atomic<uint64_t> kv_smem_set{0}, q_smem_set{0};
    cudaError_t e = ensure_dynamic_smem(bwd_kv_kernel<D, CAUSAL, RHO>, KvLayout<D>::SMEM_BYTES,
                                        kv_smem_set);
    if (e == cudaSuccess)
        e = ensure_dynamic_smem(bwd_q_kernel<D, CAUSAL, RHO>, QLayout<D>::SMEM_BYTES, q_smem_set);
    if (e != cudaSuccess) return e;
    const size_t rows = (size_t)a.BH * a.Lp;
    bwd_pre_kernel<D><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(a);
    bwd_kv_kernel<D, CAUSAL, RHO><<<(unsigned)((size_t)a.n_kt * a.BH), kKvThreads,
                                    KvLayout<D>::SMEM_BYTES, stream>>>(q32, r32, k128, v128, o32,
                                                                       dv128, dk128, a);
    bwd_q_kernel<D, CAUSAL, RHO><<<(unsigned)((size_t)a.n_qt * a.BH), kThreads,
                                   QLayout<D>::SMEM_BYTES, stream>>>(q16, r16, k128, v128, o32,
                                                                     dq64, dr64, a);
    return cudaGetLastError();
}

}  // namespace

size_t prefill_backward_workspace_bytes(int B, int H, int L) {
    return (size_t)B * H * 4 * ((L + 63) / 64 * 64) * sizeof(float);
}

cudaError_t prefill_backward_launch(const PrefillShape& s, const void* q, const void* rho,
                                    const void* k, const void* v, const float* o,
                                    const float* mu, const float* lse, const float* rbar,
                                    const void* dout, float* dq, float* drho, float* dk,
                                    float* dv, void* ws, cudaStream_t stream) {
    BwdArgs a;
    a.o = o;
    a.mu = mu;
    a.dout = static_cast<const __nv_bfloat16*>(dout);
    a.lse = lse;
    a.rbar = rbar;
    a.rs = static_cast<float*>(ws);
    a.dq = dq;
    a.drho = drho;
    a.dk = dk;
    a.dv = dv;
    a.L = s.L;
    a.BH = s.B * s.H;
    a.Lp = (s.L + 63) / 64 * 64;
    a.n_kt = (s.L + 127) / 128;
    a.n_qt = (s.L + 63) / 64;
    a.scale = s.scale;
    a.qscale = s.scale * kLog2e;
    const bool r = rho != nullptr;
#define PARALLAX_BWD_CASE(DD)                                                                   \
    if (s.d == DD) {                                                                            \
        if (s.causal)                                                                           \
            return r ? launch_all<DD, true, true>(a, q, rho, k, v, stream)                      \
                     : launch_all<DD, true, false>(a, q, rho, k, v, stream);                    \
        return r ? launch_all<DD, false, true>(a, q, rho, k, v, stream)                         \
                 : launch_all<DD, false, false>(a, q, rho, k, v, stream);                       \
    }
    PARALLAX_BWD_CASE(64)
    PARALLAX_BWD_CASE(128)
#undef PARALLAX_BWD_CASE
    return cudaErrorInvalidValue;
}

unsigned prefill_backward_take_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_bwd_err, sizeof(v)) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_bwd_err, &zero, sizeof(zero));
    return v;
}

}  // namespace parallax
