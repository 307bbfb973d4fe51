// Parallax prefill on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// One CTA computes a 128-query tile of one head.  For every 128-key tile of
// K and V (fetched once by TMA and shared by both branches -- the pages' "same
// KV stream for both branches", "Parallax mantem softmax ...", paragraph 2):
//
//   MMA-1   S = Q K^T   and   R = rho K^T            (bf16 in, fp32 in TMEM)
//   softmax P = 2^(S*scale*log2e - m)  (row max m, lazily rescaled),
//           PR = P o (R - c)           (c: per-row shift, see below)
//   MMA-2   U += P V    and   W += PR V               (P, PR read from TMEM)
//
// and at the end o = U/l - (W/l - (A/l)(U/l)) with l = sum P, A = sum PR.
//
// Roles (192 threads): warp 0 issues TMA loads, warp 1 owns TMEM and issues
// the MMAs (one elected thread), warps 2-5 (one TMEM lane quarter each, one
// query row per thread) do the softmax, the correction-branch elementwise
// work and the epilogue.
//
// TMEM (512 columns x 128 lanes): S [0,128), R [128,256), U [256,256+d),
// W [256+d, 256+2d).  P (bf16) overwrites S columns [0,64) and PR overwrites R
// columns [0,64) after the softmax threads have read S and R.
//
// Numerics:
//  * the row shift c (Cov_p(r - c, v) = Cov_p(r, v) for any constant c) is set
//    to the p-weighted mean of r over the first key tile processed, so PR is
//    centred and its bf16 rounding error stays proportional to the spread of
//    r rather than its size.  Key tiles are processed in order 0, 1, ..., with
//    the causal diagonal tile last, so that the first tile is a full one and c
//    is a mean over 128 keys (for the first query tile it is the only tile);
//  * rows that see few keys (the first query tile of a causal head, or a
//    non-causal head with L <= 128) also feed the bf16 rounding residual of PR
//    (PR - bf16(PR), stored in S columns [64,128)) through one more MMA, so the
//    correction branch is accurate to ~2^-16 there;
//  * the running max m is only moved when a tile's max exceeds it by more
//    than 2^8 (lazy rescale); the final normalisation uses the same m, so the
//    result is exact in exact arithmetic.
#include "tcgen05.cuh"
#include "kernels.h"

namespace parallax {
namespace {

__device__ unsigned g_tc_err = 0;

constexpr int BM = 128;  // queries per tile
constexpr int BN = 128;  // keys per tile
constexpr int kThreads = 192;
constexpr int kStages = 2;
constexpr float kRescaleThreshold = 8.f;  // log2 units

template <int D, bool RHO>
struct TcLayout {
    static constexpr int SUB = D / 64;                // 128-byte swizzle column blocks per row
    static constexpr int SUB_BYTES = BM * 128;        // one [128 rows x 64] bf16 block
    static constexpr int TILE_BYTES = BM * D * 2;     // one [128 x D] bf16 tile
    static constexpr int Q_OFF = 0;
    static constexpr int RHO_OFF = Q_OFF + TILE_BYTES;
    static constexpr int KV_OFF = RHO_OFF + (RHO ? TILE_BYTES : 0);
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K then V
    static constexpr int BAR_OFF = KV_OFF + kStages * STAGE_BYTES;
    static constexpr int NBARS = 1 + 3 * kStages + 3;
    static constexpr int SMEM_BYTES = BAR_OFF + NBARS * 8 + 16 + 1024;  // + alignment slack
    static constexpr uint32_t S_COL = 0;
    static constexpr uint32_t R_COL = 128;
    static constexpr uint32_t U_COL = RHO ? 256 : 128;
    static constexpr uint32_t W_COL = U_COL + D;
    static constexpr uint32_t TMEM_COLS = RHO ? 512 : 256;
};

struct TcArgs {
    float* o;
    int L;
    int BH;
    int n_qt;
    float qscale;  // scale * log2(e)
};

__device__ __forceinline__ void tmem_scale_cols(uint32_t addr, int ncols, float alpha) {
    for (int c0 = 0; c0 < ncols; c0 += 32) {
        uint32_t v[32];
        tc::tmem_ld32(addr + c0, v);
        tc::tmem_ld_wait();
#pragma unroll
        for (int x = 0; x < 32; ++x) v[x] = __float_as_uint(__uint_as_float(v[x]) * alpha);
        tc::tmem_st32(addr + c0, v);
    }
}

template <int D, bool RHO, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmR,
                      const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const TcArgs a) {
    using LY = TcLayout<D, RHO>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LY::BAR_OFF);
    uint64_t* q_full = bars;
    uint64_t* k_full = bars + 1;
    uint64_t* v_full = k_full + kStages;
    uint64_t* kv_empty = v_full + kStages;
    uint64_t* s_full = kv_empty + kStages;
    uint64_t* p_full = s_full + 1;
    uint64_t* o_full = s_full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + LY::NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int tile = blockIdx.x;
    // heaviest (most key tiles) first when causal
    const int qt = CAUSAL ? a.n_qt - 1 - tile / a.BH : tile / a.BH;
    const int bh = tile % a.BH;
    const int q0 = qt * BM;
    const int n_kv = CAUSAL ? qt + 1 : (a.L + BN - 1) / BN;
    const bool precise = RHO && (CAUSAL ? qt == 0 : n_kv == 1);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&v_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(p_full, 128);
        mbar_init(o_full, 1);
        *abort_flag = (*(volatile unsigned*)&g_tc_err & PARALLAX_DEVERR_WAIT_TIMEOUT) ? 1 : 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tmap(&tmQ);
        tc::prefetch_tmap(&tmK);
        tc::prefetch_tmap(&tmV);
        if (RHO) tc::prefetch_tmap(&tmR);
    }
    if (warp == 1) tc::tmem_alloc(tmem_slot, LY::TMEM_COLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const bool skip = *abort_flag != 0;

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0 && !skip) {
            const int z = bh;
            int it = 0;
            bool ok = true;
            mbar_arrive_expect_tx(q_full, (RHO ? 2 : 1) * LY::TILE_BYTES);
#pragma unroll
            for (int sub = 0; sub < LY::SUB; ++sub) {
                tc::tma_load_3d(smem + LY::Q_OFF + sub * LY::SUB_BYTES, &tmQ, sub * 64, q0, z, q_full);
                if (RHO)
                    tc::tma_load_3d(smem + LY::RHO_OFF + sub * LY::SUB_BYTES, &tmR, sub * 64, q0, z,
                                    q_full);
            }
            for (; it < n_kv; ++it) {
                const int j = it;
                const int s = it % kStages;
                if (it >= kStages &&
                    !mbar_wait(&kv_empty[s], ((it / kStages) - 1) & 1, &g_tc_err)) {
                    ok = false;
                    break;
                }
                unsigned char* kb = smem + LY::KV_OFF + s * LY::STAGE_BYTES;
                unsigned char* vb = kb + LY::TILE_BYTES;
                mbar_arrive_expect_tx(&k_full[s], LY::TILE_BYTES);
#pragma unroll
                for (int sub = 0; sub < LY::SUB; ++sub)
                    tc::tma_load_3d(kb + sub * LY::SUB_BYTES, &tmK, sub * 64, j * BN, z, &k_full[s]);
                mbar_arrive_expect_tx(&v_full[s], LY::TILE_BYTES);
#pragma unroll
                for (int sub = 0; sub < LY::SUB; ++sub)
                    tc::tma_load_3d(vb + sub * LY::SUB_BYTES, &tmV, sub * 64, j * BN, z, &v_full[s]);
            }
            if (!ok) {
                *abort_flag = 1;
                // wait (bounded) for the copies already issued into this CTA's shared memory
                mbar_wait(q_full, 0, &g_tc_err);
                for (int k = (it >= kStages ? it - kStages : 0); k < it; ++k) {
                    mbar_wait(&k_full[k % kStages], (k / kStages) & 1, &g_tc_err);
                    mbar_wait(&v_full[k % kStages], (k / kStages) & 1, &g_tc_err);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0 && !skip) {
            constexpr uint32_t kIdescS = tc::idesc_bf16_f32(BM, BN, false);
            constexpr uint32_t kIdescV = tc::idesc_bf16_f32(BM, D, true);
            bool ok = mbar_wait(q_full, 0, &g_tc_err);
            tc::fence_after_sync();
            // Descriptors are built once; a K-step only adds a constant to the
            // start-address field (bits 0..13, in 16-byte units).
            const uint64_t dQ = tc::smem_desc_sw128(smem_u32(smem + LY::Q_OFF), 16, 1024);
            const uint64_t dR = tc::smem_desc_sw128(smem_u32(smem + LY::RHO_OFF), 16, 1024);
            const uint32_t kv0 = smem_u32(smem + LY::KV_OFF);
            for (int it = 0; it < n_kv && ok; ++it) {
                const int s = it % kStages;
                const uint32_t ph = (it / kStages) & 1;
                const uint32_t sK = kv0 + s * LY::STAGE_BYTES;
                const uint64_t dK = tc::smem_desc_sw128(sK, 16, 1024);
                const uint64_t dV = tc::smem_desc_sw128(sK + LY::TILE_BYTES, LY::SUB_BYTES, 1024);
                if (!mbar_wait(&k_full[s], ph, &g_tc_err)) { ok = false; break; }
                tc::fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk / 4) * LY::SUB_BYTES + (kk % 4) * 32) >> 4;
                    tc::mma_ss(tmem + LY::S_COL, dQ + off, dK + off, kIdescS, kk > 0);
                    if (RHO) tc::mma_ss(tmem + LY::R_COL, dR + off, dK + off, kIdescS, kk > 0);
                }
                tc::commit(s_full);
                if (!mbar_wait(p_full, it & 1, &g_tc_err)) { ok = false; break; }
                tc::fence_after_sync();
                if (!mbar_wait(&v_full[s], ph, &g_tc_err)) { ok = false; break; }
                tc::fence_after_sync();
                const uint32_t acc0 = it > 0 ? 1u : 0u;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    // 16 keys = 16 rows of 128 bytes in each 64-column block; the second
                    // column block of V (d >= 64) sits LBO = one block further on.
                    const uint32_t off = (kk * 16 * 128) >> 4;
                    const uint32_t acc = kk > 0 ? 1u : acc0;
                    tc::mma_ts(tmem + LY::U_COL, tmem + LY::S_COL + kk * 8, dV + off, kIdescV, acc);
                    if (RHO) {
                        tc::mma_ts(tmem + LY::W_COL, tmem + LY::R_COL + kk * 8, dV + off, kIdescV, acc);
                        if (precise)
                            tc::mma_ts(tmem + LY::W_COL, tmem + LY::S_COL + 64 + kk * 8, dV + off,
                                       kIdescV, 1u);
                    }
                }
                tc::commit(&kv_empty[s]);
            }
            tc::commit(o_full);
            if (!ok) {
                *abort_flag = 1;
                mbar_wait(o_full, 0, &g_tc_err);  // MMAs already issued have drained
            }
        }
    } else {
        // ---------------------------------------------------------------- softmax / epilogue
        const int quarter = warp % 4;  // TMEM lanes this warp may touch
        const int row = quarter * 32 + lane;
        const int i = q0 + row;
        const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
        const float qscale = a.qscale;
        float m = -INFINITY, l = 0.f, A = 0.f, c = 0.f;
        bool ok = !skip;
        for (int it = 0; it < n_kv && ok; ++it) {
            const int k0 = it * BN;
            const bool got = !*abort_flag && mbar_wait(s_full, it & 1, &g_tc_err);
            if (!__all_sync(kFullMask, got)) { ok = false; break; }  // warp-uniform exit
            tc::fence_after_sync();
            uint32_t sv[4][32];
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) tc::tmem_ld32(taddr + LY::S_COL + ch * 32, sv[ch]);
            tc::tmem_ld_wait();

            // scale, mask, tile max
            const bool need_mask = (k0 + BN > a.L) || (CAUSAL && k0 + BN > q0);
            float mx = -INFINITY;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch)
#pragma unroll
                for (int x = 0; x < 32; ++x) {
                    float f = __uint_as_float(sv[ch][x]) * qscale;
                    if (need_mask) {
                        const int key = k0 + ch * 32 + x;
                        const bool valid = key < a.L && (!CAUSAL || key <= i);
                        f = valid ? f : -INFINITY;
                    }
                    sv[ch][x] = __float_as_uint(f);
                    mx = fmaxf(mx, f);
                }
            if (it == 0) {
                m = mx;
            } else if (__any_sync(kFullMask, mx > m + kRescaleThreshold)) {
                // the TMEM accesses are warp-collective, so the whole warp rescales;
                // rows whose max did not grow keep alpha = 1
                const float m_new = fmaxf(m, mx);
                const float alpha = fast_exp2(m - m_new);
                l *= alpha;
                A *= alpha;
                tmem_scale_cols(taddr + LY::U_COL, D, alpha);
                if (RHO) tmem_scale_cols(taddr + LY::W_COL, D, alpha);
                m = m_new;
            }

            // P = 2^(s - m), row sum, P -> bf16 into S columns [0, 64)
            float lsum = 0.f;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t packed[16];
#pragma unroll
                for (int x = 0; x < 32; ++x) {
                    const float p = fast_exp2(__uint_as_float(sv[ch][x]) - m);
                    sv[ch][x] = __float_as_uint(p);
                    lsum += p;
                }
#pragma unroll
                for (int y = 0; y < 16; ++y)
                    packed[y] = tc::pack_bf16(__uint_as_float(sv[ch][2 * y]),
                                              __uint_as_float(sv[ch][2 * y + 1]));
                tc::tmem_st16(taddr + LY::S_COL + ch * 16, packed);
            }
            l += lsum;

            if (RHO) {
                if (it == 0) {  // row shift: p-weighted mean of r over this first tile
                    float prs = 0.f;
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        uint32_t rr[32];
                        tc::tmem_ld32(taddr + LY::R_COL + ch * 32, rr);
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int x = 0; x < 32; ++x)
                            prs = fmaf(__uint_as_float(sv[ch][x]), __uint_as_float(rr[x]), prs);
                    }
                    c = prs / lsum;
                }
                float asum = 0.f;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t rr[32];
                    tc::tmem_ld32(taddr + LY::R_COL + ch * 32, rr);
                    tc::tmem_ld_wait();
                    float pr[32];
#pragma unroll
                    for (int x = 0; x < 32; ++x) {
                        pr[x] = __uint_as_float(sv[ch][x]) * (__uint_as_float(rr[x]) - c);
                        asum += pr[x];
                    }
                    uint32_t hi[16];
#pragma unroll
                    for (int y = 0; y < 16; ++y) hi[y] = tc::pack_bf16(pr[2 * y], pr[2 * y + 1]);
                    // columns [16ch, 16ch+16) of R were read above (chunk ch/2 <= ch)
                    tc::tmem_st16(taddr + LY::R_COL + ch * 16, hi);
                    if (precise) {
                        uint32_t lo[16];
#pragma unroll
                        for (int y = 0; y < 16; ++y)
                            lo[y] = tc::pack_bf16(pr[2 * y] - tc::bf16_lo_to_f32(hi[y]),
                                                  pr[2 * y + 1] - tc::bf16_hi_to_f32(hi[y]));
                        tc::tmem_st16(taddr + LY::S_COL + 64 + ch * 16, lo);
                    }
                }
                A += asum;
            }
            tc::tmem_st_wait();
            tc::fence_before_sync();
            mbar_arrive(p_full);
        }

        // ---- epilogue: o = U/l - (W/l - (A/l)(U/l))
        const bool done = ok && !*abort_flag && mbar_wait(o_full, 0, &g_tc_err);
        if (__all_sync(kFullMask, done)) {
            tc::fence_after_sync();
            const float inv_l = 1.f / l;
            const float rbar = A * inv_l;
            float* orow = a.o + ((size_t)bh * a.L + i) * D;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t u[32], w[32];
                tc::tmem_ld32(taddr + LY::U_COL + c0, u);
                if (RHO) tc::tmem_ld32(taddr + LY::W_COL + c0, w);
                tc::tmem_ld_wait();
                if (i < a.L) {
#pragma unroll
                    for (int x = 0; x < 32; x += 4) {
                        float out[4];
#pragma unroll
                        for (int y = 0; y < 4; ++y) {
                            const float mu = __uint_as_float(u[x + y]) * inv_l;
                            out[y] = RHO ? mu - (__uint_as_float(w[x + y]) * inv_l - rbar * mu) : mu;
                        }
                        *reinterpret_cast<float4*>(orow + c0 + x) =
                            make_float4(out[0], out[1], out[2], out[3]);
                    }
                }
            }
        } else {
            *abort_flag = 1;
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, LY::TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult qres;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &qres) == cudaSuccess &&
            qres == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// [B*H, L, D] bf16 viewed as a 3-D tensor; box = 64 columns (128 bytes) x 128 rows x 1 head,
// 128-byte swizzle; rows past L read as zeros.
bool make_map(CUtensorMap* m, const void* base, int BH, int L, int D) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)L, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)L * D * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool RHO, bool CAUSAL>
cudaError_t launch(const CUtensorMap& mq, const CUtensorMap& mr, const CUtensorMap& mk,
                   const CUtensorMap& mv, const TcArgs& a, cudaStream_t stream) {
    using LY = TcLayout<D, RHO>;
    auto kern = prefill_tc_kernel<D, RHO, CAUSAL>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             LY::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const unsigned grid = (unsigned)((size_t)a.n_qt * a.BH);
    kern<<<grid, kThreads, LY::SMEM_BYTES, stream>>>(mq, mr, mk, mv, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t prefill_tc_launch(const PrefillShape& s, const void* q, const void* rho,
                              const void* k, const void* v, float* o, int /*num_sms*/,
                              cudaStream_t stream) {
    const int BH = s.B * s.H;
    CUtensorMap mq, mr, mk, mv;
    if (!make_map(&mq, q, BH, s.L, s.d) || !make_map(&mk, k, BH, s.L, s.d) ||
        !make_map(&mv, v, BH, s.L, s.d))
        return cudaErrorInvalidValue;
    if (rho) {
        if (!make_map(&mr, rho, BH, s.L, s.d)) return cudaErrorInvalidValue;
    } else {
        mr = mq;
    }
    TcArgs a{o, s.L, BH, (s.L + BM - 1) / BM, s.scale * kLog2e};
    const bool r = rho != nullptr;
#define PARALLAX_TC_CASE(DD)                                                               \
    if (s.d == DD) {                                                                       \
        if (r) return s.causal ? launch<DD, true, true>(mq, mr, mk, mv, a, stream)         \
                               : launch<DD, true, false>(mq, mr, mk, mv, a, stream);       \
        return s.causal ? launch<DD, false, true>(mq, mr, mk, mv, a, stream)               \
                        : launch<DD, false, false>(mq, mr, mk, mv, a, stream);             \
    }
    PARALLAX_TC_CASE(64)
    PARALLAX_TC_CASE(128)
#undef PARALLAX_TC_CASE
    return cudaErrorInvalidValue;
}

unsigned prefill_tc_take_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_err, sizeof(v)) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_tc_err, &zero, sizeof(zero));
    return v;
}

}  // namespace parallax
