// Input projections of a Parallax layer on the tcgen05 tensor cores (sm_103a):
// q, k, v and the probe rho = W_R x ("Parallax mantem softmax ...", paragraph 2:
// the probe is a learned linear map of the layer input) as ONE product of the
// tokens x [B*L, width] with the stacked weight [W_q; W_k; W_v; W_R] of shape
// [n_out*H*d, width] (rows = output features, the usual linear-layer layout).
// Both operands are K-major, so both are fed by TMA with 128-byte swizzle
// straight into tcgen05.mma descriptors.  The epilogue converts the fp32
// accumulator to bf16 and scatters each 128-token x BN-feature tile into the
// head-major [B, H, L, d] tensors the attention kernels read.
//
// Persistent kernel, one CTA per SM, 6 warps:
//   warp 0      TMA producer: per 64-wide K block, the 128 x 64 token tile
//               and the BN x 64 weight tile into a STAGES-deep ring;
//   warp 1      TMEM owner and MMA issuer: 4 MMAs (M=128, N=BN, K=16) per K
//               block into one of two TMEM accumulators (2 x BN columns);
//   warps 2-5   epilogue: TMEM -> registers -> bf16 -> global, one token row
//               per thread; it drains accumulator i while the MMAs fill i^1.
// Tiles are ordered token-block-major: the CTAs resident at any time work on
// a few token blocks and all weight tiles, so the weight (33.5 MB at width
// 2048, H*d 2048) stays in L2 and each token block is read from HBM once.
// A token block never straddles two sequences: tiles are (b, 128-token block
// of sequence b), and rows past L are zero-filled by TMA and not stored.
#include "tcgen05.cuh"
#include "kernels.h"

namespace parallax {
namespace {

__device__ unsigned g_proj_err = 0;

constexpr int BM = 128;  // tokens per tile
constexpr int BK = 64;   // K block (one 128-byte swizzle atom of bf16)
constexpr int kThreads = 192;

template <int BN>
struct ProjLayout {
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = BN == 256 ? 4 : 6;
    static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
    // full[STAGES], empty[STAGES], acc_full[2], acc_empty[2], drain
    static constexpr int NBARS = 2 * STAGES + 5;
    static constexpr int SMEM_BYTES = BAR_OFF + NBARS * 8 + 16 + 1024;
    static constexpr uint32_t TMEM_COLS = 2 * BN;
};

struct ProjArgs {
    __nv_bfloat16* out[4];
    int L, H;
    int n_tiles_n;      // feature tiles (n_out * H * d / BN)
    int m_tiles_per_b;  // ceil(L / 128)
    int n_tiles;        // all tiles
    int kblocks;        // ceil(width / 64)
    size_t out_elems;   // B * H * L * d per output (debug bounds checks)
};

template <int BN, int D>
__global__ void __launch_bounds__(kThreads, 1)
    proj_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                const ProjArgs a) {
    using LY = ProjLayout<BN>;
    constexpr int S = LY::STAGES;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LY::BAR_OFF);
    uint64_t* full = bars;
    uint64_t* empty = bars + S;
    uint64_t* acc_full = bars + 2 * S;
    uint64_t* acc_empty = bars + 2 * S + 2;
    uint64_t* drain = bars + 2 * S + 4;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + LY::NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int hd = a.H * D;

    if (threadIdx.x == 0) {
        for (int b = 0; b < LY::NBARS; ++b)
            mbar_init(&bars[b], (b >= 2 * S + 2 && b < 2 * S + 4) ? 4 : 1);
        *abort_flag = (*(volatile unsigned*)&g_proj_err & PARALLAX_DEVERR_WAIT_TIMEOUT) ? 1 : 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tmap(&tmX);
        tc::prefetch_tmap(&tmW);
    }
    if (warp == 1) tc::tmem_alloc(tmem_slot, LY::TMEM_COLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const bool skip = *abort_flag != 0;

    auto tile_coords = [&](int t, int& b, int& l0, int& n0) {
        const int mt = t / a.n_tiles_n;
        n0 = (t - mt * a.n_tiles_n) * BN;
        b = mt / a.m_tiles_per_b;
        l0 = (mt - b * a.m_tiles_per_b) * BM;
    };

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0 && !skip) {
            uint32_t it = 0;  // stages issued
            bool ok = true;
            for (int t = blockIdx.x; t < a.n_tiles && ok; t += gridDim.x) {
                int b, l0, n0;
                tile_coords(t, b, l0, n0);
                for (int kb = 0; kb < a.kblocks; ++kb) {
                    const uint32_t st = it % S, round = it / S;
                    if (round > 0 && !mbar_wait(&empty[st], (round - 1) & 1, &g_proj_err)) {
                        ok = false;
                        break;
                    }
                    if (*abort_flag) {
                        ok = false;
                        break;
                    }
                    unsigned char* stage = smem + st * LY::STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[st], LY::STAGE_BYTES);
                    tc::tma_load_3d(stage, &tmX, kb * BK, l0, b, &full[st]);
                    tc::tma_load_2d(stage + LY::A_BYTES, &tmW, kb * BK, n0, &full[st]);
                    ++it;
                }
            }
            if (!ok) {
                *abort_flag = 1;
                // wait (bounded) for the copies still in flight into this CTA's shared memory
                for (uint32_t j = it > (uint32_t)S ? it - S : 0; j < it; ++j)
                    mbar_wait(&full[j % S], (j / S) & 1, &g_proj_err);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        // (the whole warp runs this; one elected lane issues each MMA and commit)
        if (!skip) {
            constexpr uint32_t kIdesc = tc::idesc_bf16_f32(BM, BN, false);
            const uint32_t sbase = smem_u32(smem);
            const uint64_t dA0 = tc::smem_desc_sw128(sbase, 16, 1024);
            const uint64_t dB0 = tc::smem_desc_sw128(sbase + LY::A_BYTES, 16, 1024);
            constexpr uint32_t kStageStep = LY::STAGE_BYTES >> 4;
            uint32_t it = 0;
            int local = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < a.n_tiles && ok; t += gridDim.x, ++local) {
                const int buf = local & 1, use = local >> 1;
                if (use > 0 && !mbar_wait_warp(&acc_empty[buf], (use - 1) & 1, &g_proj_err)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t dtm = tmem + (uint32_t)(buf * BN);
                for (int kb = 0; kb < a.kblocks; ++kb, ++it) {
                    const uint32_t st = it % S, round = it / S;
                    if (*abort_flag || !mbar_wait_warp(&full[st], round & 1, &g_proj_err)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint64_t dA = tc::opaque(dA0 + st * kStageStep);
                    const uint64_t dB = tc::opaque(dB0 + st * kStageStep);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        tc::mma_ss(dtm, dA + 2 * kk, dB + 2 * kk, kIdesc, (kb | kk) != 0);
                    tc::commit(&empty[st]);
                }
                if (!ok) break;
                tc::commit(&acc_full[buf]);
            }
            if (!ok) {
                *abort_flag = 1;
                tc::commit(drain);
                mbar_wait_warp(drain, 0, &g_proj_err);  // the MMAs already issued have drained
            }
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        const int q = warp & 3;            // TMEM lane quarter of this warp
        const int row = 32 * q + lane;     // token row of the tile
        const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
        int local = 0;
        bool ok = !skip;
        for (int t = blockIdx.x; t < a.n_tiles && ok; t += gridDim.x, ++local) {
            const int buf = local & 1, use = local >> 1;
            const bool got = !*abort_flag && mbar_wait(&acc_full[buf], use & 1, &g_proj_err);
            if (!__all_sync(kFullMask, got)) {
                *abort_flag = 1;
                ok = false;
                break;
            }
            tc::fence_after_sync();
            int b, l0, n0;
            tile_coords(t, b, l0, n0);
            const int which = n0 / hd;
            const int f0 = n0 - which * hd;  // first feature of the tile within its block
            const int l = l0 + row;
            __nv_bfloat16* base = which == 0 ? a.out[0] : which == 1 ? a.out[1]
                                : which == 2 ? a.out[2] : a.out[3];
#pragma unroll 1
            for (int ch = 0; ch < BN / 32; ch += 2) {
                uint32_t r0[32], r1[32];
                tc::tmem_ld32(trow + (uint32_t)(buf * BN + 32 * ch), r0);
                tc::tmem_ld32(trow + (uint32_t)(buf * BN + 32 * ch + 32), r1);
                tc::tmem_ld_wait();
                if (l < a.L) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const uint32_t(&r)[32] = e ? r1 : r0;
                        const int f = f0 + 32 * (ch + e);
                        const int h = f / D, c = f % D;
                        const size_t at = (((size_t)b * a.H + h) * a.L + l) * D + c;
                        if (!in_bounds(&g_proj_err, at + 32, a.out_elems)) continue;
                        uint4* dst = reinterpret_cast<uint4*>(base + at);
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            dst[v] = make_uint4(
                                tc::pack_bf16(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1])),
                                tc::pack_bf16(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3])),
                                tc::pack_bf16(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5])),
                                tc::pack_bf16(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7])));
                    }
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, LY::TMEM_COLS);
    }
}

template <int BN, int D>
cudaError_t launch(const CUtensorMap& mx, const CUtensorMap& mw, const ProjArgs& a, int num_sms,
                   cudaStream_t stream) {
    using LY = ProjLayout<BN>;
    auto kern = proj_kernel<BN, D>;
    static std::atomic<uint64_t> smem_set{0};
    if (cudaError_t e = ensure_dynamic_smem(kern, (int)LY::SMEM_BYTES, smem_set)) return e;
    const int grid = a.n_tiles < num_sms ? a.n_tiles : num_sms;
    kern<<<grid, kThreads, LY::SMEM_BYTES, stream>>>(mx, mw, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t proj_tc_launch(const ProjShape& s, const void* x, const void* w, void* const out[4],
                           int num_sms, cudaStream_t stream) {
    const int hd = s.H * s.d;
    const int BN = hd % 256 == 0 ? 256 : 128;
    if (hd % 128 != 0 || (s.d != 64 && s.d != 128) || s.width % 8 != 0)
        return cudaErrorInvalidValue;
    CUtensorMap mx, mw;
    {
        const uint64_t dims[3] = {(uint64_t)s.width, (uint64_t)s.L, (uint64_t)s.B};
        const uint64_t strides[2] = {(uint64_t)s.width * 2, (uint64_t)s.L * s.width * 2};
        const uint32_t box[3] = {BK, BM, 1};
        if (!make_tmap_bf16(&mx, x, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[2] = {(uint64_t)s.width, (uint64_t)s.n_out * hd};
        const uint64_t strides[1] = {(uint64_t)s.width * 2};
        const uint32_t box[2] = {BK, (uint32_t)BN};
        if (!make_tmap_bf16(&mw, w, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    ProjArgs a;
    for (int t = 0; t < 4; ++t)
        a.out[t] = static_cast<__nv_bfloat16*>(t < s.n_out ? out[t] : nullptr);
    a.L = s.L;
    a.H = s.H;
    a.n_tiles_n = s.n_out * hd / BN;
    a.m_tiles_per_b = (s.L + BM - 1) / BM;
    const long long tiles = (long long)s.B * a.m_tiles_per_b * a.n_tiles_n;
    if (tiles > 2147483647LL) return cudaErrorInvalidValue;
    a.n_tiles = (int)tiles;
    a.kblocks = (s.width + BK - 1) / BK;
    a.out_elems = (size_t)s.B * s.H * s.L * s.d;
    if (BN == 256)
        return s.d == 64 ? launch<256, 64>(mx, mw, a, num_sms, stream)
                         : launch<256, 128>(mx, mw, a, num_sms, stream);
    return s.d == 64 ? launch<128, 64>(mx, mw, a, num_sms, stream)
                     : launch<128, 128>(mx, mw, a, num_sms, stream);
}

unsigned proj_tc_take_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_proj_err, sizeof(v)) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_proj_err, &zero, sizeof(zero));
    return v;
}

}  // namespace parallax
