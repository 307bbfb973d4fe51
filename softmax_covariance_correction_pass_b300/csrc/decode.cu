// Parallax split-KV decode (one query token per sequence and head).
//
// Kernel 1 (decode_kernel): a persistent CTA walks work items (key/value
// head, key chunk).  One producer warp streams the chunk's K and V rows --
// contiguous in the [B, H_kv, Lmax, d] cache, or looked up page by page
// through a block table in a paged cache [num_pages, H_kv, page_size, d] --
// into a ring of shared-memory stages with bulk asynchronous copies
// (cp.async.bulk, completion on mbarriers, L2 evict-first).  Eight consumer
// warps update the online state of BOTH Parallax branches from the same bytes
// (Parallax, "Parallax mantem softmax ...", paragraph 2: one KV stream feeds
// the softmax and the covariance branch).  With G query heads per key/value
// head (grouped-query attention), the warps are split into G teams of 8/G
// warps; team g serves query head g of the group and each of its warps takes
// a 1/(8/G) share of every stage, so each K/V byte leaves HBM once for all G
// heads.  At the end of an item each team's warps merge their states in
// shared memory; the result is either the finished output (a single chunk per
// head) or a partial state (m, l, A, U, W) in the workspace.
// Kernel 2 (combine_kernel): per head, rescales the partial states to a common
// maximum (log-sum-exp), sums them and finishes o = U/l - (W/l - (A/l)(U/l)).
#include <mutex>

#include "tcgen05.cuh"
#include "warp_stream.cuh"
#include "kernels.h"

namespace parallax {
namespace {

__device__ unsigned g_decode_err = 0;

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
// Two CTAs per SM (18 warps) with 3 stages each: 192 KB of K/V in flight per SM and
// twice the warps of one CTA to hide the latency of the per-key dependency chains.
constexpr int kStages = 3;
constexpr int kCtasPerSm = 2;
constexpr int kStageRowBytes = 16384;  // bytes of K (and of V) per stage

constexpr int kMaxPageIds = 288;  // page ids of one work item held in shared memory

template <typename T, int D, int G = 1>
struct DecodeShape {
    using KL = KeyLayout<T, D>;
    static constexpr int STAGE_KEYS = kStageRowBytes / KL::ROW_BYTES;
    static constexpr int WARPS_PER_HEAD = kConsumerWarps / G;
    static constexpr int KEYS_PER_WARP = STAGE_KEYS / WARPS_PER_HEAD;
    static constexpr int BLOCKS_PER_WARP = KEYS_PER_WARP / KL::BLOCK_KEYS;
    static_assert(kConsumerWarps % G == 0, "group size must divide the consumer warps");
    static_assert(BLOCKS_PER_WARP >= 1 && KEYS_PER_WARP % KL::BLOCK_KEYS == 0, "stage shape");
    static constexpr int MERGE_FLOATS = kConsumerWarps * (4 + 2 * D);
    static constexpr size_t SMEM_BYTES = (size_t)kStages * 2 * kStageRowBytes +
                                         MERGE_FLOATS * sizeof(float) + 2 * kStages * 8 + 16 +
                                         kMaxPageIds * sizeof(int);
};

struct DecodeArgs {
    const void* q;
    const void* rho;
    const void* kc;
    const void* vc;
    const int32_t* seqlens;
    float* o;
    float4* ws_stats;  // [B*H][nsplit]   (m, l, A, -)
    float* ws_uw;      // [B*H][nsplit][2][D]
    const int32_t* block_table;  // paged cache: [B][max_pages] page ids
    int B, H, Hkv, Lmax, chunk, nsplit;
    int page_size, max_pages, num_pages;  // paged cache only
    float qscale;  // softmax scale * log2(e)
};

__device__ __forceinline__ int clamp_seqlen(const int32_t* seqlens, int b, int Lmax) {
    int n = seqlens[b];
    if (n < 0 || n > Lmax) {
        raise_error(&g_decode_err, PARALLAX_DEVERR_SEQLEN_CLAMPED);
        n = n < 0 ? 0 : Lmax;
    }
    return n;
}

// Item (key/value head bh, chunk ch) -> key range [start, end); returns false if the item
// is empty and produces nothing.  Without split every head has exactly one item (it may
// be empty: a zero-length sequence still writes o = 0).
__device__ __forceinline__ bool item_range(const DecodeArgs& a, int slot, int BH, int& bh,
                                           int& ch, int& start, int& end, bool split) {
    ch = slot / BH;
    bh = slot - ch * BH;
    const int n = clamp_seqlen(a.seqlens, bh / a.Hkv, a.Lmax);
    start = ch * a.chunk;
    end = min(start + a.chunk, n);
    return split ? start < n : true;
}

// A page id from the block table; an id outside [0, num_pages) is replaced by
// page 0 (so that no copy leaves the pool) and flagged.
__device__ __forceinline__ int checked_page(const DecodeArgs& a, int id) {
    if (id < 0 || id >= a.num_pages) {
        raise_error(&g_decode_err, PARALLAX_DEVERR_PAGE_OUT_OF_RANGE);
        return 0;
    }
    return id;
}

template <typename T, int D, bool RHO, bool SPLIT, int G, bool PAGED>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) decode_kernel(const DecodeArgs a) {
    using KL = KeyLayout<T, D>;
    using SH = DecodeShape<T, D, G>;
    constexpr int VEC = KL::VEC;
    extern __shared__ __align__(1024) unsigned char smem[];
    T* stage_k = reinterpret_cast<T*>(smem);                               // [kStages][STAGE_KEYS][D]
    T* stage_v = reinterpret_cast<T*>(smem + kStages * kStageRowBytes);    // [kStages][STAGE_KEYS][D]
    float* merge = reinterpret_cast<float*>(smem + 2 * kStages * kStageRowBytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(merge + SH::MERGE_FLOATS);
    uint64_t* empty = full + kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStages);
    int* page_ids = const_cast<int*>(abort_flag) + 4;  // [kMaxPageIds], producer only

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int BHkv = a.B * a.Hkv;
    const int total = BHkv * a.nsplit;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (*(volatile unsigned*)&g_decode_err & PARALLAX_DEVERR_WAIT_TIMEOUT) return;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        // Lane 0 issues every copy; with a paged cache the whole warp first
        // loads the item's page ids into shared memory.
        if (!PAGED && lane != 0) return;
        const uint64_t pol = l2_evict_first_policy();
        uint32_t it = 0;
        bool ok = true;
        for (int slot = blockIdx.x; slot < total && ok; slot += gridDim.x) {
            int bh, ch, start, end;
            if (!item_range(a, slot, BHkv, bh, ch, start, end, SPLIT)) continue;
            int p0 = 0, b = 0, hk = 0;
            if (PAGED) {
                b = bh / a.Hkv;
                hk = bh - b * a.Hkv;
                p0 = start / a.page_size;
                const int np = end > start ? (end - 1) / a.page_size - p0 + 1 : 0;
                for (int i = lane; i < np; i += 32)
                    page_ids[i] = checked_page(a, a.block_table[(size_t)b * a.max_pages + p0 + i]);
                __syncwarp();
            }
            if (lane == 0) {
                const size_t head = (size_t)bh * a.Lmax;
                for (int t0 = start; t0 < end; t0 += SH::STAGE_KEYS, ++it) {
                    const int s = it % kStages;
                    if (!mbar_wait(&empty[s], ((it / kStages) & 1) ^ 1, &g_decode_err)) {
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    const int nk = min(SH::STAGE_KEYS, end - t0);
                    mbar_arrive_expect_tx(&full[s], 2u * (uint32_t)nk * KL::ROW_BYTES);
                    T* dk = stage_k + (size_t)s * SH::STAGE_KEYS * D;
                    T* dv = stage_v + (size_t)s * SH::STAGE_KEYS * D;
                    if (!PAGED) {
                        const uint32_t bytes = (uint32_t)nk * KL::ROW_BYTES;
                        const size_t src =
                            in_bounds(&g_decode_err, (head + t0 + nk) * D, (size_t)BHkv * a.Lmax * D)
                                ? (head + t0) * D : 0;
                        bulk_copy_g2s(dk, static_cast<const T*>(a.kc) + src, bytes, &full[s], pol);
                        bulk_copy_g2s(dv, static_cast<const T*>(a.vc) + src, bytes, &full[s], pol);
                    } else {
                        // one copy per page the stage touches
                        for (int t = t0; t < t0 + nk;) {
                            const int pg = t / a.page_size, row = t - pg * a.page_size;
                            const int seg = min(a.page_size - row, t0 + nk - t);
                            size_t src =
                                (((size_t)page_ids[pg - p0] * a.Hkv + hk) * a.page_size + row) * D;
                            if (!in_bounds(&g_decode_err, src + (size_t)seg * D,
                                           (size_t)a.num_pages * a.Hkv * a.page_size * D))
                                src = 0;
                            const uint32_t bytes = (uint32_t)seg * KL::ROW_BYTES;
                            bulk_copy_g2s(dk + (size_t)(t - t0) * D,
                                          static_cast<const T*>(a.kc) + src, bytes, &full[s], pol);
                            bulk_copy_g2s(dv + (size_t)(t - t0) * D,
                                          static_cast<const T*>(a.vc) + src, bytes, &full[s], pol);
                            t += seg;
                        }
                    }
                }
            }
            if (PAGED) ok = __shfl_sync(kFullMask, ok, 0) != 0;  // also orders page_ids reuse
        }
        if (!ok && lane == 0) {
            // drain the copies still in flight into this CTA's shared memory
            for (uint32_t k = (it >= kStages ? it - kStages : 0); k < it; ++k)
                mbar_wait(&full[k % kStages], (k / kStages) & 1, &g_decode_err);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    // warp -> (query head of the group, share of every stage)
    const int hg = warp / SH::WARPS_PER_HEAD, share = warp - hg * SH::WARPS_PER_HEAD;
    const int g = lane / KL::LPK, e = lane % KL::LPK;
    uint32_t it = 0;
    for (int slot = blockIdx.x; slot < total; slot += gridDim.x) {
        int bh, ch, start, end;
        if (!item_range(a, slot, BHkv, bh, ch, start, end, SPLIT)) continue;
        const int bhq = bh * G + hg;  // this warp's query head
        float qf[VEC], rf[VEC];
        load_row_slice<T, D>(static_cast<const T*>(a.q) + (size_t)bhq * D, e, a.qscale, qf);
        if (RHO) load_row_slice<T, D>(static_cast<const T*>(a.rho) + (size_t)bhq * D, e, 1.f, rf);
        else
#pragma unroll
            for (int x = 0; x < VEC; ++x) rf[x] = 0.f;

        RowState<T, D> st;
        st.reset();
        bool ok = true;
        for (int t0 = start; t0 < end; t0 += SH::STAGE_KEYS, ++it) {
            const int s = it % kStages;
            if (*abort_flag || !mbar_wait(&full[s], (it / kStages) & 1, &g_decode_err)) {
                *abort_flag = 1;
                ok = false;
                break;
            }
            const int nk = min(SH::STAGE_KEYS, end - t0);
            const T* sK = stage_k + (size_t)s * SH::STAGE_KEYS * D;
            const T* sV = stage_v + (size_t)s * SH::STAGE_KEYS * D;
#pragma unroll
            for (int blk = 0; blk < SH::BLOCKS_PER_WARP; ++blk) {
                const int kb = share * SH::KEYS_PER_WARP + blk * KL::BLOCK_KEYS;
                if (kb < nk) warp_block<T, D, RHO>(st, qf, rf, sK, sV, kb, nk, lane);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        // After a timeout every warp still walks the remaining items (without
        // waiting) so that all of them meet at the same named barriers; nothing
        // is written.
        warp_merge_groups<T, D, RHO>(st);

        // ---- merge the states of each query head's warps
        float* mw = merge + warp * (4 + 2 * D);
        if (lane == 0) {
            mw[0] = st.m;
            mw[1] = st.l;
            mw[2] = st.A;
        }
        if (g == 0) {
#pragma unroll
            for (int x = 0; x < VEC; ++x) {
                mw[4 + e * VEC + x] = st.U[x];
                mw[4 + D + e * VEC + x] = st.W[x];
            }
        }
        named_bar_sync(1, kConsumerWarps * 32);
        if (ok && !*abort_flag) {
            for (int idx = threadIdx.x; idx < G * D; idx += kConsumerWarps * 32) {
                const int h2 = idx / D, c = idx - h2 * D;
                const float* m0 = merge + h2 * SH::WARPS_PER_HEAD * (4 + 2 * D);
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < SH::WARPS_PER_HEAD; ++w) M = fmaxf(M, m0[w * (4 + 2 * D)]);
                float l = 0.f, A = 0.f, U = 0.f, W = 0.f;
                if (M > -INFINITY) {
#pragma unroll
                    for (int w = 0; w < SH::WARPS_PER_HEAD; ++w) {
                        const float* m2 = m0 + w * (4 + 2 * D);
                        const float f = fast_exp2(m2[0] - M);
                        l = fmaf(f, m2[1], l);
                        A = fmaf(f, m2[2], A);
                        U = fmaf(f, m2[4 + c], U);
                        W = fmaf(f, m2[4 + D + c], W);
                    }
                }
                const int bq = bh * G + h2;
                if (SPLIT) {
                    const size_t idx2 = (size_t)bq * a.nsplit + ch;
                    if (in_bounds(&g_decode_err, idx2 + 1, (size_t)a.B * a.H * a.nsplit)) {
                        a.ws_uw[idx2 * 2 * D + c] = U;
                        a.ws_uw[idx2 * 2 * D + D + c] = W;
                        if (c == 0) a.ws_stats[idx2] = make_float4(M, l, A, 0.f);
                    }
                } else if (in_bounds(&g_decode_err, (size_t)bq * D + c + 1, (size_t)a.B * a.H * D)) {
                    const float inv_l = l > 0.f ? 1.f / l : 0.f;
                    const float mu = U * inv_l;
                    a.o[(size_t)bq * D + c] = RHO ? mu - (W * inv_l - (A * inv_l) * mu) : mu;
                }
            }
        }
        named_bar_sync(1, kConsumerWarps * 32);
    }
}

// One CTA of D threads per query head.  The chunks' maxima are reduced in parallel, then
// the chunks are taken D at a time: thread t forms the weight 2^(m_t - M) of chunk t of the
// batch (and its l, A terms) into shared memory, and thread c sums column c of U and W over
// the batch with independent, unrolled loads.
template <int D, bool RHO>
__global__ void __launch_bounds__(D) combine_kernel(const DecodeArgs a) {
    __shared__ float s_f[D];
    __shared__ float s_red[3][D / 32];
    const int bh = blockIdx.x, c = threadIdx.x, w = c / 32, lane = c % 32;
    const int n = clamp_seqlen(a.seqlens, bh / a.H, a.Lmax);
    int nch = (n + a.chunk - 1) / a.chunk;
    if (!in_bounds(&g_decode_err, (size_t)nch, (size_t)a.nsplit)) nch = a.nsplit;
    const float4* stats = a.ws_stats + (size_t)bh * a.nsplit;
    const float* uw = a.ws_uw + (size_t)bh * a.nsplit * 2 * D;
    float M = -INFINITY;
    for (int k = c; k < nch; k += D) M = fmaxf(M, stats[k].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, o));
    if (lane == 0) s_red[0][w] = M;
    __syncthreads();
    M = s_red[0][0];
#pragma unroll
    for (int i = 1; i < D / 32; ++i) M = fmaxf(M, s_red[0][i]);
    float l = 0.f, A = 0.f, U = 0.f, W = 0.f;
    for (int k0 = 0; k0 < nch; k0 += D) {
        const int nb = min(D, nch - k0);
        __syncthreads();  // s_f of the previous batch has been read
        if (c < nb) {
            const float4 st = stats[k0 + c];
            const float f = M > -INFINITY ? fast_exp2(st.x - M) : 0.f;
            s_f[c] = f;
            l = fmaf(f, st.y, l);
            A = fmaf(f, st.z, A);
        }
        __syncthreads();
        const float* col = uw + (size_t)k0 * 2 * D + c;
#pragma unroll 8
        for (int k = 0; k < nb; ++k) {
            const float f = s_f[k];
            U = fmaf(f, __ldg(col + (size_t)k * 2 * D), U);
            if (RHO) W = fmaf(f, __ldg(col + (size_t)k * 2 * D + D), W);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        l += __shfl_xor_sync(kFullMask, l, o);
        A += __shfl_xor_sync(kFullMask, A, o);
    }
    __syncthreads();
    if (lane == 0) {
        s_red[1][w] = l;
        s_red[2][w] = A;
    }
    __syncthreads();
    l = 0.f;
    A = 0.f;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) {
        l += s_red[1][i];
        A += s_red[2][i];
    }
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    const float mu = U * inv_l;
    if (in_bounds(&g_decode_err, (size_t)bh * D + c + 1, (size_t)a.B * a.H * D))
        a.o[(size_t)bh * D + c] = RHO ? mu - (W * inv_l - (A * inv_l) * mu) : mu;
}

// ---------------------------------------------------------------------------
// Grouped-query decode on the tensor cores (bf16, G = 2, 4 or 8 query heads per
// key/value head).  The G query rows and their G probe rows form one 16-row
// operand [q; rho] (rows g and 8 + g: head g), so that per 16-key block one
// warp computes
//     [S; R] = [q; rho] K^T            (16 x 16, fp32, warp-level mma m16n8k16)
// takes the online-softmax step on the scores it holds in registers, and
//     [U; W] += [P; P o R] V           (16 x D, fp32)
// with the MMA outputs of the first product reused in registers as the A
// operand of the second.  Per key and head this replaces the SIMT decode's two
// dot products and two axpys on the FMA pipes by a share of two tensor-core
// products; the SIMT decode is issue-bound at G >= 2.  The operand has only 2G
// real rows, below the 64-row minimum of tcgen05.mma, so the warp-level form
// is the one that fits.
//
// The producer lane loads each stage of keys and values with TMA tile copies
// (boxes of 64 columns x STAGE_KEYS rows, 128-byte swizzle), so that the
// ldmatrix fragment loads of eight consecutive rows hit eight different bank
// groups.  A paged cache is loaded the same way when its pages hold whole
// stages (page_size a multiple of STAGE_KEYS); other page sizes use the SIMT
// decode.  Four consumer warps take 16 keys (D = 128) or 32 keys (D = 64) of
// every stage; at the end of an item their states are merged in shared memory
// into the same partial-state / output format as decode_kernel (same plan,
// workspace and combine kernel).
constexpr int kMmaWarps = 4;
constexpr int kMmaThreads = (kMmaWarps + 1) * 32;

template <int D, int G>
struct MmaShape {
    static constexpr int STAGE_KEYS = kStageRowBytes / (D * 2);
    static constexpr int NCB = D / 64;                  // 64-column (128-byte) blocks per row
    static constexpr int CB_BYTES = STAGE_KEYS * 128;   // one swizzled column block of a stage
    static constexpr int KPW = STAGE_KEYS / kMmaWarps;  // keys per warp per stage
    static_assert(KPW % 16 == 0, "16-key blocks");
    static constexpr int STAGE_BYTES = NCB * CB_BYTES;
    // three stages while two CTAs still fit an SM (groups of 1 and 2: small merge slots),
    // two for the groups of 4 and 8, whose merge slots take the room of a third
    static constexpr int STAGES = G <= 2 ? 3 : 2;
    static constexpr int SLOT_FLOATS = G * (2 * D + 4);  // per warp: G heads x (U, W, m, l, A)
    static constexpr int MERGE_OFF = 2 * STAGES * STAGE_BYTES;
    static constexpr int BAR_OFF = MERGE_OFF + kMmaWarps * SLOT_FLOATS * 4;
    static constexpr size_t SMEM_BYTES = BAR_OFF + 2 * STAGES * 8 + 16 + 1024;
    static_assert(2 * (SMEM_BYTES + 1024) <= 228 * 1024, "two CTAs per SM");
};

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Byte offset in a stage of (row, 16-byte chunk c16 of the row): 128-byte swizzle
// within each 64-column block.
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int c16) {
    using MS = MmaShape<D, 1>;
    return (uint32_t)((c16 >> 3) * MS::CB_BYTES + row * 128 + (((c16 & 7) ^ (row & 7)) << 4));
}

template <int D, bool RHO, bool SPLIT, int G, bool PAGED>
__global__ void __launch_bounds__(kMmaThreads, 2)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const DecodeArgs a) {
    using MS = MmaShape<D, G>;
    constexpr int kMmaStages = MS::STAGES;
    using T = __nv_bfloat16;
    constexpr int ROW_BYTES = D * 2;
    extern __shared__ unsigned char smem_raw[];
    // 128-byte swizzled TMA tiles need 1024-byte aligned destinations
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* stage_k = smem;
    unsigned char* stage_v = smem + kMmaStages * MS::STAGE_BYTES;
    float* merge = reinterpret_cast<float*>(smem + MS::MERGE_OFF);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + MS::BAR_OFF);
    uint64_t* empty = full + kMmaStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kMmaStages);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int BHkv = a.B * a.Hkv;
    const int total = BHkv * a.nsplit;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kMmaStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kMmaWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (*(volatile unsigned*)&g_decode_err & PARALLAX_DEVERR_WAIT_TIMEOUT) return;

    if (warp == kMmaWarps) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        uint32_t it = 0;
        bool ok = true;
        for (int slot = blockIdx.x; slot < total && ok; slot += gridDim.x) {
            int bh, ch, start, end;
            if (!item_range(a, slot, BHkv, bh, ch, start, end, SPLIT)) continue;
            const int b = bh / a.Hkv, hk = bh - b * a.Hkv;
            for (int t0 = start; t0 < end; t0 += MS::STAGE_KEYS, ++it) {
                const int s = it % kMmaStages;
                if (!mbar_wait(&empty[s], ((it / kMmaStages) & 1) ^ 1, &g_decode_err)) {
                    ok = false;
                    break;
                }
                // row of the first key of the stage in the [rows, D] view of the cache
                int row0;
                if (PAGED) {
                    const int pg = t0 / a.page_size;  // a stage never crosses a page
                    row0 = (checked_page(a, a.block_table[(size_t)b * a.max_pages + pg]) * a.Hkv + hk) *
                               a.page_size + (t0 - pg * a.page_size);
                } else {
                    row0 = bh * a.Lmax + t0;
                }
                mbar_arrive_expect_tx(&full[s], 2u * MS::STAGE_BYTES);
                for (int cb = 0; cb < MS::NCB; ++cb) {
                    tc::tma_load_2d(stage_k + s * MS::STAGE_BYTES + cb * MS::CB_BYTES, &tmK, cb * 64,
                                    row0, &full[s]);
                    tc::tma_load_2d(stage_v + s * MS::STAGE_BYTES + cb * MS::CB_BYTES, &tmV, cb * 64,
                                    row0, &full[s]);
                }
            }
        }
        if (!ok) {
            *abort_flag = 1;
            // drain the copies still in flight into this CTA's shared memory
            for (uint32_t k = (it >= kMmaStages ? it - kMmaStages : 0); k < it; ++k)
                mbar_wait(&full[k % kMmaStages], (k / kMmaStages) & 1, &g_decode_err);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int g = lane >> 2, t = lane & 3;  // mma fragment coordinates: row g (and g + 8)
    const float qs = a.qscale;
    const uint32_t sk = smem_u32(stage_k), sv = smem_u32(stage_v);
    float* slot = merge + warp * MS::SLOT_FLOATS;
    uint32_t it = 0;
    for (int item = blockIdx.x; item < total; item += gridDim.x) {
        int bh, ch, start, end;
        if (!item_range(a, item, BHkv, bh, ch, start, end, SPLIT)) continue;
        // A fragments of [q; rho]: row g = query head g of the group, row 8 + g its probe
        uint32_t aq[D / 16][4];
        {
            const bool real = g < G;
            const T* qr = static_cast<const T*>(a.q) + (size_t)(bh * G + (real ? g : 0)) * D;
            const T* rr = RHO ? static_cast<const T*>(a.rho) + (size_t)(bh * G + (real ? g : 0)) * D
                              : qr;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int c = 16 * kk + 2 * t;
                aq[kk][0] = real ? __ldg(reinterpret_cast<const uint32_t*>(qr + c)) : 0u;
                aq[kk][1] = real && RHO ? __ldg(reinterpret_cast<const uint32_t*>(rr + c)) : 0u;
                aq[kk][2] = real ? __ldg(reinterpret_cast<const uint32_t*>(qr + c + 8)) : 0u;
                aq[kk][3] = real && RHO ? __ldg(reinterpret_cast<const uint32_t*>(rr + c + 8)) : 0u;
            }
        }
        float acc[D / 8][4];
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        float m = -INFINITY, l = 0.f, A = 0.f;
        bool ok = true;
        for (int t0 = start; t0 < end; t0 += MS::STAGE_KEYS, ++it) {
            const int s = it % kMmaStages;
            if (*abort_flag || !mbar_wait(&full[s], (it / kMmaStages) & 1, &g_decode_err)) {
                *abort_flag = 1;
                ok = false;
                break;
            }
            const int nk = min(MS::STAGE_KEYS, end - t0);
            const uint32_t kbase = sk + s * MS::STAGE_BYTES, vbase = sv + s * MS::STAGE_BYTES;
#pragma unroll
            for (int blk = 0; blk < MS::KPW / 16; ++blk) {
                const int key0 = warp * MS::KPW + 16 * blk;
                if (key0 >= nk) break;  // warp-uniform
                // ---- [S; R] for keys key0 .. key0 + 15 (two n-tiles of 8 keys)
                float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
                {
                    const int mi = lane >> 3, r = lane & 7;
                    const int row = key0 + (mi >> 1) * 8 + r;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(kbase + swz<D>(row, 2 * kk + (mi & 1)), b0, b1, b2, b3);
                        mma_bf16_16816(c0, aq[kk], b0, b1);
                        mma_bf16_16816(c1, aq[kk], b2, b3);
                    }
                }
                // keys of this thread: key0 + 2t, +1 (c0) and key0 + 8 + 2t, +1 (c1)
                const int kx = key0 + 2 * t;
                const bool v0 = kx < nk, v1 = kx + 1 < nk, v2 = kx + 8 < nk, v3 = kx + 9 < nk;
                const float s0 = v0 ? c0[0] * qs : -INFINITY, s1 = v1 ? c0[1] * qs : -INFINITY;
                const float s2 = v2 ? c1[0] * qs : -INFINITY, s3 = v3 ? c1[1] * qs : -INFINITY;
                float bm = fmaxf(fmaxf(s0, s1), fmaxf(s2, s3));
                bm = fmaxf(bm, __shfl_xor_sync(kFullMask, bm, 1));
                bm = fmaxf(bm, __shfl_xor_sync(kFullMask, bm, 2));
                if (bm > m) {  // uniform over the 4 lanes of head g
                    const float alpha = m == -INFINITY ? 0.f : fast_exp2(m - bm);
                    l *= alpha;
                    A *= alpha;
#pragma unroll
                    for (int nt = 0; nt < D / 8; ++nt) {
                        acc[nt][0] *= alpha;
                        acc[nt][1] *= alpha;
                        acc[nt][2] *= alpha;
                        acc[nt][3] *= alpha;
                    }
                    m = bm;
                }
                const float p0 = fast_exp2(s0 - m), p1 = fast_exp2(s1 - m);
                const float p2 = fast_exp2(s2 - m), p3 = fast_exp2(s3 - m);
                const float q0 = v0 ? p0 * c0[2] : 0.f, q1 = v1 ? p1 * c0[3] : 0.f;
                const float q2 = v2 ? p2 * c1[2] : 0.f, q3 = v3 ? p3 * c1[3] : 0.f;
                l += (p0 + p1) + (p2 + p3);
                A += (q0 + q1) + (q2 + q3);
                const uint32_t pa[4] = {pack2_bf16(p0, p1), pack2_bf16(q0, q1), pack2_bf16(p2, p3),
                                        pack2_bf16(q2, q3)};
                if (key0 + 16 > nk) {
                    // value rows past the chunk hold stale shared memory: zero them, since a
                    // zero weight times a NaN would still be NaN in the product
                    const int nz = key0 + 16 - nk;
                    for (int e = lane; e < nz * (ROW_BYTES / 16); e += 32) {
                        const int row = nk + e / (ROW_BYTES / 16), c16 = e % (ROW_BYTES / 16);
                        *reinterpret_cast<uint4*>(stage_v + s * MS::STAGE_BYTES + swz<D>(row, c16)) =
                            make_uint4(0, 0, 0, 0);
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                }
                // ---- [U; W] += [P; P o R] V
                {
                    const int mi = lane >> 3, r = lane & 7;
                    const int row = key0 + (mi & 1) * 8 + r;
#pragma unroll
                    for (int np = 0; np < D / 16; ++np) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_trans(vbase + swz<D>(row, 2 * np + (mi >> 1)), b0, b1, b2, b3);
                        mma_bf16_16816(acc[2 * np], pa, b0, b1);
                        mma_bf16_16816(acc[2 * np + 1], pa, b2, b3);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        // ---- this warp's state -> its merge slot (rows of head g)
        l += __shfl_xor_sync(kFullMask, l, 1);
        l += __shfl_xor_sync(kFullMask, l, 2);
        A += __shfl_xor_sync(kFullMask, A, 1);
        A += __shfl_xor_sync(kFullMask, A, 2);
        if (g < G) {  // rows past the group are padding
            float* hs = slot + g * (2 * D + 4);
            if (t == 0) {
                hs[0] = m;
                hs[1] = l;
                hs[2] = A;
            }
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt) {
                *reinterpret_cast<float2*>(hs + 4 + 8 * nt + 2 * t) =
                    make_float2(acc[nt][0], acc[nt][1]);
                *reinterpret_cast<float2*>(hs + 4 + D + 8 * nt + 2 * t) =
                    make_float2(acc[nt][2], acc[nt][3]);
            }
        }
        named_bar_sync(1, kMmaWarps * 32);
        if (ok && !*abort_flag) {
            for (int idx = threadIdx.x; idx < G * D; idx += kMmaWarps * 32) {
                const int h2 = idx / D, c = idx - h2 * D;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kMmaWarps; ++w)
                    M = fmaxf(M, merge[w * MS::SLOT_FLOATS + h2 * (2 * D + 4)]);
                float ls = 0.f, As = 0.f, U = 0.f, W = 0.f;
                if (M > -INFINITY) {
#pragma unroll
                    for (int w = 0; w < kMmaWarps; ++w) {
                        const float* x = merge + w * MS::SLOT_FLOATS + h2 * (2 * D + 4);
                        const float f = fast_exp2(x[0] - M);
                        ls = fmaf(f, x[1], ls);
                        As = fmaf(f, x[2], As);
                        U = fmaf(f, x[4 + c], U);
                        W = fmaf(f, x[4 + D + c], W);
                    }
                }
                const int bq = bh * G + h2;
                if (SPLIT) {
                    const size_t idx2 = (size_t)bq * a.nsplit + ch;
                    if (in_bounds(&g_decode_err, idx2 + 1, (size_t)a.B * a.H * a.nsplit)) {
                        a.ws_uw[idx2 * 2 * D + c] = U;
                        a.ws_uw[idx2 * 2 * D + D + c] = W;
                        if (c == 0) a.ws_stats[idx2] = make_float4(M, ls, As, 0.f);
                    }
                } else if (in_bounds(&g_decode_err, (size_t)bq * D + c + 1, (size_t)a.B * a.H * D)) {
                    const float inv_l = ls > 0.f ? 1.f / ls : 0.f;
                    const float mu = U * inv_l;
                    a.o[(size_t)bq * D + c] = RHO ? mu - (W * inv_l - (As * inv_l) * mu) : mu;
                }
            }
        }
        named_bar_sync(1, kMmaWarps * 32);
    }
}

template <int D, bool RHO, bool SPLIT, int G, bool PAGED>
cudaError_t launch_decode_mma_kernel(const DecodeArgs& a, int grid, cudaStream_t stream) {
    using MS = MmaShape<D, G>;
    auto kern = decode_mma_kernel<D, RHO, SPLIT, G, PAGED>;
    static std::atomic<uint64_t> smem_set{0};
    if (cudaError_t e = ensure_dynamic_smem(kern, (int)MS::SMEM_BYTES, smem_set)) return e;
    // the caches as [rows, D] bf16 tensors: (b, h_kv, key) -> row (b*H_kv + h_kv)*Lmax + key,
    // or, paged, (page, h_kv, row) -> (page*H_kv + h_kv)*page_size + row
    const uint64_t rows = PAGED ? (uint64_t)a.num_pages * a.Hkv * a.page_size
                                : (uint64_t)a.B * a.Hkv * a.Lmax;
    const uint64_t dims[2] = {(uint64_t)D, rows};
    const uint64_t strides[1] = {(uint64_t)D * 2};
    const uint32_t box[2] = {64, (uint32_t)MS::STAGE_KEYS};
    CUtensorMap mk, mv;
    if (!make_tmap_bf16(&mk, a.kc, 2, dims, strides, box) ||
        !make_tmap_bf16(&mv, a.vc, 2, dims, strides, box))
        return cudaErrorInvalidValue;
    kern<<<grid, kMmaThreads, MS::SMEM_BYTES, stream>>>(mk, mv, a);
    return cudaGetLastError();
}

template <typename T, int D, bool RHO, bool SPLIT, int G, bool PAGED>
cudaError_t launch_decode_kernel(const DecodeArgs& a, int grid, cudaStream_t stream) {
    using SH = DecodeShape<T, D, G>;
    auto kern = decode_kernel<T, D, RHO, SPLIT, G, PAGED>;
    static std::atomic<uint64_t> smem_set{0};
    if (cudaError_t e = ensure_dynamic_smem(kern, (int)SH::SMEM_BYTES, smem_set)) return e;
    kern<<<grid, kThreads, SH::SMEM_BYTES, stream>>>(a);
    return cudaGetLastError();
}

template <typename T, int D, bool RHO, int G, bool PAGED>
cudaError_t run_decode(const DecodePlan& plan, const void* q, const void* rho, const void* kc,
                       const void* vc, const int32_t* seqlens, float* o, void* ws,
                       const int32_t* block_table, cudaStream_t stream) {
    DecodeArgs a;
    a.q = q;
    a.rho = rho;
    a.kc = kc;
    a.vc = vc;
    a.seqlens = seqlens;
    a.o = o;
    a.block_table = block_table;
    a.B = plan.B;
    a.H = plan.H;
    a.Hkv = plan.Hkv;
    a.Lmax = plan.Lmax;
    a.chunk = plan.chunk;
    a.nsplit = plan.nsplit;
    a.page_size = plan.page_size;
    a.max_pages = plan.max_pages;
    a.num_pages = plan.num_pages;
    a.qscale = plan.scale * kLog2e;
    const size_t BH = (size_t)plan.B * plan.H;
    a.ws_stats = static_cast<float4*>(ws);
    a.ws_uw = reinterpret_cast<float*>(static_cast<char*>(ws) + BH * plan.nsplit * sizeof(float4));
    cudaError_t e = cudaSuccess;
    // grouped heads: the tensor-core decode (a paged cache only when every stage lies in one page)
    constexpr bool kMmaOk = sizeof(T) == 2;
    const bool mma = kMmaOk && decode_uses_mma(plan, true);
    if (plan.nsplit > 1) {
        if constexpr (kMmaOk) {
            if (mma) e = launch_decode_mma_kernel<D, RHO, true, G, PAGED>(a, plan.grid, stream);
            else e = launch_decode_kernel<T, D, RHO, true, G, PAGED>(a, plan.grid, stream);
        } else {
            e = launch_decode_kernel<T, D, RHO, true, G, PAGED>(a, plan.grid, stream);
        }
        if (e != cudaSuccess) return e;
        combine_kernel<D, RHO><<<(unsigned)BH, D, 0, stream>>>(a);
    } else {
        if constexpr (kMmaOk) {
            if (mma) e = launch_decode_mma_kernel<D, RHO, false, G, PAGED>(a, plan.grid, stream);
            else e = launch_decode_kernel<T, D, RHO, false, G, PAGED>(a, plan.grid, stream);
        } else {
            e = launch_decode_kernel<T, D, RHO, false, G, PAGED>(a, plan.grid, stream);
        }
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

// bf16: every group size and both cache layouts; fp32: plain attention only.
template <typename T, int D, bool RHO>
cudaError_t run_decode_any(const DecodePlan& plan, const void* q, const void* rho, const void* kc,
                           const void* vc, const int32_t* seqlens, float* o, void* ws,
                           const int32_t* block_table, cudaStream_t stream) {
    const int G = plan.H / plan.Hkv;
    const bool paged = plan.page_size > 0;
    if constexpr (sizeof(T) == 2) {
#define PARALLAX_DECODE_G(GG)                                                                     \
    if (G == GG)                                                                                  \
        return paged ? run_decode<T, D, RHO, GG, true>(plan, q, rho, kc, vc, seqlens, o, ws,      \
                                                       block_table, stream)                       \
                     : run_decode<T, D, RHO, GG, false>(plan, q, rho, kc, vc, seqlens, o, ws,     \
                                                        block_table, stream);
        PARALLAX_DECODE_G(1)
        PARALLAX_DECODE_G(2)
        PARALLAX_DECODE_G(4)
        PARALLAX_DECODE_G(8)
#undef PARALLAX_DECODE_G
        return cudaErrorInvalidValue;
    } else {
        if (G != 1 || paged) return cudaErrorInvalidValue;
        return run_decode<T, D, RHO, 1, false>(plan, q, rho, kc, vc, seqlens, o, ws, block_table,
                                               stream);
    }
}

}  // namespace

bool decode_uses_mma(const DecodePlan& plan, bool bf16) {
    if (!bf16 || plan.Hkv <= 0) return false;
    const int G = plan.H / plan.Hkv;
    const int stage_keys = kStageRowBytes / (plan.d * 2);  // MmaShape<D, G>::STAGE_KEYS
    const bool pages_fit = plan.page_size == 0 || (plan.page_size % stage_keys == 0 &&
                                                   plan.chunk % stage_keys == 0);
    return (G >= 2 || plan.mma) && pages_fit;
}

size_t decode_workspace_bytes(const DecodePlan& plan) {
    if (plan.nsplit <= 1) return 0;
    const size_t items = (size_t)plan.B * plan.H * plan.nsplit;
    return items * sizeof(float4) + items * 2 * plan.d * sizeof(float);
}

int decode_stage_keys(int d, int elem_bytes) { return kStageRowBytes / (d * elem_bytes); }

int decode_threads() { return kThreads; }

int decode_ctas_per_sm() { return kCtasPerSm; }

int decode_paged_max_chunk(int page_size) { return (kMaxPageIds - 1) * page_size; }

cudaError_t decode_launch(const DecodePlan& plan, bool bf16, const void* q, const void* rho,
                          const void* kc, const void* vc, const int32_t* seqlens, float* o,
                          void* ws, cudaStream_t stream, const int32_t* block_table) {
    const bool r = rho != nullptr;
    if (plan.Hkv <= 0 || plan.H % plan.Hkv != 0) return cudaErrorInvalidValue;
    if (plan.page_size > 0 && (!block_table || plan.chunk > decode_paged_max_chunk(plan.page_size)))
        return cudaErrorInvalidValue;
#define PARALLAX_DECODE_CASE(T, DD)                                                              \
    if (plan.d == DD)                                                                            \
        return r ? run_decode_any<T, DD, true>(plan, q, rho, kc, vc, seqlens, o, ws, block_table, \
                                               stream)                                           \
                 : run_decode_any<T, DD, false>(plan, q, rho, kc, vc, seqlens, o, ws,             \
                                                block_table, stream);
    if (bf16) {
        PARALLAX_DECODE_CASE(__nv_bfloat16, 64)
        PARALLAX_DECODE_CASE(__nv_bfloat16, 128)
    } else {
        PARALLAX_DECODE_CASE(float, 64)
        PARALLAX_DECODE_CASE(float, 128)
    }
#undef PARALLAX_DECODE_CASE
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// Fixed scratch for decode callers that cannot allocate device memory.
//
// Some callers cannot let a library call cudaMalloc: serving engines that
// reserve nearly all device memory for their own KV-cache pool up front (a
// late allocation would fail or eat into the pool), and latency-critical
// decode loops where cudaMalloc/cudaFree would synchronise the device and
// stall every other stream.  For them the split-KV partial states go to this
// file-scope array instead of the grown-on-demand workspace.  It exists once
// per device that loads the library and stays until the process exits.
// Nothing in it needs to start at zero: the combine kernel reads only the
// partial states that the decode kernel of the same call wrote.  All calls on
// a device share it, so calls that overlap on the GPU race on it.
// ---------------------------------------------------------------------------
namespace {
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};
}  // namespace

size_t decode_noalloc_capacity() { return kNoAllocScratchBytes; }

cudaError_t decode_launch_noalloc(const DecodePlan& plan, bool bf16, const void* q,
                                  const void* rho, const void* kc, const void* vc,
                                  const int32_t* seqlens, float* o, cudaStream_t stream) {
    if (decode_workspace_bytes(plan) > kNoAllocScratchBytes) return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void* ptr = nullptr;
    {
        // Set-up, once per device, with that device current: the symbol's name
        // is only a host-side stand-in, so fetch the device address of the array.
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_addr[dev]) {
            e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
            if (e != cudaSuccess) return e;
            g_noalloc_addr[dev] = ptr;
        }
        ptr = g_noalloc_addr[dev];
    }
    return decode_launch(plan, bf16, q, rho, kc, vc, seqlens, o, ptr, stream, nullptr);
}

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing ever
// arrives on, with a wait limit of limit_ns; the wait gives up, raises
// PARALLAX_DEVERR_WAIT_TIMEOUT in the decode kernels' error word and the kernel returns.
// Until the host clears the word, later decode launches see the bit and exit at once.
namespace {
__global__ void decode_wait_selftest_kernel(uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        mbar_wait(&bar, 0, &g_decode_err, limit_ns);
    }
}
}  // namespace

cudaError_t decode_wait_selftest(uint64_t limit_ns, cudaStream_t stream) {
    decode_wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
    return cudaGetLastError();
}

unsigned decode_take_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_decode_err, sizeof(v)) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_decode_err, &zero, sizeof(zero));
    return v;
}

}  // namespace parallax
