// Parallax prefill on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// For every 128-key tile of K and V (fetched once by TMA and shared by both
// branches -- the pages' "same KV stream for both branches", "Parallax mantem
// softmax ...", paragraph 2) a CTA computes, for its query rows,
//
//   MMA-1   S = Q K^T   and   R = rho K^T            (bf16 in, fp32 in TMEM)
//   softmax P = 2^(S*scale*log2e - m)  (row max m, lazily rescaled),
//           PR = P o (R - c)           (c: per-row shift, see below)
//   MMA-2   U += P V    and   W += PR V               (P, PR read from TMEM)
//
// and at the end o = U/l - (W/l - (A/l)(U/l)) with l = sum P, A = sum PR.
// With rho == NULL (W_R = 0) only S, P and U exist and o = U/l: plain softmax
// attention.
//
// A CTA owns two query sub-tiles that take turns on the tensor core: while
// the softmax warps of one sub-tile work, the MMAs of the other run.
//
//  * correction path (RHO): a sub-tile is 64 queries and the A operand of
//    MMA-1 stacks, per 16-query group g, the 16 query rows (operand rows
//    32g..32g+15) and the same 16 queries' probe rows (rows 32g+16..32g+31).
//    One M=128 MMA per sub-tile yields S and R for its 64 queries, and one
//    M=128 MMA with A = [P; PR] (from TMEM) yields U and W.  TMEM lane 32g+i
//    holds query 16g+i's S row (then P, then U) and lane 32g+16+i its R row
//    (then PR, then W).  The half-split TMEM access (.16x32bx2) gives thread
//    t < 16 and thread t + 16 of a softmax warp the same query's S and R rows,
//    each with half of the key columns, so every thread computes s, r, p and
//    p(r - c) for 64 keys of one query with no data exchange.
//  * W_R = 0 path: a sub-tile is 128 queries (one per TMEM lane and softmax
//    thread), A of MMA-1 is the Q tile, A of MMA-2 is P.
//
// TMEM columns: D_sub at 128*sub (S|R, then P|PR packed into its first 64
// columns, the few-key residuals into the next 64), O_sub at 256 + sub*d.
//
// Warps (12 = 3 warpgroups): warp 0 issues TMA loads, warp 1 owns TMEM and
// issues the MMAs (warps 2-3 idle), warps 4-7 / 8-11 are the softmax and
// epilogue warps of sub-tile 0 / 1.  The first warpgroup hands registers to
// the other two (setmaxnreg).
//
// Numerics of the correction path:
//  * the row shift c (Cov_p(r - c, v) = Cov_p(r, v) for any constant c) is set
//    to the p-weighted mean of r over the first key tile processed, so PR is
//    centred and its bf16 rounding error stays proportional to the spread of
//    r rather than its size.  Key tiles are processed in order 0, 1, ..., with
//    the causal diagonal tile last, so that the first tile is a full one and c
//    is a mean over 128 keys (for the first query block it is the only tile);
//  * rows that see few keys (the first query block of a causal head, or a
//    non-causal head with L <= 128) also feed the bf16 rounding residuals of
//    P and PR (stored in D columns [64,128)) through one more MMA, so U and W
//    are accurate to ~2^-16 there;
//  * the running max m is only moved when a tile's max exceeds it by more
//    than 2^8 (lazy rescale); the final normalisation uses the same m, so the
//    result is exact in exact arithmetic.
#include "tcgen05.cuh"
#include "kernels.h"

namespace parallax {
namespace {

__device__ unsigned g_tc_err = 0;

constexpr int BN = 128;  // keys per tile
constexpr float kRescaleThreshold = 8.f;  // log2 units
constexpr int kThreads = 384;
// Register hand-over: the launch gives every thread kRegsLaunch registers
// (3 warps per SM sub-partition x 32 x 168 <= 16384); afterwards 4 warps x 64
// + 8 warps x 216 use no more than that total.  The build checks that ptxas
// assigned kRegsLaunch registers to this kernel: with fewer, the raising
// warpgroups would wait forever.
constexpr int kRegsLaunch = 168;
constexpr int kRegsSupport = 64;
constexpr int kRegsSoftmax = 216;
static_assert(128 * kRegsSupport + 256 * kRegsSoftmax <= kThreads * kRegsLaunch,
              "register hand-over exceeds the launch allocation");
constexpr int kHeadGroup = 16;  // heads per CTA-scheduling group (keeps their K/V in L2)
// K tiles are needed half a tile step before V tiles (S of tile j+1 is computed while P of
// tile j is pending), so the K ring is one stage deeper than the V ring; K and V are loaded
// by two producer warps so that neither ring's wait holds up the other's loads.
constexpr int kKStages = 3;
constexpr int kVStages = 2;

template <int D, bool RHO>
struct PairLayout {
    static constexpr int QROWS = RHO ? 64 : 128;        // queries per sub-tile
    static constexpr int BLOCK = 2 * QROWS;             // queries per CTA
    static constexpr int SUB_BYTES = 128 * 128;         // [128 rows x 64 cols] bf16, 128B-swizzled
    static constexpr int NCB = D / 64;                  // 64-column blocks per row
    static constexpr int OP_BYTES = NCB * SUB_BYTES;    // one 128 x D bf16 operand
    static constexpr int QR_OFF = 0;                    // A operands of MMA-1, sub-tiles 0 and 1
    static constexpr int K_OFF = 2 * OP_BYTES;                     // K ring
    static constexpr int V_OFF = K_OFF + kKStages * OP_BYTES;      // V ring
    static constexpr int BAR_OFF = V_OFF + kVStages * OP_BYTES;
    // q_full, k_full[kKStages], v_full[kVStages], k_empty[kKStages], v_empty[kVStages],
    // s_full[2], p_full[2], o_full, o_full0 (sub-tile 0's last P.V has completed)
    static constexpr int B_KFULL = 1;
    static constexpr int B_VFULL = B_KFULL + kKStages;
    static constexpr int B_KEMPTY = B_VFULL + kVStages;
    static constexpr int B_VEMPTY = B_KEMPTY + kKStages;
    static constexpr int B_SFULL = B_VEMPTY + kVStages;
    static constexpr int B_PFULL = B_SFULL + 2;
    static constexpr int B_OFULL = B_PFULL + 2;
    static constexpr int B_OFULL0 = B_OFULL + 1;
    static constexpr int NBARS = B_OFULL0 + 1;
    // Epilogue: each sub-tile's fp32 output is staged as boxes of [QROWS rows x 32 columns]
    // (128 bytes a row, 128-byte swizzle) and each softmax warp stores its WROWS rows with its
    // own TMA tensor stores (boxes of [WROWS rows x 32 columns]), without waiting for the other
    // warps.  With W_R = 0 a causal sub-tile 1 has one key tile more than sub-tile 0, and
    // sub-tile 0 stages as soon as its own last P.V has completed, into the two K stages that
    // sub-tile 1's last S does not read (n1 % 3 and (n1 + 1) % 3: their tiles were consumed by
    // MMAs that completed before that P.V, and no load targets them any more); sub-tile 1
    // stages into the V ring once every MMA has completed.  On the correction path, whose
    // sub-tiles end together, both stage into the rings from K_OFF once every MMA has completed.
    static constexpr int OUT_BOX = QROWS * 128;
    static constexpr int WROWS = QROWS / 4;
    static constexpr int BOXES_PER_K_STAGE = OP_BYTES / OUT_BOX;
    static_assert(kKStages == 3 && D / 32 <= 2 * BOXES_PER_K_STAGE, "sub-tile 0 staging fits two K stages");
    static_assert(2 * (D / 32) * OUT_BOX <= BAR_OFF - K_OFF, "output staging fits the rings");
    static_assert((D / 32) * OUT_BOX <= kVStages * OP_BYTES, "sub-tile 1 staging fits the V ring");
    static constexpr int SMEM_BYTES = BAR_OFF + NBARS * 8 + 16 + 1024;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
    __host__ __device__ static constexpr uint32_t dcol(int sub) { return 128u * sub; }
    __host__ __device__ static constexpr uint32_t ocol(int sub) { return 256u + (uint32_t)(D * sub); }
};

struct TcArgs {
    float* o;
    // chunked prefill: keys already cached per sequence, or null (plain prefill).  Query
    // row i of sequence b then sits at position cache_lens[b] + i and sees the keys at
    // positions 0 .. cache_lens[b] + i of the K/V tensors.
    const int32_t* cache_lens;
    int L;         // query rows per head (also the key rows without a cache)
    int Lcap;      // rows of the K/V tensors per head (L without a cache)
    int H;
    int BH;
    int n_qb;      // query blocks per head
    float qscale;  // scale * log2(e)
    // training forward (all three set or all null): per-row log-sum-exp of the scaled
    // scores (natural log) and rbar = sum_j p_j r_j, [B*H, L]; mu_v = sum_j p_j v_j [B*H, L, D]
    float* lse;
    float* rbar;
    float* mu;
};

// Keys already cached for the sequence of head bh, clamped so that the chunk fits.
__device__ __forceinline__ int cached_keys(const TcArgs& a, int bh, unsigned* err, bool report) {
    if (!a.cache_lens) return 0;
    int off = __ldg(a.cache_lens + bh / a.H);
    if (off < 0 || off > a.Lcap - a.L) {
        if (report) raise_error(err, PARALLAX_DEVERR_SEQLEN_CLAMPED);
        off = off < 0 ? 0 : a.Lcap - a.L;
    }
    return off;
}

// p = 2^(s*qs - m) for 32 consecutive values (in place), their sum into ls0/ls1,
// and the bf16 pairs into pk.  Every exponential runs on the SFU: on sm_103a its
// ex2 rate (measured: about 32 per clock per SM) leaves the SFU far from busy.
__device__ __forceinline__ void exp_block32(uint32_t (&v)[32], float2 qs2, float2 nm2,
                                            float2& ls0, float2& ls1, uint32_t (&pk)[16]) {
#pragma unroll
    for (int y = 0; y < 16; ++y) {
        const float2 t = __ffma2_rn(
            make_float2(__uint_as_float(v[2 * y]), __uint_as_float(v[2 * y + 1])), qs2, nm2);
        const float2 p2 = make_float2(fast_exp2(t.x), fast_exp2(t.y));
        v[2 * y] = __float_as_uint(p2.x);
        v[2 * y + 1] = __float_as_uint(p2.y);
        if (y & 1) ls1 = __fadd2_rn(ls1, p2);
        else ls0 = __fadd2_rn(ls0, p2);
        pk[y] = tc::pack_bf16(p2.x, p2.y);
    }
}

// Maximum of the 128 values of v[4][32] (or 64 of v[2][32]) in eight independent chains of
// three-input max, then a short tree.
template <int NB>
__device__ __forceinline__ float max_blocks(const uint32_t (&v)[NB][32]) {
    float c[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) c[k] = -INFINITY;
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int x = 0; x < 32; x += 16)
#pragma unroll
            for (int k = 0; k < 8; ++k)
                c[k] = fmax3(c[k], __uint_as_float(v[b][x + 2 * k]), __uint_as_float(v[b][x + 2 * k + 1]));
    return fmaxf(fmaxf(fmax3(c[0], c[1], c[2]), fmax3(c[3], c[4], c[5])), fmaxf(c[6], c[7]));
}

// bf16 rounding residual of the 32 values packed in pk.
__device__ __forceinline__ void residual_block32(const uint32_t (&v)[32], uint32_t (&pk)[16]) {
#pragma unroll
    for (int y = 0; y < 16; ++y)
        pk[y] = tc::pack_bf16(__uint_as_float(v[2 * y]) - tc::bf16_lo_to_f32(pk[y]),
                              __uint_as_float(v[2 * y + 1]) - tc::bf16_hi_to_f32(pk[y]));
}

template <int D, bool CAUSAL, bool RHO>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmR,
                        const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmO, const TcArgs a) {
    using LY = PairLayout<D, RHO>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LY::BAR_OFF);
    uint64_t* q_full = bars;
    uint64_t* k_full = bars + LY::B_KFULL;
    uint64_t* v_full = bars + LY::B_VFULL;
    uint64_t* k_empty = bars + LY::B_KEMPTY;
    uint64_t* v_empty = bars + LY::B_VEMPTY;
    uint64_t* s_full = bars + LY::B_SFULL;
    uint64_t* p_full = bars + LY::B_PFULL;
    uint64_t* o_full = bars + LY::B_OFULL;
    uint64_t* o_full0 = bars + LY::B_OFULL0;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + LY::NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    // CTA -> (head, query block): heads in groups of kHeadGroup, heaviest
    // block (most key tiles) first within a group, so that the CTAs resident
    // at any time share the K/V of a few heads in L2.
    const int n_qb = a.n_qb;
    const int group = blockIdx.x / (kHeadGroup * n_qb);
    const int gsize = min(kHeadGroup, a.BH - group * kHeadGroup);
    const int r_in = blockIdx.x - group * kHeadGroup * n_qb;
    const int qb = CAUSAL ? n_qb - 1 - r_in / gsize : r_in / gsize;
    const int bh = group * kHeadGroup + r_in % gsize;
    const int q0 = qb * LY::BLOCK;
    // keys: `off` cached ones (chunked prefill) followed by the L rows of this call;
    // query row i sits at key position off + i
    // (a cached prefix only exists for causal attention)
    const int off = CAUSAL ? cached_keys(a, bh, &g_tc_err, threadIdx.x == 0) : 0;
    const int Lk = off + a.L;
    // key tiles of each sub-tile: causal rows q0 + QROWS*sub .. see keys up to
    // their own position (the last tile is the diagonal one); sub-tile 0 may need
    // one tile fewer than sub-tile 1
    const int n_all = (Lk + BN - 1) / BN;
    const int n1 = CAUSAL ? min(n_all, (off + q0 + LY::BLOCK - 1) / BN + 1) : n_all;
    const int n0 = CAUSAL ? min(n1, (off + q0 + LY::QROWS - 1) / BN + 1) : n_all;
    const bool precise = RHO && n1 == 1;

    // The first Q, K and V loads go out before the CTA-wide set-up (TMEM allocation and
    // the barrier below): thread 0 initialises the barriers and issues them, and the
    // producer loops continue after these tiles.
    const int k_pre = min(n1, kKStages), v_pre = min(n1, kVStages);
    if (threadIdx.x == 0) {
        for (int b = 0; b < LY::NBARS; ++b)
            mbar_init(&bars[b], (b == LY::B_PFULL || b == LY::B_PFULL + 1) ? 128 : 1);
        const bool abort0 = (*(volatile unsigned*)&g_tc_err & PARALLAX_DEVERR_WAIT_TIMEOUT) != 0;
        *abort_flag = abort0 ? 1 : 0;
        fence_mbar_init();
        tc::prefetch_tmap(&tmQ);
        if (RHO) tc::prefetch_tmap(&tmR);
        tc::prefetch_tmap(&tmK);
        tc::prefetch_tmap(&tmV);
        tc::prefetch_tmap(&tmO);
        if (!abort0) {
            mbar_arrive_expect_tx(q_full, 2 * LY::OP_BYTES);
            for (int sub = 0; sub < 2; ++sub)
                for (int cb = 0; cb < LY::NCB; ++cb) {
                    unsigned char* dst = smem + LY::QR_OFF + sub * LY::OP_BYTES + cb * LY::SUB_BYTES;
                    if (RHO) {
                        for (int g = 0; g < 4; ++g) {
                            const int row = q0 + 64 * sub + 16 * g;
                            tc::tma_load_3d(dst + (32 * g) * 128, &tmQ, cb * 64, row, bh, q_full);
                            tc::tma_load_3d(dst + (32 * g + 16) * 128, &tmR, cb * 64, row, bh, q_full);
                        }
                    } else {
                        tc::tma_load_3d(dst, &tmQ, cb * 64, q0 + 128 * sub, bh, q_full);
                    }
                }
            for (int j = 0; j < k_pre; ++j) {
                mbar_arrive_expect_tx(&k_full[j], LY::OP_BYTES);
                for (int cb = 0; cb < LY::NCB; ++cb)
                    tc::tma_load_3d(smem + LY::K_OFF + j * LY::OP_BYTES + cb * LY::SUB_BYTES, &tmK,
                                    cb * 64, j * BN, bh, &k_full[j]);
            }
            for (int j = 0; j < v_pre; ++j) {
                mbar_arrive_expect_tx(&v_full[j], LY::OP_BYTES);
                for (int cb = 0; cb < LY::NCB; ++cb)
                    tc::tma_load_3d(smem + LY::V_OFF + j * LY::OP_BYTES + cb * LY::SUB_BYTES, &tmV,
                                    cb * 64, j * BN, bh, &v_full[j]);
            }
        }
    }
    if (warp == 1) tc::tmem_alloc(tmem_slot, 512);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const bool skip = *abort_flag != 0;
    if (warp < 4) {
        tc::setmaxnreg_dec<kRegsSupport>();
        if (warp == 0) {
            // ------------------------------------------------------------ TMA producer: K
            // (Q and the first k_pre K tiles went out at set-up)
            if (lane == 0 && !skip) {
                const int z = bh;
                bool ok = true;
                int kj = k_pre;  // K tiles issued
                for (int j = k_pre; j < n1; ++j) {
                    const int st = j % kKStages;
                    if (j >= kKStages &&
                        !mbar_wait(&k_empty[st], (j / kKStages - 1) & 1, &g_tc_err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&k_full[st], LY::OP_BYTES);
                    for (int cb = 0; cb < LY::NCB; ++cb)
                        tc::tma_load_3d(smem + LY::K_OFF + st * LY::OP_BYTES + cb * LY::SUB_BYTES,
                                        &tmK, cb * 64, j * BN, z, &k_full[st]);
                    kj = j + 1;
                }
                if (!ok) {
                    *abort_flag = 1;
                    // wait (bounded) for the copies already issued into this CTA's shared memory
                    mbar_wait(q_full, 0, &g_tc_err);
                    for (int k = (kj >= kKStages ? kj - kKStages : 0); k < kj; ++k)
                        mbar_wait(&k_full[k % kKStages], (k / kKStages) & 1, &g_tc_err);
                }
            }
        } else if (warp == 2) {
            // ------------------------------------------------------------ TMA producer: V
            // (the first v_pre V tiles went out at set-up)
            if (lane == 0 && !skip) {
                bool ok = true;
                int vj = v_pre;  // V tiles issued
                for (int j = v_pre; j < n1; ++j) {
                    const int st = j % kVStages;
                    if (j >= kVStages &&
                        !mbar_wait(&v_empty[st], (j / kVStages - 1) & 1, &g_tc_err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&v_full[st], LY::OP_BYTES);
                    for (int cb = 0; cb < LY::NCB; ++cb)
                        tc::tma_load_3d(smem + LY::V_OFF + st * LY::OP_BYTES + cb * LY::SUB_BYTES,
                                        &tmV, cb * 64, j * BN, bh, &v_full[st]);
                    vj = j + 1;
                }
                if (!ok) {
                    *abort_flag = 1;
                    for (int k = (vj >= kVStages ? vj - kVStages : 0); k < vj; ++k)
                        mbar_wait(&v_full[k % kVStages], (k / kVStages) & 1, &g_tc_err);
                }
            }
        } else if (warp == 1) {
            // ------------------------------------------------------------ MMA issuer
            // (the whole warp runs this; one elected lane issues each MMA and commit)
            if (!skip) {
                constexpr uint32_t kIdesc1 = tc::idesc_bf16_f32(128, BN, false);
                constexpr uint32_t kIdesc2 = tc::idesc_bf16_f32(128, D, true);
                const uint32_t sbase = smem_u32(smem);
                // descriptors: one base each; a stage / sub-tile / K-step only adds a
                // constant to the 16-byte start-address field
                const uint64_t dQR0 = tc::smem_desc_sw128(sbase + LY::QR_OFF, 16, 1024);
                const uint64_t dK0 = tc::smem_desc_sw128(sbase + LY::K_OFF, 16, 1024);
                const uint64_t dV0 = tc::smem_desc_sw128(sbase + LY::V_OFF, LY::SUB_BYTES, 1024);
                constexpr uint32_t kOpStep = LY::OP_BYTES >> 4;
                // (the per-call bases pass through tc::opaque so that the compiler
                // does not hoist every K-step's descriptor out of the tile loop and
                // keep them all live in registers)
                auto mma1 = [&](int sub, int st) {  // D_sub = A_sub K^T
                    const uint64_t dA = tc::opaque(dQR0 + (uint32_t)sub * kOpStep);
                    const uint64_t dB = tc::opaque(dK0 + (uint32_t)st * kOpStep);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = ((kk / 4) * LY::SUB_BYTES + (kk % 4) * 32) >> 4;
                        tc::mma_ss(tmem + LY::dcol(sub), dA + off, dB + off, kIdesc1, kk > 0);
                    }
                };
                auto mma2 = [&](int sub, int st, bool first) {  // O_sub += [P;PR]_sub V
                    const uint64_t dB = tc::opaque(dV0 + (uint32_t)st * kOpStep);
                    const uint32_t acc0 = first ? 0u : 1u;
                    if (precise) {
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk) {
                            const uint32_t off = (kk * 16 * 128) >> 4;
                            tc::mma_ts(tmem + LY::ocol(sub), tmem + LY::dcol(sub) + kk * 8,
                                       dB + off, kIdesc2, kk == 0 ? acc0 : 1u);
                            tc::mma_ts(tmem + LY::ocol(sub), tmem + LY::dcol(sub) + 64 + kk * 8,
                                       dB + off, kIdesc2, 1u);
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk) {
                            const uint32_t off = (kk * 16 * 128) >> 4;
                            tc::mma_ts(tmem + LY::ocol(sub), tmem + LY::dcol(sub) + kk * 8,
                                       dB + off, kIdesc2, kk == 0 ? acc0 : 1u);
                        }
                    }
                };
                bool ok = mbar_wait_warp(q_full, 0, &g_tc_err) &&
                          mbar_wait_warp(&k_full[0], 0, &g_tc_err);
                tc::fence_after_sync();
                if (ok) {
                    mma1(0, 0);
                    tc::commit(&s_full[0]);
                    mma1(1, 0);
                    tc::commit(&s_full[1]);
                    tc::commit(&k_empty[0]);
                }
                bool o0_committed = false;
                for (int j = 0; j < n1 && ok; ++j) {
                    const int vs = j % kVStages, ks = (j + 1) % kKStages;  // V of j, K of j + 1
                    const bool do0 = j < n0, more0 = j + 1 < n0, more1 = j + 1 < n1;
                    // V first: it is normally resident long before P is ready
                    if (!mbar_wait_warp(&v_full[vs], (j / kVStages) & 1, &g_tc_err)) {
                        ok = false;
                        break;
                    }
                    if (do0) {
                        if (!mbar_wait_warp(&p_full[0], j & 1, &g_tc_err)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after_sync();
                        mma2(0, vs, j == 0);
                        if constexpr (!RHO) {  // sub-tile 0's output may be staged early
                            if (j + 1 == n0) {
                                tc::commit(o_full0);
                                o0_committed = true;
                            }
                        }
                    }
                    if (more1 &&
                        !mbar_wait_warp(&k_full[ks], ((j + 1) / kKStages) & 1, &g_tc_err)) {
                        ok = false;
                        break;
                    }
                    if (more0) {
                        tc::fence_after_sync();
                        mma1(0, ks);  // in order after mma2(0): P_0 is read before D_0 is rewritten
                        tc::commit(&s_full[0]);
                    }
                    if (!mbar_wait_warp(&p_full[1], j & 1, &g_tc_err)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    mma2(1, vs, j == 0);
                    tc::commit(&v_empty[vs]);
                    if (more1) {
                        mma1(1, ks);
                        tc::commit(&s_full[1]);
                        tc::commit(&k_empty[ks]);
                    }
                }
                if (!RHO && !o0_committed) tc::commit(o_full0);
                tc::commit(o_full);
                if (!ok) {
                    *abort_flag = 1;
                    mbar_wait_warp(o_full, 0, &g_tc_err);  // the MMAs already issued have drained
                }
            }
        }
    } else {
        tc::setmaxnreg_inc<kRegsSoftmax>();
        // ---------------------------------------------------------------- softmax / epilogue
        const int sub = (warp - 4) >> 2;
        const int g = warp & 3;  // TMEM lane quarter of this warp
        const int n_tiles = sub ? n1 : n0;
        const int first_row = q0 + LY::QROWS * sub;  // first query of this sub-tile
        const float qs = a.qscale;
        const float2 qs2 = make_float2(qs, qs);
        float m = -INFINITY, l = 0.f;
        bool ok = !skip;
        if constexpr (RHO) {
            const int h = lane >> 4;              // which half of the key (and d) columns
            const int i = first_row + 16 * g + (lane & 15);  // query index
            const uint32_t rowS = tmem + ((uint32_t)(32 * g) << 16);
            const uint32_t rowR = tmem + ((uint32_t)(32 * g + 16) << 16);
            const uint32_t tS = rowS + LY::dcol(sub), tR = rowR + LY::dcol(sub);
            const uint32_t tU = rowS + LY::ocol(sub), tW = rowR + LY::ocol(sub);
            float A = 0.f, c = 0.f;
            for (int it = 0; it < n_tiles && ok; ++it) {
                // this thread owns keys it*128 + 64h + 32b + x, b in {0,1}, x in [0,32)
                const int k0 = it * BN + 64 * h;
                const bool got = !*abort_flag && mbar_wait(&s_full[sub], it & 1, &g_tc_err);
                if (!__all_sync(kFullMask, got)) {  // warp-uniform exit
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                // S and R of this thread's 64 keys, behind a single wait
                uint32_t sv[2][32], rv[2][32];
                tc::tmem_ld32_split<64>(tS, sv[0]);
                tc::tmem_ld32_split<64>(tS + 32, sv[1]);
                tc::tmem_ld32_split<64>(tR, rv[0]);
                tc::tmem_ld32_split<64>(tR + 32, rv[1]);
                tc::tmem_ld_wait();

                // causal: keys past the row's position (for a real row that includes every
                // key >= Lk; padding rows past L may see zero-filled keys); full: keys >= Lk
                const bool need_mask = CAUSAL ? it * BN + BN - 1 > off + first_row : it * BN + BN > Lk;
                if (need_mask) {
                    const int lim = CAUSAL ? off + i : Lk - 1;
#pragma unroll
                    for (int b = 0; b < 2; ++b)
#pragma unroll
                        for (int x = 0; x < 32; ++x) {
                            const int key = k0 + 32 * b + x;
                            if (key > lim)
                                sv[b][x] = __float_as_uint(-INFINITY);
                        }
                }
                // row max: this thread's half of the row, then the other half's
                float mx = max_blocks<2>(sv);
                mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 16)) * qs;
                if (it == 0) {
                    m = mx;
                } else if (__any_sync(kFullMask, mx > m + kRescaleThreshold)) {
                    // TMEM accesses are warp-collective: the whole warp rescales, rows
                    // whose max did not grow use alpha = 1
                    const float m_new = fmaxf(m, mx);
                    const float alpha = fast_exp2(m - m_new);
                    l *= alpha;
                    A *= alpha;
#pragma unroll 1
                    for (int b = 0; b < D / 64; ++b) {
                        uint32_t u[32];
                        tc::tmem_ld32_split<D / 2>(tU + 32 * b, u);
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int x = 0; x < 32; ++x) u[x] = __float_as_uint(__uint_as_float(u[x]) * alpha);
                        tc::tmem_st32_split<D / 2>(tU + 32 * b, u);
                        tc::tmem_ld32_split<D / 2>(tW + 32 * b, u);
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int x = 0; x < 32; ++x) u[x] = __float_as_uint(__uint_as_float(u[x]) * alpha);
                        tc::tmem_st32_split<D / 2>(tW + 32 * b, u);
                    }
                    m = m_new;
                }
                // P -> packed columns 16b.. of this thread's half of the row (split 32);
                // p overwrites s in registers
                const float2 nm2 = make_float2(-m, -m);
                float2 ls0 = make_float2(0.f, 0.f), ls1 = make_float2(0.f, 0.f);
                auto do_p = [&](int b) {
                    uint32_t pk[16];
                    exp_block32(sv[b], qs2, nm2, ls0, ls1, pk);
                    tc::tmem_st16_split<32>(tS + 16 * b, pk);
                    if (precise) {
                        residual_block32(sv[b], pk);
                        tc::tmem_st16_split<32>(tS + 64 + 16 * b, pk);
                    }
                };
                // PR = p (r - c) -> packed columns of the R rows.  R was read in full
                // above, so these stores may land on columns that the other half of
                // the row read as R.
                float2 as0 = make_float2(0.f, 0.f), as1 = make_float2(0.f, 0.f);
                auto do_pr = [&](int b) {
                    const float2 nc2 = make_float2(-c, -c);
                    uint32_t pk[16];
#pragma unroll
                    for (int y = 0; y < 16; ++y) {
                        const float2 p2 = make_float2(__uint_as_float(sv[b][2 * y]),
                                                      __uint_as_float(sv[b][2 * y + 1]));
                        const float2 r2 = make_float2(__uint_as_float(rv[b][2 * y]),
                                                      __uint_as_float(rv[b][2 * y + 1]));
                        const float2 pr = __fmul2_rn(p2, __fadd2_rn(r2, nc2));
                        rv[b][2 * y] = __float_as_uint(pr.x);
                        rv[b][2 * y + 1] = __float_as_uint(pr.y);
                        if (y & 1) as1 = __fadd2_rn(as1, pr);
                        else as0 = __fadd2_rn(as0, pr);
                        pk[y] = tc::pack_bf16(pr.x, pr.y);
                    }
                    tc::tmem_st16_split<32>(tR + 16 * b, pk);
                    if (precise) {
                        residual_block32(rv[b], pk);
                        tc::tmem_st16_split<32>(tR + 64 + 16 * b, pk);
                    }
                };
                if (it == 0) {
                    // row shift c: p-weighted mean of r over the first (full) key tile,
                    // needed before any PR
                    do_p(0);
                    do_p(1);
                    float2 pr0 = make_float2(0.f, 0.f), pr1 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int b = 0; b < 2; ++b)
#pragma unroll
                        for (int y = 0; y < 16; ++y) {
                            const float2 p2 = make_float2(__uint_as_float(sv[b][2 * y]),
                                                          __uint_as_float(sv[b][2 * y + 1]));
                            const float2 r2 = make_float2(__uint_as_float(rv[b][2 * y]),
                                                          __uint_as_float(rv[b][2 * y + 1]));
                            if (y & 1) pr1 = __ffma2_rn(p2, r2, pr1);
                            else pr0 = __ffma2_rn(p2, r2, pr0);
                        }
                    const float2 ls = __fadd2_rn(ls0, ls1);
                    const float2 pr = __fadd2_rn(pr0, pr1);
                    float prs = pr.x + pr.y;
                    prs += __shfl_xor_sync(kFullMask, prs, 16);
                    c = prs / (ls.x + ls.y + __shfl_xor_sync(kFullMask, ls.x + ls.y, 16));
                    do_pr(0);
                    do_pr(1);
                } else {
                    // one pass per 32-key block keeps fewer values live
                    do_p(0);
                    do_pr(0);
                    do_p(1);
                    do_pr(1);
                }
                const float2 ls = __fadd2_rn(ls0, ls1);
                const float2 as = __fadd2_rn(as0, as1);
                l += ls.x + ls.y;
                A += as.x + as.y;
                tc::tmem_st_wait();
                tc::fence_before_sync();
                mbar_arrive(&p_full[sub]);
            }

            // ---- epilogue: o = U/l - (W/l - (A/l)(U/l)) = ((U (1 + A/l)) - W) / l
            const bool done = ok && !*abort_flag && mbar_wait(o_full, 0, &g_tc_err);
            const int rl = 16 * g + (lane & 15);  // row within the sub-tile
            // 32-column box cb of this sub-tile's staged output: the two sub-tiles have the same
            // number of key tiles here, so both stage into the K/V rings once every MMA has
            // completed
            auto box_at = [&](int cb) -> unsigned char* {
                return smem + LY::K_OFF + (sub * (D / 32) + cb) * LY::OUT_BOX;
            };
            if (__all_sync(kFullMask, done)) {
                tc::fence_after_sync();
                const float lt = l + __shfl_xor_sync(kFullMask, l, 16);
                const float At = A + __shfl_xor_sync(kFullMask, A, 16);
                const float inv_l = 1.f / lt;
                const float gain = 1.f + At * inv_l;
                const bool row_ok =
                    i < a.L && in_bounds(&g_tc_err, ((size_t)bh * a.L + i + 1) * D, (size_t)a.BH * a.L * D);
                // all of this thread's U and W columns behind one wait
                uint32_t uu[D / 64][32], ww[D / 64][32];
#pragma unroll
                for (int b = 0; b < D / 64; ++b) {
                    tc::tmem_ld32_split<D / 2>(tU + 32 * b, uu[b]);
                    tc::tmem_ld32_split<D / 2>(tW + 32 * b, ww[b]);
                }
                tc::tmem_ld_wait();
#pragma unroll
                for (int b = 0; b < D / 64; ++b) {
                    const uint32_t(&u)[32] = uu[b];
                    const uint32_t(&w)[32] = ww[b];
                    // columns h D/2 + 32 b .. : 32-column box h (D/64) + b
                    unsigned char* box = box_at(h * (D / 64) + b) + rl * 128;
#pragma unroll
                    for (int x = 0; x < 8; ++x) {
                        float out[4];
#pragma unroll
                        for (int y = 0; y < 4; ++y)
                            out[y] = (__uint_as_float(u[4 * x + y]) * gain - __uint_as_float(w[4 * x + y])) *
                                     inv_l;
                        *reinterpret_cast<float4*>(box + ((x ^ (rl & 7)) << 4)) =
                            make_float4(out[0], out[1], out[2], out[3]);
                    }
                    if (a.mu && row_ok) {
                        float* mrow = a.mu + ((size_t)bh * a.L + i) * D + h * (D / 2);
#pragma unroll
                        for (int x = 0; x < 32; x += 4)
                            *reinterpret_cast<float4*>(mrow + 32 * b + x) = make_float4(
                                __uint_as_float(u[x]) * inv_l, __uint_as_float(u[x + 1]) * inv_l,
                                __uint_as_float(u[x + 2]) * inv_l, __uint_as_float(u[x + 3]) * inv_l);
                    }
                }
                if (a.lse && h == 0 && row_ok) {
                    a.lse[(size_t)bh * a.L + i] = (m + __log2f(lt)) * kLn2;
                    a.rbar[(size_t)bh * a.L + i] = At * inv_l + c;
                }
            } else {
                *abort_flag = 1;
            }
            // this warp's rows, once all of its threads have written them (rows past L are
            // clipped by the tensor map)
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && !*abort_flag) {
                const uint64_t pol = l2_evict_first_policy();
#pragma unroll 1
                for (int cb = 0; cb < D / 32; ++cb)
                    tc::tma_store_3d_hint(&tmO, 32 * cb, first_row + LY::WROWS * g, bh,
                                          box_at(cb) + LY::WROWS * g * 128, pol);
                tc::bulk_commit_group();
                tc::bulk_wait_group_read0();
            }
        } else {
            // ------------------------------------------------ W_R = 0: one query row per thread
            const int i = first_row + 32 * g + lane;
            const uint32_t row = tmem + ((uint32_t)(32 * g) << 16);
            const uint32_t tS = row + LY::dcol(sub), tU = row + LY::ocol(sub);
            for (int it = 0; it < n_tiles && ok; ++it) {
                const int k0 = it * BN;
                const bool got = !*abort_flag && mbar_wait(&s_full[sub], it & 1, &g_tc_err);
                if (!__all_sync(kFullMask, got)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                uint32_t sv[4][32];
                const bool need_mask = CAUSAL ? k0 + BN - 1 > off + first_row : k0 + BN > Lk;
                // S of the tile into registers, masked
                auto load_s = [&]() {
#pragma unroll
                    for (int b = 0; b < 4; ++b) tc::tmem_ld32(tS + 32 * b, sv[b]);
                    tc::tmem_ld_wait();
                    if (need_mask) {
                        const int lim = CAUSAL ? off + i : Lk - 1;
#pragma unroll
                        for (int b = 0; b < 4; ++b)
#pragma unroll
                            for (int x = 0; x < 32; ++x)
                                if (k0 + 32 * b + x > lim) sv[b][x] = __float_as_uint(-INFINITY);
                    }
                };
                float2 ls0, ls1;
                uint32_t pk[4][16];  // P as bf16 pairs: keys 32b.. -> packed columns 16b..
                auto exps = [&]() {
                    const float2 nm2 = make_float2(-m, -m);
                    ls0 = ls1 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int b = 0; b < 4; ++b) exp_block32(sv[b], qs2, nm2, ls0, ls1, pk[b]);
                };
                // the row maximum sets m (first tile) or, when it exceeds m by more than the
                // lazy-rescale threshold, moves m and rescales U and l
                auto max_pass = [&]() {
                    const float mx = max_blocks<4>(sv) * qs;
                    if (it == 0) {
                        m = mx;
                    } else if (__any_sync(kFullMask, mx > m + kRescaleThreshold)) {
                        const float m_new = fmaxf(m, mx);
                        const float alpha = fast_exp2(m - m_new);
                        l *= alpha;
#pragma unroll 1
                        for (int b = 0; b < D / 32; ++b) {
                            uint32_t u[32];
                            tc::tmem_ld32(tU + 32 * b, u);
                            tc::tmem_ld_wait();
#pragma unroll
                            for (int x = 0; x < 32; ++x) u[x] = __float_as_uint(__uint_as_float(u[x]) * alpha);
                            tc::tmem_st32(tU + 32 * b, u);
                        }
                        m = m_new;
                    }
                };
                load_s();
                if (it == 0) {
                    max_pass();
                    exps();
                } else {
                    // Later tiles skip the row maximum: P is taken against the running m,
                    // and a row whose P sums to at most 2^8 has no p above 2^8, i.e. its
                    // maximum has not passed m by more than the lazy-rescale threshold and
                    // these are the values the maximum would have given.  Otherwise (rare)
                    // the maximum is formed from S, reloaded from TMEM (P is stored below).
                    exps();
                    const float2 lt = __fadd2_rn(ls0, ls1);
                    if (__any_sync(kFullMask, lt.x + lt.y > 256.f)) {
                        load_s();
                        max_pass();
                        exps();
                    }
                }
#pragma unroll
                for (int b = 0; b < 4; ++b) tc::tmem_st16(tS + 16 * b, pk[b]);
                const float2 ls = __fadd2_rn(ls0, ls1);
                l += ls.x + ls.y;
                tc::tmem_st_wait();
                tc::fence_before_sync();
                mbar_arrive(&p_full[sub]);
            }
            // ---- epilogue: o = U / l
            const bool done = ok && !*abort_flag && mbar_wait(sub ? o_full : o_full0, 0, &g_tc_err);
            const int rl = 32 * g + lane;  // row within the sub-tile
            // 32-column box cb of this sub-tile's staged output
            auto box_at = [&](int cb) -> unsigned char* {
                return sub ? smem + LY::V_OFF + cb * LY::OUT_BOX
                           : smem + LY::K_OFF +
                                 ((n1 + cb / LY::BOXES_PER_K_STAGE) % kKStages) * LY::OP_BYTES +
                                 (cb % LY::BOXES_PER_K_STAGE) * LY::OUT_BOX;
            };
            if (__all_sync(kFullMask, done)) {
                tc::fence_after_sync();
                const float inv_l = 1.f / l;
                const bool row_ok =
                    i < a.L && in_bounds(&g_tc_err, ((size_t)bh * a.L + i + 1) * D, (size_t)a.BH * a.L * D);
                // all of this thread's U columns behind one wait
                uint32_t uu[D / 32][32];
#pragma unroll
                for (int b = 0; b < D / 32; ++b) tc::tmem_ld32(tU + 32 * b, uu[b]);
                tc::tmem_ld_wait();
#pragma unroll
                for (int b = 0; b < D / 32; ++b) {
                    const uint32_t(&u)[32] = uu[b];
                    unsigned char* box = box_at(b) + rl * 128;
#pragma unroll
                    for (int x = 0; x < 8; ++x) {
                        const float4 v4 = make_float4(
                            __uint_as_float(u[4 * x]) * inv_l, __uint_as_float(u[4 * x + 1]) * inv_l,
                            __uint_as_float(u[4 * x + 2]) * inv_l, __uint_as_float(u[4 * x + 3]) * inv_l);
                        *reinterpret_cast<float4*>(box + ((x ^ (rl & 7)) << 4)) = v4;
                        if (a.mu && row_ok)
                            *reinterpret_cast<float4*>(a.mu + ((size_t)bh * a.L + i) * D + 32 * b + 4 * x) = v4;
                    }
                }
                if (a.lse && row_ok) {
                    a.lse[(size_t)bh * a.L + i] = (m + __log2f(l)) * kLn2;
                    a.rbar[(size_t)bh * a.L + i] = 0.f;
                }
            } else {
                *abort_flag = 1;
            }
            // this warp's rows, once all of its threads have written them (rows past L are
            // clipped by the tensor map)
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && !*abort_flag) {
                const uint64_t pol = l2_evict_first_policy();
#pragma unroll 1
                for (int cb = 0; cb < D / 32; ++cb)
                    tc::tma_store_3d_hint(&tmO, 32 * cb, first_row + LY::WROWS * g, bh,
                                          box_at(cb) + LY::WROWS * g * 128, pol);
                tc::bulk_commit_group();
                tc::bulk_wait_group_read0();
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- host side
// [B*H, L, D] bf16 viewed as a 3-D tensor; box = 64 columns (128 bytes) x box_rows rows x 1 head,
// 128-byte swizzle; rows past L read as zeros.
bool make_map(CUtensorMap* m, const void* base, int BH, int L, int D, int box_rows = 128) {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)L, (uint64_t)BH};
    const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)L * D * 2};
    const uint32_t box[3] = {64, (uint32_t)box_rows, 1};
    return make_tmap_bf16(m, base, 3, dims, strides, box);
}

template <int D, bool CAUSAL, bool RHO>
cudaError_t launch(const CUtensorMap& mq, const CUtensorMap& mr, const CUtensorMap& mk,
                   const CUtensorMap& mv, const CUtensorMap& mo, const TcArgs& a,
                   cudaStream_t stream) {
    using LY = PairLayout<D, RHO>;
    auto kern = prefill_pair_kernel<D, CAUSAL, RHO>;
    static std::atomic<uint64_t> smem_set{0};
    if (cudaError_t e = ensure_dynamic_smem(kern, (int)LY::SMEM_BYTES, smem_set)) return e;
    const unsigned grid = (unsigned)((size_t)a.n_qb * a.BH);
    kern<<<grid, kThreads, LY::SMEM_BYTES, stream>>>(mq, mr, mk, mv, mo, a);
    return cudaGetLastError();
}

template <int D, bool RHO>
cudaError_t launch_d(const PrefillShape& s, const CUtensorMap& mq, const CUtensorMap& mr,
                     const CUtensorMap& mk, const CUtensorMap& mv, float* o,
                     const int32_t* cache_lens, int Lcap, const TrainStats& ts,
                     cudaStream_t stream) {
    using LY = PairLayout<D, RHO>;
    const TcArgs a{o,      cache_lens, s.L,    Lcap,  s.H,  s.B * s.H, (s.L + LY::BLOCK - 1) / LY::BLOCK,
                   s.scale * kLog2e, ts.lse, ts.rbar, ts.mu};
    // o [B*H, L, D] fp32 for the TMA stores of the epilogue: boxes of 32 columns x WROWS rows
    // (one softmax warp's rows)
    CUtensorMap mo;
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)s.L, (uint64_t)s.B * s.H};
    const uint64_t strides[2] = {(uint64_t)D * 4, (uint64_t)s.L * D * 4};
    const uint32_t box[3] = {32, (uint32_t)LY::WROWS, 1};
    if (!make_tmap_f32(&mo, o, 3, dims, strides, box)) return cudaErrorInvalidValue;
    return s.causal ? launch<D, true, RHO>(mq, mr, mk, mv, mo, a, stream)
                    : launch<D, false, RHO>(mq, mr, mk, mv, mo, a, stream);
}

// Query-side maps (q, rho: L rows per head) and key-side maps (k, v: Lcap rows per head).
cudaError_t launch_any(const PrefillShape& s, const void* q, const void* rho, const void* k,
                       const void* v, float* o, const int32_t* cache_lens, int Lcap,
                       cudaStream_t stream, const TrainStats& ts = TrainStats{}) {
    const int BH = s.B * s.H;
    CUtensorMap mq, mr, mk, mv;
    if (!make_map(&mk, k, BH, Lcap, s.d) || !make_map(&mv, v, BH, Lcap, s.d))
        return cudaErrorInvalidValue;
    if (rho) {
        // correction path: query and probe maps use 16-row boxes (stacked operand)
        if (!make_map(&mq, q, BH, s.L, s.d, 16) || !make_map(&mr, rho, BH, s.L, s.d, 16))
            return cudaErrorInvalidValue;
        if (s.d == 64) return launch_d<64, true>(s, mq, mr, mk, mv, o, cache_lens, Lcap, ts, stream);
        if (s.d == 128) return launch_d<128, true>(s, mq, mr, mk, mv, o, cache_lens, Lcap, ts, stream);
        return cudaErrorInvalidValue;
    }
    if (!make_map(&mq, q, BH, s.L, s.d)) return cudaErrorInvalidValue;
    mr = mq;  // unused
    if (s.d == 64) return launch_d<64, false>(s, mq, mr, mk, mv, o, cache_lens, Lcap, ts, stream);
    if (s.d == 128) return launch_d<128, false>(s, mq, mr, mk, mv, o, cache_lens, Lcap, ts, stream);
    return cudaErrorInvalidValue;
}

// Copy the chunk's K and V rows [B, H, L, D] into the caches [B, H, Lcap, D] at rows
// cache_lens[b] .. cache_lens[b] + L - 1 (16-byte vectors, grid-stride), and zero the
// cache rows from there up to the end of that 128-key tile (at most Lcap): the
// attention kernel multiplies those rows by zero weights, and they must not hold
// NaN or Inf left over in unwritten memory.  A length that leaves no room for the
// chunk is clamped exactly as the attention kernel does.
constexpr int kPadRows = BN - 1;
__global__ void __launch_bounds__(256) append_kernel(const uint4* __restrict__ k_new,
                                                     const uint4* __restrict__ v_new,
                                                     uint4* __restrict__ k_cache,
                                                     uint4* __restrict__ v_cache,
                                                     const int32_t* __restrict__ cache_lens, int H,
                                                     int L, int Lcap, int vec_per_row,
                                                     size_t total_vec) {
    const int rows = L + kPadRows;  // per head: the chunk, then the padding of its last tile
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total_vec;
         idx += (size_t)gridDim.x * blockDim.x) {
        const size_t row = idx / vec_per_row;  // (bh, i)
        const int c = (int)(idx - row * vec_per_row);
        const int bh = (int)(row / rows), i = (int)(row - (size_t)bh * rows);
        int off = __ldg(cache_lens + bh / H);
        off = off < 0 ? 0 : (off > Lcap - L ? Lcap - L : off);
        const size_t dst = ((size_t)bh * Lcap + off + i) * vec_per_row + c;
        if (!in_bounds(&g_tc_err, dst + 1, total_vec / rows * Lcap)) continue;
        if (i < L) {
            const size_t src = ((size_t)bh * L + i) * vec_per_row + c;
            k_cache[dst] = k_new[src];
            v_cache[dst] = v_new[src];
        } else {
            const int end = off + L, tile_end = min(Lcap, (end + BN - 1) / BN * BN);
            if (off + i < tile_end) {
                k_cache[dst] = make_uint4(0, 0, 0, 0);
                v_cache[dst] = make_uint4(0, 0, 0, 0);
            }
        }
    }
}

}  // namespace

cudaError_t prefill_tc_launch(const PrefillShape& s, const void* q, const void* rho,
                              const void* k, const void* v, float* o, int /*num_sms*/,
                              cudaStream_t stream, const TrainStats& ts) {
    return launch_any(s, q, rho, k, v, o, nullptr, s.L, stream, ts);
}

cudaError_t prefill_tc_chunk_launch(const PrefillShape& s, const void* q, const void* rho,
                                    const void* k_new, const void* v_new, void* k_cache,
                                    void* v_cache, const int32_t* cache_lens, int Lmax, float* o,
                                    int num_sms, cudaStream_t stream) {
    const int vec_per_row = s.d * 2 / 16;
    const size_t total_vec = (size_t)s.B * s.H * (s.L + kPadRows) * vec_per_row;
    const size_t want = (total_vec + 255) / 256;
    const unsigned grid = (unsigned)(want < (size_t)num_sms * 8 ? want : (size_t)num_sms * 8);
    append_kernel<<<grid, 256, 0, stream>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), cache_lens, s.H, s.L, Lmax,
        vec_per_row, total_vec);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_any(s, q, rho, k_cache, v_cache, o, cache_lens, Lmax, stream);
}

// Self-test of the bounded wait for the tensor-core prefill's error word (see
// decode_wait_selftest); later prefill CTAs see the bit, skip their work, free their
// TMEM and return.
namespace {
__global__ void tc_wait_selftest_kernel(uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        mbar_wait(&bar, 0, &g_tc_err, limit_ns);
    }
}
}  // namespace

cudaError_t prefill_tc_wait_selftest(uint64_t limit_ns, cudaStream_t stream) {
    tc_wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
    return cudaGetLastError();
}

unsigned prefill_tc_take_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_err, sizeof(v)) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_tc_err, &zero, sizeof(zero));
    return v;
}

}  // namespace parallax
