// One warp streaming keys/values out of shared memory for ONE query row,
// updating the online state of both Parallax branches from the same K/V bytes.
//
// State (log2 domain, s_j = (scale*log2 e) q.k_j, r_j = rho.k_j):
//   m          running max of s
//   l = sum 2^(s_j-m)          A = sum 2^(s_j-m) r_j
//   U = sum 2^(s_j-m) v_j      W = sum 2^(s_j-m) r_j v_j
// and at the end   o = U/l - (W/l - (A/l)(U/l))   -- softmax attention minus
// the probe-projected key/value covariance (Parallax, "Parallax mantem
// softmax ...", paragraph 2), written in the one-pass form
// o = mu_v - (sum p r v - (sum p r) mu_v).
//
// Lane layout: a key row of D elements is read as D/VEC 16-byte vectors, one
// per lane, so LPK = D/VEC lanes cover one key and a warp covers KPS = 32/LPK
// keys per step.  Lane (g, e) = (lane / LPK, lane % LPK) owns elements
// [e*VEC, e*VEC+VEC) of the keys of group g.  A block is 4 steps = 4*KPS keys.
// The two dot products of the 4 steps are reduced over the LPK lanes by a
// transposing butterfly (each level halves the values held per lane), so a
// block costs 2 + 1 + log2(LPK) - 2 shuffles per dot product instead of
// 4*log2(LPK).
#pragma once

#include "common.cuh"

namespace parallax {

template <typename T, int D>
struct KeyLayout {
    static constexpr int VEC = Vec16<T>::N;                 // elements per 16-byte vector
    static constexpr int LPK = D / VEC;                     // lanes per key
    static constexpr int KPS = 32 / LPK;                    // keys per warp step
    static constexpr int ROW_BYTES = D * (int)sizeof(T);    // bytes per key row
    static constexpr int BLOCK_KEYS = 4 * KPS;              // keys per 4-step block
    static_assert(LPK >= 8 && LPK <= 32, "unsupported (T, D)");
};

template <typename T, int D>
struct RowState {
    static constexpr int VEC = KeyLayout<T, D>::VEC;
    float m, l, A;
    float U[VEC], W[VEC];
    __device__ __forceinline__ void reset() {
        m = -INFINITY;
        l = 0.f;
        A = 0.f;
#pragma unroll
        for (int x = 0; x < VEC; ++x) U[x] = W[x] = 0.f;
    }
};

// Sum v[0..3] over the LPK lanes of a key group; lane e ends up holding the
// complete sum for step 2*bit(LPK/2) + bit(LPK/4) of e.
template <int LPK>
__device__ __forceinline__ float transpose_reduce4(const float (&v)[4], int e) {
    const bool h1 = (e & (LPK / 2)) != 0;
    const float s0 = h1 ? v[0] : v[2], s1 = h1 ? v[1] : v[3];
    float k0 = h1 ? v[2] : v[0], k1 = h1 ? v[3] : v[1];
    k0 += __shfl_xor_sync(kFullMask, s0, LPK / 2);
    k1 += __shfl_xor_sync(kFullMask, s1, LPK / 2);
    const bool h2 = (e & (LPK / 4)) != 0;
    const float s = h2 ? k0 : k1;
    float k = h2 ? k1 : k0;
    k += __shfl_xor_sync(kFullMask, s, LPK / 4);
#pragma unroll
    for (int off = LPK / 8; off >= 1; off >>= 1) k += __shfl_xor_sync(kFullMask, k, off);
    return k;
}

// Process keys kb .. kb + BLOCK_KEYS - 1 of the tiles sK / sV (row-major,
// ROW_BYTES per key); keys with index >= nvalid are masked out (their shared
// memory may hold anything).  qf is pre-scaled by scale*log2(e).
template <typename T, int D, bool RHO>
__device__ __forceinline__ void warp_block(RowState<T, D>& st,
                                           const float (&qf)[KeyLayout<T, D>::VEC],
                                           const float (&rf)[KeyLayout<T, D>::VEC],
                                           const T* sK, const T* sV, int kb, int nvalid,
                                           int lane) {
    using KL = KeyLayout<T, D>;
    constexpr int VEC = KL::VEC, LPK = KL::LPK, KPS = KL::KPS;
    const int g = lane / LPK, e = lane % LPK;

    float sp[4], rp[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const int key = kb + s * KPS + g;
        float kf[VEC];
        Vec16<T>::unpack(ld_shared_16(sK + key * D + e * VEC), kf);
        float a = 0.f, b = 0.f;
#pragma unroll
        for (int x = 0; x < VEC; ++x) {
            a = fmaf(qf[x], kf[x], a);
            if (RHO) b = fmaf(rf[x], kf[x], b);
        }
        sp[s] = a;
        rp[s] = b;
    }
    float s_mine = transpose_reduce4<LPK>(sp, e);
    float r_mine = RHO ? transpose_reduce4<LPK>(rp, e) : 0.f;
    const int my_step = ((e & (LPK / 2)) ? 2 : 0) + ((e & (LPK / 4)) ? 1 : 0);
    const bool valid = (kb + my_step * KPS + g) < nvalid;
    s_mine = valid ? s_mine : -INFINITY;

    // block max over all keys the warp holds
    float mb = fmaxf(s_mine, __shfl_xor_sync(kFullMask, s_mine, LPK / 2));
    mb = fmaxf(mb, __shfl_xor_sync(kFullMask, mb, LPK / 4));
#pragma unroll
    for (int off = LPK; off < 32; off <<= 1) mb = fmaxf(mb, __shfl_xor_sync(kFullMask, mb, off));
    if (mb > st.m) {  // warp-uniform; never taken when every key is masked
        const float alpha = fast_exp2(st.m - mb);
        st.l *= alpha;
        st.A *= alpha;
#pragma unroll
        for (int x = 0; x < VEC; ++x) {
            st.U[x] *= alpha;
            st.W[x] *= alpha;
        }
        st.m = mb;
    }
    const float p = valid ? fast_exp2(s_mine - st.m) : 0.f;
    const float pr = (RHO && valid) ? p * r_mine : 0.f;

    // broadcast the 4 weights of this lane's key group and accumulate values
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const int src = g * LPK + (s >> 1) * (LPK / 2) + (s & 1) * (LPK / 4);
        const float ps = __shfl_sync(kFullMask, p, src);
        const float prs = RHO ? __shfl_sync(kFullMask, pr, src) : 0.f;
        st.l += ps;
        if (RHO) st.A += prs;
        const int key = kb + s * KPS + g;
        if (key < nvalid) {
            float vf[VEC];
            Vec16<T>::unpack(ld_shared_16(sV + key * D + e * VEC), vf);
#pragma unroll
            for (int x = 0; x < VEC; ++x) {
                st.U[x] = fmaf(ps, vf[x], st.U[x]);
                if (RHO) st.W[x] = fmaf(prs, vf[x], st.W[x]);
            }
        }
    }
}

// Sum the per-group partial states of a warp (all groups share m); afterwards
// every group holds the warp total.
template <typename T, int D, bool RHO>
__device__ __forceinline__ void warp_merge_groups(RowState<T, D>& st) {
    using KL = KeyLayout<T, D>;
#pragma unroll
    for (int off = KL::LPK; off < 32; off <<= 1) {
        st.l += __shfl_xor_sync(kFullMask, st.l, off);
        if (RHO) st.A += __shfl_xor_sync(kFullMask, st.A, off);
#pragma unroll
        for (int x = 0; x < KL::VEC; ++x) {
            st.U[x] += __shfl_xor_sync(kFullMask, st.U[x], off);
            if (RHO) st.W[x] += __shfl_xor_sync(kFullMask, st.W[x], off);
        }
    }
}

// Load this lane's VEC-slice of a query-side vector (q or rho) of length D.
template <typename T, int D>
__device__ __forceinline__ void load_row_slice(const T* row, int e, float scale,
                                               float (&out)[KeyLayout<T, D>::VEC]) {
    constexpr int VEC = KeyLayout<T, D>::VEC;
    float f[VEC];
    Vec16<T>::unpack(ld_global_16(row + e * VEC), f);
#pragma unroll
    for (int x = 0; x < VEC; ++x) out[x] = f[x] * scale;
}

// Finished output slice from a merged state: o = U/l - (W/l - (A/l)(U/l)).
// A row with no keys (l == 0) yields 0.
template <typename T, int D, bool RHO>
__device__ __forceinline__ void finish_slice(const RowState<T, D>& st, float* o_slice) {
    constexpr int VEC = KeyLayout<T, D>::VEC;
    const float inv_l = st.l > 0.f ? 1.f / st.l : 0.f;
    const float rbar = st.A * inv_l;
    float out[VEC];
#pragma unroll
    for (int x = 0; x < VEC; ++x) {
        const float mu = st.U[x] * inv_l;
        out[x] = RHO ? mu - (st.W[x] * inv_l - rbar * mu) : mu;
    }
#pragma unroll
    for (int x = 0; x < VEC; x += 4)
        *reinterpret_cast<float4*>(o_slice + x) = make_float4(out[x], out[x + 1], out[x + 2], out[x + 3]);
}

}  // namespace parallax
