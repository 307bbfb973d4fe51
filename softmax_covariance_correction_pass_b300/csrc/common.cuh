// Device helpers shared by the Parallax attention kernels (sm_103a).
//
// Every pipeline wait in these kernels is bounded: a wait that has not
// completed after kWaitLimitNs of wall time records PARALLAX_DEVERR_WAIT_TIMEOUT
// in the device error word and returns false, and the caller then winds its
// CTA down instead of hanging the GPU.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/parallax_attn.h"

namespace parallax {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ----------------------------------------------------------------------------
// host: per-device one-time kernel set-up
// ----------------------------------------------------------------------------
// Raise a kernel's dynamic shared-memory limit to `bytes` on the current device, once per
// device: the attribute is held by each device's context, so a process that launches on
// several devices sets it on each.  `done` is the kernel's own mask of devices already set
// (devices 0..63; a later device sets it on every launch).  Threads racing on a first
// launch may both set it, which is harmless.
template <typename Kernel>
inline cudaError_t ensure_dynamic_smem(Kernel kern, int bytes, std::atomic<uint64_t>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? 1ull << dev : 0ull;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// ----------------------------------------------------------------------------
// error word: one per translation unit, read and cleared by the host
// ----------------------------------------------------------------------------
__device__ __forceinline__ void raise_error(unsigned* err, unsigned bits) { atomicOr(err, bits); }

// Debug builds (-DPARALLAX_DEBUG_CHECKS; `build.py --debug`) check, before each global
// write and bulk copy they cover, that the element range [begin, end) lies inside its
// tensor of `extent` elements.  A failed check raises PARALLAX_DEVERR_BOUNDS in the kernel's
// error word; the caller then skips the write, or points a copy at the start of its tensor
// so that every byte count the pipeline waits for still arrives.  Release builds compile
// the checks away.
#ifdef PARALLAX_DEBUG_CHECKS
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif
__device__ __forceinline__ bool in_bounds(unsigned* err, size_t end, size_t extent) {
    if (!kDebugChecks || end <= extent) return true;
    raise_error(err, PARALLAX_DEVERR_BOUNDS);
    return false;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ----------------------------------------------------------------------------
// shared-memory addresses and mbarriers
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false (and
// raises the timeout bit) if it did not complete within limit_ns.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned* err,
                                          uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    uint32_t n = 0;
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((++n & 63u) == 0 && global_timer_ns() - t0 > limit_ns) {
            raise_error(err, PARALLAX_DEVERR_WAIT_TIMEOUT);
            return false;
        }
    }
}

// Warp-collective form of mbar_wait for code that the whole warp runs (the
// MMA issuer): every lane polls, and the result is the same on all lanes, so
// that a timeout seen by one lane takes the whole warp down the same path.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, unsigned* err) {
    return __all_sync(kFullMask, mbar_wait(bar, parity, err));
}

// ----------------------------------------------------------------------------
// bulk (non-tensor) asynchronous copies global -> shared, completing on an mbarrier
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// ----------------------------------------------------------------------------
// arithmetic helpers
// ----------------------------------------------------------------------------
// 2^x on the SFU (approximate, flushes subnormals; 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max(a, b, c) in one instruction (three-input max of the sm_100 family).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Unpack 16 bytes of T into fp32.
template <typename T>
struct Vec16;

template <>
struct Vec16<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void unpack(const uint4& u, float (&f)[4]) {
        f[0] = __uint_as_float(u.x);
        f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z);
        f[3] = __uint_as_float(u.w);
    }
};

template <>
struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    // bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32 word.
    __device__ __forceinline__ static void unpack(const uint4& u, float (&f)[8]) {
        f[0] = __uint_as_float(u.x << 16);
        f[1] = __uint_as_float(u.x & 0xffff0000u);
        f[2] = __uint_as_float(u.y << 16);
        f[3] = __uint_as_float(u.y & 0xffff0000u);
        f[4] = __uint_as_float(u.z << 16);
        f[5] = __uint_as_float(u.z & 0xffff0000u);
        f[6] = __uint_as_float(u.w << 16);
        f[7] = __uint_as_float(u.w & 0xffff0000u);
    }
};

template <typename T>
__device__ __forceinline__ uint4 ld_shared_16(const T* p) {
    return *reinterpret_cast<const uint4*>(p);
}

template <typename T>
__device__ __forceinline__ uint4 ld_global_16(const T* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

}  // namespace parallax
