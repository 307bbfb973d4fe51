// C-ABI layer of libparallax_attn: argument validation (on the host, before
// anything is launched), split-KV planning, the per-device decode workspace,
// and the device error word.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/parallax_attn.h"
#include "kernels.h"

namespace {

thread_local std::string t_last_error;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return code;
}

int succeed() {
    t_last_error.clear();
    return PARALLAX_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(PARALLAX_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

std::atomic<int> g_chunk_override{0};

struct DeviceState {
    void* ws = nullptr;
    size_t ws_bytes = 0;
    int num_sms = 0;
};
std::mutex g_mu;
std::vector<DeviceState> g_dev;

DeviceState* device_state(int* dev_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if ((int)g_dev.size() <= dev) g_dev.resize(dev + 1);
    DeviceState& s = g_dev[dev];
    if (s.num_sms == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return nullptr;
        s.num_sms = n;
    }
    if (dev_out) *dev_out = dev;
    return &s;
}

// Keys per split-KV chunk.  Aim for about 16 work items per SM so the
// persistent CTAs balance well (also for ragged lengths), with chunks of
// 256..4096 keys: long enough that the 1 KB partial state per chunk is noise
// next to the chunk's K/V bytes.
int plan_chunk(int B, int H, int Lmax, int num_sms) {
    const int forced = g_chunk_override.load();
    int c;
    if (forced > 0) {
        c = forced;
    } else {
        const double per_item = (double)B * H * Lmax / (16.0 * num_sms);
        c = 256;
        while (c < 4096 && (double)(2 * c) <= per_item) c *= 2;
    }
    return c >= Lmax ? Lmax : c;
}

int validate_common(const void* q, const void* k, const void* v, const void* o, const void* rho,
                    int B, int H, int L, int d, const char* Lname) {
    if (!q || !k || !v || !o)
        return fail(PARALLAX_ERR_INVALID, "null tensor pointer (q=%p k=%p v=%p o=%p)", q, k, v, o);
    if (B <= 0 || H <= 0 || L <= 0)
        return fail(PARALLAX_ERR_INVALID, "B=%d, H=%d, %s=%d must all be >= 1", B, H, Lname, L);
    if (d != 64 && d != 128)
        return fail(PARALLAX_ERR_UNSUPPORTED, "head dimension d=%d (supported: 64, 128)", d);
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(rho))
        return fail(PARALLAX_ERR_INVALID, "every tensor pointer must be 16-byte aligned");
    const double elems = (double)B * H * L * d;
    if (elems > 9.0e15 || (double)B * H > 2147483647.0 || (double)L * d > 2147483647.0)
        return fail(PARALLAX_ERR_INVALID, "tensor too large");
    return PARALLAX_OK;
}

int prefill_common(const void* q, const void* rho, const void* k, const void* v, void* o, int B,
                   int H, int L, int d, int causal, float scale, cudaStream_t stream, bool bf16) {
    int rc = validate_common(q, k, v, o, rho, B, H, L, d, "L");
    if (rc != PARALLAX_OK) return rc;
    if (causal != 0 && causal != 1)
        return fail(PARALLAX_ERR_INVALID, "causal=%d must be 0 or 1", causal);
    if (!std::isfinite(scale)) return fail(PARALLAX_ERR_INVALID, "scale must be finite");
    int dev = 0;
    DeviceState* ds = device_state(&dev);
    if (!ds) return fail(PARALLAX_ERR_CUDA, "no usable CUDA device");
    parallax::PrefillShape s{B, H, L, d, causal, scale};
    cudaError_t e;
    if (bf16)
        e = parallax::prefill_tc_launch(s, q, rho, k, v, static_cast<float*>(o), ds->num_sms,
                                        stream);
    else
        e = parallax::prefill_simt_launch(s, false, q, rho, k, v, static_cast<float*>(o), stream);
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return succeed();
}

int decode_common(const void* q, const void* rho, const void* kc, const void* vc,
                  const int32_t* seqlens, void* o, int B, int H, int Lmax, int d,
                  cudaStream_t stream, bool bf16) {
    int rc = validate_common(q, kc, vc, o, rho, B, H, Lmax, d, "Lmax");
    if (rc != PARALLAX_OK) return rc;
    if (!seqlens) return fail(PARALLAX_ERR_INVALID, "null seqlens pointer");
    int dev = 0;
    DeviceState* ds = device_state(&dev);
    if (!ds) return fail(PARALLAX_ERR_CUDA, "no usable CUDA device");

    parallax::DecodePlan plan;
    plan.B = B;
    plan.H = H;
    plan.Lmax = Lmax;
    plan.d = d;
    plan.scale = 1.0f / std::sqrt((float)d);
    plan.chunk = plan_chunk(B, H, Lmax, ds->num_sms);
    plan.nsplit = (Lmax + plan.chunk - 1) / plan.chunk;
    const long long items = (long long)B * H * plan.nsplit;
    plan.grid = (int)std::min<long long>(items, (long long)ds->num_sms);

    const size_t need = parallax::decode_workspace_bytes(plan);
    void* ws = nullptr;
    if (need > 0) {
        std::lock_guard<std::mutex> lock(g_mu);
        DeviceState& s = g_dev[dev];
        if (s.ws_bytes < need) {
            if (s.ws) {
                cudaError_t e = cudaFree(s.ws);  // synchronises the device
                s.ws = nullptr;
                s.ws_bytes = 0;
                if (e != cudaSuccess) return cuda_fail(e, "workspace free");
            }
            cudaError_t e = cudaMalloc(&s.ws, need);
            if (e != cudaSuccess) {
                s.ws = nullptr;
                return cuda_fail(e, "workspace allocation");
            }
            s.ws_bytes = need;
        }
        ws = s.ws;
    }
    cudaError_t e = parallax::decode_launch(plan, bf16, q, rho, kc, vc, seqlens,
                                            static_cast<float*>(o), ws, stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return succeed();
}

}  // namespace

extern "C" {

int parallax_attn_prefill(const void* q, const void* rho, const void* k, const void* v, void* o,
                          int B, int H, int L, int d, int causal, float scale,
                          cudaStream_t stream) {
    return prefill_common(q, rho, k, v, o, B, H, L, d, causal, scale, stream, true);
}

int parallax_attn_prefill_f32(const void* q, const void* rho, const void* k, const void* v,
                              void* o, int B, int H, int L, int d, int causal, float scale,
                              cudaStream_t stream) {
    return prefill_common(q, rho, k, v, o, B, H, L, d, causal, scale, stream, false);
}

int parallax_attn_decode(const void* q, const void* rho, const void* k_cache,
                         const void* v_cache, const int32_t* seqlens, void* o, int B, int H,
                         int Lmax, int d, cudaStream_t stream) {
    return decode_common(q, rho, k_cache, v_cache, seqlens, o, B, H, Lmax, d, stream, true);
}

int parallax_attn_decode_f32(const void* q, const void* rho, const void* k_cache,
                             const void* v_cache, const int32_t* seqlens, void* o, int B, int H,
                             int Lmax, int d, cudaStream_t stream) {
    return decode_common(q, rho, k_cache, v_cache, seqlens, o, B, H, Lmax, d, stream, false);
}

int parallax_attn_decode_noalloc(const void* q, const void* rho, const void* k_cache,
                                 const void* v_cache, const int32_t* seqlens, void* o, int B,
                                 int H, int Lmax, int d, cudaStream_t stream) {
    int rc = validate_common(q, k_cache, v_cache, o, rho, B, H, Lmax, d, "Lmax");
    if (rc != PARALLAX_OK) return rc;
    if (!seqlens) return fail(PARALLAX_ERR_INVALID, "null seqlens pointer");
    DeviceState* ds = device_state(nullptr);
    if (!ds) return fail(PARALLAX_ERR_CUDA, "no usable CUDA device");
    // the same split plan as parallax_attn_decode, so both give the same result
    parallax::DecodePlan plan;
    plan.B = B;
    plan.H = H;
    plan.Lmax = Lmax;
    plan.d = d;
    plan.scale = 1.0f / std::sqrt((float)d);
    plan.chunk = plan_chunk(B, H, Lmax, ds->num_sms);
    plan.nsplit = (Lmax + plan.chunk - 1) / plan.chunk;
    plan.grid = (int)std::min<long long>((long long)B * H * plan.nsplit, (long long)ds->num_sms);
    const size_t need = parallax::decode_workspace_bytes(plan);
    const size_t cap = parallax::decode_noalloc_capacity();
    if (need > cap)
        return fail(PARALLAX_ERR_UNSUPPORTED,
                    "decode of B=%d H=%d Lmax=%d d=%d needs %zu bytes of split-KV scratch; the "
                    "no-allocation entry point holds at most %zu bytes (use "
                    "parallax_attn_decode for this size)",
                    B, H, Lmax, d, need, cap);
    cudaError_t e = parallax::decode_launch_noalloc(plan, true, q, rho, k_cache, v_cache,
                                                    seqlens, static_cast<float*>(o), stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode (no-allocation) launch");
    return succeed();
}

int parallax_attn_decode_chunk_keys(int B, int H, int Lmax, int d, int elem_bytes) {
    if (B <= 0 || H <= 0 || Lmax <= 0)
        return fail(PARALLAX_ERR_INVALID, "B, H, Lmax must be >= 1");
    if (d != 64 && d != 128) return fail(PARALLAX_ERR_UNSUPPORTED, "d=%d", d);
    if (elem_bytes != 2 && elem_bytes != 4)
        return fail(PARALLAX_ERR_INVALID, "elem_bytes=%d must be 2 or 4", elem_bytes);
    int num_sms = 148;
    if (DeviceState* ds = device_state(nullptr)) num_sms = ds->num_sms;
    succeed();
    return plan_chunk(B, H, Lmax, num_sms);
}

int parallax_attn_set_decode_chunk_keys(int keys) {
    if (keys < 0 || keys % 256 != 0)
        return fail(PARALLAX_ERR_INVALID, "chunk keys %d must be 0 or a positive multiple of 256",
                    keys);
    g_chunk_override.store(keys);
    return succeed();
}

size_t parallax_attn_workspace_bytes(void) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(g_mu);
    return (int)g_dev.size() > dev ? g_dev[dev].ws_bytes : 0;
}

int parallax_attn_release_workspace(void) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lock(g_mu);
    if ((int)g_dev.size() > dev && g_dev[dev].ws) {
        e = cudaFree(g_dev[dev].ws);
        g_dev[dev].ws = nullptr;
        g_dev[dev].ws_bytes = 0;
        if (e != cudaSuccess) return cuda_fail(e, "workspace free");
    }
    return succeed();
}

const char* parallax_last_error(void) { return t_last_error.c_str(); }

int parallax_check_device_error(cudaStream_t stream, unsigned int* bits) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    const unsigned v = parallax::decode_take_error() | parallax::prefill_simt_take_error() |
                       parallax::prefill_tc_take_error();
    if (bits) *bits = v;
    if (v) return fail(PARALLAX_ERR_DEVICE, "device error word 0x%x", v);
    return succeed();
}

int parallax_version(void) { return 100; }

}  // extern "C"
