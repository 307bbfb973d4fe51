// C-ABI layer of libparallax_attn: argument validation (on the host, before
// anything is launched), split-KV planning, the per-device decode workspace,
// and the device error word.
#include <algorithm>
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
thread_local unsigned t_last_bits = 0;  // device error bits of this thread's last check

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

// A library-owned device buffer, grown in stream order.  `last_use` is recorded on the
// stream of every launch that reads or writes the buffer, so that a later call that grows
// it (on any stream) frees the old buffer only after that launch.  The usable bytes
// [ptr, ptr + bytes) sit between two guard bands of kGuardBytes filled with kGuardFill,
// which parallax_workspace_guards_intact() checks (a kernel that overran its workspace
// would have changed them).
constexpr size_t kGuardBytes = 4096;
constexpr unsigned char kGuardFill = 0xA5;

struct Workspace {
    void* ptr = nullptr;  // usable region (base + kGuardBytes)
    size_t bytes = 0;
    cudaEvent_t last_use = nullptr;
    bool used = false;  // last_use has been recorded since the buffer was allocated
    unsigned char* base() const { return static_cast<unsigned char*>(ptr) - kGuardBytes; }
};

struct DeviceState {
    Workspace ws;   // decode split-KV partials
    Workspace bws;  // prefill backward row statistics
    int num_sms = 0;
};

// Make `w` at least `need` bytes for a launch on `stream`: the old buffer is freed with
// cudaFreeAsync on `stream` after `stream` has waited for the buffer's last use, and the new
// one comes from cudaMallocAsync on `stream`; nothing synchronises the device.  Call with
// g_mu held, and keep holding it until the launch that uses the buffer is recorded.
int grow(Workspace& w, size_t need, cudaStream_t stream, const char* what);
// Record the launch just issued on `stream` as the buffer's last use (g_mu held).  A call
// captured into a CUDA graph is not recorded: its launches run when the graph does.
int mark_used(Workspace& w, cudaStream_t stream, const char* what);
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

// Keys per split-KV chunk for grouped heads: about `items_per_sm` work items per SM, with
// chunks of 256..4096 keys (long enough that the 1 KB partial state per chunk is noise next
// to the chunk's K/V bytes).
int plan_chunk(int B, int H, int Lmax, int num_sms, double items_per_sm) {
    const int forced = g_chunk_override.load();
    int c;
    if (forced > 0) {
        c = forced;
    } else {
        const double per_item = (double)B * H * Lmax / (items_per_sm * num_sms);
        c = 256;
        while (c < 4096 && (double)(2 * c) <= per_item) c *= 2;
    }
    return c >= Lmax ? Lmax : c;
}

// One query head per key/value head: the longest chunk (256..4096 keys, powers of two) that
// still leaves about one work item per resident CTA (at least 85% of them).  Every item ends
// with a merge of its warps' states, and every split adds partial states for the combine
// kernel, so few long items beat many short ones as long as the CTAs stay busy; heads of at
// most 1024 keys are not split at all (their stream is shorter than a second launch costs).
// Measured at H=16, d=128 over chunks 256..4096: B=1 with 32768 keys runs best at 2048-key
// items (256 items), B=8 with 8192 keys at 4096 (256 items), B=1 with 8192 keys at 512-1024,
// B=8 with 1024 keys unsplit.  The 4096-key cap keeps ragged batches splitting.
int plan_chunk_single(int B, int H, int Lmax, int ctas) {
    const int forced = g_chunk_override.load();
    if (forced > 0) return forced >= Lmax ? Lmax : forced;
    if (Lmax <= 1024) return Lmax;
    const long long heads = (long long)B * H;
    const double target = 0.85 * ctas;
    int c = 4096;
    while (c > 256 && (double)heads * ((Lmax + c - 1) / c) < target) c /= 2;
    return c >= Lmax ? Lmax : c;
}

int grow(Workspace& w, size_t need, cudaStream_t stream, const char* what) {
    if (w.bytes >= need) return PARALLAX_OK;
    cudaError_t e;
    if (!w.last_use) {
        e = cudaEventCreateWithFlags(&w.last_use, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            w.last_use = nullptr;
            return cuda_fail(e, what);
        }
    }
    if (w.ptr) {
        if (w.used) {
            e = cudaStreamWaitEvent(stream, w.last_use, 0);
            if (e != cudaSuccess) return cuda_fail(e, what);
        }
        e = cudaFreeAsync(w.base(), stream);
        w.ptr = nullptr;
        w.bytes = 0;
        w.used = false;
        if (e != cudaSuccess) return cuda_fail(e, what);
    }
    void* base = nullptr;
    e = cudaMallocAsync(&base, need + 2 * kGuardBytes, stream);
    if (e != cudaSuccess) return cuda_fail(e, what);
    unsigned char* b = static_cast<unsigned char*>(base);
    e = cudaMemsetAsync(b, kGuardFill, kGuardBytes, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(b + kGuardBytes + need, kGuardFill, kGuardBytes, stream);
    if (e != cudaSuccess) {
        cudaFreeAsync(base, stream);
        return cuda_fail(e, what);
    }
    w.ptr = b + kGuardBytes;
    w.bytes = need;
    return PARALLAX_OK;
}

int mark_used(Workspace& w, cudaStream_t stream, const char* what) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess) return cuda_fail(e, what);
    if (cap != cudaStreamCaptureStatusNone) return PARALLAX_OK;
    e = cudaEventRecord(w.last_use, stream);
    if (e != cudaSuccess) return cuda_fail(e, what);
    w.used = true;
    return PARALLAX_OK;
}

// Free a buffer after the whole device has finished with it (release path).
int release(Workspace& w, const char* what) {
    if (!w.ptr) return PARALLAX_OK;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaFreeAsync(w.base(), nullptr);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    w.ptr = nullptr;
    w.bytes = 0;
    w.used = false;
    return e == cudaSuccess ? PARALLAX_OK : cuda_fail(e, what);
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

// The split plan shared by every decode entry point.  Work items are (key/value
// head, chunk); a paged cache caps the chunk so that an item's page ids fit the
// kernel's per-item table.
parallax::DecodePlan make_plan(int B, int H, int Hkv, int Lmax, int d, int num_sms,
                               int page_size = 0, int max_pages = 0, int num_pages = 0) {
    parallax::DecodePlan plan;
    plan.B = B;
    plan.H = H;
    plan.Hkv = Hkv;
    plan.Lmax = Lmax;
    plan.d = d;
    plan.page_size = page_size;
    plan.max_pages = max_pages;
    plan.num_pages = num_pages;
    plan.scale = 1.0f / std::sqrt((float)d);
    // grouped heads run the tensor-core decode, whose per-item merge and combine cost more:
    // groups of 4 or 8 take the longest chunk that still leaves at least 1.7 items per SM,
    // groups of 2 about 8 items per SM (chunks capped at 4096 keys in every case, so ragged
    // lengths keep splitting).  Measured at B=64, H=16, 8192 keys, forced chunks 256..8192:
    // H_kv = 2 and 4 run fastest at 4096 keys among the chunks this allows, H_kv = 8 at 2048.
    const int ctas = num_sms * parallax::decode_ctas_per_sm();
    plan.chunk = H == Hkv ? plan_chunk_single(B, H, Lmax, ctas)
                          : plan_chunk(B, Hkv, Lmax, num_sms, H >= 4 * Hkv ? 1.7 : 8.0);
    // a paged cache usually holds a ragged batch, which balances better on shorter items:
    // grouped heads on a paged cache take at most 2048 keys per item (B=512, lengths
    // U{128..16384}, page 256, H=16, H_kv=4: 1.39 ms at 2048 keys, 1.45 ms at 4096)
    if (page_size > 0 && H > Hkv && g_chunk_override.load() == 0)
        plan.chunk = std::min(plan.chunk, 2048);
    if (page_size > 0 && plan.chunk > parallax::decode_paged_max_chunk(page_size)) plan.chunk = 4096;
    plan.nsplit = (Lmax + plan.chunk - 1) / plan.chunk;
    const long long items = (long long)B * Hkv * plan.nsplit;
    plan.grid = (int)std::min<long long>(items, (long long)ctas);
    // One query head per key/value head (bf16): the tensor-core decode streams faster once
    // every CTA has at least two items of 512 keys or more (B=64, 8192 keys: 7.1 against
    // 6.8 TB/s; B=2048, 1024 keys: 7.2 against 6.9); with fewer, shorter items the SIMT
    // decode's deeper per-CTA pipeline wins (B=8, 8192 keys: 6.3 against 6.1 TB/s; 128-key
    // heads: 6.3 against 5.8).
    plan.mma = items >= 2LL * ctas && plan.chunk >= 512;
    return plan;
}

int decode_run(const parallax::DecodePlan& plan, int dev, const void* q, const void* rho,
               const void* kc, const void* vc, const int32_t* seqlens, void* o,
               cudaStream_t stream, bool bf16, const int32_t* block_table) {
    const size_t need = parallax::decode_workspace_bytes(plan);
    if (need == 0) {
        cudaError_t e = parallax::decode_launch(plan, bf16, q, rho, kc, vc, seqlens,
                                                static_cast<float*>(o), nullptr, stream,
                                                block_table);
        if (e != cudaSuccess) return cuda_fail(e, "decode launch");
        return succeed();
    }
    // the buffer is grown, used and marked under one lock, so that another thread's call
    // cannot free it between this call's growth and its launch
    std::lock_guard<std::mutex> lock(g_mu);
    Workspace& w = g_dev[dev].ws;
    int rc = grow(w, need, stream, "decode workspace");
    if (rc != PARALLAX_OK) return rc;
    cudaError_t e = parallax::decode_launch(plan, bf16, q, rho, kc, vc, seqlens,
                                            static_cast<float*>(o), w.ptr, stream, block_table);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    rc = mark_used(w, stream, "decode workspace");
    if (rc != PARALLAX_OK) return rc;
    return succeed();
}

int validate_groups(int H, int Hkv) {
    if (Hkv <= 0 || H % Hkv != 0)
        return fail(PARALLAX_ERR_INVALID, "H=%d must be a positive multiple of H_kv=%d", H, Hkv);
    const int G = H / Hkv;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return fail(PARALLAX_ERR_UNSUPPORTED, "query heads per key/value head %d (supported: "
                    "1, 2, 4, 8)", G);
    return PARALLAX_OK;
}

int decode_common(const void* q, const void* rho, const void* kc, const void* vc,
                  const int32_t* seqlens, void* o, int B, int H, int Hkv, int Lmax, int d,
                  cudaStream_t stream, bool bf16) {
    int rc = validate_common(q, kc, vc, o, rho, B, H, Lmax, d, "Lmax");
    if (rc != PARALLAX_OK) return rc;
    if (!seqlens) return fail(PARALLAX_ERR_INVALID, "null seqlens pointer");
    rc = validate_groups(H, Hkv);
    if (rc != PARALLAX_OK) return rc;
    if (!bf16 && Hkv != H)
        return fail(PARALLAX_ERR_UNSUPPORTED, "shared key/value heads need bf16 inputs");
    int dev = 0;
    DeviceState* ds = device_state(&dev);
    if (!ds) return fail(PARALLAX_ERR_CUDA, "no usable CUDA device");
    const parallax::DecodePlan plan = make_plan(B, H, Hkv, Lmax, d, ds->num_sms);
    return decode_run(plan, dev, q, rho, kc, vc, seqlens, o, stream, bf16, nullptr);
}

}  // namespace

extern "C" {

int parallax_attn_prefill(const void* q, const void* rho, const void* k, const void* v, void* o,
                          int B, int H, int L, int d, int causal, float scale,
                          cudaStream_t stream) {
    return prefill_common(q, rho, k, v, o, B, H, L, d, causal, scale, stream, true);
}

int parallax_attn_prefill_train(const void* q, const void* rho, const void* k, const void* v,
                                void* o, float* lse, float* rbar, float* mu_v, int B, int H, int L,
                                int d, int causal, float scale, cudaStream_t stream) {
    int rc = validate_common(q, k, v, o, rho, B, H, L, d, "L");
    if (rc != PARALLAX_OK) return rc;
    if (!lse || !rbar || !mu_v)
        return fail(PARALLAX_ERR_INVALID, "null statistics pointer (lse=%p rbar=%p mu_v=%p)",
                    (void*)lse, (void*)rbar, (void*)mu_v);
    if (!aligned16(mu_v) || !aligned16(lse) || !aligned16(rbar))
        return fail(PARALLAX_ERR_INVALID, "every tensor pointer must be 16-byte aligned");
    if (causal != 0 && causal != 1)
        return fail(PARALLAX_ERR_INVALID, "causal=%d must be 0 or 1", causal);
    if (!std::isfinite(scale)) return fail(PARALLAX_ERR_INVALID, "scale must be finite");
    DeviceState* ds = device_state(nullptr);
    if (!ds) return fail(PARALLAX_ERR_CUDA, "no usable CUDA device");
    parallax::PrefillShape s{B, H, L, d, causal, scale};
    parallax::TrainStats ts;
    ts.lse = lse;
    ts.rbar = rbar;
    ts.mu = mu_v;
    cudaError_t e = parallax::prefill_tc_launch(s, q, rho, k, v, static_cast<float*>(o),
                                                ds->num_sms, stream, ts);
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return succeed();
}

int parallax_attn_prefill_backward(const void* q, const void* rho, const void* k, const void* v,
                                   const float* o, const float* mu_v, const float* lse,
                                   const float* rbar, const void* dout, float* dq, float* drho,
                                   float* dk, float* dv, int B, int H, int L, int d, int causal,
                                   float scale, cudaStream_t stream) {
    int rc = validate_common(q, k, v, o, rho, B, H, L, d, "L");
    if (rc != PARALLAX_OK) return rc;
    if (!mu_v || !lse || !rbar || !dout || !dq || !dk || !dv || (rho && !drho))
        return fail(PARALLAX_ERR_INVALID, "null pointer among mu_v, lse, rbar, dout, dq, drho, "
                    "dk, dv (drho may be null only when rho is)");
    if (!aligned16(mu_v) || !aligned16(lse) || !aligned16(rbar) || !aligned16(dout) ||
        !aligned16(dq) || !aligned16(drho) || !aligned16(dk) || !aligned16(dv))
        return fail(PARALLAX_ERR_INVALID, "every tensor pointer must be 16-byte aligned");
    if (causal != 0 && causal != 1)
        return fail(PARALLAX_ERR_INVALID, "causal=%d must be 0 or 1", causal);
    if (!std::isfinite(scale)) return fail(PARALLAX_ERR_INVALID, "scale must be finite");
    int dev = 0;
    DeviceState* ds = device_state(&dev);
    if (!ds) return fail(PARALLAX_ERR_CUDA, "no usable CUDA device");
    parallax::PrefillShape s{B, H, L, d, causal, scale};
    std::lock_guard<std::mutex> lock(g_mu);
    Workspace& w = g_dev[dev].bws;
    rc = grow(w, parallax::prefill_backward_workspace_bytes(B, H, L), stream,
              "backward workspace");
    if (rc != PARALLAX_OK) return rc;
    cudaError_t e = parallax::prefill_backward_launch(s, q, rho, k, v, o, mu_v, lse, rbar, dout,
                                                      dq, drho, dk, dv, w.ptr, stream);
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    rc = mark_used(w, stream, "backward workspace");
    if (rc != PARALLAX_OK) return rc;
    return succeed();
}

int parallax_attn_prefill_f32(const void* q, const void* rho, const void* k, const void* v,
                              void* o, int B, int H, int L, int d, int causal, float scale,
                              cudaStream_t stream) {
    return prefill_common(q, rho, k, v, o, B, H, L, d, causal, scale, stream, false);
}

int parallax_attn_decode(const void* q, const void* rho, const void* k_cache,
                         const void* v_cache, const int32_t* seqlens, void* o, int B, int H,
                         int Lmax, int d, cudaStream_t stream) {
    return decode_common(q, rho, k_cache, v_cache, seqlens, o, B, H, H, Lmax, d, stream, true);
}

int parallax_attn_decode_f32(const void* q, const void* rho, const void* k_cache,
                             const void* v_cache, const int32_t* seqlens, void* o, int B, int H,
                             int Lmax, int d, cudaStream_t stream) {
    return decode_common(q, rho, k_cache, v_cache, seqlens, o, B, H, H, Lmax, d, stream, false);
}

int parallax_attn_decode_gqa(const void* q, const void* rho, const void* k_cache,
                             const void* v_cache, const int32_t* seqlens, void* o, int B, int H,
                             int H_kv, int Lmax, int d, cudaStream_t stream) {
    return decode_common(q, rho, k_cache, v_cache, seqlens, o, B, H, H_kv, Lmax, d, stream, true);
}

int parallax_attn_decode_paged(const void* q, const void* rho, const void* k_pages,
                               const void* v_pages, const int32_t* block_table,
                               const int32_t* seqlens, void* o, int B, int H, int H_kv,
                               int page_size, int max_pages, int num_pages, int d,
                               cudaStream_t stream) {
    if (!block_table) return fail(PARALLAX_ERR_INVALID, "null block_table pointer");
    if (page_size <= 0 || max_pages <= 0 || num_pages <= 0)
        return fail(PARALLAX_ERR_INVALID, "page_size=%d, max_pages=%d, num_pages=%d must all be "
                    ">= 1", page_size, max_pages, num_pages);
    if (page_size % 16 != 0)
        return fail(PARALLAX_ERR_UNSUPPORTED, "page_size=%d must be a multiple of 16", page_size);
    if ((long long)page_size * max_pages > 2147483647LL)
        return fail(PARALLAX_ERR_INVALID, "max_pages * page_size exceeds the int range");
    const int Lmax = page_size * max_pages;
    int rc = validate_common(q, k_pages, v_pages, o, rho, B, H, Lmax, d, "Lmax");
    if (rc != PARALLAX_OK) return rc;
    if (!seqlens) return fail(PARALLAX_ERR_INVALID, "null seqlens pointer");
    rc = validate_groups(H, H_kv);
    if (rc != PARALLAX_OK) return rc;
    if ((double)num_pages * H_kv * page_size * d > 9.0e15)
        return fail(PARALLAX_ERR_INVALID, "page pool too large");
    int dev = 0;
    DeviceState* ds = device_state(&dev);
    if (!ds) return fail(PARALLAX_ERR_CUDA, "no usable CUDA device");
    const parallax::DecodePlan plan =
        make_plan(B, H, H_kv, Lmax, d, ds->num_sms, page_size, max_pages, num_pages);
    return decode_run(plan, dev, q, rho, k_pages, v_pages, seqlens, o, stream, true,
                      block_table);
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
    const parallax::DecodePlan plan = make_plan(B, H, H, Lmax, d, ds->num_sms);
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

int parallax_attn_prefill_chunk(const void* q, const void* rho, const void* k_new,
                                const void* v_new, void* k_cache, void* v_cache,
                                const int32_t* cache_lens, void* o, int B, int H, int Lq,
                                int Lmax, int d, float scale, cudaStream_t stream) {
    int rc = validate_common(q, k_new, v_new, o, rho, B, H, Lq, d, "Lq");
    if (rc != PARALLAX_OK) return rc;
    if (!k_cache || !v_cache || !cache_lens)
        return fail(PARALLAX_ERR_INVALID, "null cache pointer (k_cache=%p v_cache=%p "
                    "cache_lens=%p)", k_cache, v_cache, (const void*)cache_lens);
    if (!aligned16(k_cache) || !aligned16(v_cache))
        return fail(PARALLAX_ERR_INVALID, "every tensor pointer must be 16-byte aligned");
    if (Lmax < Lq) return fail(PARALLAX_ERR_INVALID, "Lmax=%d is smaller than the chunk Lq=%d",
                               Lmax, Lq);
    if ((double)B * H * Lmax * d > 9.0e15 || (double)Lmax * d > 2147483647.0)
        return fail(PARALLAX_ERR_INVALID, "cache too large");
    if (!std::isfinite(scale)) return fail(PARALLAX_ERR_INVALID, "scale must be finite");
    DeviceState* ds = device_state(nullptr);
    if (!ds) return fail(PARALLAX_ERR_CUDA, "no usable CUDA device");
    parallax::PrefillShape s{B, H, Lq, d, 1, scale};
    cudaError_t e = parallax::prefill_tc_chunk_launch(s, q, rho, k_new, v_new, k_cache, v_cache,
                                                      cache_lens, Lmax, static_cast<float*>(o),
                                                      ds->num_sms, stream);
    if (e != cudaSuccess) return cuda_fail(e, "chunked prefill launch");
    return succeed();
}

int parallax_attn_qkvr_projection(const void* x, const void* w, void* q, void* k, void* v,
                                  void* rho, int B, int L, int width, int H, int d,
                                  cudaStream_t stream) {
    if (!x || !w || !q || !k || !v)
        return fail(PARALLAX_ERR_INVALID, "null tensor pointer (x=%p w=%p q=%p k=%p v=%p)", x, w,
                    q, k, v);
    if (B <= 0 || L <= 0 || width <= 0 || H <= 0)
        return fail(PARALLAX_ERR_INVALID, "B=%d, L=%d, width=%d, H=%d must all be >= 1", B, L,
                    width, H);
    if (d != 64 && d != 128)
        return fail(PARALLAX_ERR_UNSUPPORTED, "head dimension d=%d (supported: 64, 128)", d);
    if ((H * d) % 128 != 0)
        return fail(PARALLAX_ERR_UNSUPPORTED, "H*d=%d must be a multiple of 128", H * d);
    if (width % 8 != 0)
        return fail(PARALLAX_ERR_UNSUPPORTED, "width=%d must be a multiple of 8", width);
    if (!aligned16(x) || !aligned16(w) || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
        !aligned16(rho))
        return fail(PARALLAX_ERR_INVALID, "every tensor pointer must be 16-byte aligned");
    if ((double)B * L * width > 9.0e15 || (double)B * H * L * d > 9.0e15 ||
        (double)B * H > 2147483647.0 || (double)L * width > 9.0e15)
        return fail(PARALLAX_ERR_INVALID, "tensor too large");
    DeviceState* ds = device_state(nullptr);
    if (!ds) return fail(PARALLAX_ERR_CUDA, "no usable CUDA device");
    parallax::ProjShape s{B, L, width, H, d, rho ? 4 : 3};
    void* const out[4] = {q, k, v, rho};
    cudaError_t e = parallax::proj_tc_launch(s, x, w, out, ds->num_sms, stream);
    if (e != cudaSuccess) return cuda_fail(e, "projection launch");
    return succeed();
}

int parallax_lla_decode(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* seqlens, void* o, float* rho, int B, int H, int Lmax,
                        int d, int cg_iters, cudaStream_t stream) {
    int rc = validate_common(q, k_cache, v_cache, o, rho, B, H, Lmax, d, "Lmax");
    if (rc != PARALLAX_OK) return rc;
    if (!seqlens || !rho) return fail(PARALLAX_ERR_INVALID, "null seqlens or rho pointer");
    if (cg_iters < 0) return fail(PARALLAX_ERR_INVALID, "cg_iters=%d must be >= 0", cg_iters);
    int dev = 0;
    DeviceState* ds = device_state(&dev);
    if (!ds) return fail(PARALLAX_ERR_CUDA, "no usable CUDA device");
    cudaError_t e = parallax::lla_launch(q, k_cache, v_cache, seqlens, rho, static_cast<float*>(o),
                                         B, H, Lmax, d, cg_iters > 0 ? cg_iters : d, stream);
    if (e != cudaSuccess) return cuda_fail(e, "LLA launch");
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
    const parallax::DecodePlan plan = make_plan(B, H, H, Lmax, d, num_sms);
    succeed();
    return plan.chunk;
}

int parallax_attn_decode_plan_keys(int B, int H, int H_kv, int Lmax, int d, int page_size) {
    if (B <= 0 || H <= 0 || Lmax <= 0)
        return fail(PARALLAX_ERR_INVALID, "B, H, Lmax must be >= 1");
    if (d != 64 && d != 128) return fail(PARALLAX_ERR_UNSUPPORTED, "d=%d", d);
    int rc = validate_groups(H, H_kv);
    if (rc != PARALLAX_OK) return rc;
    if (page_size < 0) return fail(PARALLAX_ERR_INVALID, "page_size=%d must be >= 0", page_size);
    if (page_size % 16 != 0)
        return fail(PARALLAX_ERR_UNSUPPORTED, "page_size=%d must be a multiple of 16", page_size);
    int num_sms = 148;
    if (DeviceState* ds = device_state(nullptr)) num_sms = ds->num_sms;
    const int max_pages = page_size > 0 ? (Lmax + page_size - 1) / page_size : 0;
    const parallax::DecodePlan plan =
        make_plan(B, H, H_kv, Lmax, d, num_sms, page_size, max_pages, page_size > 0 ? 1 : 0);
    succeed();
    return plan.chunk;
}

int parallax_attn_decode_plan_kernel(int B, int H, int H_kv, int Lmax, int d, int page_size) {
    const int chunk = parallax_attn_decode_plan_keys(B, H, H_kv, Lmax, d, page_size);
    if (chunk < 0) return chunk;
    int num_sms = 148;
    if (DeviceState* ds = device_state(nullptr)) num_sms = ds->num_sms;
    const int max_pages = page_size > 0 ? (Lmax + page_size - 1) / page_size : 0;
    const parallax::DecodePlan plan =
        make_plan(B, H, H_kv, Lmax, d, num_sms, page_size, max_pages, page_size > 0 ? 1 : 0);
    succeed();
    return parallax::decode_uses_mma(plan, true) ? 1 : 0;
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
    return (int)g_dev.size() > dev ? g_dev[dev].ws.bytes : 0;
}

int parallax_attn_release_workspace(void) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lock(g_mu);
    if ((int)g_dev.size() > dev) {
        int rc = release(g_dev[dev].ws, "workspace free");
        if (rc != PARALLAX_OK) return rc;
        rc = release(g_dev[dev].bws, "workspace free");
        if (rc != PARALLAX_OK) return rc;
    }
    return succeed();
}

const char* parallax_last_error(void) { return t_last_error.c_str(); }

int parallax_check_device_error(cudaStream_t stream) {
    t_last_bits = 0;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    const unsigned v = parallax::decode_take_error() | parallax::prefill_simt_take_error() |
                       parallax::prefill_tc_take_error() | parallax::proj_tc_take_error() |
                       parallax::prefill_backward_take_error() | parallax::lla_take_error();
    t_last_bits = v;
    if (v) return fail(PARALLAX_ERR_DEVICE, "device error word 0x%x", v);
    return succeed();
}

unsigned int parallax_last_device_error_bits(void) { return t_last_bits; }

int parallax_workspace_guards_intact(void) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "device synchronize");
    std::lock_guard<std::mutex> lock(g_mu);
    if ((int)g_dev.size() <= dev) {
        succeed();
        return 1;
    }
    std::vector<unsigned char> band(kGuardBytes);
    for (Workspace* w : {&g_dev[dev].ws, &g_dev[dev].bws}) {
        if (!w->ptr) continue;
        for (unsigned char* g : {w->base(), static_cast<unsigned char*>(w->ptr) + w->bytes}) {
            e = cudaMemcpy(band.data(), g, kGuardBytes, cudaMemcpyDeviceToHost);
            if (e != cudaSuccess) return cuda_fail(e, "guard band copy");
            for (unsigned char c : band)
                if (c != kGuardFill) {
                    succeed();
                    return 0;
                }
        }
    }
    succeed();
    return 1;
}

int parallax_selftest_wait_timeout(int family, unsigned int limit_us, cudaStream_t stream) {
    if (family != PARALLAX_SELFTEST_DECODE && family != PARALLAX_SELFTEST_PREFILL)
        return fail(PARALLAX_ERR_INVALID, "kernel family %d (0: decode, 1: tensor-core prefill)",
                    family);
    if (limit_us < 1 || limit_us > 1000000)
        return fail(PARALLAX_ERR_INVALID, "limit_us=%u must lie in [1, 1000000]", limit_us);
    const uint64_t ns = 1000ull * limit_us;
    cudaError_t e = family == PARALLAX_SELFTEST_DECODE ? parallax::decode_wait_selftest(ns, stream)
                                                      : parallax::prefill_tc_wait_selftest(ns, stream);
    if (e != cudaSuccess) return cuda_fail(e, "wait self-test launch");
    return succeed();
}

int parallax_version(void) { return 100; }

int parallax_debug_checks(void) {
#ifdef PARALLAX_DEBUG_CHECKS
    return 1;
#else
    return 0;
#endif
}

}  // extern "C"
