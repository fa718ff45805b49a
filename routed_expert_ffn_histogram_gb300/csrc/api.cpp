// C entry points: status text, validation, expert packing and dispatch to
// the kernel launchers.  Every argument is checked before anything is
// enqueued; nothing here allocates device memory.
#include <chrono>
#include <cstring>
#include <thread>
#include <mutex>

#include "internal.h"

namespace moe {

static thread_local int g_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
    g_last_cuda_error = int(e);
    cudaGetLastError();  // clear the sticky-free error state of this thread
    return MOE_ERR_CUDA;
}

int current_device_info(DeviceInfo* out) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(mu);
    if (cache[dev].device != dev) {
        DeviceInfo d;
        d.device = dev;
        MOE_CUDA_TRY(cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev));
        MOE_CUDA_TRY(cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev));
        MOE_CUDA_TRY(cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev));
        int optin = 0;
        MOE_CUDA_TRY(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
        d.smem_optin = size_t(optin);
        cache[dev] = d;
    }
    *out = cache[dev];
    return MOE_OK;
}

const Layout* pool_layout(const moe_pool_t* p);
const moe_pool_desc* pool_desc(const moe_pool_t* p);

}  // namespace moe

using moe::Layout;

extern "C" const char* moe_status_str(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID: return "invalid argument";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_CAPACITY: return "unique routed experts exceed the pool's slots";
        case MOE_ERR_TIMEOUT: return "bounded wait timed out";
        case MOE_ERR_STATE: return "object in the wrong state";
        case MOE_ERR_UNSUPPORTED: return "shape or device not supported";
        default: return "unknown status";
    }
}

extern "C" int moe_last_cuda_error(void) { return moe::g_last_cuda_error; }

extern "C" int moe_device_count(void) {
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

extern "C" int moe_expert_bytes(int hidden, int inter, size_t* out) {
    Layout L;
    if (!out || !Layout::make(hidden, inter, &L)) return MOE_ERR_INVALID;
    *out = L.expert_bytes;
    return MOE_OK;
}

extern "C" int moe_pack_expert(const uint8_t* gc, const uint8_t* gs, const uint8_t* uc, const uint8_t* us,
                               const uint8_t* dc, const uint8_t* ds, int hidden, int inter, void* dst) {
    Layout L;
    if (!gc || !gs || !uc || !us || !dc || !ds || !dst || !Layout::make(hidden, inter, &L))
        return MOE_ERR_INVALID;
    uint8_t* o = static_cast<uint8_t*>(dst);
    std::memset(o, 0, L.expert_bytes);
    const size_t hc = size_t(hidden) / 2, hsc = size_t(hidden) / 32;
    const size_t ic = size_t(inter) / 2, isc = size_t(inter) / 32;
    for (int r = 0; r < inter; ++r) {
        uint8_t* grow = o + Layout::gate_row(r) * L.rs_gu;
        uint8_t* urow = grow + Layout::kChunk * L.rs_gu;
        std::memcpy(grow, gc + size_t(r) * hc, hc);
        std::memcpy(grow + hc, gs + size_t(r) * hsc, hsc);
        std::memcpy(urow, uc + size_t(r) * hc, hc);
        std::memcpy(urow + hc, us + size_t(r) * hsc, hsc);
    }
    for (int r = 0; r < hidden; ++r) {
        uint8_t* drow = o + L.d_off + size_t(r) * L.rs_d;
        std::memcpy(drow, dc + size_t(r) * ic, ic);
        std::memcpy(drow + ic, ds + size_t(r) * isc, isc);
    }
    // column-blocked copy: block c holds, for every row n, the 8 code bytes
    // of elements 16c..16c+15 and then, for every row, its scale of block c/2
    constexpr int dc_cols = Layout::kDtCols;
    for (int c = 0; c < inter / dc_cols; ++c) {
        uint8_t* blk = o + L.dt_off + size_t(c) * L.dt_stride;
        for (int r = 0; r < hidden; ++r) {
            std::memcpy(blk + size_t(r) * (dc_cols / 2), dc + size_t(r) * ic + size_t(c) * (dc_cols / 2), dc_cols / 2);
            blk[size_t(hidden) * (dc_cols / 2) + r] = ds[size_t(r) * isc + size_t(c) * dc_cols / 32];
        }
    }
    return MOE_OK;
}

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

extern "C" int moe_route_workspace_bytes(int T, int E, int k, size_t* out) {
    if (!out || T < 0 || E < 1 || E > MOE_MAX_EXPERTS || k < 1 || k > E || k > MOE_MAX_TOPK)
        return MOE_ERR_INVALID;
    const int tiles = moe::route_tiles(T, k);
    *out = tiles > 1 ? moe::round_up(size_t(tiles) * E * sizeof(int32_t), 256) : 0;
    return MOE_OK;
}

extern "C" int moe_route_plan(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                              int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                              int32_t* counts_host, void* workspace, size_t ws_bytes, moe_stream_t stream) {
    size_t need = 0;
    if (moe_route_workspace_bytes(T, E, k, &need) != MOE_OK) return MOE_ERR_INVALID;
    if (!counts || !offsets || (T > 0 && (!logits || !ids || !w || !perm || !inv))) return MOE_ERR_INVALID;
    if (size_t(T) * k > size_t(INT32_MAX)) return MOE_ERR_INVALID;
    if (need > 0 && (!workspace || ws_bytes < need || !aligned(workspace, 16))) return MOE_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int tiles = moe::route_tiles(T, k);
    int rc = moe::launch_route_plan(logits, T, E, k, ids, w, counts, offsets, perm, inv,
                                    static_cast<int32_t*>(workspace), tiles, s);
    if (rc != MOE_OK) return rc;
    if (counts_host)
        MOE_CUDA_TRY(cudaMemcpyAsync(counts_host, counts, sizeof(int32_t) * E, cudaMemcpyDeviceToHost, s));
    return MOE_OK;
}

extern "C" int moe_route_plan_noalloc(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                                      int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                                      int32_t* counts_host, moe_stream_t stream) {
    if (T < 0 || E < 1 || E > MOE_MAX_EXPERTS || k < 1 || k > E || k > MOE_MAX_TOPK) return MOE_ERR_INVALID;
    if (!counts || !offsets || (T > 0 && (!logits || !ids || !w || !perm || !inv))) return MOE_ERR_INVALID;
    if (T > moe::route_noalloc_max_tokens()) return MOE_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc = moe::route_plan_noalloc(logits, T, E, k, ids, w, counts, offsets, perm, inv, s);
    if (rc != MOE_OK) return rc;
    if (counts_host)
        MOE_CUDA_TRY(cudaMemcpyAsync(counts_host, counts, sizeof(int32_t) * E, cudaMemcpyDeviceToHost, s));
    return MOE_OK;
}

static int resolve_path(int path, int T, int k) {
    if (path & ~(MOE_FFN_ACCUMULATE | MOE_FFN_SKIP_ABSENT | 3)) return -1;
    path &= 3;
    if (path == MOE_PATH_AUTO) return size_t(T) * k <= MOE_DECODE_MAX_ASSIGN ? MOE_PATH_DECODE : MOE_PATH_PREFILL;
    return path;
}

extern "C" int moe_ffn_workspace_bytes(int T, int k, int hidden, int inter, int path, size_t* out) {
    Layout L;
    if (!out || T < 0 || k < 1 || k > MOE_MAX_TOPK || !Layout::make(hidden, inter, &L)) return MOE_ERR_INVALID;
    path = resolve_path(path, T, k);
    if (path == MOE_PATH_DECODE) *out = moe::decode_workspace_bytes(T, k, hidden, inter);
    else if (path == MOE_PATH_PREFILL) *out = moe::prefill_workspace_bytes(T, k, hidden, inter);
    else return MOE_ERR_INVALID;
    return MOE_OK;
}

extern "C" int moe_expert_ffn(const moe_pool_t* pool, int layer, const void* x_bf16, int T, int k,
                              const int32_t* ids, const float* w, const int32_t* offsets,
                              const int32_t* perm, const int32_t* inv, const int32_t* slot_of,
                              int path, void* workspace, size_t ws_bytes, float* out, moe_stream_t stream) {
    if (!pool) return MOE_ERR_INVALID;
    const moe_pool_desc& d = *moe::pool_desc(pool);
    const Layout& L = *moe::pool_layout(pool);
    if (d.dry_run || !d.dev_slots) return MOE_ERR_STATE;
    if (layer < 0 || layer >= d.layers || T < 0 || k < 1 || k > d.experts || k > MOE_MAX_TOPK)
        return MOE_ERR_INVALID;
    const bool accumulate = (path & MOE_FFN_ACCUMULATE) != 0;
    const bool skip_absent = (path & MOE_FFN_SKIP_ABSENT) != 0;
    path = resolve_path(path, T, k);
    if (path != MOE_PATH_DECODE && path != MOE_PATH_PREFILL) return MOE_ERR_INVALID;
    if (skip_absent && path != MOE_PATH_DECODE) return MOE_ERR_UNSUPPORTED;
    size_t need = 0;
    moe_ffn_workspace_bytes(T, k, d.hidden, d.inter, path, &need);
    if (T > 0) {
        if (!x_bf16 || !ids || !w || !slot_of || !out) return MOE_ERR_INVALID;
        if (path == MOE_PATH_PREFILL && (!offsets || !perm || !inv)) return MOE_ERR_INVALID;
        if (!aligned(x_bf16, 16) || !aligned(out, 16)) return MOE_ERR_INVALID;
        if (need > 0 && (!workspace || ws_bytes < need || !aligned(workspace, 256))) return MOE_ERR_INVALID;
    }
    moe::FfnArgs a;
    a.slots = static_cast<const uint8_t*>(d.dev_slots) + size_t(layer) * d.slots_per_layer * L.expert_bytes;
    a.expert_bytes = L.expert_bytes;
    a.S = d.slots_per_layer;
    a.E = d.experts;
    a.L = &L;
    a.x = static_cast<const uint16_t*>(x_bf16);
    a.T = T;
    a.k = k;
    a.ids = ids;
    a.w = w;
    a.offsets = offsets;
    a.perm = perm;
    a.inv = inv;
    a.slot_of = slot_of;
    a.out = out;
    a.accumulate = accumulate;
    a.skip_absent = skip_absent;
    a.decode_parts_only = d.stage_parts == MOE_STAGE_DECODE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (path == MOE_PATH_DECODE) return moe::launch_decode_ffn(a, workspace, ws_bytes, s);
    if (a.decode_parts_only) return MOE_ERR_UNSUPPORTED;
    return moe::launch_prefill_ffn(a, workspace, ws_bytes, s);
}

static int decode_layer(const moe_pool_t* pool, int layer, const float* logits, const void* x_bf16, int T, int k,
                        int32_t* ids, float* w, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                        const int32_t* slot_of, void* workspace, size_t ws_bytes, float* out, moe_stream_t stream,
                        bool accumulate) {
    if (!pool) return MOE_ERR_INVALID;
    const moe_pool_desc& d = *moe::pool_desc(pool);
    const Layout& L = *moe::pool_layout(pool);
    if (d.dry_run || !d.dev_slots) return MOE_ERR_STATE;
    if (layer < 0 || layer >= d.layers || T < 1 || k < 1 || k > d.experts || k > MOE_MAX_TOPK || T * k > 32)
        return MOE_ERR_INVALID;
    if (!logits || !x_bf16 || !ids || !w || !counts || !offsets || !perm || !inv || !slot_of || !out)
        return MOE_ERR_INVALID;
    size_t need = 0;
    moe_ffn_workspace_bytes(T, k, d.hidden, d.inter, MOE_PATH_DECODE, &need);
    if (!workspace || ws_bytes < need || !aligned(workspace, 256) || !aligned(x_bf16, 16) || !aligned(out, 16))
        return MOE_ERR_INVALID;
    moe::FfnArgs a;
    a.slots = static_cast<const uint8_t*>(d.dev_slots) + size_t(layer) * d.slots_per_layer * L.expert_bytes;
    a.expert_bytes = L.expert_bytes;
    a.S = d.slots_per_layer;
    a.E = d.experts;
    a.L = &L;
    a.x = static_cast<const uint16_t*>(x_bf16);
    a.T = T;
    a.k = k;
    a.ids = ids;
    a.w = w;
    a.offsets = offsets;
    a.perm = perm;
    a.inv = inv;
    a.slot_of = slot_of;
    a.out = out;
    a.accumulate = accumulate;
    moe::RouteOut ro;
    ro.logits = logits;
    ro.ids = ids;
    ro.w = w;
    ro.counts = counts;
    ro.offsets = offsets;
    ro.perm = perm;
    ro.inv = inv;
    return moe::launch_decode_layer(a, ro, workspace, static_cast<cudaStream_t>(stream));
}

extern "C" int moe_decode_layer(const moe_pool_t* pool, int layer, const float* logits, const void* x_bf16, int T,
                                int k, int32_t* ids, float* w, int32_t* counts, int32_t* offsets, int32_t* perm,
                                int32_t* inv, const int32_t* slot_of, void* workspace, size_t ws_bytes, float* out,
                                moe_stream_t stream) {
    return decode_layer(pool, layer, logits, x_bf16, T, k, ids, w, counts, offsets, perm, inv, slot_of, workspace,
                        ws_bytes, out, stream, false);
}

extern "C" int moe_decode_layer_acc(const moe_pool_t* pool, int layer, const float* logits, const void* x_bf16,
                                    int T, int k, int32_t* ids, float* w, int32_t* counts, int32_t* offsets,
                                    int32_t* perm, int32_t* inv, const int32_t* slot_of, void* workspace,
                                    size_t ws_bytes, float* out, moe_stream_t stream) {
    return decode_layer(pool, layer, logits, x_bf16, T, k, ids, w, counts, offsets, perm, inv, slot_of, workspace,
                        ws_bytes, out, stream, true);
}

namespace moe {
// Wait, polling an event (at most timeout_ms), until the work enqueued so
// far on `s` is done.  One event per host thread, created on first use.
static int bounded_stream_wait(cudaStream_t s, int timeout_ms) {
    thread_local cudaEvent_t ev = nullptr;
    if (ev == nullptr) MOE_CUDA_TRY(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
    MOE_CUDA_TRY(cudaEventRecord(ev, s));
    const auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        const cudaError_t q = cudaEventQuery(ev);
        if (q == cudaSuccess) return MOE_OK;
        if (q != cudaErrorNotReady) return cuda_fail(q);
        if (std::chrono::steady_clock::now() - t0 > std::chrono::milliseconds(timeout_ms)) return MOE_ERR_TIMEOUT;
        std::this_thread::yield();
    }
}
}  // namespace moe

extern "C" int moe_ffn_status(void* workspace, int path, moe_stream_t stream, uint32_t* bits) {
    if (!workspace || !bits || (path != MOE_PATH_DECODE && path != MOE_PATH_PREFILL)) return MOE_ERR_INVALID;
    if (!aligned(workspace, 256)) return MOE_ERR_INVALID;
    // decode: word 2 of the 256-byte control block; prefill: the first word
    uint32_t* dev = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + (path == MOE_PATH_DECODE ? 8 : 0));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    constexpr int kStatusWaitMs = 10000;
    int rc = moe::bounded_stream_wait(s, kStatusWaitMs);
    if (rc != MOE_OK) return rc;
    uint32_t h = 0;
    MOE_CUDA_TRY(cudaMemcpy(&h, dev, sizeof h, cudaMemcpyDeviceToHost));   // the stream's work is done
    if (h != 0) {
        MOE_CUDA_TRY(cudaMemsetAsync(dev, 0, sizeof h, s));
        rc = moe::bounded_stream_wait(s, kStatusWaitMs);
        if (rc != MOE_OK) return rc;
    }
    *bits = h;
    return MOE_OK;
}

extern "C" int moe_debug_stall_next_decode(int n) {
    if (n < 0) return MOE_ERR_INVALID;
    moe::g_stall_decode.store(n);
    return MOE_OK;
}

extern "C" int moe_combine(const float* y_perm, const float* w, const int32_t* inv, int T, int k, int H,
                           float* out, moe_stream_t stream) {
    if (T < 0 || k < 1 || k > MOE_MAX_TOPK || H < 1) return MOE_ERR_INVALID;
    if (T == 0) return MOE_OK;
    if (!y_perm || !w || !inv || !out) return MOE_ERR_INVALID;
    return moe::launch_combine(y_perm, w, inv, T, k, H, out, static_cast<cudaStream_t>(stream));
}

extern "C" int moe_quant_mxfp4(const void* x_bf16, int K, int rows, uint8_t* q, uint8_t* scales, int scale_stride,
                               moe_stream_t stream) {
    if (K <= 0 || K % 32 || rows < 0 || scale_stride < K / 32) return MOE_ERR_INVALID;
    if (rows == 0) return MOE_OK;
    if (!x_bf16 || !q || !scales || !aligned(x_bf16, 16) || !aligned(q, 16)) return MOE_ERR_INVALID;
    return moe::launch_quant_mxfp4(static_cast<const uint16_t*>(x_bf16), K, rows, q, scales, scale_stride,
                                   static_cast<cudaStream_t>(stream));
}

extern "C" int moe_quant_mxfp8(const void* x_bf16, int K, const int32_t* perm, int k, int rows, uint8_t* q,
                               uint8_t* scales, int scale_stride, moe_stream_t stream) {
    if (K <= 0 || K % 32 || rows < 0 || k < 1 || scale_stride < K / 32) return MOE_ERR_INVALID;
    if (rows == 0) return MOE_OK;
    if (!x_bf16 || !q || !scales || !aligned(x_bf16, 16) || !aligned(q, 16)) return MOE_ERR_INVALID;
    return moe::launch_quant_mxfp8(static_cast<const uint16_t*>(x_bf16), K, perm, k, rows, q, scales,
                                   scale_stride, static_cast<cudaStream_t>(stream));
}

extern "C" int moe_gguf_expert_bytes(int fmt, int hidden, int inter, size_t* out) {
    if (!out) return MOE_ERR_INVALID;
    const size_t b = moe::gguf_expert_bytes(fmt, hidden, inter);
    if (!b) return MOE_ERR_INVALID;
    *out = b;
    return MOE_OK;
}

extern "C" int moe_gguf_workspace_bytes(int T, int k, int hidden, int inter, size_t* out) {
    if (!out || T < 0 || k < 1 || k > MOE_MAX_TOPK || hidden <= 0 || inter <= 0) return MOE_ERR_INVALID;
    *out = moe::gguf_workspace_bytes(T, k, hidden, inter);
    return MOE_OK;
}

extern "C" int moe_decode_layer_gguf(int fmt, const void* slots, int n_slots, int hidden, int inter,
                                     const float* logits, const void* x_bf16, int T, int k, int32_t* ids, float* w,
                                     int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                                     const int32_t* slot_of, int E, void* workspace, size_t ws_bytes, float* out,
                                     int accumulate, moe_stream_t stream) {
    if (fmt != MOE_GGUF_Q8_0 && fmt != MOE_GGUF_Q4_K) return MOE_ERR_INVALID;
    if (!moe::gguf_expert_bytes(fmt, hidden, inter)) return MOE_ERR_INVALID;
    if (T < 1 || k < 1 || k > MOE_MAX_TOPK || k > E || E > MOE_MAX_EXPERTS || n_slots < 1 || T * k > 32)
        return MOE_ERR_INVALID;
    if (!slots || !logits || !x_bf16 || !ids || !w || !counts || !offsets || !perm || !inv || !slot_of || !out ||
        !workspace)
        return MOE_ERR_INVALID;
    if (!aligned(slots, 256) || !aligned(workspace, 256) || !aligned(x_bf16, 16)) return MOE_ERR_INVALID;
    if (ws_bytes < moe::gguf_workspace_bytes(T, k, hidden, inter)) return MOE_ERR_INVALID;
    if (!moe::gguf_fused_supported(fmt, T, k, hidden, inter)) return MOE_ERR_UNSUPPORTED;
    moe::RouteOut ro;
    ro.logits = logits;
    ro.ids = ids;
    ro.w = w;
    ro.counts = counts;
    ro.offsets = offsets;
    ro.perm = perm;
    ro.inv = inv;
    return moe::launch_gguf_fused(fmt, static_cast<const uint8_t*>(slots), n_slots, E, hidden, inter,
                                  static_cast<const uint16_t*>(x_bf16), T, k, nullptr, nullptr, slot_of, &ro,
                                  workspace, out, accumulate != 0, static_cast<cudaStream_t>(stream));
}

extern "C" int moe_expert_ffn_gguf(int fmt, const void* slots, int n_slots, int hidden, int inter, const void* x_bf16,
                                   int T, int k, const int32_t* ids, const float* w, const int32_t* slot_of, int E,
                                   void* workspace, size_t ws_bytes, float* out, int accumulate,
                                   moe_stream_t stream) {
    if (fmt != MOE_GGUF_Q8_0 && fmt != MOE_GGUF_Q4_K) return MOE_ERR_INVALID;
    if (!moe::gguf_expert_bytes(fmt, hidden, inter)) return MOE_ERR_INVALID;
    if (T < 0 || k < 1 || k > MOE_MAX_TOPK || E < 1 || E > MOE_MAX_EXPERTS || n_slots < 1) return MOE_ERR_INVALID;
    if (T == 0) return MOE_OK;
    if (!slots || !x_bf16 || !ids || !w || !slot_of || !out || !workspace) return MOE_ERR_INVALID;
    if (!aligned(slots, 256) || !aligned(workspace, 256) || !aligned(x_bf16, 4)) return MOE_ERR_INVALID;
    if (ws_bytes < moe::gguf_workspace_bytes(T, k, hidden, inter)) return MOE_ERR_INVALID;
    return moe::launch_gguf_ffn(fmt, static_cast<const uint8_t*>(slots), n_slots, E, hidden, inter,
                                static_cast<const uint16_t*>(x_bf16), T, k, ids, w, slot_of, workspace, out,
                                accumulate != 0, static_cast<cudaStream_t>(stream));
}
