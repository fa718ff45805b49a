// Host-side definitions shared by the library's translation units.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "moe.h"

namespace moe {

// Remember a CUDA error for moe_last_cuda_error() and map it to a status.
int cuda_fail(cudaError_t e);

#define MOE_CUDA_TRY(expr)                                  \
    do {                                                    \
        cudaError_t _e = (expr);                            \
        if (_e != cudaSuccess) return ::moe::cuda_fail(_e); \
    } while (0)

inline size_t pad16(size_t x) { return (x + 15) & ~size_t(15); }
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// GPU-native packed expert.  Every row stores its K/2 code bytes followed by
// its K/32 E8M0 scale bytes, zero-padded to a multiple of 32 bytes.  The gate/up
// matrix has 2I rows interleaved in chunks of 32: chunk c holds gate rows
// 32c..32c+31 then up rows 32c..32c+31, so a 32-wide block of h = SwiGLU(g, u)
// comes from one 64-row pair of chunks.  The down matrix (H rows) follows,
// then a column-blocked copy of it for decode: for each block of 16 columns
// (16 consecutive elements of h), the H rows' 8 code bytes of that block,
// then the H rows' E8M0 scale bytes of the 32-block it lies in.
struct Layout {
    int H = 0, I = 0;
    size_t rs_gu = 0;        // bytes per gate/up row (K = H)
    size_t rs_d = 0;         // bytes per down row (K = I)
    size_t d_off = 0;        // byte offset of the down matrix
    size_t dt_off = 0;       // byte offset of the column-blocked down copy
    size_t dt_stride = 0;    // bytes per 16-column block of it (H*8 codes + H scales, padded)
    size_t expert_bytes = 0; // whole expert, a multiple of 1024

    static bool make(int hidden, int inter, Layout* L) {
        if (hidden <= 0 || inter <= 0 || hidden % 64 || inter % 64) return false;
        L->H = hidden;
        L->I = inter;
        // rows are multiples of 32 bytes: a TMA rule for the unpacked-FP4 tile type
        L->rs_gu = round_up(size_t(hidden) / 2 + pad16(size_t(hidden) / 32), 32);
        L->rs_d = round_up(size_t(inter) / 2 + pad16(size_t(inter) / 32), 32);
        L->d_off = 2 * size_t(inter) * L->rs_gu;
        L->dt_off = round_up(L->d_off + size_t(hidden) * L->rs_d, 128);
        L->dt_stride = round_up(size_t(hidden) * (kDtCols / 2 + 1), 128);
        L->expert_bytes = round_up(L->dt_off + size_t(inter / kDtCols) * L->dt_stride, 1024);
        return true;
    }
    static constexpr int kChunk = 32;
    static constexpr int kDtCols = 16;   // columns per block of the column-blocked down copy
    // Row of the gate/up matrix that holds gate row r (its up row: + kChunk).
    __host__ __device__ static inline size_t gate_row(int r) {
        return size_t(r / kChunk) * (2 * kChunk) + size_t(r % kChunk);
    }
};

struct DeviceInfo {
    int device = -1;
    int sms = 0;
    int cc_major = 0, cc_minor = 0;
    size_t smem_optin = 0;
};
// Properties of the current device (cached per device).
int current_device_info(DeviceInfo* out);

// One bit per device (ordinal < 64), set once a kernel's launch attributes
// are in place on that device.  Atomic, so host threads may launch
// concurrently; two threads that both find the bit clear both set the same
// attribute, which is harmless.
struct DeviceOnce {
    std::atomic<uint64_t> bits{0};
    bool done(int dev) const { return (bits.load(std::memory_order_acquire) >> dev) & 1u; }
    void mark(int dev) { bits.fetch_or(uint64_t(1) << dev, std::memory_order_release); }
};

// ---- kernel launchers (route.cu, decode.cu, prefill.cu) -------------------

int launch_route_plan(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                      int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                      int32_t* tile_hist, int n_tiles, cudaStream_t s);
int route_tiles(int T, int k);
int route_plan_noalloc(const float* logits, int T, int E, int k, int32_t* ids, float* w, int32_t* counts,
                       int32_t* offsets, int32_t* perm, int32_t* inv, cudaStream_t s);
int route_noalloc_max_tokens();

struct FfnArgs {
    const uint8_t* slots;      // base of this layer's slots
    size_t expert_bytes;
    bool decode_parts_only = false;  // the pool staged only what the fused decode kernel reads
    int S, E;
    const Layout* L;
    const uint16_t* x;         // bf16 [T][H]
    int T, k;
    const int32_t* ids;
    const float* w;
    const int32_t* offsets;
    const int32_t* perm;
    const int32_t* inv;
    const int32_t* slot_of;
    float* out;
    bool accumulate = false;   // out += result instead of out = result
    bool skip_absent = false;  // decode: serve only assignments whose expert's slot is >= 0
};

struct RouteOut {
    const float* logits;
    int32_t *ids, *counts, *offsets, *perm, *inv;
    float* w;
};

size_t decode_workspace_bytes(int T, int k, int H, int I);
size_t decode_acc_offset(int T, int k, int I);
int launch_decode_layer(const FfnArgs& a, const RouteOut& ro, void* ws, cudaStream_t s);
size_t decode_fused_smem(int T, int k, int H, int I);
extern std::atomic<int> g_stall_decode;  // test hook: fused decode launches to stall
int launch_decode_fused(const FfnArgs& a, void* ws, cudaStream_t s);
int launch_decode_ffn(const FfnArgs& a, void* ws, size_t ws_bytes, cudaStream_t s);

size_t prefill_workspace_bytes(int T, int k, int H, int I);
int launch_prefill_ffn(const FfnArgs& a, void* ws, size_t ws_bytes, cudaStream_t s);
// The prefill path in two parts: zeroing + activation quantisation once,
// then the grouped GEMMs of the expert groups [e0, e1) (slots from the host
// table slot_tab when it is given, else from the device map a.slot_of).
int launch_prefill_prepare(const FfnArgs& a, void* ws, size_t ws_bytes, cudaStream_t s);
int launch_prefill_experts(const FfnArgs& a, void* ws, int e0, int e1, const int32_t* slot_tab, int max_mtiles,
                           cudaStream_t s);

// Decode on GGUF expert weights (gguf_decode.cu: three launches;
// gguf_fused.cu: one launch, its workspace layout and counters).
size_t gguf_row_bytes(int fmt, int K);
size_t gguf_expert_bytes(int fmt, int H, int I);
size_t gguf_workspace_bytes(int T, int k, int H, int I);
size_t gguf_h_offset();
size_t gguf_y_offset(int T, int k, int I);
int launch_gguf_ffn(int fmt, const uint8_t* slots, int S, int E, int H, int I, const uint16_t* x, int T, int k,
                    const int32_t* ids, const float* w, const int32_t* slot_of, void* ws, float* out,
                    bool accumulate, cudaStream_t s);
bool gguf_fused_supported(int fmt, int T, int k, int H, int I);
int launch_gguf_fused(int fmt, const uint8_t* slots, int S, int E, int H, int I, const uint16_t* x, int T, int k,
                      const int32_t* ids, const float* w, const int32_t* slot_of, const RouteOut* ro, void* ws,
                      float* out, bool accumulate, cudaStream_t s);

// Device-planned pool staging (pool_dev.cu): `rec` is the layer's record in
// the device state (pool_plan.h, dev_record).
int launch_pool_plan(uint8_t* rec, int S, int E, int policy, const int32_t* counts, int32_t* slot_of,
                     int32_t* split, uint64_t bytes_per_load, cudaStream_t s);
// Routing of T tokens (T * k <= 32; the one-warp plan of launch_route_plan)
// and the planning of the layer's event in one launch.
int launch_pool_route_plan(const float* logits, int T, int k, int32_t* ids, float* w, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv, uint8_t* rec, int S, int E, int policy,
                           int32_t* slot_of, int32_t* split, uint64_t bytes_per_load, cudaStream_t s);
int launch_pool_gather(const uint8_t* rec, int S, int E, const uint8_t* host_layer, uint8_t* slots_layer,
                       size_t eb, size_t len0, size_t off1, size_t len1, cudaStream_t s);

// Tensor-core rate probe (mma_probe.cu).
int launch_mma_probe(int stages, uint32_t* err, int* ctas, cudaStream_t s);

int launch_combine(const float* y_perm, const float* w, const int32_t* inv, int T, int k, int H,
                   float* out, cudaStream_t s);
int launch_quant_mxfp8(const uint16_t* x, int K, const int32_t* perm, int k, int rows, uint8_t* q,
                       uint8_t* scales, int scale_stride, cudaStream_t s);
// MXFP4 (E2M1 + E8M0 per 32) of bf16 rows, codes packed two per byte.
int launch_quant_mxfp4(const uint16_t* x, int K, int rows, uint8_t* q, uint8_t* scales, int scale_stride,
                       cudaStream_t s);
// Prefill operand: token t's MXFP8 row written to grouped rows inv[t*k + j].
int launch_quant_mxfp8_scatter(const uint16_t* x, int K, const int32_t* inv, int k, int T, uint8_t* q,
                               uint8_t* scales, int scale_stride, cudaStream_t s);

}  // namespace moe
