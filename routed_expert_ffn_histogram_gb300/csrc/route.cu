// Routing and grouping: top-k + softmax over the selected experts, a
// shared-memory atomic histogram per tile of tokens, an exclusive prefix sum
// over experts and a stable permutation of the assignments by expert.
//
// Source: tinyserve README, "Performance" (top_k=4 routing of GPT-OSS-20B)
// and "How it works" item 6 (batched prefill groups tokens by expert so each
// unique expert is loaded once); llama.cpp discussion "fixed GPU expert
// working set with Native CPU miss execution", main post (selected expert IDs
// are split per step before the experts run).
//
// Layout: one warp per token for the top-k (each lane holds E/32 logits,
// k rounds of a warp-wide arg-best); tiles of 256 tokens per CTA.  With one
// tile the whole plan is a single launch; otherwise a second launch turns
// the per-tile histograms into global offsets and scatters the permutation.
// Ranks inside a warp come from __match_any_sync + __popc, so the order is
// fixed by the assignment index, never by the order atomics land in.
#include <cfloat>
#include <cmath>
#include <mutex>

#include "internal.h"
#include "route_warp.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTileTokens = 256;

struct Smem {
    int hist[MOE_MAX_EXPERTS];
    int base[MOE_MAX_EXPERTS];
    int scan_tmp[kWarps];
    int warp_cnt[kWarps][MOE_MAX_EXPERTS];
};

// Top-k + softmax for the tokens [t0, t0 + ntok) of this CTA, one warp per
// token at a time; accumulates the histogram into hist (zeroed by the caller).
template <int EPL>
__device__ void topk_tokens(const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ ids,
                            float* __restrict__ w, int t0, int ntok, int* hist) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int t1 = min(T, t0 + ntok);
    for (int t = t0 + warp; t < t1; t += nwarps) {
        float sel_v;
        int sel_id;
        topk_warp<EPL>(logits + (size_t)t * E, E, k, sel_v, sel_id);
        const float wv = softmax_lane(sel_v, k);
        if (lane < k) {
            ids[(size_t)t * k + lane] = sel_id;
            w[(size_t)t * k + lane] = wv;
            if (hist) atomicAdd(&hist[sel_id], 1);
        }
    }
}

// Exclusive scan of tot[e] over e < E (E <= kThreads) into out[e]; returns
// the total to every thread.
__device__ int block_exclusive_scan(int v, int* out, Smem& sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += n;
    }
    if (lane == 31) sm.scan_tmp[warp] = incl;
    __syncthreads();
    int wbase = 0, total = 0;
    for (int i = 0; i < kWarps; ++i) {
        const int s = sm.scan_tmp[i];
        if (i < warp) wbase += s;
        total += s;
    }
    out[threadIdx.x] = wbase + incl - v;
    __syncthreads();
    return total;
}

// Offsets + stable scatter of the assignments [a0, a1) of one tile, given
// this tile's first position per expert in sm.base.
__device__ void scatter_tile(const int32_t* __restrict__ ids, int a0, int a1, int E,
                             int32_t* __restrict__ perm, int32_t* __restrict__ inv, Smem& sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kWarps * MOE_MAX_EXPERTS; i += kThreads) (&sm.warp_cnt[0][0])[i] = 0;
    __syncthreads();
    const int n = a1 - a0;
    const int seg = ((n + kWarps - 1) / kWarps + 31) / 32 * 32;
    const int ws = a0 + warp * seg, we = min(a1, ws + seg);
    const uint32_t lt = (1u << lane) - 1u;
    for (int c = ws; c < we; c += 32) {
        const int a = c + lane;
        const int e = (a < we) ? ids[a] : -1;
        const uint32_t mask = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && (mask & lt) == 0) sm.warp_cnt[warp][e] += __popc(mask);
    }
    __syncthreads();
    if (threadIdx.x < E) {
        int run = sm.base[threadIdx.x];
        for (int i = 0; i < kWarps; ++i) {
            const int c = sm.warp_cnt[i][threadIdx.x];
            sm.warp_cnt[i][threadIdx.x] = run;
            run += c;
        }
    }
    __syncthreads();
    for (int c = ws; c < we; c += 32) {
        const int a = c + lane;
        const int e = (a < we) ? ids[a] : -1;
        const uint32_t mask = __match_any_sync(0xffffffffu, e);
        int pos = 0;
        if (e >= 0) pos = sm.warp_cnt[warp][e] + __popc(mask & lt);
        __syncwarp();
        if (e >= 0) {
            perm[pos] = a;
            inv[a] = pos;
            if ((mask & lt) == 0) sm.warp_cnt[warp][e] += __popc(mask);
        }
        __syncwarp();
    }
}

// Whole plan in one CTA (T <= one tile).
template <int EPL>
__global__ void __launch_bounds__(kThreads) route_single_kernel(
    const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ ids,
    float* __restrict__ w, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
    __shared__ Smem sm;
    if (threadIdx.x < MOE_MAX_EXPERTS) sm.hist[threadIdx.x] = 0;
    __syncthreads();
    topk_tokens<EPL>(logits, T, E, k, ids, w, 0, kTileTokens, sm.hist);
    __syncthreads();
    const int tot = (threadIdx.x < E) ? sm.hist[threadIdx.x] : 0;
    const int total = block_exclusive_scan(tot, sm.base, sm);
    if (threadIdx.x < E) {
        counts[threadIdx.x] = tot;
        offsets[threadIdx.x] = sm.base[threadIdx.x];
    }
    if (threadIdx.x == 0) offsets[E] = total;
    __syncthreads();
    scatter_tile(ids, 0, T * k, E, perm, inv, sm);
}

// Multi-tile, pass 1: top-k + softmax, one warp per token and kTopkWarps
// tokens per CTA, so every SM has tokens in flight (the per-token work is a
// latency chain of shuffles); each token adds its k experts to the
// histogram of its kTileTokens tile in tile_hist (zeroed before launch).
constexpr int kTopkWarps = 8;
template <int EPL>
__global__ void __launch_bounds__(32 * kTopkWarps) route_topk_kernel(
    const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ ids,
    float* __restrict__ w, int32_t* __restrict__ tile_hist) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kTopkWarps + (threadIdx.x >> 5);
    if (t >= T) return;  // whole warp
    float sel_v;
    int sel_id;
    topk_warp<EPL>(logits + (size_t)t * E, E, k, sel_v, sel_id);
    const float wv = softmax_lane(sel_v, k);
    if (lane < k) {
        ids[(size_t)t * k + lane] = sel_id;
        w[(size_t)t * k + lane] = wv;
        atomicAdd(&tile_hist[(size_t)(t / kTileTokens) * E + sel_id], 1);
    }
}

// Whole plan in one warp when T * k <= 32 (the decode shapes): no block
// barriers (route_tiny_warp).
template <int EPL>
__global__ void __launch_bounds__(32) route_tiny_kernel(
    const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ ids,
    float* __restrict__ w, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
    // launched with programmatic stream serialisation: nothing is read
    // before the previous kernel in the stream has finished
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ int sel_id[32];
    __shared__ float sel_v[32];
    route_tiny_warp<EPL>(logits, T, E, k, ids, w, counts, offsets, perm, inv, sel_id, sel_v);
}

// Multi-tile, pass 2: global offsets from all tile histograms, then the
// stable scatter of this tile.
__global__ void __launch_bounds__(kThreads) route_scatter_kernel(
    const int32_t* __restrict__ ids, int T, int E, int k, const int32_t* __restrict__ tile_hist,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
    int32_t* __restrict__ inv) {
    __shared__ Smem sm;
    const int tile = blockIdx.x, n_tiles = gridDim.x;
    int tot = 0, pre = 0;
    if (threadIdx.x < E) {
        for (int i = 0; i < n_tiles; ++i) {
            const int c = tile_hist[(size_t)i * E + threadIdx.x];
            tot += c;
            if (i < tile) pre += c;
        }
    }
    const int total = block_exclusive_scan(tot, sm.base, sm);
    if (threadIdx.x < E) {
        if (tile == 0) {
            counts[threadIdx.x] = tot;
            offsets[threadIdx.x] = sm.base[threadIdx.x];
        }
        sm.base[threadIdx.x] += pre;
    }
    if (tile == 0 && threadIdx.x == 0) offsets[E] = total;
    __syncthreads();
    const int a0 = tile * kTileTokens * k;
    const int a1 = min(T, (tile + 1) * kTileTokens) * k;
    scatter_tile(ids, a0, a1, E, perm, inv, sm);
}

}  // namespace

int route_tiles(int T, int k) {
    (void)k;
    return T <= kTileTokens ? 1 : (T + kTileTokens - 1) / kTileTokens;
}

template <int EPL>
int launch_route_epl(const float* logits, int T, int E, int k, int32_t* ids, float* w, int32_t* counts,
                     int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* tile_hist, int n_tiles,
                     cudaStream_t s) {
    if (T * k <= 32) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1);
        cfg.blockDim = dim3(32);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, route_tiny_kernel<EPL>, logits, T, E, k, ids, w, counts, offsets,
                                        perm, inv));
    } else if (n_tiles <= 1) {
        route_single_kernel<EPL><<<1, kThreads, 0, s>>>(logits, T, E, k, ids, w, counts, offsets, perm, inv);
    } else {
        MOE_CUDA_TRY(cudaMemsetAsync(tile_hist, 0, sizeof(int32_t) * size_t(n_tiles) * E, s));
        route_topk_kernel<EPL><<<(T + kTopkWarps - 1) / kTopkWarps, 32 * kTopkWarps, 0, s>>>(logits, T, E, k, ids,
                                                                                             w, tile_hist);
        MOE_CUDA_TRY(cudaGetLastError());
        route_scatter_kernel<<<n_tiles, kThreads, 0, s>>>(ids, T, E, k, tile_hist, counts, offsets, perm, inv);
    }
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

int launch_route_plan(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                      int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                      int32_t* tile_hist, int n_tiles, cudaStream_t s) {
    if (E <= 32) return launch_route_epl<1>(logits, T, E, k, ids, w, counts, offsets, perm, inv, tile_hist, n_tiles, s);
    if (E <= 64) return launch_route_epl<2>(logits, T, E, k, ids, w, counts, offsets, perm, inv, tile_hist, n_tiles, s);
    if (E <= 128) return launch_route_epl<4>(logits, T, E, k, ids, w, counts, offsets, perm, inv, tile_hist, n_tiles, s);
    return launch_route_epl<8>(logits, T, E, k, ids, w, counts, offsets, perm, inv, tile_hist, n_tiles, s);
}

// ---------------------------------------------------------------------------
// Routing without caller-provided scratch (moe_route_plan_noalloc).
//
// Some callers cannot allocate device memory where they route: engines
// whose device memory is carved up in advance by their own allocator under a
// fixed budget, and real-time decode loops that must never call into the
// driver's allocator, which can block or synchronise.  For them the per-tile histograms live in this
// file-scope device array instead of a workspace.  It holds
// kNoallocMaxTiles * MOE_MAX_EXPERTS int32 (64 KB), enough for up to
// kNoallocMaxTiles * 256 = 16384 tokens; every GPU that loads the library
// keeps it until the process exits.  Each call clears the entries it uses
// (an asynchronous memset on the caller's stream, not an allocation) before
// counting into them.  All calls share it, so calls that
// can overlap on the GPU (different streams, or different host threads
// without ordering) race on it.
// ---------------------------------------------------------------------------
namespace {
constexpr int kNoallocMaxTiles = 64;
__device__ __align__(256) int32_t g_route_noalloc_scratch[kNoallocMaxTiles * MOE_MAX_EXPERTS];

// Device address of the scratch array on the current device, resolved once
// per device (with that device current) on the first call made there and
// kept for the life of the process (the header asks callers not to use the
// entry after a device reset, which could move the array).
int noalloc_scratch(int32_t** out) {
    static std::mutex mu;
    static int32_t* addr[64] = {};
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        MOE_CUDA_TRY(cudaGetSymbolAddress(&p, g_route_noalloc_scratch));
        addr[dev] = static_cast<int32_t*>(p);
    }
    *out = addr[dev];
    return MOE_OK;
}
}  // namespace

int route_plan_noalloc(const float* logits, int T, int E, int k, int32_t* ids, float* w, int32_t* counts,
                       int32_t* offsets, int32_t* perm, int32_t* inv, cudaStream_t s) {
    const int tiles = route_tiles(T, k);
    if (tiles > kNoallocMaxTiles) return MOE_ERR_INVALID;
    int32_t* scratch = nullptr;
    const int rc = noalloc_scratch(&scratch);
    if (rc != MOE_OK) return rc;
    return launch_route_plan(logits, T, E, k, ids, w, counts, offsets, perm, inv, scratch, tiles, s);
}

int route_noalloc_max_tokens() { return kNoallocMaxTiles * kTileTokens; }

}  // namespace moe
