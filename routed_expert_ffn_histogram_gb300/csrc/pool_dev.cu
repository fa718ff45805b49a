// Device-planned staging of the expert-slot pool: the policy state of every
// layer lives in a caller-provided device buffer (one record per layer, laid
// out by pool_plan.h's dev_record), each staging event is planned on the GPU
// from the device counts that routing wrote, and the SMs copy the missed
// experts out of the pinned host store through its mapped device address.
//
// Sources: tinyserve README, "How it works" item 1 (experts kept as raw
// quantised bytes in pinned CPU memory), item 3 (cache keyed by (layer,
// expert_id) with a GPU slot map) and item 4 (host-to-device traffic
// overlapped with compute); llama.cpp discussion "fixed GPU expert working
// set", main post (routed ids split into resident hits and misses).  The
// decisions are those of the host pool (the planning code is shared); what
// differs is where they are taken: on a Grace host the GPU reads pinned host
// memory at the link rate itself, so the route -> plan -> copy -> FFN chain
// of a layer is enqueued once and runs with no host round trip between
// routing and the copies (the copy on a second stream, beside the FFN of the
// event's hits, when the caller asks for it).
//
// Kernels:
//   pool_plan_kernel    one CTA of 256 threads: the layer's record is loaded
//                       into shared memory by all threads, thread 0 plans
//                       the event (pool_plan.h) and updates the counters,
//                       all threads write the record back and the slot map.
//   pool_route_plan_kernel  the same planning, with the routing of the event's
//                       tokens (T * k <= 32) done by warp 0 in the same launch
//                       while the other warps load the record.
//   pool_gather_kernel  one CTA of 64 threads per SM: 64 KB chunks of the
//                       planned loads (both staged parts of each expert),
//                       16-byte loads from host memory, sixteen in flight
//                       per thread (≈ 2.5 MB in flight: the link, ≈ 0.2
//                       TB/s, stays the limit; eight gave 1 % less).  Small
//                       CTAs so that the FFN of a layer's hits runs beside
//                       the copy: an SM holding one of them (93 registers a
//                       thread) still takes a decode FFN CTA (with 128-thread
//                       CTAs the FFN waited for the copy to end; the CTA
//                       scheduler does not spread them one per SM).
#include <cstdint>

#include "internal.h"
#include "pool_plan.h"
#include "route_warp.cuh"

namespace moe {
namespace {

constexpr int kPlanThreads = 256;
static_assert(kPlanThreads >= MOE_MAX_EXPERTS, "one thread per expert in the planner");
constexpr int kGatherThreads = 64;
constexpr int kGatherUnroll = 16;
constexpr unsigned long long kChunk = 64ull << 10;

// The planner's shared-memory copy of a layer's record and the event.
struct PlanSmem {
    int32_t se[MOE_MAX_EXPERTS], es[MOE_MAX_EXPERTS], cnt[MOE_MAX_EXPERTS], hit_e[MOE_MAX_EXPERTS],
        miss_e[MOE_MAX_EXPERTS];
    int warp_hits[kPlanThreads / 32], warp_misses[kPlanThreads / 32];
    int64_t st[MOE_MAX_EXPERTS], uses[MOE_MAX_EXPERTS];
    int8_t seg[MOE_MAX_EXPERTS];
    PlanLoad loads[MOE_MAX_EXPERTS];
    int ok_s;
};

// Slot-indexed fields of the record into shared memory (threads t0, t0 +
// nt, ...); the expert-indexed ones are loaded by the callers.
__device__ __forceinline__ void load_slots(PlanSmem& sm, const uint8_t* rec, const DevRecord& dr, int S, int t0,
                                           int nt) {
    const int32_t* g_se = reinterpret_cast<const int32_t*>(rec + dr.se);
    const int64_t* g_st = reinterpret_cast<const int64_t*>(rec + dr.st);
    const int64_t* g_uses = reinterpret_cast<const int64_t*>(rec + dr.uses);
    const int8_t* g_seg = reinterpret_cast<const int8_t*>(rec + dr.seg);
    for (int i = t0; i < S; i += nt) {
        sm.se[i] = g_se[i];
        sm.st[i] = g_st[i];
        sm.uses[i] = g_uses[i];
        sm.seg[i] = g_seg[i];
    }
}

// One event planned by the whole CTA once the record and the counts are in
// shared memory; c and es0: this thread's expert's count and slot before the
// event (0 and -1 past E).
__device__ void plan_block(PlanSmem& sm, int c, int es0, uint8_t* rec, const DevRecord& dr, int S, int E,
                           int policy, int32_t* __restrict__ slot_of, int32_t* __restrict__ split,
                           unsigned long long bytes_per_load) {
    const int t = threadIdx.x;
    int32_t* g_se = reinterpret_cast<int32_t*>(rec + dr.se);
    int32_t* g_es = reinterpret_cast<int32_t*>(rec + dr.es);
    int64_t* g_st = reinterpret_cast<int64_t*>(rec + dr.st);
    int64_t* g_uses = reinterpret_cast<int64_t*>(rec + dr.uses);
    int8_t* g_seg = reinterpret_cast<int8_t*>(rec + dr.seg);
    int64_t* g_freq = reinterpret_cast<int64_t*>(rec + dr.freq);
    uint8_t* g_fresh = rec + dr.fresh;
    int32_t* se = sm.se;
    int32_t* es = sm.es;
    int32_t* cnt = sm.cnt;
    int32_t* hit_e = sm.hit_e;
    int32_t* miss_e = sm.miss_e;
    int64_t* st = sm.st;
    int64_t* uses = sm.uses;
    int8_t* seg = sm.seg;
    PlanLoad* loads = sm.loads;
    int* warp_hits = sm.warp_hits;
    int* warp_misses = sm.warp_misses;
    int& ok_s = sm.ok_s;
    // the event's routed experts, split into resident (hits) and absent
    // (misses), each list in ascending expert id, built by all threads so
    // that the planning thread walks only the routed experts
    const int lane = t & 31, wid = t >> 5;
    const bool is_hit = c > 0 && es0 >= 0, is_miss = c > 0 && es0 < 0;
    const unsigned bh = __ballot_sync(0xffffffffu, is_hit), bm = __ballot_sync(0xffffffffu, is_miss);
    if (lane == 0) {
        warp_hits[wid] = __popc(bh);
        warp_misses[wid] = __popc(bm);
    }
    const int any_negative = __syncthreads_or(c < 0);
    const int uniq = __syncthreads_count(c > 0);
    int nh_all = 0, nm_all = 0, oh = 0, om = 0;
    for (int i = 0; i < kPlanThreads / 32; ++i) {
        if (i == wid) {
            oh = nh_all;
            om = nm_all;
        }
        nh_all += warp_hits[i];
        nm_all += warp_misses[i];
    }
    const unsigned below = (1u << lane) - 1u;
    if (is_hit) hit_e[oh + __popc(bh & below)] = t;
    if (is_miss) miss_e[om + __popc(bm & below)] = t;
    __syncthreads();
    if (t == 0) {
        uint64_t* ctr = reinterpret_cast<uint64_t*>(rec + dr.ctr);  // moe_counters, field order
        int64_t* g_clk = reinterpret_cast<int64_t*>(rec + dr.clk);
        int32_t* g_n = reinterpret_cast<int32_t*>(rec + dr.n_loads);
        int32_t* g_copy = reinterpret_cast<int32_t*>(rec + dr.n_copy);
        int ok = 0;
        if (!any_negative && uniq <= S) {
            PlanView v{se, es, st, uses, seg, *g_clk, S, E, policy};
            const int nh = nh_all;
            const int n = plan_event_lists(v, cnt, nullptr, hit_e, nh_all, miss_e, nm_all, loads);
            if (n >= 0) {  // always, without a keep set: U fits in the slots
                ok = 1;
                *g_clk = v.clk;
                int32_t* le = reinterpret_cast<int32_t*>(rec + dr.le);
                int32_t* ls = reinterpret_cast<int32_t*>(rec + dr.ls);
                uint64_t ev = 0;
                for (int i = 0; i < n; ++i) {
                    le[i] = loads[i].e;
                    ls[i] = loads[i].slot;
                    ev += loads[i].victim >= 0;
                }
                ctr[0] += uint64_t(nh);                     // hits
                ctr[1] += uint64_t(n);                      // misses
                ctr[2] += ev;                               // evictions
                ctr[3] += uint64_t(n) * bytes_per_load;     // h2d_bytes
                ctr[5] += 1;                                // events
                for (int i = 0; i < nh; ++i)
                    if (g_fresh[hit_e[i]]) {
                        ctr[7] += 1;                        // prefetch_hits
                        g_fresh[hit_e[i]] = 0;
                    }
                for (int i = 0; i < n; ++i) {
                    g_fresh[loads[i].e] = 0;
                    if (loads[i].victim >= 0) g_fresh[loads[i].victim] = 0;
                }
                *g_n = n;
                *g_copy = n;
            }
        }
        if (!ok) {
            // nothing changes: no copies, the slot map stays the current one
            // (routed experts that are absent stay -1), and the last loads
            // stay those of the last successful event
            *reinterpret_cast<int32_t*>(rec + dr.status) |= any_negative ? 1 : 2;
            *g_copy = 0;
        }
        ok_s = ok;
    }
    __syncthreads();
    if (ok_s) {
        if (t < S) {
            g_se[t] = se[t];
            g_st[t] = st[t];
            g_uses[t] = uses[t];
            g_seg[t] = seg[t];
        }
        if (t < E) {
            g_es[t] = es[t];
            g_freq[t] += cnt[t] > 0;
        }
    }
    if (t < E) {
        slot_of[t] = es[t];
        if (split) {
            // [0, E): the routed experts that were resident (the event's
            // hits), [E, 2E): the ones this event loads; -1 elsewhere.  After
            // an event that changed nothing, routed experts without a slot get
            // slot S in the first map (out of range: a computation over it
            // yields NaN instead of leaving them out).
            if (ok_s) {
                split[t] = (c > 0 && es0 >= 0) ? es[t] : -1;
                split[E + t] = (c > 0 && es0 < 0) ? es[t] : -1;
            } else {
                split[t] = c > 0 ? (es0 >= 0 ? es0 : S) : -1;
                split[E + t] = -1;
            }
        }
    }
}

__global__ void __launch_bounds__(kPlanThreads) pool_plan_kernel(uint8_t* rec, DevRecord dr, int S, int E,
                                                                 int policy, const int32_t* __restrict__ counts,
                                                                 int32_t* __restrict__ slot_of,
                                                                 int32_t* __restrict__ split,
                                                                 unsigned long long bytes_per_load) {
    __shared__ PlanSmem sm;
    // launched with programmatic stream serialisation: the counts and the
    // record are read only after the previous kernel has finished
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int t = threadIdx.x;
    load_slots(sm, rec, dr, S, t, kPlanThreads);
    int c = 0, es0 = -1;
    if (t < E) {
        es0 = reinterpret_cast<const int32_t*>(rec + dr.es)[t];
        sm.es[t] = es0;
        c = counts[t];
        sm.cnt[t] = c;
    }
    plan_block(sm, c, es0, rec, dr, S, E, policy, slot_of, split, bytes_per_load);
}

// Routing (T * k <= 32 assignments, warp 0, the code of the one-warp
// routing kernel) and the event's planning in one launch: the other warps
// load the layer's record while warp 0 ranks the tokens, and the counts
// reach the planner through shared memory.
template <int EPL>
__global__ void __launch_bounds__(kPlanThreads) pool_route_plan_kernel(
    const float* __restrict__ logits, int T, int k, int32_t* __restrict__ ids, float* __restrict__ w,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
    int32_t* __restrict__ inv, uint8_t* rec, DevRecord dr, int S, int E, int policy, int32_t* __restrict__ slot_of,
    int32_t* __restrict__ split, unsigned long long bytes_per_load) {
    __shared__ PlanSmem sm;
    __shared__ int sel_id[32];
    __shared__ float sel_v[32];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int t = threadIdx.x;
    if (t < 32) {
        const int my_id = route_tiny_warp<EPL>(logits, T, E, k, ids, w, counts, offsets, perm, inv, sel_id, sel_v);
        const int A = T * k;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + t;
            int eq = 0;
            for (int b = 0; b < A; ++b) eq += __shfl_sync(0xffffffffu, my_id, b) == e;
            if (e < E) sm.cnt[e] = eq;
        }
    } else {
        load_slots(sm, rec, dr, S, t - 32, kPlanThreads - 32);
        const int32_t* g_es = reinterpret_cast<const int32_t*>(rec + dr.es);
        for (int i = t - 32; i < E; i += kPlanThreads - 32) sm.es[i] = g_es[i];
    }
    __syncthreads();
    const int c = t < E ? sm.cnt[t] : 0;
    const int es0 = t < E ? sm.es[t] : -1;
    plan_block(sm, c, es0, rec, dr, S, E, policy, slot_of, split, bytes_per_load);
}

__global__ void __launch_bounds__(kGatherThreads) pool_gather_kernel(const uint8_t* rec, DevRecord dr,
                                                                     const uint8_t* host_layer, uint8_t* slots_layer,
                                                                     unsigned long long eb, unsigned long long len0,
                                                                     unsigned long long off1, unsigned long long len1) {
    // launched with programmatic stream serialisation: the planned loads are
    // read after the previous kernel in the stream has finished, and the
    // next one (the loaded experts' FFN, when the caller puts it behind the
    // copy) may launch and wait for this grid
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int n = *reinterpret_cast<const int32_t*>(rec + dr.n_copy);
    const int32_t* le = reinterpret_cast<const int32_t*>(rec + dr.le);
    const int32_t* ls = reinterpret_cast<const int32_t*>(rec + dr.ls);
    const unsigned long long c0 = (len0 + kChunk - 1) / kChunk, c1 = (len1 + kChunk - 1) / kChunk;
    const unsigned long long cpl = c0 + c1;
    for (unsigned long long c = blockIdx.x; c < (unsigned long long)n * cpl; c += gridDim.x) {
        const unsigned long long i = c / cpl;
        unsigned long long r = c - i * cpl, base, len;
        if (r < c0) {
            base = r * kChunk;
            len = min(kChunk, len0 - base);
        } else {
            r -= c0;
            base = off1 + r * kChunk;
            len = min(kChunk, len1 - r * kChunk);
        }
        const uint4* src = reinterpret_cast<const uint4*>(host_layer + (unsigned long long)le[i] * eb + base);
        uint4* dst = reinterpret_cast<uint4*>(slots_layer + (unsigned long long)ls[i] * eb + base);
        const unsigned long long n16 = len / 16;
        for (unsigned long long j = threadIdx.x; j < n16; j += (unsigned long long)kGatherUnroll * kGatherThreads) {
            uint4 v[kGatherUnroll];
#pragma unroll
            for (int u = 0; u < kGatherUnroll; ++u) {
                const unsigned long long jj = j + (unsigned long long)u * kGatherThreads;
                if (jj < n16) v[u] = __ldg(src + jj);
            }
#pragma unroll
            for (int u = 0; u < kGatherUnroll; ++u) {
                const unsigned long long jj = j + (unsigned long long)u * kGatherThreads;
                if (jj < n16) dst[jj] = v[u];
            }
        }
    }
}

}  // namespace

int launch_pool_plan(uint8_t* rec, int S, int E, int policy, const int32_t* counts, int32_t* slot_of,
                     int32_t* split, uint64_t bytes_per_load, cudaStream_t s) {
    if (E > MOE_MAX_EXPERTS || S > E) return MOE_ERR_INVALID;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kPlanThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, pool_plan_kernel, rec, dev_record(S, E), S, E, policy, counts, slot_of,
                                    split, (unsigned long long)bytes_per_load));
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

namespace {
template <int EPL>
int launch_route_plan_epl(const float* logits, int T, int k, int32_t* ids, float* w, int32_t* counts,
                          int32_t* offsets, int32_t* perm, int32_t* inv, uint8_t* rec, int S, int E, int policy,
                          int32_t* slot_of, int32_t* split, uint64_t bytes_per_load, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kPlanThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, pool_route_plan_kernel<EPL>, logits, T, k, ids, w, counts, offsets, perm,
                                    inv, rec, dev_record(S, E), S, E, policy, slot_of, split,
                                    (unsigned long long)bytes_per_load));
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}
}  // namespace

int launch_pool_route_plan(const float* logits, int T, int k, int32_t* ids, float* w, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv, uint8_t* rec, int S, int E, int policy,
                           int32_t* slot_of, int32_t* split, uint64_t bytes_per_load, cudaStream_t s) {
    if (E > MOE_MAX_EXPERTS || S > E || T < 1 || k < 1 || k > E || T * k > 32) return MOE_ERR_INVALID;
    if (E <= 32)
        return launch_route_plan_epl<1>(logits, T, k, ids, w, counts, offsets, perm, inv, rec, S, E, policy, slot_of,
                                        split, bytes_per_load, s);
    if (E <= 64)
        return launch_route_plan_epl<2>(logits, T, k, ids, w, counts, offsets, perm, inv, rec, S, E, policy, slot_of,
                                        split, bytes_per_load, s);
    if (E <= 128)
        return launch_route_plan_epl<4>(logits, T, k, ids, w, counts, offsets, perm, inv, rec, S, E, policy, slot_of,
                                        split, bytes_per_load, s);
    return launch_route_plan_epl<8>(logits, T, k, ids, w, counts, offsets, perm, inv, rec, S, E, policy, slot_of,
                                    split, bytes_per_load, s);
}

int launch_pool_gather(const uint8_t* rec, int S, int E, const uint8_t* host_layer, uint8_t* slots_layer,
                       size_t eb, size_t len0, size_t off1, size_t len1, cudaStream_t s) {
    if ((eb | len0 | off1 | len1) & 15) return MOE_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(host_layer) | reinterpret_cast<uintptr_t>(slots_layer)) & 15)
        return MOE_ERR_INVALID;
    DeviceInfo di;
    int rc = current_device_info(&di);
    if (rc != MOE_OK) return rc;
    if (di.device < 0 || di.device >= 64) return MOE_ERR_UNSUPPORTED;
    static DeviceOnce carveout_set;
    if (!carveout_set.done(di.device)) {
        // An SM configured with a small shared-memory carve-out (what a
        // kernel without shared memory would get) cannot take a decode FFN
        // CTA (about 210 KB) until it drains: ask for the largest carve-out
        // so the FFN of a layer's hits runs beside the copy.
        MOE_CUDA_TRY(cudaFuncSetAttribute(pool_gather_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                          int(cudaSharedmemCarveoutMaxShared)));
        carveout_set.mark(di.device);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(di.sms));
    cfg.blockDim = dim3(unsigned(kGatherThreads));
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, pool_gather_kernel, rec, dev_record(S, E), host_layer, slots_layer,
                                    (unsigned long long)eb, (unsigned long long)len0, (unsigned long long)off1,
                                    (unsigned long long)len1));
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

}  // namespace moe
