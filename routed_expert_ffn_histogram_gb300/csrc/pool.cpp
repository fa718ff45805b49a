// Expert-slot pool: per-layer (expert -> slot) map with policy-driven eviction and
// host-to-device staging of missed experts on a copy stream.
//
// Sources: tinyserve README, "How it works" item 1 (expert weights kept as
// raw quantised bytes in pinned CPU memory), item 3 (cache keyed by
// (layer, expert_id) with a lazily synced GPU slot map) and "Configuration"
// (cache_policy lru); llama.cpp discussion "fixed GPU expert working set with
// Native CPU miss execution", main post (a fixed set of packed experts is
// materialised in a GPU pool at load; routed IDs split into resident hits
// and misses); "Expert Offloading" topic page, replay-semantics study (one
// fused cache event per (layer, step) instead of per-access replay).
//
// Event of one (layer, step): U = routed experts with a nonzero count,
// ascending.  Resident members of U are hits and are touched first, in
// ascending id; then each absent member, ascending, takes the lowest free
// slot or evicts a resident expert that is not in U, chosen by the pool's
// policy (tinyserve README, "Configuration": cache_policy lru, lfru, slru,
// lfu, fifo; "How it works" item 3: frequency-recency eviction).  The
// planning itself (touch, victim choice, load) is pool_plan.h, shared with
// the device planner of pool_dev.cu, which keeps the state in device memory
// and plans each event on the GPU from the device counts (no host round
// trip), copying the misses with the SMs out of the mapped host store.
//
// Prefill through a pool smaller than the routed set (moe_prefill_staged):
// tinyserve README, "How it works" item 6 (batched prefill groups tokens by
// expert and loads each unique expert once).  The unique experts are cut
// into windows of at most S/2; each window is one event as above whose
// victims also exclude the previous window (its GEMMs may still read it);
// copies wait on the device for the GEMMs of the window before that.
//
// Next-layer prefetch (moe_pool_prefetch): tinyserve README, "How it works"
// item 4 (FATE: current-layer activations predict the next layer's experts,
// H2D overlapped with compute).  This path has no router weights, so the
// layer's own routing history ranks the candidates: the most often routed
// non-resident experts, each displacing only an expert routed less often.
// The Expert Offloading topic page (WiSP abstract) reports that speculative
// transfers compete with demand transfers when the link is the bottleneck;
// the same holds on GB300 for single-token decode (an expert copy outlasts
// a layer's FFN), so the call is a building block, off by default.
#include <algorithm>
#include <chrono>
#include <cstdint>
#include <cstring>
#include <new>
#include <thread>
#include <vector>

#include "internal.h"
#include "pool_plan.h"

struct moe_pool {
    moe_pool_desc d;
    moe::Layout L;
    size_t eb = 0;
    std::vector<int32_t> slot_expert;   // [L][S], -1 = free
    std::vector<int32_t> expert_slot;   // [L][E], -1 = absent
    std::vector<int64_t> stamp;         // [L][S] last touch (fifo: load)
    std::vector<int64_t> uses;          // [L][S] touches since load (lfu, lfru)
    std::vector<int8_t> seg;            // [L][S] slru: 0 probation, 1 protected
    std::vector<int64_t> clock;         // [L]
    std::vector<int64_t> freq;          // [L][E] events that routed the expert (prefetch ranking)
    std::vector<uint8_t> fresh;         // [L][E] loaded by a prefetch, not routed since
    std::vector<uint8_t> pending;       // [L] prefetch copies not yet ordered before later work
    std::vector<moe_counters> ctr;      // [L]
    size_t bytes_per_load = 0;          // bytes one miss copies
    std::vector<int32_t> last_e, last_s;  // [L][S]
    std::vector<int> last_n;            // [L]
    int32_t* map_pinned = nullptr;      // [L][E] staging for slot-map uploads
    cudaEvent_t ev_compute = nullptr, ev_copy = nullptr;
    cudaEvent_t ev_win[2] = {nullptr, nullptr};  // staged prefill: window GEMMs finished
    std::vector<cudaEvent_t> ev_pf;     // [L] the layer's last prefetch copies finished
    int inject_fail = 0;
    uint8_t* dev_state = nullptr;       // device-planned staging: the state lives here while attached
    const uint8_t* host_dev = nullptr;  // device address of host_experts (mapped pinned memory)
    cudaEvent_t ev_plan = nullptr;      // device planner done (the copy stream's copies follow it)
    std::vector<cudaEvent_t> ev_gather; // [L] the layer's last copies on the copy stream done
    std::vector<uint8_t> gather_pending;  // [L] copies on the copy stream not yet joined
};

namespace {

constexpr uint32_t kStateMagic = 0x4d4f4551u;  // "MOEQ": with routing frequencies and prefetch flags

// Per-layer policy state, planned on copies and committed on success.
struct LayerState {
    std::vector<int32_t> se, es;  // slot -> expert, expert -> slot
    std::vector<int64_t> st, uses;
    std::vector<int8_t> seg;
    int64_t clk = 0;
    moe::PlanView view(int S, int E, int policy) {
        return moe::PlanView{se.data(), es.data(), st.data(), uses.data(), seg.data(), clk, S, E, policy};
    }
};

// Copy expert e of `layer` from the host store into slot `slot`: the whole
// packed expert, or (MOE_STAGE_DECODE) the gate/up rows and the
// column-blocked down copy, skipping the row-major down matrix.
cudaError_t copy_expert(const moe_pool_t* p, int layer, int e, int slot, cudaMemcpyKind kind, cudaStream_t s,
                        bool sync) {
    const size_t E = size_t(p->d.experts), S = size_t(p->d.slots_per_layer);
    const uint8_t* src = static_cast<const uint8_t*>(p->d.host_experts) + (size_t(layer) * E + e) * p->eb;
    uint8_t* dst = static_cast<uint8_t*>(p->d.dev_slots) + (size_t(layer) * S + slot) * p->eb;
    auto cp = [&](size_t off, size_t n) {
        return sync ? cudaMemcpy(dst + off, src + off, n, kind) : cudaMemcpyAsync(dst + off, src + off, n, kind, s);
    };
    if (p->d.stage_parts != MOE_STAGE_DECODE) return cp(0, p->eb);
    cudaError_t r = cp(0, p->L.d_off);
    if (r == cudaSuccess) r = cp(p->L.dt_off, p->eb - p->L.dt_off);
    return r;
}

int wait_stream(moe_pool_t* p, cudaStream_t s, int timeout_ms) {
    MOE_CUDA_TRY(cudaEventRecord(p->ev_compute, s));
    const auto t0 = std::chrono::steady_clock::now();
    const auto limit = std::chrono::milliseconds(timeout_ms > 0 ? timeout_ms : 10000);
    for (;;) {
        cudaError_t q = cudaEventQuery(p->ev_compute);
        if (q == cudaSuccess) return MOE_OK;
        if (q != cudaErrorNotReady) return moe::cuda_fail(q);
        if (std::chrono::steady_clock::now() - t0 > limit) return MOE_ERR_TIMEOUT;
        std::this_thread::yield();
    }
}

}  // namespace

extern "C" int moe_pool_create(const moe_pool_desc* desc, moe_pool_t** out) {
    if (!desc || !out) return MOE_ERR_INVALID;
    *out = nullptr;
    const moe_pool_desc& d = *desc;
    moe::Layout L;
    if (d.layers < 1 || d.experts < 1 || d.experts > MOE_MAX_EXPERTS || d.slots_per_layer < 1 ||
        d.slots_per_layer > d.experts || !moe::Layout::make(d.hidden, d.inter, &L))
        return MOE_ERR_INVALID;
    if (!d.dry_run && (!d.host_experts || !d.dev_slots)) return MOE_ERR_INVALID;
    if (d.policy < MOE_POLICY_LRU || d.policy > MOE_POLICY_SLRU) return MOE_ERR_INVALID;
    if (d.stage_parts != MOE_STAGE_WHOLE && d.stage_parts != MOE_STAGE_DECODE) return MOE_ERR_INVALID;
    moe_pool_t* p = new (std::nothrow) moe_pool;
    if (!p) return MOE_ERR_INVALID;
    p->d = d;
    p->L = L;
    p->eb = L.expert_bytes;
    p->bytes_per_load = d.stage_parts == MOE_STAGE_DECODE ? L.d_off + (L.expert_bytes - L.dt_off) : L.expert_bytes;
    const size_t nl = size_t(d.layers), S = size_t(d.slots_per_layer), E = size_t(d.experts);
    p->slot_expert.assign(nl * S, -1);
    p->expert_slot.assign(nl * E, -1);
    p->stamp.assign(nl * S, 0);
    p->uses.assign(nl * S, 0);
    p->seg.assign(nl * S, 0);
    p->clock.assign(nl, 0);
    p->freq.assign(nl * E, 0);
    p->fresh.assign(nl * E, 0);
    p->pending.assign(nl, 0);
    p->ctr.assign(nl, moe_counters{});
    p->last_e.assign(nl * S, -1);
    p->last_s.assign(nl * S, -1);
    p->last_n.assign(nl, 0);
    if (!d.dry_run) {
        cudaError_t e = cudaHostAlloc(reinterpret_cast<void**>(&p->map_pinned), nl * E * sizeof(int32_t),
                                      cudaHostAllocDefault);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_compute, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_copy, cudaEventDisableTiming);
        for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&p->ev_win[i], cudaEventDisableTiming);
        p->ev_pf.assign(nl, nullptr);
        for (size_t l = 0; l < nl && e == cudaSuccess; ++l) e = cudaEventCreateWithFlags(&p->ev_pf[l], cudaEventDisableTiming);
        if (e != cudaSuccess) {
            moe_pool_destroy(p);
            return moe::cuda_fail(e);
        }
    }
    if (d.preload) {
        for (size_t l = 0; l < nl; ++l)
            for (size_t s = 0; s < S; ++s) {
                p->slot_expert[l * S + s] = int32_t(s);
                p->expert_slot[l * E + s] = int32_t(s);
                p->uses[l * S + s] = 1;
                if (!d.dry_run) {
                    cudaError_t e = copy_expert(p, int(l), int(s), int(s), cudaMemcpyHostToDevice, nullptr, true);
                    if (e != cudaSuccess) {
                        moe_pool_destroy(p);
                        return moe::cuda_fail(e);
                    }
                }
            }
    }
    *out = p;
    return MOE_OK;
}

namespace {

// One staging event of `layer` over U = {e : counts[e] > 0}: plan hits,
// misses and victims on a copy of the layer's state (victims never in U,
// nor in `keep`), enqueue the miss copies on `ps`, and commit.  If a copy
// cannot be enqueued, only the copies already enqueued are applied.
// *copied tells whether any copy was enqueued.
int stage_event(moe_pool_t* p, int layer, const int32_t* counts, const uint8_t* keep, cudaStream_t ps,
                bool* copied) {
    const int S = p->d.slots_per_layer, E = p->d.experts;
    *copied = false;
    int32_t* se = &p->slot_expert[size_t(layer) * S];
    int32_t* es = &p->expert_slot[size_t(layer) * E];
    int64_t* st = &p->stamp[size_t(layer) * S];
    int64_t* us = &p->uses[size_t(layer) * S];
    int8_t* sg = &p->seg[size_t(layer) * S];
    int64_t& clk = p->clock[layer];
    moe_counters& c = p->ctr[layer];
    const int policy = p->d.policy;

    int uniq = 0;
    for (int e = 0; e < E; ++e) {
        if (counts[e] < 0) return MOE_ERR_INVALID;
        uniq += counts[e] > 0;
    }
    if (uniq > S) return MOE_ERR_CAPACITY;

    // Plan the event on copies of the layer's state; commit on success.
    LayerState ls;
    ls.se.assign(se, se + S);
    ls.es.assign(es, es + E);
    ls.st.assign(st, st + S);
    ls.uses.assign(us, us + S);
    ls.seg.assign(sg, sg + S);
    ls.clk = clk;
    std::vector<moe::PlanLoad> plan(size_t(S) + 1);
    std::vector<int32_t> hit_e(size_t(S) + 1), miss_e(size_t(S) + 1);
    int n_hits = 0;
    moe::PlanView v = ls.view(S, E, policy);
    const int n_loads = moe::plan_event(v, counts, keep, plan.data(), hit_e.data(), &n_hits, miss_e.data());
    if (n_loads < 0) return MOE_ERR_CAPACITY;  // U and keep together fill the slots
    ls.clk = v.clk;
    plan.resize(size_t(n_loads));
    hit_e.resize(size_t(n_hits));
    const uint64_t hits = uint64_t(n_hits);

    size_t done = 0;
    int fail = MOE_OK;
    for (const moe::PlanLoad& q : plan) {
        if (p->inject_fail > 0) {
            --p->inject_fail;
            fail = moe::cuda_fail(cudaErrorUnknown);
            break;
        }
        if (!p->d.dry_run) {
            cudaError_t e = copy_expert(p, layer, q.e, q.slot, cudaMemcpyHostToDevice, ps, false);
            if (e != cudaSuccess) {
                fail = moe::cuda_fail(e);
                break;
            }
        }
        ++done;
    }
    *copied = done > 0 && !p->d.dry_run;

    int64_t* fq = &p->freq[size_t(layer) * E];
    uint8_t* fr = &p->fresh[size_t(layer) * E];
    if (fail != MOE_OK) {
        // Keep only the loads that were enqueued (their slots now hold the new
        // experts); everything else of the event is not applied.
        for (size_t i = 0; i < done; ++i) {
            const moe::PlanLoad& q = plan[i];
            fr[q.e] = 0;
            if (q.victim >= 0) {
                es[q.victim] = -1;
                fr[q.victim] = 0;
                ++c.evictions;
            }
            se[q.slot] = q.e;
            es[q.e] = q.slot;
            st[q.slot] = ++clk;
            us[q.slot] = 1;
            sg[q.slot] = 0;
            ++c.misses;
            c.h2d_bytes += p->bytes_per_load;
        }
        ++c.errors;
        p->last_n[layer] = 0;
    } else {
        std::memcpy(se, ls.se.data(), sizeof(int32_t) * S);
        std::memcpy(es, ls.es.data(), sizeof(int32_t) * E);
        std::memcpy(st, ls.st.data(), sizeof(int64_t) * S);
        std::memcpy(us, ls.uses.data(), sizeof(int64_t) * S);
        std::memcpy(sg, ls.seg.data(), sizeof(int8_t) * S);
        clk = ls.clk;
        c.hits += hits;
        c.misses += plan.size();
        for (const moe::PlanLoad& q : plan) c.evictions += q.victim >= 0;
        for (int e : hit_e)
            if (fr[e]) {
                ++c.prefetch_hits;
                fr[e] = 0;
            }
        for (const moe::PlanLoad& q : plan) {
            fr[q.e] = 0;
            if (q.victim >= 0) fr[q.victim] = 0;
        }
        for (int e = 0; e < E; ++e) fq[e] += counts[e] > 0;
        c.h2d_bytes += plan.size() * p->bytes_per_load;
        ++c.events;
        p->last_n[layer] = int(plan.size());
        for (size_t i = 0; i < plan.size(); ++i) {
            p->last_e[size_t(layer) * S + i] = plan[i].e;
            p->last_s[size_t(layer) * S + i] = plan[i].slot;
        }
    }
    return fail;
}

// A prefetch of `layer` may still be copying into its slots: order the
// copy stream (before it overwrites any slot) and the compute stream
// (before it reads a prefetched expert) after those copies.
int order_after_prefetch(moe_pool_t* p, int layer, cudaStream_t cs, cudaStream_t ps, bool both) {
    if (p->d.dry_run || !p->pending[layer]) return MOE_OK;
    MOE_CUDA_TRY(cudaStreamWaitEvent(ps, p->ev_pf[layer], 0));
    if (both && cs != ps) MOE_CUDA_TRY(cudaStreamWaitEvent(cs, p->ev_pf[layer], 0));
    p->pending[layer] = 0;
    return MOE_OK;
}

}  // namespace

extern "C" int moe_pool_stage(moe_pool_t* p, int layer, const int32_t* counts_host, int32_t* slot_of_dev,
                              moe_stream_t compute, moe_stream_t copy, int timeout_ms) {
    if (!p || !counts_host || layer < 0 || layer >= p->d.layers) return MOE_ERR_INVALID;
    if (p->dev_state) return MOE_ERR_STATE;
    const int E = p->d.experts;
    cudaStream_t cs = static_cast<cudaStream_t>(compute), ps = static_cast<cudaStream_t>(copy);
    if (!p->d.dry_run) {
        int rc = wait_stream(p, cs, timeout_ms);
        if (rc == MOE_OK) rc = order_after_prefetch(p, layer, cs, ps, true);
        if (rc != MOE_OK) return rc;
    }
    bool copied = false;
    const int fail = stage_event(p, layer, counts_host, nullptr, ps, &copied);
    if (fail == MOE_ERR_INVALID || fail == MOE_ERR_CAPACITY) return fail;
    if (!p->d.dry_run) {
        if (copied && ps != cs) {
            MOE_CUDA_TRY(cudaEventRecord(p->ev_copy, ps));
            MOE_CUDA_TRY(cudaStreamWaitEvent(cs, p->ev_copy, 0));
        }
        if (slot_of_dev) {
            const int32_t* es = &p->expert_slot[size_t(layer) * E];
            int32_t* stage = p->map_pinned + size_t(layer) * E;
            std::memcpy(stage, es, sizeof(int32_t) * E);
            MOE_CUDA_TRY(cudaMemcpyAsync(slot_of_dev, stage, sizeof(int32_t) * E, cudaMemcpyHostToDevice, cs));
        }
    }
    return fail;
}

extern "C" int moe_prefill_staged(moe_pool_t* p, int layer, const void* x_bf16, int T, int k, const int32_t* ids,
                                  const float* w, const int32_t* offsets, const int32_t* perm, const int32_t* inv,
                                  const int32_t* counts_host, int window, void* workspace, size_t ws_bytes,
                                  float* out, moe_stream_t compute, moe_stream_t copy, int timeout_ms) {
    if (!p || !counts_host || layer < 0 || layer >= p->d.layers || T < 0 || k < 1 || k > p->d.experts ||
        k > MOE_MAX_TOPK)
        return MOE_ERR_INVALID;
    if (p->dev_state) return MOE_ERR_STATE;
    const int S = p->d.slots_per_layer, E = p->d.experts;
    if (window < 1 || 2 * window > S) return MOE_ERR_INVALID;
    if (p->d.stage_parts == MOE_STAGE_DECODE) return MOE_ERR_UNSUPPORTED;  // no row-major down matrix
    const bool dry = p->d.dry_run;
    if (!dry && T > 0) {
        if (!x_bf16 || !ids || !w || !offsets || !perm || !inv || !out || !workspace) return MOE_ERR_INVALID;
        if (reinterpret_cast<uintptr_t>(x_bf16) % 16 || reinterpret_cast<uintptr_t>(out) % 16 ||
            reinterpret_cast<uintptr_t>(workspace) % 256)
            return MOE_ERR_INVALID;
        if (ws_bytes < moe::prefill_workspace_bytes(T, k, p->d.hidden, p->d.inter)) return MOE_ERR_INVALID;
    }
    if (T == 0) return MOE_OK;
    cudaStream_t cs = static_cast<cudaStream_t>(compute), ps = static_cast<cudaStream_t>(copy);
    if (!dry) {
        // routing finished (counts_host is final) and no earlier work still
        // reads a slot this call may overwrite
        int rc = wait_stream(p, cs, timeout_ms);
        if (rc == MOE_OK) rc = order_after_prefetch(p, layer, cs, ps, true);
        if (rc != MOE_OK) return rc;
    }
    int64_t total = 0;
    for (int e = 0; e < E; ++e) {
        if (counts_host[e] < 0) return MOE_ERR_INVALID;
        total += counts_host[e];
    }
    if (total != int64_t(T) * k) return MOE_ERR_INVALID;

    // windows: the unique routed experts, ascending, `window` at a time
    std::vector<int> uniq;
    for (int e = 0; e < E; ++e)
        if (counts_host[e] > 0) uniq.push_back(e);
    const int nu = int(uniq.size()), n_win = (nu + window - 1) / window;

    moe::FfnArgs a;
    a.slots = static_cast<const uint8_t*>(p->d.dev_slots) + size_t(layer) * S * p->eb;
    a.expert_bytes = p->eb;
    a.S = S;
    a.E = E;
    a.L = &p->L;
    a.x = static_cast<const uint16_t*>(x_bf16);
    a.T = T;
    a.k = k;
    a.ids = ids;
    a.w = w;
    a.offsets = offsets;
    a.perm = perm;
    a.inv = inv;
    a.slot_of = nullptr;
    a.out = out;
    if (!dry) {
        const int rc = moe::launch_prefill_prepare(a, workspace, ws_bytes, cs);
        if (rc != MOE_OK) return rc;
    }
    const int32_t* es = &p->expert_slot[size_t(layer) * E];
    std::vector<int32_t> cw(E);
    std::vector<uint8_t> keep(E);
    std::vector<int32_t> tab;
    int prev_lo = 0, prev_hi = 0;
    for (int wi = 0; wi < n_win; ++wi) {
        const int lo = wi * window, hi = std::min(nu, lo + window);
        std::fill(cw.begin(), cw.end(), 0);
        std::fill(keep.begin(), keep.end(), uint8_t(0));
        for (int i = lo; i < hi; ++i) cw[uniq[i]] = counts_host[uniq[i]];
        // the previous window's GEMMs may still be running: its slots stay
        for (int i = prev_lo; i < prev_hi; ++i) keep[uniq[i]] = 1;
        // victims can only be slots last read by window wi - 2 or earlier
        if (!dry && wi >= 2 && ps != cs) MOE_CUDA_TRY(cudaStreamWaitEvent(ps, p->ev_win[wi & 1], 0));
        bool copied = false;
        const int rc = stage_event(p, layer, cw.data(), keep.data(), ps, &copied);
        if (rc != MOE_OK) return rc;
        if (!dry) {
            if (copied && ps != cs) {
                MOE_CUDA_TRY(cudaEventRecord(p->ev_copy, ps));
                MOE_CUDA_TRY(cudaStreamWaitEvent(cs, p->ev_copy, 0));
            }
            const int e0 = uniq[lo], e1 = uniq[hi - 1] + 1;
            tab.assign(size_t(e1 - e0), -1);
            int rows = 0;
            for (int e = e0; e < e1; ++e)
                if (cw[e] > 0) {
                    tab[e - e0] = es[e];
                    rows += cw[e];
                }
            const int r2 = moe::launch_prefill_experts(a, workspace, e0, e1, tab.data(), rows / 128 + (hi - lo) + 1, cs);
            if (r2 != MOE_OK) return r2;
            MOE_CUDA_TRY(cudaEventRecord(p->ev_win[wi & 1], cs));
        }
        prev_lo = lo;
        prev_hi = hi;
    }
    return MOE_OK;
}

extern "C" int moe_pool_prefetch(moe_pool_t* p, int layer, int max_loads, moe_stream_t compute, moe_stream_t copy,
                                 int* loaded) {
    if (loaded) *loaded = 0;
    if (!p || layer < 0 || layer >= p->d.layers || max_loads < 0) return MOE_ERR_INVALID;
    if (p->dev_state) return MOE_ERR_STATE;
    const int S = p->d.slots_per_layer, E = p->d.experts;
    const bool dry = p->d.dry_run;
    cudaStream_t cs = static_cast<cudaStream_t>(compute), ps = static_cast<cudaStream_t>(copy);
    if (!dry) {
        int rc = order_after_prefetch(p, layer, cs, ps, false);
        if (rc != MOE_OK) return rc;
        // the slots may still be read by work enqueued so far on `compute`
        if (ps != cs) {
            MOE_CUDA_TRY(cudaEventRecord(p->ev_compute, cs));
            MOE_CUDA_TRY(cudaStreamWaitEvent(ps, p->ev_compute, 0));
        }
    }
    int32_t* se = &p->slot_expert[size_t(layer) * S];
    int32_t* es = &p->expert_slot[size_t(layer) * E];
    int64_t* fq = &p->freq[size_t(layer) * E];
    uint8_t* fr = &p->fresh[size_t(layer) * E];
    moe_counters& c = p->ctr[layer];
    std::vector<int> cand;
    for (int e = 0; e < E; ++e)
        if (es[e] < 0 && fq[e] > 0) cand.push_back(e);
    std::stable_sort(cand.begin(), cand.end(), [&](int a, int b) { return fq[a] > fq[b]; });
    std::vector<uint8_t> mine(size_t(E), 0);  // loaded by this call: never victims
    int n = 0;
    for (int e : cand) {
        if (n >= max_loads) break;
        // plan on a copy of the layer's state, commit after the copy is enqueued
        LayerState ls;
        ls.se.assign(se, se + S);
        ls.es.assign(es, es + E);
        ls.st.assign(&p->stamp[size_t(layer) * S], &p->stamp[size_t(layer) * S] + S);
        ls.uses.assign(&p->uses[size_t(layer) * S], &p->uses[size_t(layer) * S] + S);
        ls.seg.assign(&p->seg[size_t(layer) * S], &p->seg[size_t(layer) * S] + S);
        ls.clk = p->clock[layer];
        int s = -1;
        for (int i = 0; i < S; ++i)
            if (ls.se[i] < 0) { s = i; break; }
        int victim = -1;
        if (s < 0) {
            const moe::PlanView v = ls.view(S, E, p->d.policy);
            s = moe::plan_victim(v, nullptr, mine.data());
            if (s < 0) break;
            victim = ls.se[s];
            if (fq[victim] >= fq[e]) break;  // only displace experts routed less often
        }
        if (p->inject_fail > 0) {
            --p->inject_fail;
            ++c.errors;
            return moe::cuda_fail(cudaErrorUnknown);
        }
        if (!dry) {
            const cudaError_t r = copy_expert(p, layer, e, s, cudaMemcpyHostToDevice, ps, false);
            if (r != cudaSuccess) {
                ++c.errors;
                if (n > 0) {
                    MOE_CUDA_TRY(cudaEventRecord(p->ev_pf[layer], ps));
                    p->pending[layer] = 1;
                }
                return moe::cuda_fail(r);
            }
        }
        if (victim >= 0) {
            es[victim] = -1;
            fr[victim] = 0;
            ++c.evictions;
        }
        se[s] = e;
        es[e] = s;
        p->stamp[size_t(layer) * S + s] = ++p->clock[layer];
        p->uses[size_t(layer) * S + s] = 1;
        p->seg[size_t(layer) * S + s] = 0;
        fr[e] = 1;
        mine[e] = 1;
        ++c.prefetches;
        c.h2d_bytes += p->bytes_per_load;
        ++n;
    }
    if (!dry && n > 0) {
        MOE_CUDA_TRY(cudaEventRecord(p->ev_pf[layer], ps));
        p->pending[layer] = 1;
    }
    if (loaded) *loaded = n;
    return MOE_OK;
}

extern "C" int moe_pool_counters(const moe_pool_t* p, int layer, moe_counters* out) {
    if (!p || !out || layer < -1 || layer >= p->d.layers) return MOE_ERR_INVALID;
    if (p->dev_state) return MOE_ERR_STATE;
    if (layer >= 0) {
        *out = p->ctr[layer];
        return MOE_OK;
    }
    moe_counters s{};
    for (const moe_counters& c : p->ctr) {
        s.hits += c.hits;
        s.misses += c.misses;
        s.evictions += c.evictions;
        s.h2d_bytes += c.h2d_bytes;
        s.errors += c.errors;
        s.events += c.events;
        s.prefetches += c.prefetches;
        s.prefetch_hits += c.prefetch_hits;
    }
    *out = s;
    return MOE_OK;
}

extern "C" int moe_pool_slot_map(const moe_pool_t* p, int layer, int32_t* out) {
    if (!p || !out || layer < 0 || layer >= p->d.layers) return MOE_ERR_INVALID;
    if (p->dev_state) return MOE_ERR_STATE;
    std::memcpy(out, &p->expert_slot[size_t(layer) * p->d.experts], sizeof(int32_t) * p->d.experts);
    return MOE_OK;
}

extern "C" int moe_pool_last_loads(const moe_pool_t* p, int layer, int32_t* le, int32_t* ls, int* n) {
    if (!p || !le || !ls || !n || layer < 0 || layer >= p->d.layers) return MOE_ERR_INVALID;
    if (p->dev_state) return MOE_ERR_STATE;
    const int S = p->d.slots_per_layer;
    *n = p->last_n[layer];
    for (int i = 0; i < *n; ++i) {
        le[i] = p->last_e[size_t(layer) * S + i];
        ls[i] = p->last_s[size_t(layer) * S + i];
    }
    return MOE_OK;
}

namespace {
struct StateHeader {
    uint32_t magic;
    int32_t layers, experts, slots, hidden, inter, policy;
};
size_t state_bytes(const moe_pool_t* p) {
    return sizeof(StateHeader) + p->slot_expert.size() * 4 + p->expert_slot.size() * 4 +
           p->stamp.size() * 8 + p->uses.size() * 8 + p->seg.size() + p->clock.size() * 8 +
           p->ctr.size() * sizeof(moe_counters) + p->freq.size() * 8 + p->fresh.size();
}
}  // namespace

extern "C" int moe_pool_state_bytes(const moe_pool_t* p, size_t* out) {
    if (!p || !out) return MOE_ERR_INVALID;
    *out = state_bytes(p);
    return MOE_OK;
}

extern "C" int moe_pool_save(const moe_pool_t* p, void* buf, size_t bytes) {
    if (!p || !buf || bytes < state_bytes(p)) return MOE_ERR_INVALID;
    if (p->dev_state) return MOE_ERR_STATE;
    uint8_t* o = static_cast<uint8_t*>(buf);
    StateHeader h{kStateMagic, p->d.layers, p->d.experts, p->d.slots_per_layer, p->d.hidden, p->d.inter,
                  p->d.policy};
    std::memcpy(o, &h, sizeof h);
    o += sizeof h;
    auto put = [&o](const void* src, size_t n) { std::memcpy(o, src, n); o += n; };
    put(p->slot_expert.data(), p->slot_expert.size() * 4);
    put(p->expert_slot.data(), p->expert_slot.size() * 4);
    put(p->stamp.data(), p->stamp.size() * 8);
    put(p->uses.data(), p->uses.size() * 8);
    put(p->seg.data(), p->seg.size());
    put(p->clock.data(), p->clock.size() * 8);
    put(p->ctr.data(), p->ctr.size() * sizeof(moe_counters));
    put(p->freq.data(), p->freq.size() * 8);
    put(p->fresh.data(), p->fresh.size());
    return MOE_OK;
}

extern "C" int moe_pool_load(moe_pool_t* p, const void* buf, size_t bytes) {
    if (!p || !buf || bytes < state_bytes(p)) return MOE_ERR_INVALID;
    if (p->dev_state) return MOE_ERR_STATE;
    const uint8_t* i = static_cast<const uint8_t*>(buf);
    StateHeader h;
    std::memcpy(&h, i, sizeof h);
    if (h.magic != kStateMagic || h.layers != p->d.layers || h.experts != p->d.experts ||
        h.slots != p->d.slots_per_layer || h.hidden != p->d.hidden || h.inter != p->d.inter ||
        h.policy != p->d.policy)
        return MOE_ERR_STATE;
    i += sizeof h;
    // validate before committing: every map entry in range and consistent
    const size_t S = size_t(h.slots), E = size_t(h.experts);
    std::vector<int32_t> se(p->slot_expert.size()), es(p->expert_slot.size());
    std::memcpy(se.data(), i, se.size() * 4);
    std::memcpy(es.data(), i + se.size() * 4, es.size() * 4);
    for (size_t l = 0; l < size_t(h.layers); ++l) {
        for (size_t s = 0; s < S; ++s) {
            const int32_t e = se[l * S + s];
            if (e < -1 || e >= int32_t(E) || (e >= 0 && es[l * E + e] != int32_t(s))) return MOE_ERR_STATE;
        }
        for (size_t e = 0; e < E; ++e) {
            const int32_t s = es[l * E + e];
            if (s < -1 || s >= int32_t(S) || (s >= 0 && se[l * S + s] != int32_t(e))) return MOE_ERR_STATE;
        }
    }
    auto get = [&i](void* dst, size_t n) { std::memcpy(dst, i, n); i += n; };
    get(p->slot_expert.data(), p->slot_expert.size() * 4);
    get(p->expert_slot.data(), p->expert_slot.size() * 4);
    get(p->stamp.data(), p->stamp.size() * 8);
    get(p->uses.data(), p->uses.size() * 8);
    get(p->seg.data(), p->seg.size());
    get(p->clock.data(), p->clock.size() * 8);
    get(p->ctr.data(), p->ctr.size() * sizeof(moe_counters));
    get(p->freq.data(), p->freq.size() * 8);
    get(p->fresh.data(), p->fresh.size());
    return MOE_OK;
}

// ---- device-planned staging -------------------------------------------------

namespace {
// Host state of every layer <-> the device records (pool_plan.h, dev_record).
void pack_device_state(const moe_pool_t* p, uint8_t* img) {
    const int S = p->d.slots_per_layer, E = p->d.experts;
    const moe::DevRecord dr = moe::dev_record(S, E);
    for (int l = 0; l < p->d.layers; ++l) {
        uint8_t* r = img + size_t(l) * dr.bytes;
        std::memset(r, 0, dr.bytes);
        std::memcpy(r + dr.ctr, &p->ctr[l], sizeof(moe_counters));
        std::memcpy(r + dr.clk, &p->clock[l], 8);
        const int32_t n = p->last_n[l];
        std::memcpy(r + dr.n_loads, &n, 4);
        std::memcpy(r + dr.st, &p->stamp[size_t(l) * S], 8 * size_t(S));
        std::memcpy(r + dr.uses, &p->uses[size_t(l) * S], 8 * size_t(S));
        std::memcpy(r + dr.freq, &p->freq[size_t(l) * E], 8 * size_t(E));
        std::memcpy(r + dr.se, &p->slot_expert[size_t(l) * S], 4 * size_t(S));
        std::memcpy(r + dr.es, &p->expert_slot[size_t(l) * E], 4 * size_t(E));
        std::memcpy(r + dr.le, &p->last_e[size_t(l) * S], 4 * size_t(S));
        std::memcpy(r + dr.ls, &p->last_s[size_t(l) * S], 4 * size_t(S));
        std::memcpy(r + dr.seg, &p->seg[size_t(l) * S], size_t(S));
        std::memcpy(r + dr.fresh, &p->fresh[size_t(l) * E], size_t(E));
    }
}

// Returns the union of the records' status bits.
uint32_t unpack_device_state(moe_pool_t* p, const uint8_t* img) {
    const int S = p->d.slots_per_layer, E = p->d.experts;
    const moe::DevRecord dr = moe::dev_record(S, E);
    uint32_t status = 0;
    for (int l = 0; l < p->d.layers; ++l) {
        const uint8_t* r = img + size_t(l) * dr.bytes;
        std::memcpy(&p->ctr[l], r + dr.ctr, sizeof(moe_counters));
        std::memcpy(&p->clock[l], r + dr.clk, 8);
        int32_t n = 0;
        std::memcpy(&n, r + dr.n_loads, 4);
        p->last_n[l] = n;
        uint32_t st = 0;
        std::memcpy(&st, r + dr.status, 4);
        status |= st;
        std::memcpy(&p->stamp[size_t(l) * S], r + dr.st, 8 * size_t(S));
        std::memcpy(&p->uses[size_t(l) * S], r + dr.uses, 8 * size_t(S));
        std::memcpy(&p->freq[size_t(l) * E], r + dr.freq, 8 * size_t(E));
        std::memcpy(&p->slot_expert[size_t(l) * S], r + dr.se, 4 * size_t(S));
        std::memcpy(&p->expert_slot[size_t(l) * E], r + dr.es, 4 * size_t(E));
        std::memcpy(&p->last_e[size_t(l) * S], r + dr.le, 4 * size_t(S));
        std::memcpy(&p->last_s[size_t(l) * S], r + dr.ls, 4 * size_t(S));
        std::memcpy(&p->seg[size_t(l) * S], r + dr.seg, size_t(S));
        std::memcpy(&p->fresh[size_t(l) * E], r + dr.fresh, size_t(E));
    }
    return status;
}

size_t device_state_bytes(const moe_pool_t* p) {
    return size_t(p->d.layers) * moe::dev_record(p->d.slots_per_layer, p->d.experts).bytes;
}
}  // namespace

extern "C" int moe_pool_device_state_bytes(const moe_pool_t* p, size_t* out) {
    if (!p || !out) return MOE_ERR_INVALID;
    *out = device_state_bytes(p);
    return MOE_OK;
}

extern "C" int moe_pool_device_attach(moe_pool_t* p, void* dev_state, size_t bytes, moe_stream_t stream,
                                      int timeout_ms) {
    if (!p || !dev_state || (reinterpret_cast<uintptr_t>(dev_state) & 15) || bytes < device_state_bytes(p))
        return MOE_ERR_INVALID;
    if (p->d.dry_run || p->dev_state) return MOE_ERR_STATE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void* hd = nullptr;
    if (cudaHostGetDevicePointer(&hd, p->d.host_experts, 0) != cudaSuccess || !hd) {
        (void)cudaGetLastError();
        return MOE_ERR_UNSUPPORTED;  // the host store is not mapped into the device's address space
    }
    // prefetch copies still in flight write slots: the device planner's
    // copies and the FFNs that follow on `stream` come after them
    for (int l = 0; l < p->d.layers; ++l)
        if (p->pending[l]) {
            MOE_CUDA_TRY(cudaStreamWaitEvent(s, p->ev_pf[l], 0));
            p->pending[l] = 0;
        }
    if (!p->ev_plan) {
        MOE_CUDA_TRY(cudaEventCreateWithFlags(&p->ev_plan, cudaEventDisableTiming));
        p->ev_gather.assign(size_t(p->d.layers), nullptr);
        for (auto& ev : p->ev_gather) MOE_CUDA_TRY(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
        p->gather_pending.assign(size_t(p->d.layers), 0);
    }
    std::vector<uint8_t> img(device_state_bytes(p));
    pack_device_state(p, img.data());
    MOE_CUDA_TRY(cudaMemcpyAsync(dev_state, img.data(), img.size(), cudaMemcpyHostToDevice, s));
    const int rc = wait_stream(p, s, timeout_ms);  // img must outlive the copy
    if (rc != MOE_OK) return rc;
    p->dev_state = static_cast<uint8_t*>(dev_state);
    p->host_dev = static_cast<const uint8_t*>(hd);
    return MOE_OK;
}

// The copy stream's copies of `layer` come before whatever is enqueued next
// on `s`.
static int join_gather(moe_pool_t* p, int layer, cudaStream_t s) {
    if (!p->gather_pending.empty() && p->gather_pending[layer]) {
        MOE_CUDA_TRY(cudaStreamWaitEvent(s, p->ev_gather[layer], 0));
        p->gather_pending[layer] = 0;
    }
    return MOE_OK;
}

namespace {
// After the planner: the staged parts of the event's loads copied by the SMs
// out of the mapped store, on `copy` (forked from `compute` after the
// planner) or on `compute`.
int enqueue_gather(moe_pool_t* p, int layer, cudaStream_t s, cudaStream_t cp) {
    const int S = p->d.slots_per_layer, E = p->d.experts;
    uint8_t* rec = p->dev_state + size_t(layer) * moe::dev_record(S, E).bytes;
    const bool fork = cp != nullptr && cp != s;
    if (fork) {
        MOE_CUDA_TRY(cudaEventRecord(p->ev_plan, s));
        MOE_CUDA_TRY(cudaStreamWaitEvent(cp, p->ev_plan, 0));
    }
    const size_t eb = p->eb;
    const bool decode = p->d.stage_parts == MOE_STAGE_DECODE;
    const size_t len0 = decode ? p->L.d_off : eb;
    const size_t off1 = decode ? p->L.dt_off : eb;
    const size_t len1 = decode ? eb - p->L.dt_off : 0;
    const uint8_t* host_layer = p->host_dev + size_t(layer) * size_t(E) * eb;
    uint8_t* slots_layer = static_cast<uint8_t*>(p->d.dev_slots) + size_t(layer) * size_t(S) * eb;
    const int rc = moe::launch_pool_gather(rec, S, E, host_layer, slots_layer, eb, len0, off1, len1, fork ? cp : s);
    if (rc != MOE_OK || !fork) return rc;
    MOE_CUDA_TRY(cudaEventRecord(p->ev_gather[layer], cp));
    p->gather_pending[layer] = 1;
    return MOE_OK;
}
}  // namespace

extern "C" int moe_pool_stage_device(moe_pool_t* p, int layer, const int32_t* counts_dev, int32_t* slot_of_dev,
                                     int32_t* split_dev, moe_stream_t compute, moe_stream_t copy) {
    if (!p || !counts_dev || !slot_of_dev || layer < 0 || layer >= p->d.layers) return MOE_ERR_INVALID;
    if (!p->dev_state) return MOE_ERR_STATE;
    const int S = p->d.slots_per_layer, E = p->d.experts;
    cudaStream_t s = static_cast<cudaStream_t>(compute), cp = static_cast<cudaStream_t>(copy);
    // the planner rewrites the record the layer's previous copies read
    int rc = join_gather(p, layer, s);
    if (rc != MOE_OK) return rc;
    uint8_t* rec = p->dev_state + size_t(layer) * moe::dev_record(S, E).bytes;
    rc = moe::launch_pool_plan(rec, S, E, p->d.policy, counts_dev, slot_of_dev, split_dev, p->bytes_per_load, s);
    if (rc != MOE_OK) return rc;
    return enqueue_gather(p, layer, s, cp);
}

extern "C" int moe_pool_route_stage_device(moe_pool_t* p, int layer, const float* logits, int T, int k,
                                           int32_t* ids, float* w, int32_t* counts, int32_t* offsets, int32_t* perm,
                                           int32_t* inv, int32_t* slot_of_dev, int32_t* split_dev,
                                           moe_stream_t compute, moe_stream_t copy) {
    if (!p || layer < 0 || layer >= p->d.layers) return MOE_ERR_INVALID;
    if (!logits || !ids || !w || !counts || !offsets || !perm || !inv || !slot_of_dev) return MOE_ERR_INVALID;
    const int S = p->d.slots_per_layer, E = p->d.experts;
    if (T < 1 || k < 1 || k > E) return MOE_ERR_INVALID;
    if (T * k > 32) return MOE_ERR_UNSUPPORTED;
    if (!p->dev_state) return MOE_ERR_STATE;
    cudaStream_t s = static_cast<cudaStream_t>(compute), cp = static_cast<cudaStream_t>(copy);
    int rc = join_gather(p, layer, s);
    if (rc != MOE_OK) return rc;
    uint8_t* rec = p->dev_state + size_t(layer) * moe::dev_record(S, E).bytes;
    rc = moe::launch_pool_route_plan(logits, T, k, ids, w, counts, offsets, perm, inv, rec, S, E, p->d.policy,
                                     slot_of_dev, split_dev, p->bytes_per_load, s);
    if (rc != MOE_OK) return rc;
    return enqueue_gather(p, layer, s, cp);
}

extern "C" int moe_pool_device_join(moe_pool_t* p, int layer, moe_stream_t compute) {
    if (!p || layer < 0 || layer >= p->d.layers) return MOE_ERR_INVALID;
    if (!p->dev_state) return MOE_ERR_STATE;
    return join_gather(p, layer, static_cast<cudaStream_t>(compute));
}

extern "C" int moe_pool_device_detach(moe_pool_t* p, moe_stream_t stream, int timeout_ms) {
    if (!p) return MOE_ERR_INVALID;
    if (!p->dev_state) return MOE_ERR_STATE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int l = 0; l < p->d.layers; ++l) {
        const int rj = join_gather(p, l, s);
        if (rj != MOE_OK) return rj;
    }
    std::vector<uint8_t> img(device_state_bytes(p));
    MOE_CUDA_TRY(cudaMemcpyAsync(img.data(), p->dev_state, img.size(), cudaMemcpyDeviceToHost, s));
    const int rc = wait_stream(p, s, timeout_ms);
    if (rc != MOE_OK) return rc;  // still attached; the caller may retry
    const uint32_t status = unpack_device_state(p, img.data());
    p->dev_state = nullptr;
    p->host_dev = nullptr;
    if (status & 1u) return MOE_ERR_INVALID;
    if (status & 2u) return MOE_ERR_CAPACITY;
    return MOE_OK;
}

extern "C" int moe_pool_inject_copy_failures(moe_pool_t* p, int n) {
    if (!p || n < 0) return MOE_ERR_INVALID;
    p->inject_fail = n;
    return MOE_OK;
}

extern "C" void moe_pool_destroy(moe_pool_t* p) {
    if (!p) return;
    if (p->ev_compute) cudaEventDestroy(p->ev_compute);
    if (p->ev_copy) cudaEventDestroy(p->ev_copy);
    for (cudaEvent_t ev : p->ev_win)
        if (ev) cudaEventDestroy(ev);
    for (cudaEvent_t ev : p->ev_pf)
        if (ev) cudaEventDestroy(ev);
    if (p->map_pinned) cudaFreeHost(p->map_pinned);
    if (p->ev_plan) cudaEventDestroy(p->ev_plan);
    for (cudaEvent_t ev : p->ev_gather)
        if (ev) cudaEventDestroy(ev);
    delete p;
}

namespace moe {
// Accessors used by the FFN entry point (same library).
const Layout* pool_layout(const moe_pool_t* p) { return &p->L; }
const moe_pool_desc* pool_desc(const moe_pool_t* p) { return &p->d; }
}  // namespace moe
