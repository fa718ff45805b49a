// Expert-slot pool: per-layer (expert -> slot) map with LRU eviction and
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
// ascending.  Resident members of U are hits and are touched first (fresh
// recency stamps in ascending id); then each absent member, ascending, takes
// the lowest free slot or evicts the resident expert with the oldest stamp.
// Members of U were all stamped during the event, so they are never evicted.
#include <chrono>
#include <cstring>
#include <new>
#include <thread>
#include <vector>

#include "internal.h"

struct moe_pool {
    moe_pool_desc d;
    moe::Layout L;
    size_t eb = 0;
    std::vector<int32_t> slot_expert;   // [L][S], -1 = free
    std::vector<int32_t> expert_slot;   // [L][E], -1 = absent
    std::vector<int64_t> stamp;         // [L][S]
    std::vector<int64_t> clock;         // [L]
    std::vector<moe_counters> ctr;      // [L]
    std::vector<int32_t> last_e, last_s;  // [L][S]
    std::vector<int> last_n;            // [L]
    int32_t* map_pinned = nullptr;      // [L][E] staging for slot-map uploads
    cudaEvent_t ev_compute = nullptr, ev_copy = nullptr;
    int inject_fail = 0;
};

namespace {

constexpr uint32_t kStateMagic = 0x4d4f4550u;  // "MOEP"

struct Planned {
    int32_t e, slot, victim;
};

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
    moe_pool_t* p = new (std::nothrow) moe_pool;
    if (!p) return MOE_ERR_INVALID;
    p->d = d;
    p->L = L;
    p->eb = L.expert_bytes;
    const size_t nl = size_t(d.layers), S = size_t(d.slots_per_layer), E = size_t(d.experts);
    p->slot_expert.assign(nl * S, -1);
    p->expert_slot.assign(nl * E, -1);
    p->stamp.assign(nl * S, 0);
    p->clock.assign(nl, 0);
    p->ctr.assign(nl, moe_counters{});
    p->last_e.assign(nl * S, -1);
    p->last_s.assign(nl * S, -1);
    p->last_n.assign(nl, 0);
    if (!d.dry_run) {
        cudaError_t e = cudaHostAlloc(reinterpret_cast<void**>(&p->map_pinned), nl * E * sizeof(int32_t),
                                      cudaHostAllocDefault);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_compute, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_copy, cudaEventDisableTiming);
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
                if (!d.dry_run) {
                    const uint8_t* src = static_cast<const uint8_t*>(d.host_experts) + (l * E + s) * p->eb;
                    uint8_t* dst = static_cast<uint8_t*>(d.dev_slots) + (l * S + s) * p->eb;
                    cudaError_t e = cudaMemcpy(dst, src, p->eb, cudaMemcpyHostToDevice);
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

extern "C" int moe_pool_stage(moe_pool_t* p, int layer, const int32_t* counts_host, int32_t* slot_of_dev,
                              moe_stream_t compute, moe_stream_t copy, int timeout_ms) {
    if (!p || !counts_host || layer < 0 || layer >= p->d.layers) return MOE_ERR_INVALID;
    const int S = p->d.slots_per_layer, E = p->d.experts;
    cudaStream_t cs = static_cast<cudaStream_t>(compute), ps = static_cast<cudaStream_t>(copy);
    if (!p->d.dry_run) {
        const int rc = wait_stream(p, cs, timeout_ms);
        if (rc != MOE_OK) return rc;
    }
    int32_t* se = &p->slot_expert[size_t(layer) * S];
    int32_t* es = &p->expert_slot[size_t(layer) * E];
    int64_t* st = &p->stamp[size_t(layer) * S];
    int64_t& clk = p->clock[layer];
    moe_counters& c = p->ctr[layer];

    int uniq = 0;
    for (int e = 0; e < E; ++e) {
        if (counts_host[e] < 0) return MOE_ERR_INVALID;
        uniq += counts_host[e] > 0;
    }
    if (uniq > S) return MOE_ERR_CAPACITY;

    // Plan the event on scratch copies; commit load by load as copies enqueue.
    std::vector<int32_t> se2(se, se + S), es2(es, es + E);
    std::vector<int64_t> st2(st, st + S);
    int64_t clk2 = clk;
    uint64_t hits = 0;
    for (int e = 0; e < E; ++e)
        if (counts_host[e] > 0 && es2[e] >= 0) {
            st2[es2[e]] = ++clk2;
            ++hits;
        }
    std::vector<Planned> plan;
    for (int e = 0; e < E; ++e) {
        if (counts_host[e] <= 0 || es2[e] >= 0) continue;
        int s = -1;
        for (int i = 0; i < S; ++i)
            if (se2[i] < 0) { s = i; break; }
        int victim = -1;
        if (s < 0) {
            for (int i = 0; i < S; ++i)
                if (s < 0 || st2[i] < st2[s]) s = i;
            victim = se2[s];
            es2[victim] = -1;
        }
        se2[s] = e;
        es2[e] = s;
        st2[s] = ++clk2;
        plan.push_back({e, s, victim});
    }

    size_t done = 0;
    int fail = MOE_OK;
    for (const Planned& q : plan) {
        if (p->inject_fail > 0) {
            --p->inject_fail;
            fail = moe::cuda_fail(cudaErrorUnknown);
            break;
        }
        if (!p->d.dry_run) {
            const uint8_t* src = static_cast<const uint8_t*>(p->d.host_experts) +
                                 (size_t(layer) * E + q.e) * p->eb;
            uint8_t* dst = static_cast<uint8_t*>(p->d.dev_slots) + (size_t(layer) * S + q.slot) * p->eb;
            cudaError_t e = cudaMemcpyAsync(dst, src, p->eb, cudaMemcpyHostToDevice, ps);
            if (e != cudaSuccess) {
                fail = moe::cuda_fail(e);
                break;
            }
        }
        ++done;
    }

    if (fail != MOE_OK) {
        // Keep only the loads that were enqueued (their slots now hold the new
        // experts); everything else of the event is not applied.
        for (size_t i = 0; i < done; ++i) {
            const Planned& q = plan[i];
            if (q.victim >= 0) {
                es[q.victim] = -1;
                ++c.evictions;
            }
            se[q.slot] = q.e;
            es[q.e] = q.slot;
            st[q.slot] = ++clk;
            ++c.misses;
            c.h2d_bytes += p->eb;
        }
        ++c.errors;
        p->last_n[layer] = 0;
    } else {
        std::memcpy(se, se2.data(), sizeof(int32_t) * S);
        std::memcpy(es, es2.data(), sizeof(int32_t) * E);
        std::memcpy(st, st2.data(), sizeof(int64_t) * S);
        clk = clk2;
        c.hits += hits;
        c.misses += plan.size();
        for (const Planned& q : plan) c.evictions += q.victim >= 0;
        c.h2d_bytes += plan.size() * p->eb;
        ++c.events;
        p->last_n[layer] = int(plan.size());
        for (size_t i = 0; i < plan.size(); ++i) {
            p->last_e[size_t(layer) * S + i] = plan[i].e;
            p->last_s[size_t(layer) * S + i] = plan[i].slot;
        }
    }

    if (!p->d.dry_run) {
        if (done > 0 && ps != cs) {
            MOE_CUDA_TRY(cudaEventRecord(p->ev_copy, ps));
            MOE_CUDA_TRY(cudaStreamWaitEvent(cs, p->ev_copy, 0));
        }
        if (slot_of_dev) {
            int32_t* stage = p->map_pinned + size_t(layer) * E;
            std::memcpy(stage, es, sizeof(int32_t) * E);
            MOE_CUDA_TRY(cudaMemcpyAsync(slot_of_dev, stage, sizeof(int32_t) * E, cudaMemcpyHostToDevice, cs));
        }
    }
    return fail;
}

extern "C" int moe_pool_counters(const moe_pool_t* p, int layer, moe_counters* out) {
    if (!p || !out || layer < -1 || layer >= p->d.layers) return MOE_ERR_INVALID;
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
    }
    *out = s;
    return MOE_OK;
}

extern "C" int moe_pool_slot_map(const moe_pool_t* p, int layer, int32_t* out) {
    if (!p || !out || layer < 0 || layer >= p->d.layers) return MOE_ERR_INVALID;
    std::memcpy(out, &p->expert_slot[size_t(layer) * p->d.experts], sizeof(int32_t) * p->d.experts);
    return MOE_OK;
}

extern "C" int moe_pool_last_loads(const moe_pool_t* p, int layer, int32_t* le, int32_t* ls, int* n) {
    if (!p || !le || !ls || !n || layer < 0 || layer >= p->d.layers) return MOE_ERR_INVALID;
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
    int32_t layers, experts, slots, hidden, inter;
};
size_t state_bytes(const moe_pool_t* p) {
    return sizeof(StateHeader) + p->slot_expert.size() * 4 + p->expert_slot.size() * 4 +
           p->stamp.size() * 8 + p->clock.size() * 8 + p->ctr.size() * sizeof(moe_counters);
}
}  // namespace

extern "C" int moe_pool_state_bytes(const moe_pool_t* p, size_t* out) {
    if (!p || !out) return MOE_ERR_INVALID;
    *out = state_bytes(p);
    return MOE_OK;
}

extern "C" int moe_pool_save(const moe_pool_t* p, void* buf, size_t bytes) {
    if (!p || !buf || bytes < state_bytes(p)) return MOE_ERR_INVALID;
    uint8_t* o = static_cast<uint8_t*>(buf);
    StateHeader h{kStateMagic, p->d.layers, p->d.experts, p->d.slots_per_layer, p->d.hidden, p->d.inter};
    std::memcpy(o, &h, sizeof h);
    o += sizeof h;
    auto put = [&o](const void* src, size_t n) { std::memcpy(o, src, n); o += n; };
    put(p->slot_expert.data(), p->slot_expert.size() * 4);
    put(p->expert_slot.data(), p->expert_slot.size() * 4);
    put(p->stamp.data(), p->stamp.size() * 8);
    put(p->clock.data(), p->clock.size() * 8);
    put(p->ctr.data(), p->ctr.size() * sizeof(moe_counters));
    return MOE_OK;
}

extern "C" int moe_pool_load(moe_pool_t* p, const void* buf, size_t bytes) {
    if (!p || !buf || bytes < state_bytes(p)) return MOE_ERR_INVALID;
    const uint8_t* i = static_cast<const uint8_t*>(buf);
    StateHeader h;
    std::memcpy(&h, i, sizeof h);
    if (h.magic != kStateMagic || h.layers != p->d.layers || h.experts != p->d.experts ||
        h.slots != p->d.slots_per_layer || h.hidden != p->d.hidden || h.inter != p->d.inter)
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
    get(p->clock.data(), p->clock.size() * 8);
    get(p->ctr.data(), p->ctr.size() * sizeof(moe_counters));
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
    if (p->map_pinned) cudaFreeHost(p->map_pinned);
    delete p;
}

namespace moe {
// Accessors used by the FFN entry point (same library).
const Layout* pool_layout(const moe_pool_t* p) { return &p->L; }
const moe_pool_desc* pool_desc(const moe_pool_t* p) { return &p->d; }
}  // namespace moe
