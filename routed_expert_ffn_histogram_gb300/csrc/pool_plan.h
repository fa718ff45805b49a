// Policy planning of one staging event of the expert-slot pool, shared by the
// host pool (pool.cpp, compiled by the host compiler) and the device planner
// (pool_dev.cu): the same code takes every hit, miss and eviction decision on
// both sides.
//
// Event of one (layer, step) over U = {e : counts[e] > 0} (tinyserve README,
// "How it works" item 3 and "Configuration": cache_policy; Expert Offloading
// topic page, replay-semantics study: one fused cache event per (layer,
// step)): the resident members of U are hits, touched in ascending id; then
// each absent member, ascending, takes the lowest free slot or evicts the
// resident expert outside U (and outside `keep`) that the policy names.  A
// loaded expert gets a fresh stamp, count 1 and probation.
//   lru   touch: fresh stamp.             victim: oldest stamp.
//   fifo  touch: nothing (stamp = load).  victim: oldest load.
//   lfu   touch: count + 1.               victim: fewest uses, then lowest id.
//   lfru  touch: count + 1, fresh stamp.  victim: fewest uses, then oldest stamp.
//   slru  touch: fresh stamp; a probationary expert moves to the protected
//         segment (capacity S / 2, at least 1), whose least recent member,
//         if it overflows, goes back to probation with a fresh stamp.
//         victim: oldest probationary, else oldest protected.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "moe.h"

#if defined(__CUDACC__)
#define MOE_HD __host__ __device__ inline
#else
#define MOE_HD inline
#endif

namespace moe {

// One layer's policy state, seen through raw arrays (host vectors or a
// device planner's shared-memory copies).
struct PlanView {
    int32_t* se;    // [S] slot -> expert, -1 = free
    int32_t* es;    // [E] expert -> slot, -1 = absent
    int64_t* st;    // [S] recency / load stamps
    int64_t* uses;  // [S] touches since load
    int8_t* seg;    // [S] slru: 0 probation, 1 protected
    int64_t clk;    // the layer's stamp clock
    int S, E, policy;
};

struct PlanLoad {
    int32_t e, slot, victim;  // victim -1: the slot was free
};

MOE_HD void plan_touch(PlanView& v, int s) {
    switch (v.policy) {
        case MOE_POLICY_FIFO: break;
        case MOE_POLICY_LFU: ++v.uses[s]; break;
        case MOE_POLICY_LFRU:
            ++v.uses[s];
            v.st[s] = ++v.clk;
            break;
        case MOE_POLICY_SLRU: {
            v.st[s] = ++v.clk;
            if (v.seg[s] == 0) {
                v.seg[s] = 1;
                const int cap = v.S / 2 > 0 ? v.S / 2 : 1;
                int n = 0, oldest = -1;
                for (int i = 0; i < v.S; ++i)
                    if (v.se[i] >= 0 && v.seg[i] == 1) {
                        ++n;
                        if (oldest < 0 || v.st[i] < v.st[oldest]) oldest = i;
                    }
                if (n > cap) {
                    v.seg[oldest] = 0;
                    v.st[oldest] = ++v.clk;
                }
            }
            break;
        }
        default: v.st[s] = ++v.clk; break;  // lru
    }
}

// Whether slot i is a better victim than slot b under the policy.
MOE_HD bool plan_better(const PlanView& v, int i, int b) {
    switch (v.policy) {
        case MOE_POLICY_LFU: return v.uses[i] != v.uses[b] ? v.uses[i] < v.uses[b] : v.se[i] < v.se[b];
        case MOE_POLICY_LFRU: return v.uses[i] != v.uses[b] ? v.uses[i] < v.uses[b] : v.st[i] < v.st[b];
        case MOE_POLICY_SLRU: return v.seg[i] != v.seg[b] ? v.seg[i] < v.seg[b] : v.st[i] < v.st[b];
        default: return v.st[i] < v.st[b];  // lru, fifo
    }
}

// Slot to evict for a miss: a resident expert with counts[e] == 0 (when
// counts is given: not routed in this event) and keep[e] == 0 (when keep is
// given: not read by work still in flight); -1 if there is none.
MOE_HD int plan_victim(const PlanView& v, const int32_t* counts, const uint8_t* keep) {
    int best = -1;
    for (int i = 0; i < v.S; ++i) {
        const int e = v.se[i];
        if (e < 0 || (counts && counts[e] > 0) || (keep && keep[e])) continue;
        if (best < 0 || plan_better(v, i, best)) best = i;
    }
    return best;
}

MOE_HD int plan_free_slot(const PlanView& v) {
    for (int i = 0; i < v.S; ++i)
        if (v.se[i] < 0) return i;
    return -1;
}

// Put expert e into slot s (evicting its occupant, if any): fresh stamp,
// count 1, probation.
MOE_HD void plan_load(PlanView& v, int e, int s) {
    const int victim = v.se[s];
    if (victim >= 0) v.es[victim] = -1;
    v.se[s] = e;
    v.es[e] = s;
    v.st[s] = ++v.clk;
    v.uses[s] = 1;
    v.seg[s] = 0;
}

// Plans one event in place from its routed experts already split into the
// resident ones (hits, ascending expert id) and the absent ones (misses,
// ascending): the hits are touched in that order, then each miss takes the
// lowest free slot or the policy's victim.  A routed expert is never a
// victim, so the misses are exactly the routed experts absent before the
// event.  Writes the loads to `loads` in issue order; returns their number,
// or -1 if a miss found neither a free slot nor a victim (only possible
// with `keep`); the view is then partly modified, so callers plan on copies.
MOE_HD int plan_event_lists(PlanView& v, const int32_t* counts, const uint8_t* keep, const int32_t* hits, int nh,
                            const int32_t* misses, int nm, PlanLoad* loads) {
    for (int i = 0; i < nh; ++i) plan_touch(v, v.es[hits[i]]);
    int n = 0;
    for (int i = 0; i < nm; ++i) {
        const int e = misses[i];
        int s = plan_free_slot(v);
        int victim = -1;
        if (s < 0) {
            s = plan_victim(v, counts, keep);
            if (s < 0) return -1;
            victim = v.se[s];
        }
        plan_load(v, e, s);
        loads[n++] = PlanLoad{int32_t(e), int32_t(s), int32_t(victim)};
    }
    return n;
}

// Plans one event in place.  counts: [E], every entry >= 0 and at most S of
// them nonzero (the caller checks).  Writes the hits' expert ids to hit_e
// (ascending, *n_hits of them) and the loads to `loads` in issue order
// (ascending expert id); `misses` is scratch for up to S expert ids.
// Returns what plan_event_lists returns.
MOE_HD int plan_event(PlanView& v, const int32_t* counts, const uint8_t* keep, PlanLoad* loads, int32_t* hit_e,
                      int* n_hits, int32_t* misses) {
    int nh = 0, nm = 0;
    for (int e = 0; e < v.E; ++e) {
        if (counts[e] <= 0) continue;
        if (v.es[e] >= 0) hit_e[nh++] = e;
        else misses[nm++] = e;
    }
    *n_hits = nh;
    return plan_event_lists(v, counts, keep, hit_e, nh, misses, nm, loads);
}

// Device copy of the pool's per-layer state: one record per layer, fields
// at these byte offsets (16-byte aligned record).
struct DevRecord {
    size_t bytes;
    size_t ctr, clk, n_loads, status, n_copy, st, uses, freq, se, es, le, ls, seg, fresh;
};

MOE_HD size_t dev_align16(size_t n) { return (n + 15) & ~size_t(15); }

MOE_HD DevRecord dev_record(int S, int E) {
    DevRecord r{};
    size_t o = 0;
    r.ctr = o;     o += 8 * 8;               // moe_counters: eight uint64
    r.clk = o;     o += 8;
    r.n_loads = o; o += 4;                   // loads of the last successful event
    r.status = o;  o += 4;                   // bit 0: negative count, bit 1: more than S routed
    r.n_copy = o;  o += 8;                   // loads the current event's copy kernel makes (0 after a failed event)
    r.st = o;      o += 8 * size_t(S);
    r.uses = o;    o += 8 * size_t(S);
    r.freq = o;    o += 8 * size_t(E);       // events that routed each expert
    r.se = o;      o += 4 * size_t(S);
    r.es = o;      o += 4 * size_t(E);
    r.le = o;      o += 4 * size_t(S);       // last event's loads: expert, slot
    r.ls = o;      o += 4 * size_t(S);
    r.seg = o;     o += size_t(S);
    r.fresh = o;   o += size_t(E);           // loaded by a prefetch, not routed since
    r.bytes = dev_align16(o);
    return r;
}

}  // namespace moe
