// Warp-level routing pieces shared by the routing kernels and the fused
// decode kernel: top-k of one token's logits (larger logit first, equal
// logits by lower id, NaN last) and the softmax over the k selected logits
// (fp64, summed in rank order, rounded to fp32).
#pragma once

#include <cmath>
#include <cstdint>

namespace moe {
namespace {

__device__ __forceinline__ bool ranks_before(float la, int a, float lb, int b) {
    const bool na = isnan(la), nb = isnan(lb);
    if (na != nb) return nb;
    if (!na && la != lb) return la > lb;
    return a < b;
}

// Top-k of one token's logits by one warp: lane j < k ends with the j-th
// ranked (logit, id).  EPL = candidates per lane (E <= 32 * EPL).
template <int EPL>
__device__ __forceinline__ void topk_warp(const float* __restrict__ row, int E, int k, float& sel_v, int& sel_id) {
    const int lane = threadIdx.x & 31;
    float v[EPL];
    uint32_t taken = 0;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        v[i] = (e < E) ? __ldg(row + e) : 0.0f;
        if (e >= E) taken |= 1u << i;
    }
    sel_v = 0.0f;
    sel_id = -1;
    for (int j = 0; j < k; ++j) {
        float bv = 0.0f;
        int bid = -1;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            if (taken & (1u << i)) continue;
            const int e = lane + 32 * i;
            if (bid < 0 || ranks_before(v[i], e, bv, bid)) { bv = v[i]; bid = e; }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oid = __shfl_xor_sync(0xffffffffu, bid, off);
            if (oid >= 0 && (bid < 0 || ranks_before(ov, oid, bv, bid))) { bv = ov; bid = oid; }
        }
        // every lane now holds the same winner
        if ((bid & 31) == lane) taken |= 1u << (bid >> 5);
        if (lane == j) { sel_v = bv; sel_id = bid; }
    }
}

// Softmax over the k selected logits in fp64: lane j < k evaluates its own
// exponential, the sum is folded in rank order, lane j divides.
__device__ __forceinline__ float softmax_lane(float sel_v, int k) {
    const int lane = threadIdx.x & 31;
    const double m = (double)__shfl_sync(0xffffffffu, sel_v, 0);
    const double d = (lane < k) ? exp((double)sel_v - m) : 0.0;
    double sum = 0.0;
    for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, d, j);
    return (float)(d / sum);
}

// Grouping of A <= 32 assignments by one warp: lane a holds the expert id
// of assignment a (lanes >= A hold any id >= E).  Writes counts[E],
// offsets[E+1] (exclusive prefix sum), perm (assignments grouped by expert,
// stable) and inv.  A lane's grouped position is (# assignments with a
// smaller id) + (# earlier assignments with the same id).
__device__ __forceinline__ void plan_warp(int my_id, int A, int E, int32_t* __restrict__ counts,
                                          int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                                          int32_t* __restrict__ inv) {
    const int lane = threadIdx.x & 31;
    const uint32_t lt = (1u << lane) - 1u;
    const uint32_t same = __match_any_sync(0xffffffffu, my_id);
    int below = 0;
    for (int b = 0; b < A; ++b) below += __shfl_sync(0xffffffffu, my_id, b) < my_id;
    if (lane < A) {
        const int pos = below + __popc(same & lt);
        perm[pos] = lane;
        inv[lane] = pos;
    }
    for (int e0 = 0; e0 <= E; e0 += 32) {
        const int e = e0 + lane;
        int lt_e = 0, eq_e = 0;
        for (int b = 0; b < A; ++b) {
            const int idb = __shfl_sync(0xffffffffu, my_id, b);
            lt_e += idb < e;
            eq_e += idb == e;
        }
        if (e < E) counts[e] = eq_e;
        if (e <= E) offsets[e] = lt_e;
    }
}

}  // namespace
}  // namespace moe
