// Warp-level routing pieces shared by the routing kernels and the fused
// decode kernel: top-k of one token's logits (larger logit first, equal
// logits by lower id, NaN last; one round = two redux.sync warp reductions
// on an order-preserving key) and the softmax over the k selected logits
// (float-float, about 48 bits, summed in rank order, rounded to fp32).
#pragma once

#include <cmath>
#include <cstdint>

namespace moe {
namespace {

// Order-preserving 32-bit key of a logit for the top-k: a larger logit has
// a larger key, -0 and +0 share one key, and NaN has key 0, below every
// number (the lowest non-NaN key, that of -inf, is 0x007fffff).
__device__ __forceinline__ uint32_t rank_key(float f) {
    if (isnan(f)) return 0u;
    uint32_t u = __float_as_uint(f);
    if ((u << 1) == 0u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One round of a warp top-k: candidate i of this lane is expert lane + 32 i
// with key key[i]; bit i of `taken` marks a candidate already selected or
// absent.  The round's winner (largest key, then lowest expert id) is found
// with two warp reductions (redux.sync max over the lanes' best keys, then
// min over the expert ids of the lanes holding that key), marked taken, and
// returned to every lane.
template <int EPL>
__device__ __forceinline__ int topk_round(const uint32_t (&key)[EPL], uint32_t& taken) {
    const int lane = threadIdx.x & 31;
    uint32_t best = 0u;
    int bi = -1;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
        if (!((taken >> i) & 1u) && (bi < 0 || key[i] > best)) {
            best = key[i];
            bi = i;
        }
    const uint32_t top = __reduce_max_sync(0xffffffffu, bi >= 0 ? best : 0u);
    const uint32_t cand = (bi >= 0 && best == top) ? uint32_t(lane + 32 * bi) : 0xffffffffu;
    const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
    if (int(win & 31u) == lane) taken |= 1u << (win >> 5);
    return int(win);
}

// Value v[win >> 5] of the lane holding expert `win`, on every lane.
template <int EPL, typename T>
__device__ __forceinline__ T from_winner(const T (&v)[EPL], int win) {
    T mine = v[0];
#pragma unroll
    for (int i = 1; i < EPL; ++i)
        if ((win >> 5) == i) mine = v[i];
    return __shfl_sync(0xffffffffu, mine, win & 31);
}

// Top-k of one token's logits by one warp: lane j < k ends with the j-th
// ranked (logit, id): larger logit first, equal logits by lower id, NaN
// last.  EPL = candidates per lane (E <= 32 * EPL).
template <int EPL>
__device__ __forceinline__ void topk_warp(const float* __restrict__ row, int E, int k, float& sel_v, int& sel_id) {
    const int lane = threadIdx.x & 31;
    float v[EPL];
    uint32_t key[EPL];
    uint32_t taken = 0;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        v[i] = (e < E) ? __ldg(row + e) : 0.0f;
        key[i] = rank_key(v[i]);
        if (e >= E) taken |= 1u << i;
    }
    sel_v = 0.0f;
    sel_id = -1;
    for (int j = 0; j < k; ++j) {
        const int win = topk_round<EPL>(key, taken);
        const float wv = from_winner<EPL>(v, win);
        if (lane == j) {
            sel_v = wv;
            sel_id = win;
        }
    }
}

// Prefetch a contiguous array of n floats into L1, a 128-byte line per lane
// at a time, so the rows a warp ranks one after another are all in flight at
// once instead of costing a memory round trip each.
__device__ __forceinline__ void prefetch_l1(const float* base, int n) {
    const int lane = threadIdx.x & 31;
    for (int c = lane; c * 32 < n; c += 32)
        asm volatile("prefetch.global.L1 [%0];" ::"l"(base + c * 32) : "memory");
}

// ---- float-float ("double-single") arithmetic --------------------------
// A value is an unevaluated sum hi + lo of two floats (about 48 bits).  The
// error-free transforms are Knuth's two-sum and the fma-based two-product;
// exp uses Cody-Waite reduction by ln 2 (split in three floats so n * c1 and
// n * c2 are exact), a further reduction by 8, a degree-10 Taylor series and
// three squarings.  GB300's fp64 rate is a small fraction of its fp32 rate,
// so this is much faster than double while matching a double evaluation
// after rounding to fp32 except in rare near-ties.
struct FF {
    float hi, lo;
};

__device__ __forceinline__ FF ff_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float v = __fsub_rn(s, a);
    return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, v)), __fsub_rn(b, v))};
}
__device__ __forceinline__ FF ff_fast_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ FF ff_two_prod(float a, float b) {
    const float p = __fmul_rn(a, b);
    return {p, __fmaf_rn(a, b, -p)};
}
__device__ __forceinline__ FF ff_add(FF x, FF y) {
    const FF s = ff_two_sum(x.hi, y.hi);
    return ff_fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo)));
}
__device__ __forceinline__ FF ff_mul(FF x, FF y) {
    const FF p = ff_two_prod(x.hi, y.hi);
    return ff_fast_two_sum(p.hi, __fadd_rn(p.lo, __fadd_rn(__fmul_rn(x.hi, y.lo), __fmul_rn(x.lo, y.hi))));
}

// e^d for d <= 0 given as a float-float.
__device__ __forceinline__ FF ff_exp_nonpos(FF d) {
    if (d.hi < -110.0f) return {0.0f, 0.0f};
    // ln 2 = c1 + c2 + c3 (c1 has 16 significant bits)
    const float c1 = 0.693145751953125f, c2 = 1.428606765330187e-06f, c3 = 5.497923148104107e-14f;
    const float n = rintf(d.hi * 1.4426950216293335f);
    FF r = ff_add(d, FF{-n * c1, 0.0f});
    r = ff_add(r, ff_two_prod(-n, c2));
    r = ff_add(r, FF{-n * c3, 0.0f});
    r.hi *= 0.125f;
    r.lo *= 0.125f;
    // 1/i! as float-float pairs, i = 0..10
    const float ch[11] = {1.0f, 1.0f, 0.5f, 0.1666666716337204f, 0.0416666679084301f, 0.008333333767950535f,
                          0.0013888889225199819f, 0.00019841270113829523f, 2.4801587642286904e-05f,
                          2.7557318844628753e-06f, 2.755731998149713e-07f};
    const float cl[11] = {0.0f, 0.0f, 0.0f, -4.967053879312289e-09f, -1.2417634698280722e-09f, -4.34617203337595e-10f,
                          -3.3631094437103215e-11f, -2.725596874933456e-12f, -3.40699609366682e-13f,
                          3.793571224297229e-14f, -7.575112209051195e-15f};
    FF p{ch[10], cl[10]};
#pragma unroll
    for (int i = 9; i >= 0; --i) p = ff_add(ff_mul(p, r), FF{ch[i], cl[i]});
    p = ff_mul(p, p);
    p = ff_mul(p, p);
    p = ff_mul(p, p);
    const int ni = int(n);
    return {ldexpf(p.hi, ni), ldexpf(p.lo, ni)};
}

// Softmax over the k selected logits: lane j < k evaluates its own
// exponential of (l_j - l_0) in float-float, the sum is folded in rank
// order, lane j divides; the result is rounded once to fp32.
__device__ __forceinline__ float softmax_lane(float sel_v, int k) {
    const int lane = threadIdx.x & 31;
    const float m = __shfl_sync(0xffffffffu, sel_v, 0);
    FF e{0.0f, 0.0f};
    if (lane < k) e = ff_exp_nonpos(ff_two_sum(sel_v, -m));
    FF s{0.0f, 0.0f};
    for (int j = 0; j < k; ++j) {
        const FF ej{__shfl_sync(0xffffffffu, e.hi, j), __shfl_sync(0xffffffffu, e.lo, j)};
        s = ff_add(s, ej);
    }
    const float q1 = __fdiv_rn(e.hi, s.hi);
    FF qs = ff_two_prod(s.hi, q1);
    qs.lo = __fmaf_rn(s.lo, q1, qs.lo);
    const FF r = ff_add(e, FF{-qs.hi, -qs.lo});
    return __fadd_rn(q1, __fdiv_rn(r.hi, s.hi));
}

// Softmax over each token's k selected logits for all A = T * k <= 32
// assignments at once: lane a < A holds the selected logit of assignment a
// (token a / k, rank a % k) and gets its weight; the same arithmetic as
// softmax_lane (float-float exponentials of l_j - l_0, summed in rank order,
// rounded once), every token in parallel.
__device__ __forceinline__ float softmax_assign(float sel_v, int k, int A) {
    const int lane = threadIdx.x & 31;
    const int t0 = (lane < A && A > k) ? (lane / k) * k : 0;   // first assignment of the lane's token
    const float m = __shfl_sync(0xffffffffu, sel_v, t0);
    FF e{0.0f, 0.0f};
    if (lane < A) e = ff_exp_nonpos(ff_two_sum(sel_v, -m));
    FF s{0.0f, 0.0f};
    for (int j = 0; j < k; ++j) {
        const FF ej{__shfl_sync(0xffffffffu, e.hi, t0 + j), __shfl_sync(0xffffffffu, e.lo, t0 + j)};
        s = ff_add(s, ej);
    }
    const float q1 = __fdiv_rn(e.hi, s.hi);
    FF qs = ff_two_prod(s.hi, q1);
    qs.lo = __fmaf_rn(s.lo, q1, qs.lo);
    const FF r = ff_add(e, FF{-qs.hi, -qs.lo});
    return __fadd_rn(q1, __fdiv_rn(r.hi, s.hi));
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

// The whole routing plan of T tokens (T * k <= 32) in one warp: lane a
// owns assignment a = t*k + j; its grouped position is (# assignments with a
// smaller expert id) + (# earlier assignments with the same id).  Every
// token's logits are put in flight at once, then each token is ranked (the
// lane holding a winner records it for its assignment in sel_id / sel_v,
// 32 entries of shared memory), then one softmax pass serves every
// assignment.  Returns the lane's expert id (MOE_MAX_EXPERTS past A).
template <int EPL>
__device__ __forceinline__ int route_tiny_warp(const float* __restrict__ logits, int T, int E, int k,
                                               int32_t* __restrict__ ids, float* __restrict__ w,
                                               int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                               int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                                               int* sel_id, float* sel_v) {
    const int lane = threadIdx.x & 31;
    const int A = T * k;
    if (T > 1) prefetch_l1(logits, T * E);
    for (int t = 0; t < T; ++t) {
        const float* row = logits + (size_t)t * E;
        float v[EPL];
        uint32_t key[EPL], taken = 0;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            v[i] = e < E ? __ldg(row + e) : 0.0f;
            key[i] = rank_key(v[i]);
            if (e >= E) taken |= 1u << i;
        }
        for (int j = 0; j < k; ++j) {
            const int bid = topk_round<EPL>(key, taken);
            const float bv = from_winner<EPL>(v, bid);
            if (lane == 0) {
                sel_id[t * k + j] = bid;
                sel_v[t * k + j] = bv;
            }
        }
    }
    __syncwarp();
    const int my_id = lane < A ? sel_id[lane] : MOE_MAX_EXPERTS;   // MOE_MAX_EXPERTS sorts after every real id
    const float wv = softmax_assign(lane < A ? sel_v[lane] : 0.0f, k, A);
    if (lane < A) {
        ids[lane] = my_id;
        w[lane] = wv;
    }
    plan_warp(my_id, A, E, counts, offsets, perm, inv);
    return my_id;
}

}  // namespace
}  // namespace moe
