// Decode path, fused: the whole expert FFN of one layer (gate/up + SwiGLU,
// down + weighted combine) in one kernel, with the routing of the token(s)
// folded in for moe_decode_layer.
//
// Source: tinyserve README, "How it works" item 2 -- gate, up and down run
// directly on the quantised bytes, with no intermediate BF16 weights;
// llama.cpp discussion "fixed GPU expert working set with Native CPU miss
// execution", main post -- outputs merged with the routing weights, and CUDA
// graphs matter for decode because launches dominate a one-token step.
// Formats: OCP MX v1.0 (E2M1 elements, E8M0 scale per 32 along K).
//
// Arithmetic is the decode path's: bf16 activation x fp32-dequantised fp4
// (every product exact in fp32), fp32 sums, SwiGLU in fp32 rounded to bf16,
// down product on bf16(h), combine of w_j * y_j in fp32.  The down sums
// and the combine are split over CTAs and folded with fp32 atomics, so
// their rounding order (not their value beyond fp32 rounding) varies
// between runs.
//
// Shape: one CTA per SM, 18 warps in three roles.
//   routing  warp 0, and for several tokens up to 16 consumer warps too,
//            each rank their own tokens: the slot map and the first token's
//            logits in one memory round trip (later tokens' logits
//            prefetched into L1 at the same time), each top-k round two
//            redux.sync warp reductions; each assignment's expert and slot
//            are published through an mbarrier of their own as soon as its
//            rank is decided.  Once every router has reported, warp 0 weighs
//            every assignment in one softmax pass.
//   copies   warp 1 (one lane) streams the CTA's work items: items of 16
//            consecutive rows of h for one assignment.  The 16 gate and 16
//            up rows (contiguous in the packed layout) go into a 3-slot ring
//            as eight bulk copies, one arrival barrier per group of four row
//            pairs; the matching 16-column block of the column-blocked down
//            copy goes into a 2-slot ring.  An item is issued as soon as its
//            assignment is published and its slots are free.
//   consumers warps 2..17 stage x (while warp 0 routes) and then, per item:
//   gate/up  warp j takes row pair j of the item once its group of rows has
//            landed: one 16-byte load = one MX block per lane; x is staged
//            once per CTA in shared memory as f16 scaled per 32-block by a
//            power of two (exact for every value within 2^-31 of the block
//            maximum) in XOR-swizzled 16-byte chunks; E2M1 pairs become f16x2
//            by hardware conversion and multiply-add into fp32 (products
//            exact); h = bf16(silu(g)*u).  The gate/up slot is handed back
//            before the per-item barrier, so its next rows stream in while
//            the down block is applied.
//   down     the 16 h values (f16 under one power-of-2 scale, taken from the
//            item's largest |h|, which the gate/up warps record with a
//            shared atomic max) times the block's codes, every consumer
//            thread owning fixed output rows; partial sums stay in registers
//            across an assignment's items.  E8M0 scales come from a
//            256-entry table in shared memory.
//   combine  w_a * y added with float4 atomics (a lane quad's four rows) to
//            `out` directly when the caller accumulates (out += result, a
//            residual stream), else to an fp32 accumulator in the
//            workspace that the last CTA to finish (a ticket counter, no
//            waiting) copies to the output and clears for the next call.
// Skip-absent launches (MOE_FFN_SKIP_ABSENT; kernel instances of their own)
// serve only the assignments whose expert has a slot: every warp forms the
// same bit mask of them, and the work items run over those assignments
// alone, spread over all CTAs -- a layer then computes in two launches over
// complementary slot maps (the event's hits beside the copy of its misses,
// then the loaded experts).
// No CTA waits for another: there is no grid barrier and no cooperative
// launch.  Waits inside the CTA are bounded mbarrier waits (about a second,
// then an error bit and NaN output instead of a hang).  The kernel is
// launched with programmatic stream serialisation: each CTA runs its
// shared-memory-only prologue, lets the next kernel launch, and waits for the
// previous one (griddepcontrol) before touching global memory, so
// consecutive layers hand SMs over CTA by CTA.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <type_traits>
#include <cmath>

#include "internal.h"
#include "route_warp.cuh"
#include "tc_ptx.cuh"


namespace moe {
namespace {

constexpr int kGroup = 16;             // row pairs per ring slot (one bulk copy each for gate and up)
constexpr int kThreads = 32 * (kGroup + 2);  // warp 0: routing; warp 1: copy producer; warps 2..17: one row pair each
static_assert(Layout::kChunk % kGroup == 0, "a group of gate rows stays inside one interleave chunk");

// Value of an E8M0 scale byte: 2^(b - 127), byte 255 NaN (OCP MX v1.0).
__device__ __forceinline__ float e8m0_value_f(int b) {
    if (b == 255) return __int_as_float(0x7fc00000);
    return b >= 1 ? __int_as_float(b << 23) : __int_as_float(0x00400000);  // b = 0: 2^-127 (subnormal)
}

// acc0 += w.lo * x.lo, acc1 += w.hi * x.hi: f16 x f16 products formed
// exactly and added in fp32 (mixed-precision FMA).
__device__ __forceinline__ void fma2_f16_f32(float& acc0, float& acc1, uint32_t w2, uint32_t x2) {
    asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
        "mov.b32 {wl, wh}, %2;\n\tmov.b32 {xl, xh}, %3;\n\t"
        "fma.rn.f32.f16 %0, wl, xl, %0;\n\tfma.rn.f32.f16 %1, wh, xh, %1;\n\t}"
        : "+f"(acc0), "+f"(acc1)
        : "r"(w2), "r"(x2));
}

// Eight E2M1 codes (element 2i in the low nibble of byte i) -> four f16x2.
__device__ __forceinline__ void e2m1x8_f16(uint32_t word, uint32_t (&h)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(word));
}

// Staged activation block b (32 f16 = 4 chunks of 16 bytes), chunk q;
// XOR-swizzled so the 8 lanes of an LDS.128 phase hit distinct banks.
__device__ __forceinline__ int hswz(int b, int q) { return b * 4 + (q ^ ((b >> 1) & 3)); }

// Two rows (gate, up) against the same staged block b.
__device__ __forceinline__ void block_dot2_f16(const uint4 cg, const uint4 cu, const uint4* __restrict__ xs,
                                               int b, float& dg, float& du) {
    const uint32_t wg[4] = {cg.x, cg.y, cg.z, cg.w};
    const uint32_t wu[4] = {cu.x, cu.y, cu.z, cu.w};
    float g0 = 0.f, g1 = 0.f, u0 = 0.f, u1 = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 xv = xs[hswz(b, q)];
        uint32_t fg[4], fu[4];
        e2m1x8_f16(wg[q], fg);
        e2m1x8_f16(wu[q], fu);
        fma2_f16_f32(g0, g1, fg[0], xv.x);
        fma2_f16_f32(u0, u1, fu[0], xv.x);
        fma2_f16_f32(g0, g1, fg[1], xv.y);
        fma2_f16_f32(u0, u1, fu[1], xv.y);
        fma2_f16_f32(g0, g1, fg[2], xv.z);
        fma2_f16_f32(u0, u1, fu[2], xv.z);
        fma2_f16_f32(g0, g1, fg[3], xv.w);
        fma2_f16_f32(u0, u1, fu[3], xv.w);
    }
    dg = g0 + g1;
    du = u0 + u1;
}

// Served assignments as a bit mask: the n-th set bit (n counted from 0),
// and the next set bit after a (64 when there is none).
__device__ __forceinline__ int nth_active(uint64_t m, int n) {
    for (int i = 0; i < n && m; ++i) m &= m - 1;
    return m ? __ffsll((long long)m) - 1 : 64;
}
__device__ __forceinline__ int next_active(uint64_t m, int a) {
    const uint64_t rest = (a >= 63) ? 0ull : (m >> (a + 1));
    return rest ? a + __ffsll((long long)rest) : 64;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Stage nb blocks of 32 bf16 values as f16 scaled per block by a power of
// two 2^-e (e from the block's largest magnitude, so every value fits f16):
// x * 2^-e is exact in f16 for all values within 2^-31 of the block maximum
// (smaller ones round by less than 2^-24 of the block's dot product).
// The block's factor 2^e is kept as fp32 (e in [-140, 113]: exact).
// One thread per block.
__device__ __forceinline__ void stage_block_f16(const uint16_t* __restrict__ src, uint4* dst, int b,
                                                float* factors) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src) + b * 4;
    uint4 v[4];
    float amax = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        v[q] = __ldcg(s4 + q);
        const uint32_t u[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            amax = fmaxf(amax, fabsf(__uint_as_float(u[i] << 16)));
            amax = fmaxf(amax, fabsf(__uint_as_float(u[i] & 0xffff0000u)));
        }
    }
    // e: unbiased exponent of amax minus 14 (scaled maximum in [2^14, 2^15))
    const int ef = int((__float_as_uint(amax) >> 23) & 0xffu);
    const int e = (amax == 0.f) ? 0 : (ef == 0 ? -126 - 14 : ef - 127 - 14);
    const float m = ldexpf(1.0f, -e);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t u[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 hh = __floats2half2_rn(__uint_as_float(u[i] << 16) * m,
                                                 __uint_as_float(u[i] & 0xffff0000u) * m);
            o[i] = *reinterpret_cast<const uint32_t*>(&hh);
        }
        dst[hswz(b, q)] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    factors[b] = ldexpf(1.0f, e);
}

struct FusedParams {
    int stall;         // test hook: the first item's copies are not issued
    const uint8_t* slots;
    size_t expert_bytes;
    int S, E, H, I, k, T;
    size_t rs_gu, dt_off, dt_stride;
    const uint16_t* x;
    const int32_t* ids;
    const float* w;
    const int32_t* slot_of;
    uint16_t* h;       // bf16 [T*k][I]: the SwiGLU output, kept for inspection
    float* acc;        // fp32 [T][H] accumulator, all zero between calls
    float* out;        // fp32 [T][H]
    unsigned* ctl;     // [0] CTAs finished (zero between calls), [2] error bits
    int accumulate;    // out += result: partial sums go to out, no completion pass
    // fused routing (logits != nullptr): the kernel selects the experts itself
    // and CTA 0 writes the routing outputs below
    const float* logits;
    int32_t* r_ids;
    float* r_w;
    int32_t* r_counts;
    int32_t* r_offsets;
    int32_t* r_perm;
    int32_t* r_inv;
};

constexpr int kMaxAssign = MOE_DECODE_MAX_ASSIGN;
constexpr int kConsumers = kThreads - 64;   // threads of warps 2..kGroup+1
constexpr int kGuGroups = 4;                // arrival barriers per gate/up slot (4 consumer warps each)
constexpr int kRowsPerGroup = kGroup / kGuGroups;
constexpr int kMaxGuSlots = 8, kMaxDSlots = 8;

// Per-CTA table of the routed assignments.
struct AssignTable {
    int slot_of[MOE_MAX_EXPERTS];
    const uint8_t* base[kMaxAssign];
    float w[kMaxAssign];
    float sel_v[kMaxAssign];
    int id[kMaxAssign];
};

__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            tc::smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void named_bar_consumers() {
    asm volatile("bar.sync 1, %0;" ::"r"(kConsumers) : "memory");
}

struct Ring {
    uint64_t full_gu[kMaxGuSlots][kGuGroups];  // gate/up rows of a group of 4 row pairs landed
    uint64_t empty_gu[kMaxGuSlots];            // 16 consumer warps done with the slot's rows
    uint64_t full_d[kMaxDSlots];               // down block landed
    uint64_t empty_d[kMaxDSlots];              // 16 consumer warps done with the block
    uint64_t ranked;                           // every routing warp has published its tokens' ranks
    uint64_t routed;                           // routing table (ids, weights, bases) written
    uint64_t assigned[kMaxAssign];             // assignment a's expert and slot known
};

// Work item (a, c): gate/up rows 16c..16c+15 of assignment a, and block c of
// the column-blocked down copy.  The rows and the block travel in separate
// rings: a gate/up slot is handed back as soon as the 16 h values exist, so
// its next rows stream in while the down block is applied.  Warp j (1..16)
// computes h[16c + j - 1], waiting only for the rows of its group of four;
// then the 512 consumer threads apply the 16 h values to the block: thread
// q owns output rows n = q + 512 m and accumulates y[n] in registers while
// the items of one assignment follow each other.  When the assignment
// changes (and at the end) the thread adds w_a * y[n] into out (residual
// form) or into the fp32 accumulator of its token, which the last CTA to
// finish copies to `out` and clears.  No CTA ever waits for another one.
template <int NG, int NN, bool kSkip>
__global__ void __launch_bounds__(kThreads, 1)
decode_fused_kernel(FusedParams p, int n_gu, int n_d, int gu_off, int d_off) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ AssignTable tab;
    __shared__ __align__(8) Ring rb;
    __shared__ __align__(16) float hval[2][kGroup];
    __shared__ unsigned hmax_bits[3];
    __shared__ float e8m0_lut[256];
    __shared__ int last_cta;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = gridDim.x;
    const int A = p.T * p.k;
    volatile uint32_t* err = p.ctl + 2;
    // Prologue that touches no global memory, then the programmatic launch
    // hand-off: the next kernel in the stream may launch now (its CTAs take
    // SMs as ours exit and run their own prologue), and nothing below reads
    // an input or writes an output before the previous kernel has finished.
    for (int i = threadIdx.x; i < 256; i += kThreads) e8m0_lut[i] = e8m0_value_f(i);
    if (threadIdx.x == 0) {
        for (int s = 0; s < n_gu; ++s) {
            for (int q = 0; q < kGuGroups; ++q) tc::mbar_init(&rb.full_gu[s][q], 1);
            tc::mbar_init(&rb.empty_gu[s], kGroup);
        }
        for (int s = 0; s < n_d; ++s) {
            tc::mbar_init(&rb.full_d[s], 1);
            tc::mbar_init(&rb.empty_d[s], kGroup);
        }
        tc::mbar_init(&rb.routed, 1);
        tc::mbar_init(&rb.ranked, p.logits != nullptr ? unsigned(min(p.T, 1 + kConsumers / 32)) : 1u);
        hmax_bits[0] = hmax_bits[1] = hmax_bits[2] = 0u;
        for (int a = 0; a < A; ++a) tc::mbar_init(&rb.assigned[a], 1);
        tc::fence_barrier_init();
    }
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // The assignments this launch serves: all of them, or (kSkip, the
    // skip-absent launches) those whose expert has a slot (>= 0; a slot >= S
    // still counts and yields NaN).  Every warp forms the same mask.
    uint64_t act = (A >= 64) ? ~0ull : ((1ull << A) - 1ull);
    if (kSkip) {
        uint64_t m = 0;
        for (int base = 0; base < A; base += 32) {
            const int a = base + lane;
            bool on = false;
            if (a < A) {
                const int e = __ldg(p.ids + a);
                on = e >= 0 && e < p.E && __ldg(p.slot_of + e) >= 0;
            }
            m |= uint64_t(__ballot_sync(0xffffffffu, on)) << base;
        }
        act = m;
    }
    // This CTA's items: a contiguous range of the n_act * I / 16 items in
    // (served assignment, column block) order.
    const int items = (kSkip ? __popcll(act) : A) * p.I / kGroup;
    const int per = (items + G - 1) / G;
    const int g0 = min(items, (int)blockIdx.x * per), g1 = min(items, g0 + per);
    const int cnt = g1 - g0;
    const int nbx = p.H / 32;
    const size_t row_bytes = p.rs_gu;
    const uint32_t gu_bytes = uint32_t(2 * kGroup * row_bytes);       // gate rows, then up rows
    const uint32_t dt_bytes = uint32_t(p.H) * (kGroup / 2 + 1);          // codes, then scales
    const uint32_t dt_slot = (dt_bytes + 127u) / 128u * 128u;
    uint8_t* ring_gu = smem + gu_off;
    uint8_t* ring_d = smem + d_off;

    // ---- routing: with logits, warp 0 and up to 16 consumer warps each rank
    // their own tokens (t = r, r + R, ...; warp 0 is router 0, warp w >= 2
    // router w - 1), before the consumers stage x.  Each assignment's expert
    // and slot are published (an mbarrier per assignment) as soon as its
    // rank is decided, so the producer issues that assignment's copies while
    // the remaining ranks are still being found; warp 0 weighs every
    // assignment once all routers have reported ----
    const int R = (p.logits != nullptr) ? min(p.T, 1 + kConsumers / 32) : 0;
    const int rw = (warp == 0) ? 0 : warp - 1;
    if (p.logits != nullptr && (warp == 0 || (warp >= 2 && rw < R))) {
        auto route_tokens = [&](auto epl_tag) {
            constexpr int EPL = decltype(epl_tag)::value;
            // the slot map and this router's first token's logits are fetched
            // together (one memory round trip); its later tokens' logits are
            // prefetched at the same time; lane l keeps slot_of[l + 32 i]
            const int epl = (p.E + 31) / 32;
            for (int t = rw + R; t < p.T; t += R) prefetch_l1(p.logits + (size_t)t * p.E, p.E);
            int sl[EPL];
            float v[EPL];
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int e = lane + 32 * i;
                const bool in = i < epl && e < p.E;
                v[i] = in ? __ldg(p.logits + (size_t)rw * p.E + e) : 0.0f;
                sl[i] = in ? __ldg(p.slot_of + e) : -1;
            }
            for (int t = rw; t < p.T; t += R) {
                const float* row = p.logits + (size_t)t * p.E;
                uint32_t taken = 0, key[EPL];
#pragma unroll
                for (int i = 0; i < EPL; ++i) {
                    const int e = lane + 32 * i;
                    const bool in = i < epl && e < p.E;
                    if (t > rw) v[i] = in ? __ldg(row + e) : 0.0f;
                    key[i] = rank_key(v[i]);
                    if (!in) taken |= 1u << i;
                }
                for (int j = 0; j < p.k; ++j) {
                    const int bid = topk_round<EPL>(key, taken);
                    const int ws = from_winner<EPL>(sl, bid);   // the winner's slot
                    const float bv = from_winner<EPL>(v, bid);
                    if (lane == 0) {
                        const int a = t * p.k + j;
                        const int slot = (bid >= 0 && bid < p.E) ? ws : -1;
                        tab.id[a] = bid;
                        tab.sel_v[a] = bv;
                        tab.base[a] = (slot >= 0 && slot < p.S) ? p.slots + (size_t)slot * p.expert_bytes : nullptr;
                        tc::mbar_arrive(&rb.assigned[a]);
                    }
                }
            }
        };
        if (p.E <= 32) route_tokens(std::integral_constant<int, 1>{});
        else if (p.E <= 64) route_tokens(std::integral_constant<int, 2>{});
        else if (p.E <= 128) route_tokens(std::integral_constant<int, 4>{});
        else route_tokens(std::integral_constant<int, 8>{});
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&rb.ranked);
    }
    if (warp == 0) {
        if (p.logits != nullptr) {
            // every assignment's weight in one pass (lane a: assignment a)
            const bool ranked = tc::mbar_wait_suspend(&rb.ranked, 0u, err, 8u);
            const float sv = (ranked && lane < A) ? tab.sel_v[lane] : __int_as_float(0x7fc00000);
            const float wv = softmax_assign(sv, p.k, A);
            if (lane < A) tab.w[lane] = wv;
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&rb.routed);
            if (blockIdx.x == 0) {
                int my_id = MOE_MAX_EXPERTS;
                if (lane < A) {
                    my_id = ranked ? tab.id[lane] : -1;
                    p.r_ids[lane] = my_id;
                    p.r_w[lane] = tab.w[lane];
                }
                plan_warp(my_id, A, p.E, p.r_counts, p.r_offsets, p.r_perm, p.r_inv);
            }
        } else {
            for (int a = lane; a < A; a += 32) {
                const int e = p.ids[a];
                const int s = (e >= 0 && e < p.E) ? p.slot_of[e] : -1;
                tab.id[a] = e;
                tab.base[a] = (s >= 0 && s < p.S) ? p.slots + (size_t)s * p.expert_bytes : nullptr;
                tab.w[a] = p.w[a];
            }
            __syncwarp();
            if (lane == 0) {
                for (int a = 0; a < A; ++a) tc::mbar_arrive(&rb.assigned[a]);
                tc::mbar_arrive(&rb.routed);
            }
        }
    } else if (warp == 1) {
        // ---- copy producer (lane 0): gate/up rows and down blocks of the
        // CTA's items in the order the consumers take them, each as soon as
        // its assignment is known and its ring slot is free ----
        if (lane == 0) {
        // per ring: next slot, its phase, and the next item's (assignment, row)
        const int it0 = g0 * kGroup;
        const int ai0 = it0 / p.I;
        const int a0 = kSkip ? nth_active(act, ai0) : ai0;
        int gu_slot = 0, gu_a = a0, gu_r = it0 - ai0 * p.I;
        uint32_t gu_ph = 0;
        int d_slot = 0, d_a = a0, d_r = gu_r;
        uint32_t d_ph = 0;
        auto issue_gu = [&](int n) -> bool {
            const int slot = gu_slot;
            const uint32_t ph = gu_ph;
            const int a = gu_a, r = gu_r;
            if (++gu_slot == n_gu) { gu_slot = 0; gu_ph ^= 1u; }
            if ((gu_r += kGroup) == p.I) { gu_r = 0; gu_a = kSkip ? next_active(act, gu_a) : gu_a + 1; }
            if (!tc::mbar_wait_suspend(&rb.empty_gu[slot], ph ^ 1u, err, 4u)) return false;
            if (n == 0 && p.stall) return true;   // test hook: the first item never lands
            if (!tc::mbar_wait_suspend(&rb.assigned[a], 0u, err, 4u)) return false;
            const uint8_t* eb = tab.base[a];
            uint8_t* dst = ring_gu + (size_t)slot * gu_bytes;
            for (int q = 0; q < kGuGroups; ++q) {
                if (eb != nullptr) {
                    const uint8_t* g = eb + Layout::gate_row(r + kRowsPerGroup * q) * row_bytes;
                    const uint32_t part = uint32_t(kRowsPerGroup * row_bytes);
                    tc::mbar_arrive_expect_tx(&rb.full_gu[slot][q], 2 * part);
                    bulk_copy_g2s(dst + (size_t)kRowsPerGroup * q * row_bytes, g, part, &rb.full_gu[slot][q]);
                    bulk_copy_g2s(dst + (size_t)(kGroup + kRowsPerGroup * q) * row_bytes, g + Layout::kChunk * row_bytes,
                                  part, &rb.full_gu[slot][q]);
                } else {
                    tc::mbar_arrive(&rb.full_gu[slot][q]);
                }
            }
            return true;
        };
        auto issue_d = [&](int n) -> bool {
            const int slot = d_slot;
            const uint32_t ph = d_ph;
            const int a = d_a, r = d_r;
            if (++d_slot == n_d) { d_slot = 0; d_ph ^= 1u; }
            if ((d_r += kGroup) == p.I) { d_r = 0; d_a = kSkip ? next_active(act, d_a) : d_a + 1; }
            if (!tc::mbar_wait_suspend(&rb.empty_d[slot], ph ^ 1u, err, 4u)) return false;
            if (n == 0 && p.stall) return true;
            if (!tc::mbar_wait_suspend(&rb.assigned[a], 0u, err, 4u)) return false;
            const uint8_t* eb = tab.base[a];
            if (eb != nullptr) {
                tc::mbar_arrive_expect_tx(&rb.full_d[slot], dt_bytes);
                bulk_copy_g2s(ring_d + (size_t)slot * dt_slot, eb + p.dt_off + (size_t)(r / kGroup) * p.dt_stride,
                              dt_bytes, &rb.full_d[slot]);
            } else {
                tc::mbar_arrive(&rb.full_d[slot]);
            }
            return true;
        };
            bool ok = true;
            int next_gu = 0, next_d = 0;
            while (ok && (next_gu < cnt || next_d < cnt)) {
                if (next_gu < cnt && (next_gu <= next_d || next_d >= cnt)) {
                    ok = issue_gu(next_gu);
                    ++next_gu;
                } else {
                    ok = issue_d(next_d);
                    ++next_d;
                }
            }
        }
    } else {
        // ---- consumers (warps 2..17) ----
        uint4* xs = reinterpret_cast<uint4*>(smem);
        float* xe = reinterpret_cast<float*>(smem + (size_t)p.T * nbx * 64);
        for (int c = threadIdx.x - 64; c < p.T * nbx; c += kConsumers) {
            const int t = c / nbx, b = c - t * nbx;
            stage_block_f16(p.x + (size_t)t * p.H, xs + (size_t)t * nbx * 4, b, xe + t * nbx);
        }
        named_bar_consumers();
        const int j = warp - 2;
        const int grp = j / kRowsPerGroup;
        const int ct = threadIdx.x - 64;
        float y[NN];
#pragma unroll
        for (int m = 0; m < NN; ++m) y[m] = 0.0f;
        int cur_a = -1;
        bool routed = false;
        // Lanes 4i..4i+3 of a warp own four consecutive rows (H is a
        // multiple of 32, so a quad is all inside or all outside [0, H));
        // lane 4i adds the quad with one float4 atomic.
        auto flush = [&](int a) {
            if (a < 0) return;
            if (!routed) routed = tc::mbar_wait_suspend(&rb.routed, 0u, err, 8u);
            const float wa = routed ? tab.w[a] : __int_as_float(0x7fc00000);
            float* dst = (p.accumulate ? p.out : p.acc) + (size_t)(a / p.k) * p.H;
#pragma unroll
            for (int m = 0; m < NN; ++m) {
                const int n = ct + kConsumers * m;
                const float v = wa * y[m];
                const float v1 = __shfl_down_sync(0xffffffffu, v, 1);
                const float v2 = __shfl_down_sync(0xffffffffu, v, 2);
                const float v3 = __shfl_down_sync(0xffffffffu, v, 3);
                if ((lane & 3) == 0 && n < p.H) atomicAdd(reinterpret_cast<float4*>(dst + n), make_float4(v, v1, v2, v3));
                y[m] = 0.0f;
            }
        };
        // item state carried from item to item: assignment and row, ring
        // slots and phases, the token's staged x, the h-exponent word
        const int it0 = g0 * kGroup;
        const int ai0 = it0 / p.I;
        int a = kSkip ? nth_active(act, ai0) : ai0, r = it0 - ai0 * p.I;
        int sg = 0, sd = 0, hm = 0;
        uint32_t ph_gu = 0, ph_d = 0;
        const uint4* xt = xs;
        const float* et = xe;
        for (int n = 0; n < cnt; ++n) {
            if (a != cur_a) {
                flush(cur_a);
                cur_a = a;
                const int t = a / p.k;
                xt = xs + (size_t)t * nbx * 4;
                et = xe + t * nbx;
            }
            // (1) h for row r0 + j, once this warp's group of rows has landed
            const bool got = tc::mbar_wait_suspend(&rb.full_gu[sg][grp], ph_gu, err, 8u);
            const uint8_t* eb = tab.base[a];
            const bool have = got && eb != nullptr;
            const uint8_t* sl = ring_gu + (size_t)sg * gu_bytes;
            float hj = __int_as_float(0x7fc00000);
            if (have) {
                const uint8_t* g = sl + (size_t)j * row_bytes;
                const uint8_t* u = g + kGroup * row_bytes;
                float ag = 0.0f, au = 0.0f;
#pragma unroll
                for (int i = 0; i < NG; ++i) {
                    const int b = lane + 32 * i;
                    // NG = ceil(nbx / 32): only the last group has lanes past nbx
                    if (i < NG - 1 || b < nbx) {
                        const uint4 cg = *reinterpret_cast<const uint4*>(g + 16 * b);
                        const uint4 cu = *reinterpret_cast<const uint4*>(u + 16 * b);
                        const float xf = et[b];
                        float dg, du;
                        block_dot2_f16(cg, cu, xt, b, dg, du);
                        ag = fmaf(dg, e8m0_lut[g[p.H / 2 + b]] * xf, ag);
                        au = fmaf(du, e8m0_lut[u[p.H / 2 + b]] * xf, au);
                    }
                }
                __syncwarp();
                if (lane == 0 && got) tc::mbar_arrive(&rb.empty_gu[sg]);
                ag = warp_sum(ag);
                au = warp_sum(au);
                // fast exponential and division: a few fp32 ulps, far below
                // the bf16 rounding of h that follows
                const float silu = __fdividef(ag, 1.0f + __expf(-ag));
                hj = __bfloat162float(__float2bfloat16_rn(silu * au));
            } else if (lane == 0 && got) {
                tc::mbar_arrive(&rb.empty_gu[sg]);
            }
            if (lane == 0) {
                hval[n & 1][j] = hj;
                atomicMax(&hmax_bits[hm], __float_as_uint(fabsf(hj)));
                const __nv_bfloat16 hb = __float2bfloat16_rn(hj);
                p.h[(size_t)(g0 + n) * kGroup + j] = *reinterpret_cast<const uint16_t*>(&hb);
            }
            named_bar_consumers();
            // the word of item n - 1 was last read before this barrier and is
            // next written after the following one
            if (ct == 0 && n >= 1) hmax_bits[hm == 0 ? 2 : hm - 1] = 0u;
            // (2) y[n] += W[n][r0..r0+15] . h[r0..r0+15], once the block has landed
            const bool gotd = tc::mbar_wait_suspend(&rb.full_d[sd], ph_d, err, 8u);
            if (have && gotd) {
                // the 16 h values as f16 pairs under one power-of-2 scale (bf16 -> f16 is exact)
                float hv[kGroup];
#pragma unroll
                for (int i = 0; i < kGroup / 4; ++i) {
                    const float4 v4 = reinterpret_cast<const float4*>(hval[n & 1])[i];
                    hv[4 * i] = v4.x;
                    hv[4 * i + 1] = v4.y;
                    hv[4 * i + 2] = v4.z;
                    hv[4 * i + 3] = v4.w;
                }
                // scale 2^-e with e = exponent of the item's largest |h| minus 14
                const uint32_t hbits = hmax_bits[hm];
                const int ef = int(hbits >> 23);
                float mul, hf;
                if (ef >= 15 && ef <= 254) {
                    mul = __uint_as_float(uint32_t(268 - ef) << 23);
                    hf = __uint_as_float(uint32_t(ef - 14) << 23);
                } else {
                    const int e = (hbits == 0u) ? 0 : (ef == 0 ? -126 - 14 : ef - 127 - 14);
                    mul = ldexpf(1.0f, -e);
                    hf = ldexpf(1.0f, e);
                }
                uint32_t h2[kGroup / 2];
#pragma unroll
                for (int i = 0; i < kGroup / 2; ++i) {
                    const __half2 hh = __floats2half2_rn(hv[2 * i] * mul, hv[2 * i + 1] * mul);
                    h2[i] = *reinterpret_cast<const uint32_t*>(&hh);
                }
                const uint8_t* codes = ring_d + (size_t)sd * dt_slot;
                const uint8_t* scales = codes + (size_t)p.H * (kGroup / 2);
#pragma unroll
                for (int m = 0; m < NN; ++m) {
                    const int nn = ct + kConsumers * m;
                    // NN = ceil(H / 512): only the last row group reaches past H
                    if (m < NN - 1 || nn < p.H) {
                        const uint2 cw = *reinterpret_cast<const uint2*>(codes + (size_t)nn * (kGroup / 2));
                        uint32_t w0[4], w1[4];
                        e2m1x8_f16(cw.x, w0);
                        e2m1x8_f16(cw.y, w1);
                        float s0 = 0.0f, s1 = 0.0f;
                        fma2_f16_f32(s0, s1, w0[0], h2[0]);
                        fma2_f16_f32(s0, s1, w0[1], h2[1]);
                        fma2_f16_f32(s0, s1, w0[2], h2[2]);
                        fma2_f16_f32(s0, s1, w0[3], h2[3]);
                        fma2_f16_f32(s0, s1, w1[0], h2[4]);
                        fma2_f16_f32(s0, s1, w1[1], h2[5]);
                        fma2_f16_f32(s0, s1, w1[2], h2[6]);
                        fma2_f16_f32(s0, s1, w1[3], h2[7]);
                        y[m] = fmaf(s0 + s1, e8m0_lut[scales[nn]] * hf, y[m]);
                    }
                }
            } else {
#pragma unroll
                for (int m = 0; m < NN; ++m) y[m] = __int_as_float(0x7fc00000);
            }
            __syncwarp();
            if (lane == 0 && gotd) tc::mbar_arrive(&rb.empty_d[sd]);
            if ((r += kGroup) == p.I) { r = 0; a = kSkip ? next_active(act, a) : a + 1; }
            if (++sg == n_gu) { sg = 0; ph_gu ^= 1u; }
            if (++sd == n_d) { sd = 0; ph_d ^= 1u; }
            hm = (hm == 2) ? 0 : hm + 1;
        }
        flush(cur_a);
    }

    // ---- completion: the last CTA to finish moves the sums to `out` ----
    if (p.accumulate) return;  // the partial sums went to out directly
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned done = atomicAdd(p.ctl, 1u);
        last_cta = (done == unsigned(G) - 1u);
    }
    __syncthreads();
    if (last_cta) {
        __threadfence();
        const int n4 = p.T * p.H / 4;
        float4* acc4 = reinterpret_cast<float4*>(p.acc);
        float4* out4 = reinterpret_cast<float4*>(p.out);
        for (int i = threadIdx.x; i < n4; i += kThreads) {
            out4[i] = __ldcg(acc4 + i);
            acc4[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
        if (threadIdx.x == 0) p.ctl[0] = 0u;
    }
}

}  // namespace

// Shared memory of the fused kernel: the activation staging, then the ring
// of gate/up rows (16 gate + 16 up rows per slot), then the ring of down
// blocks.
static size_t staging_bytes(int T, int H) {
    return round_up(size_t(T) * H * 2 + size_t(T) * (H / 32) * 4, 128);
}
static size_t gu_slot_bytes(const Layout& L) { return 2 * size_t(kGroup) * L.rs_gu; }
static size_t d_slot_bytes(const Layout& L) { return round_up(size_t(L.H) * (kGroup / 2 + 1), 128); }

constexpr size_t kFusedSmemBudget = 216 * 1024;

// Ring depths: the deepest gate/up ring that fits (at most 8 slots, at
// least 2), then the deepest down ring beside it (2 up to as many slots).
// At the GPT-OSS shape that is 3 and 2; small shapes get 8 and 8, so their
// many small items keep enough bytes in flight.
static bool fused_rings(int T, const Layout& L, int* n_gu, int* n_d, size_t* bytes) {
    const size_t st = staging_bytes(T, L.H);
    for (int g = kMaxGuSlots; g >= 2; --g)
        for (int d = g < kMaxDSlots ? g : kMaxDSlots; d >= 2; --d) {
            const size_t need = st + g * gu_slot_bytes(L) + d * d_slot_bytes(L);
            if (need <= kFusedSmemBudget) {
                *n_gu = g;
                *n_d = d;
                *bytes = need;
                return true;
            }
        }
    return false;
}

size_t decode_fused_smem(int T, int k, int H, int I) {
    Layout L;
    if (!Layout::make(H, I, &L) || T * k > kMaxAssign || I % kGroup || Layout::kDtCols != kGroup || H > 4096) return 0;
    int g, d;
    size_t bytes;
    return fused_rings(T, L, &g, &d, &bytes) ? bytes : 0;
}

// Test hook (moe_debug_stall_next_decode): launches still to stall.
std::atomic<int> g_stall_decode{0};

int launch_decode_fused_impl(const FfnArgs& a, void* ws, cudaStream_t s, const RouteOut* ro) {
    const Layout& L = *a.L;
    DeviceInfo di;
    int rc = current_device_info(&di);
    if (rc != MOE_OK) return rc;
    if (decode_fused_smem(a.T, a.k, L.H, L.I) == 0) return MOE_ERR_UNSUPPORTED;
    int n_gu = 0, n_d = 0;
    size_t smem = 0;
    if (!fused_rings(a.T, L, &n_gu, &n_d, &smem)) return MOE_ERR_UNSUPPORTED;
    const size_t st = staging_bytes(a.T, L.H);
    const size_t d_off = st + size_t(n_gu) * gu_slot_bytes(L);
    FusedParams p;
    p.stall = 0;
    for (int n = g_stall_decode.load(); n > 0; n = g_stall_decode.load())
        if (g_stall_decode.compare_exchange_weak(n, n - 1)) {
            p.stall = 1;
            break;
        }
    p.slots = a.slots;
    p.expert_bytes = a.expert_bytes;
    p.S = a.S;
    p.E = a.E;
    p.H = L.H;
    p.I = L.I;
    p.k = a.k;
    p.T = a.T;
    p.rs_gu = L.rs_gu;
    p.dt_off = L.dt_off;
    p.dt_stride = L.dt_stride;
    p.x = a.x;
    p.ids = a.ids;
    p.w = a.w;
    p.slot_of = a.slot_of;
    p.ctl = static_cast<unsigned*>(ws);
    p.h = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + 256);
    p.acc = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + decode_acc_offset(a.T, a.k, L.I));
    p.out = a.out;
    p.accumulate = a.accumulate ? 1 : 0;
    p.logits = ro ? ro->logits : nullptr;
    p.r_ids = ro ? ro->ids : nullptr;
    p.r_w = ro ? ro->w : nullptr;
    p.r_counts = ro ? ro->counts : nullptr;
    p.r_offsets = ro ? ro->offsets : nullptr;
    p.r_perm = ro ? ro->perm : nullptr;
    p.r_inv = ro ? ro->inv : nullptr;
    if (ro && (a.T * a.k > 32 || a.E > MOE_MAX_EXPERTS)) return MOE_ERR_UNSUPPORTED;
    const int ng = (L.H / 32 + 31) / 32, nn = (L.H + kConsumers - 1) / kConsumers;
    using Kern = void (*)(FusedParams, int, int, int, int);
    struct Variant {
        int ng, nn;
        bool skip;
        Kern kern;
    };
    // ng = ceil(H / 1024) groups of 32 scale blocks per row, nn = ceil(H / 512)
    // outputs per consumer thread; H <= 4096 gives exactly these pairs.  The
    // skip-absent launches have kernels of their own, so the others keep
    // their code exactly.
    static const Variant variants[] = {
        {1, 1, false, decode_fused_kernel<1, 1, false>}, {1, 2, false, decode_fused_kernel<1, 2, false>},
        {2, 3, false, decode_fused_kernel<2, 3, false>}, {2, 4, false, decode_fused_kernel<2, 4, false>},
        {3, 5, false, decode_fused_kernel<3, 5, false>}, {3, 6, false, decode_fused_kernel<3, 6, false>},
        {4, 7, false, decode_fused_kernel<4, 7, false>}, {4, 8, false, decode_fused_kernel<4, 8, false>},
        {1, 1, true, decode_fused_kernel<1, 1, true>},   {1, 2, true, decode_fused_kernel<1, 2, true>},
        {2, 3, true, decode_fused_kernel<2, 3, true>},   {2, 4, true, decode_fused_kernel<2, 4, true>},
        {3, 5, true, decode_fused_kernel<3, 5, true>},   {3, 6, true, decode_fused_kernel<3, 6, true>},
        {4, 7, true, decode_fused_kernel<4, 7, true>},   {4, 8, true, decode_fused_kernel<4, 8, true>},
    };
    constexpr int kVariants = int(sizeof(variants) / sizeof(variants[0]));
    static DeviceOnce attr_set[kVariants];
    int vi = -1;
    for (int i = 0; i < kVariants; ++i)
        if (variants[i].ng == ng && variants[i].nn == nn && variants[i].skip == a.skip_absent) vi = i;
    if (vi < 0) return MOE_ERR_UNSUPPORTED;
    const Kern kern = variants[vi].kern;
    if (di.device < 0 || di.device >= 64) return MOE_ERR_UNSUPPORTED;
    if (!attr_set[vi].done(di.device)) {
        MOE_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kFusedSmemBudget)));
        attr_set[vi].mark(di.device);
    }
    // programmatic stream serialisation: the kernel may launch while the
    // previous kernel in the stream finishes; it waits for it (griddepcontrol)
    // before touching global memory
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(di.sms));
    cfg.blockDim = dim3(unsigned(kThreads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, p, n_gu, n_d, int(st), int(d_off)));
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

int launch_decode_fused(const FfnArgs& a, void* ws, cudaStream_t s) { return launch_decode_fused_impl(a, ws, s, nullptr); }

int launch_decode_layer(const FfnArgs& a, const RouteOut& ro, void* ws, cudaStream_t s) {
    return launch_decode_fused_impl(a, ws, s, &ro);
}

}  // namespace moe
