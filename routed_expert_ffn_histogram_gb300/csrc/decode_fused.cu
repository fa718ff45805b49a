// Decode path, fused: the whole expert FFN of one layer (gate/up + SwiGLU,
// down + weighted combine) in one persistent cooperative kernel.
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
// down product on bf16(h), combine sum_j w_j * y_j in ascending j.
//
// Shape: one CTA per SM, 24 warps each, all co-resident (cooperative
// launch).  Each CTA owns a contiguous range of (assignment, row) items of
// the gate/up product and a contiguous range of output rows of the down
// product, and first asks L2 to prefetch exactly those weight bytes
// (cp.async.bulk.prefetch), gate/up first: HBM then streams the layer's
// experts at full rate whatever the warps are doing, and the warps' loads
// meet the data in L2.
//   phase 1  a warp takes one item at a time: the gate row and the up row
//            (32 rows apart in the packed layout), one 16-byte load = one MX
//            block per lane; x is staged once per CTA in shared memory as
//            f16 scaled per 32-block by a power of two (exact for every
//            value within 2^-31 of the block maximum) in XOR-swizzled
//            16-byte chunks; E2M1 pairs become f16x2 by hardware conversion
//            and multiply-add into fp32 (products exact); lane 0 writes
//            bf16(silu(g) * u).
//   barrier  bounded grid barrier (arrival counter zeroed before launch).
//   phase 2  h of a token staged per CTA the same way; a warp takes an
//            output row, reads that row of all k experts, and folds
//            w_j * y_j in rank order.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>

#include "internal.h"
#include "route_warp.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int kGroup = 16;             // row pairs per ring slot (one bulk copy each for gate and up)
constexpr int kThreads = 32 * (kGroup + 1);  // warp 0: copy producer; warps 1..16: one row pair each
static_assert(Layout::kChunk % kGroup == 0, "a group of gate rows stays inside one interleave chunk");
constexpr int kMaxSlots = 16;
constexpr int kMaxRows2 = 64;          // output rows per CTA in phase 2
constexpr int kWarps = kThreads / 32;
constexpr uint32_t kBarrierLimit = 1u << 23;  // polls (~1 s) before the grid barrier gives up

__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 2^(e - 127) for an integer biased exponent e (any range), as fp32.
__device__ __forceinline__ float pow2_biased(int e) {
    if (e >= 1 && e <= 254) return __int_as_float(e << 23);
    return ldexpf(1.0f, e - 127);
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

// Dot of one MX block (16 code bytes = 32 elements) with staged block b.
// Eight independent accumulation chains keep the FMA latency hidden.
__device__ __forceinline__ float block_dot_f16(const uint4 c, const uint4* __restrict__ xs, int b) {
    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 xv = xs[hswz(b, q)];
        uint32_t wv[4];
        e2m1x8_f16(cw[q], wv);
        fma2_f16_f32(a[0], a[1], wv[0], xv.x);
        fma2_f16_f32(a[2], a[3], wv[1], xv.y);
        fma2_f16_f32(a[4], a[5], wv[2], xv.z);
        fma2_f16_f32(a[6], a[7], wv[3], xv.w);
    }
    return ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
}

// Two rows (gate, up) against the same staged block b.
__device__ __forceinline__ void block_dot2_f16(const uint4 cg, const uint4 cu, const uint4* __restrict__ xs,
                                               int b, float& dg, float& du) {
    const uint32_t wg[4] = {cg.x, cg.y, cg.z, cg.w};
    const uint32_t wu[4] = {cu.x, cu.y, cu.z, cu.w};
    float g[4] = {0.f, 0.f, 0.f, 0.f}, u[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 xv = xs[hswz(b, q)];
        uint32_t fg[4], fu[4];
        e2m1x8_f16(wg[q], fg);
        e2m1x8_f16(wu[q], fu);
        fma2_f16_f32(g[0], g[1], fg[0], xv.x);
        fma2_f16_f32(u[0], u[1], fu[0], xv.x);
        fma2_f16_f32(g[2], g[3], fg[1], xv.y);
        fma2_f16_f32(u[2], u[3], fu[1], xv.y);
        fma2_f16_f32(g[0], g[1], fg[2], xv.z);
        fma2_f16_f32(u[0], u[1], fu[2], xv.z);
        fma2_f16_f32(g[2], g[3], fg[3], xv.w);
        fma2_f16_f32(u[2], u[3], fu[3], xv.w);
    }
    dg = (g[0] + g[1]) + (g[2] + g[3]);
    du = (u[0] + u[1]) + (u[2] + u[3]);
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
// One thread per block.
__device__ __forceinline__ void stage_block_f16(const uint16_t* __restrict__ src, uint4* dst, int b,
                                                int* exps) {
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
    exps[b] = e;
}

struct FusedParams {
    const uint8_t* slots;
    size_t expert_bytes;
    int S, E, H, I, k, T;
    size_t rs_gu, rs_d, d_off;
    const uint16_t* x;
    const int32_t* ids;
    const float* w;
    const int32_t* slot_of;
    uint16_t* h;       // bf16 [T*k][I]
    float* out;        // fp32 [T][H]
    unsigned* bar;     // [0] arrivals (zero when idle), [1] generation, [2] error bits
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

__device__ __forceinline__ const uint8_t* expert_of(const FusedParams& p, int a) {
    const int e = p.ids[a];
    if (e < 0 || e >= p.E) return nullptr;
    const int s = p.slot_of[e];
    if (s < 0 || s >= p.S) return nullptr;
    return p.slots + (size_t)s * p.expert_bytes;
}

// Per-CTA table of the routed assignments, filled once so the work loops
// never wait on dependent loads of ids / slot_of / w.
struct AssignTable {
    int slot_of[MOE_MAX_EXPERTS];
    const uint8_t* base[kMaxAssign];
    float w[kMaxAssign];
    float sel_v[kMaxAssign];
    int id[kMaxAssign];
};

// Sense-reversing grid barrier in the workspace's first bytes: bar[0]
// counts arrivals and is reset to zero by the last arriver, which then
// advances the generation bar[1] that the others wait on; bar[2] collects
// error bits.  bar[0] must be zero when the workspace is first used; the
// kernel leaves it zero.  A wait that runs out (about one second) sets an
// error bit instead of spinning on.
__device__ bool grid_barrier(unsigned* bar, unsigned G, int* ok_smem) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        unsigned gen;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(gen) : "l"(bar + 1) : "memory");
        const unsigned arrived = atomicAdd(bar, 1u);
        int ok = 1;
        if (arrived == G - 1) {
            atomicExch(bar, 0u);
            __threadfence();
            asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(bar + 1), "r"(gen + 1) : "memory");
        } else {
            for (uint32_t i = 0;; ++i) {
                unsigned v;
                asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(bar + 1) : "memory");
                if (v != gen) break;
                if (i >= kBarrierLimit) {
                    atomicOr(bar + 2, 1u);
                    ok = 0;
                    break;
                }
                if (i > 256) __nanosleep(32);
            }
        }
        __threadfence();
        *ok_smem = ok;
    }
    __syncthreads();
    return *ok_smem != 0;
}

__device__ __forceinline__ void prefetch_l2(const void* p, size_t bytes) {
    if (bytes >= 16)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(uint32_t(bytes & ~size_t(15)))
                     : "memory");
}

__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            tc::smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
        : "memory");
}

template <int NG, int ND>
__global__ void __launch_bounds__(kThreads, 1) decode_fused_kernel(FusedParams p, int slots, int ring_off) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int ok_smem;
    __shared__ AssignTable tab;
    __shared__ __align__(8) uint64_t full[kMaxSlots];
    __shared__ __align__(8) uint64_t empty[kMaxSlots];
    __shared__ __align__(8) uint64_t down_full;
    __shared__ float ypart[kMaxRows2][kMaxAssign];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = gridDim.x;
    const int A = p.T * p.k;
    volatile uint32_t* err = p.bar + 2;
    if (p.logits != nullptr) {
        // routing in every CTA: warp 0 ranks each token's logits while the
        // other warps fetch the slot map
        if (warp == 0) {
            for (int t = 0; t < p.T; ++t) {
                float sv;
                int sid;
                const float* row = p.logits + (size_t)t * p.E;
                if (p.E <= 32) topk_warp<1>(row, p.E, p.k, sv, sid);
                else if (p.E <= 64) topk_warp<2>(row, p.E, p.k, sv, sid);
                else if (p.E <= 128) topk_warp<4>(row, p.E, p.k, sv, sid);
                else topk_warp<8>(row, p.E, p.k, sv, sid);
                if (lane < p.k) {
                    tab.id[t * p.k + lane] = sid;
                    tab.sel_v[t * p.k + lane] = sv;
                }
            }
        } else {
            for (int e = threadIdx.x - 32; e < p.E; e += kThreads - 32) tab.slot_of[e] = p.slot_of[e];
        }
        __syncthreads();
        for (int a = threadIdx.x; a < A; a += kThreads) {
            const int e = tab.id[a];
            const int sl = (e >= 0 && e < p.E) ? tab.slot_of[e] : -1;
            tab.base[a] = (sl >= 0 && sl < p.S) ? p.slots + (size_t)sl * p.expert_bytes : nullptr;
        }
    } else {
        for (int a = threadIdx.x; a < A; a += kThreads) {
            tab.base[a] = expert_of(p, a);
            tab.w[a] = p.w[a];
        }
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < slots; ++i) {
            tc::mbar_init(&full[i], 1);
            tc::mbar_init(&empty[i], kGroup);
        }
        tc::mbar_init(&down_full, 1);
        tc::fence_barrier_init();
    }
    __syncthreads();

    // This CTA's work: a contiguous range of groups of kGroup (assignment,
    // row) gate/up items -- kGroup consecutive gate rows, and the matching up
    // rows, are contiguous in the packed layout -- and a contiguous range of
    // output rows for the down product.
    const int groups = A * p.I / kGroup;
    const int perg = (groups + G - 1) / G;
    const int g0 = min(groups, (int)blockIdx.x * perg), g1 = min(groups, g0 + perg);
    const int per2 = (p.H + G - 1) / G;
    const int r0 = min(p.H, (int)blockIdx.x * per2), r1 = min(p.H, r0 + per2);
    const int nbx = p.H / 32;
    const size_t row_bytes = p.rs_gu;
    const size_t slot_bytes = 2 * kGroup * row_bytes;
    uint8_t* ring = smem + ring_off;

    if (warp == 0) {
        // ---- producer: the down rows this CTA needs go to L2 first; then
        //      gate/up rows stream through the ring, kGroup pairs per slot ----
        if (lane == 0) {
            if (r1 > r0)
                for (int a = 0; a < A; ++a) {
                    const uint8_t* eb = tab.base[a];
                    if (eb != nullptr) prefetch_l2(eb + p.d_off + (size_t)r0 * p.rs_d, size_t(r1 - r0) * p.rs_d);
                }
            for (int n = 0; g0 + n < g1; ++n) {
                const int slot = n % slots;
                const uint32_t phase = uint32_t(n / slots) & 1u;
                if (!tc::mbar_wait(&empty[slot], phase ^ 1u, err, 4u)) break;
                const int it = (g0 + n) * kGroup;
                const int a = it / p.I, r = it - a * p.I;
                const uint8_t* eb = tab.base[a];
                if (eb != nullptr) {
                    const uint8_t* g = eb + Layout::gate_row(r) * p.rs_gu;
                    tc::mbar_arrive_expect_tx(&full[slot], uint32_t(slot_bytes));
                    bulk_copy_g2s(ring + (size_t)slot * slot_bytes, g, uint32_t(kGroup * row_bytes), &full[slot]);
                    bulk_copy_g2s(ring + (size_t)slot * slot_bytes + kGroup * row_bytes, g + Layout::kChunk * p.rs_gu,
                                  uint32_t(kGroup * row_bytes), &full[slot]);
                } else {
                    tc::mbar_arrive(&full[slot]);
                }
            }
            // once every slot is released, this CTA's down rows of all
            // assignments are copied into the ring: they land while the grid
            // barrier is in progress, and phase 2 reads shared memory only.
            const int issued = g1 - g0;
            bool free_all = true;
            for (int n = issued; n < issued + slots && free_all; ++n)
                free_all = tc::mbar_wait(&empty[n % slots], (uint32_t(n / slots) & 1u) ^ 1u, err, 4u);
            const size_t dbytes = size_t(r1 - r0) * p.rs_d;
            if (free_all && r1 > r0) {
                tc::mbar_arrive_expect_tx(&down_full, uint32_t(dbytes * A));
                for (int a = 0; a < A; ++a) {
                    const uint8_t* eb = tab.base[a];
                    const uint8_t* src = eb != nullptr ? eb + p.d_off + (size_t)r0 * p.rs_d : nullptr;
                    if (src != nullptr) bulk_copy_g2s(ring + (size_t)a * dbytes, src, uint32_t(dbytes), &down_full);
                    else asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(tc::smem_u32(&down_full)),
                                      "r"(uint32_t(dbytes)) : "memory");
                }
            } else {
                tc::mbar_arrive(&down_full);
            }
        }
    } else {
        // ---- consumers: warp w computes row pair w - 1 of every slot ----
        uint4* xs = reinterpret_cast<uint4*>(smem);
        int* xe = reinterpret_cast<int*>(smem + (size_t)p.T * nbx * 64);
        for (int c = threadIdx.x - 32; c < p.T * nbx; c += kThreads - 32) {
            const int t = c / nbx, b = c - t * nbx;
            stage_block_f16(p.x + (size_t)t * p.H, xs + (size_t)t * nbx * 4, b, xe + t * nbx);
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kThreads - 32) : "memory");
        if (p.logits != nullptr && warp == 1) {
            // softmax weights (needed only by phase 2), computed while the first
            // copies are in flight; CTA 0 also writes the routing outputs
            int my_id = MOE_MAX_EXPERTS;
            for (int t = 0; t < p.T; ++t) {
                const int a0 = t * p.k;
                const float sv = lane < p.k ? tab.sel_v[a0 + lane] : 0.0f;
                const float wv = softmax_lane(sv, p.k);
                if (lane < p.k) tab.w[a0 + lane] = wv;
            }
            __syncwarp();
            if (blockIdx.x == 0) {
                if (lane < A) {
                    my_id = tab.id[lane];
                    p.r_ids[lane] = my_id;
                    p.r_w[lane] = tab.w[lane];
                }
                plan_warp(my_id, A, p.E, p.r_counts, p.r_offsets, p.r_perm, p.r_inv);
            }
        }
        const int j = warp - 1;
        for (int n = 0; g0 + n < g1; ++n) {
            const int slot = n % slots;
            const uint32_t phase = uint32_t(n / slots) & 1u;
            const bool got = tc::mbar_wait(&full[slot], phase, err, 8u);
            const int it = (g0 + n) * kGroup + j;
            const int a = it / p.I, r = it - a * p.I;
            const uint8_t* eb = tab.base[a];
            if (!got || eb == nullptr) {
                if (lane == 0) p.h[(size_t)a * p.I + r] = 0x7fc0;
            } else {
                const uint8_t* g = ring + (size_t)slot * slot_bytes + (size_t)j * row_bytes;
                const uint8_t* u = g + kGroup * row_bytes;
                const int t = a / p.k;
                const uint4* xt = xs + (size_t)t * nbx * 4;
                const int* et = xe + t * nbx;
                float ag = 0.0f, au = 0.0f;
#pragma unroll
                for (int i = 0; i < NG; ++i) {
                    const int b = lane + 32 * i;
                    if (b < nbx) {
                        const uint4 cg = *reinterpret_cast<const uint4*>(g + 16 * b);
                        const uint4 cu = *reinterpret_cast<const uint4*>(u + 16 * b);
                        const int e = et[b];
                        float dg, du;
                        block_dot2_f16(cg, cu, xt, b, dg, du);
                        ag = fmaf(dg, pow2_biased(int(g[p.H / 2 + b]) + e), ag);
                        au = fmaf(du, pow2_biased(int(u[p.H / 2 + b]) + e), au);
                    }
                }
                ag = warp_sum(ag);
                au = warp_sum(au);
                if (lane == 0) {
                    const float silu = ag / (1.0f + expf(-ag));
                    const __nv_bfloat16 hv = __float2bfloat16_rn(silu * au);
                    p.h[(size_t)a * p.I + r] = *reinterpret_cast<const uint16_t*>(&hv);
                }
            }
            __syncwarp();
            if (lane == 0 && got) tc::mbar_arrive(&empty[slot]);
        }
    }

    const bool ok0 = grid_barrier(p.bar, (unsigned)G, &ok_smem);
    const bool ok = ok0 && tc::mbar_wait(&down_full, 0, err, 16u);

    // ---- phase 2: down + weighted combine (rows prefetched into L2) ----
    // Items are (row, expert) pairs; y of each lands in shared memory and
    // one pass per row folds w_j * y_j in rank order.
    constexpr int kWarpsAll = kThreads / 32;
    uint4* hs = reinterpret_cast<uint4*>(smem);
    const int nbh = p.I / 32;
    int* he = reinterpret_cast<int*>(smem + (size_t)p.k * nbh * 64);
    const int nrows = r1 - r0;
    for (int t = 0; t < p.T; ++t) {
        __syncthreads();
        for (int c = threadIdx.x; c < p.k * nbh; c += kThreads) {
            const int jj = c / nbh, b = c - jj * nbh;
            stage_block_f16(p.h + ((size_t)t * p.k + jj) * p.I, hs + (size_t)jj * nbh * 4, b, he + jj * nbh);
        }
        __syncthreads();
        const int items2 = nrows * p.k;
        for (int q0 = warp * 2; q0 < items2; q0 += kWarpsAll * 2) {
            uint4 c[2][ND];
            int sc[2][ND];
#pragma unroll
            for (int u2 = 0; u2 < 2; ++u2) {
                const int q = q0 + u2;
                if (q >= items2) break;
                const int rr = q / p.k, jj = q % p.k;
                if (tab.base[t * p.k + jj] == nullptr || !ok) continue;
                const uint8_t* row = ring + (size_t)(t * p.k + jj) * nrows * p.rs_d + (size_t)rr * p.rs_d;
#pragma unroll
                for (int i = 0; i < ND; ++i) {
                    const int b = lane + 32 * i;
                    if (b < nbh) {
                        c[u2][i] = *reinterpret_cast<const uint4*>(row + 16 * b);
                        sc[u2][i] = row[p.I / 2 + b];
                    }
                }
            }
#pragma unroll
            for (int u2 = 0; u2 < 2; ++u2) {
                const int q = q0 + u2;
                if (q >= items2) break;
                const int jj = q % p.k;
                float y = __int_as_float(0x7fc00000);
                if (tab.base[t * p.k + jj] != nullptr && ok) {
                    const uint4* hj = hs + (size_t)jj * nbh * 4;
                    const int* ej = he + jj * nbh;
                    float acc = 0.0f;
#pragma unroll
                    for (int i = 0; i < ND; ++i) {
                        const int b = lane + 32 * i;
                        if (b < nbh)
                            acc = fmaf(block_dot_f16(c[u2][i], hj, b), pow2_biased(sc[u2][i] + ej[b]), acc);
                    }
                    y = warp_sum(acc);
                }
                if (lane == 0) ypart[q / p.k][jj] = y;
            }
        }
        __syncthreads();
        for (int q = threadIdx.x; q < nrows; q += kThreads) {
            float out = 0.0f;
            for (int jj = 0; jj < p.k; ++jj) out = __fadd_rn(out, __fmul_rn(tab.w[t * p.k + jj], ypart[q][jj]));
            p.out[(size_t)t * p.H + r0 + q] = out;
        }
    }
}

}  // namespace

// Shared memory of the fused kernel: the activation staging (phase 1) or
// the h staging (phase 2), then the copy ring of gate/up row pairs.
static size_t staging_bytes(int T, int k, int H, int I) {
    const size_t x = size_t(T) * H * 2 + size_t(T) * (H / 32) * 4;
    const size_t h = size_t(k) * I * 2 + size_t(k) * (I / 32) * 4;
    return round_up(x > h ? x : h, 128);
}

size_t decode_fused_smem(int T, int k, int H, int I) {
    Layout L;
    if (!Layout::make(H, I, &L) || T * k > kMaxAssign || I % kGroup) return 0;
    if (k * ((H + 151) / 152) > kMaxRows2 * kMaxAssign) return 0;
    const size_t st = staging_bytes(T, k, H, I);
    const size_t ring_min = 2 * 2 * kGroup * L.rs_gu;
    return st + ring_min <= 200 * 1024 ? st + ring_min : 0;
}

int launch_decode_fused_impl(const FfnArgs& a, void* ws, cudaStream_t s, const RouteOut* ro) {
    const Layout& L = *a.L;
    DeviceInfo di;
    int rc = current_device_info(&di);
    if (rc != MOE_OK) return rc;
    if (decode_fused_smem(a.T, a.k, L.H, L.I) == 0) return MOE_ERR_UNSUPPORTED;
    const size_t st = staging_bytes(a.T, a.k, L.H, L.I);
    const size_t slot_bytes = 2 * kGroup * L.rs_gu;
    const size_t budget = 200 * 1024;
    if ((L.H + di.sms - 1) / di.sms > kMaxRows2) return MOE_ERR_UNSUPPORTED;
    const int slots = int(std::min<size_t>(kMaxSlots, (budget - st) / slot_bytes));
    const size_t down_bytes = size_t(a.T) * a.k * ((L.H + di.sms - 1) / di.sms) * L.rs_d;
    if (slots < 2 || down_bytes > size_t(slots) * slot_bytes) return MOE_ERR_UNSUPPORTED;
    const size_t smem = st + size_t(slots) * slot_bytes;
    FusedParams p;
    p.slots = a.slots;
    p.expert_bytes = a.expert_bytes;
    p.S = a.S;
    p.E = a.E;
    p.H = L.H;
    p.I = L.I;
    p.k = a.k;
    p.T = a.T;
    p.rs_gu = L.rs_gu;
    p.rs_d = L.rs_d;
    p.d_off = L.d_off;
    p.x = a.x;
    p.ids = a.ids;
    p.w = a.w;
    p.slot_of = a.slot_of;
    p.bar = static_cast<unsigned*>(ws);
    p.h = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + 256);
    p.out = a.out;
    p.logits = ro ? ro->logits : nullptr;
    p.r_ids = ro ? ro->ids : nullptr;
    p.r_w = ro ? ro->w : nullptr;
    p.r_counts = ro ? ro->counts : nullptr;
    p.r_offsets = ro ? ro->offsets : nullptr;
    p.r_perm = ro ? ro->perm : nullptr;
    p.r_inv = ro ? ro->inv : nullptr;
    if (ro && (a.T * a.k > 32 || a.E > MOE_MAX_EXPERTS)) return MOE_ERR_UNSUPPORTED;
    const int ng = (L.H / 32 + 31) / 32, nd = (L.I / 32 + 31) / 32;
    void (*kern)(FusedParams, int, int) = nullptr;
#define MOE_PICK(G_, D_) \
    if (ng == G_ && nd == D_) kern = decode_fused_kernel<G_, D_>;
    MOE_PICK(1, 1) MOE_PICK(1, 2) MOE_PICK(2, 1) MOE_PICK(2, 2) MOE_PICK(3, 3) MOE_PICK(3, 1)
    MOE_PICK(1, 3) MOE_PICK(4, 4) MOE_PICK(2, 4) MOE_PICK(4, 2) MOE_PICK(3, 2) MOE_PICK(2, 3)
#undef MOE_PICK
    if (kern == nullptr) return MOE_ERR_UNSUPPORTED;
    static bool attr_set[16][64] = {};  // per kernel variant and device
    const int variant = (ng - 1) * 4 + (nd - 1);
    if (di.device >= 64) return MOE_ERR_UNSUPPORTED;
    if (!attr_set[variant][di.device]) {
        MOE_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(budget)));
        attr_set[variant][di.device] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(di.sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, p, slots, int(st)));
    return MOE_OK;
}

int launch_decode_fused(const FfnArgs& a, void* ws, cudaStream_t s) { return launch_decode_fused_impl(a, ws, s, nullptr); }

int launch_decode_layer(const FfnArgs& a, const RouteOut& ro, void* ws, cudaStream_t s) {
    return launch_decode_fused_impl(a, ws, s, &ro);
}

}  // namespace moe
