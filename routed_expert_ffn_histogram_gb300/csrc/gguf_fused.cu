// Single-launch decode on GGUF expert weights (Q8_0, Q4_K) read in place:
// optional routing, gate/up + SwiGLU, down, and the rank-order combine.
//
// Source: tinyserve README, "How it works" item 2 -- the expert runs on its
// native quantised bytes (Q4_K ... Q8_0) -- and "Supported models", Formats.
// The block layouts are the published GGUF / ggml ones:
//   Q8_0  per 32 elements 34 bytes: binary16 d, 32 int8 q; element = d * q.
//   Q4_K  per 256 elements 144 bytes: binary16 d and dmin, 12 bytes packing
//         eight 6-bit scales and mins, 128 bytes of 4-bit values (sub-blocks
//         2g and 2g+1 in the low and high nibbles of bytes 32g .. 32g+31);
//         element = d * sc * q - dmin * m.
// Arithmetic: bf16 activations times the exactly dequantised weights, fp32
// sums, h = bf16(silu(g) * u), each block summed in its own factors
// (d * sum(q x); d*sc * sum(q x) - dmin*m * sum(x)), the k terms of a token
// summed in rank order.  The activations are held as f16 scaled per block
// of 32 by a power of two (exact for every value within 2^-31 of the
// block's largest) and the codes as exact f16 values (Q8_0: the integer q;
// Q4_K: 8 + q/2, its bias taken out with the min term through sum(x)), so
// each product is exact in fp32 (mixed-precision FMA).
//
// Shape: one persistent CTA per SM, 18 warps, launched cooperatively (all
// CTAs resident at once, which the waits between CTAs below rely on).
//   warp 0   routing when logits are given, with up to 16 consumer warps
//            ranking further tokens of a batch (slot map and logits in one
//            round trip, later tokens' logits prefetched into L1; top-k by
//            two warp reductions per rank; each assignment's expert and slot
//            published through their own mbarrier as soon as its rank is
//            decided; then one softmax pass for all assignments by warp 0),
//            else the given ids and weights.  CTA 0 writes the routing
//            outputs.
//   warp 1   lane 0 copies: the CTA's gate/up work items (up to 8 rows of h of
//            one assignment: 8 gate and 8 up rows, two bulk copies) into a ring
//            of shared-memory slots, and, once the ring is first full, the down
//            rows behind the CTA's output rows (one bulk copy per rank) into a
//            buffer of their own, where they wait for the down phase (or, when
//            they do not fit, a prefetch of them into L2).
//   warps 2..17, two groups of eight taking alternate items: warp j of a
//            group forms h for row j of its item, lane u taking unit u (64
//            elements) of both the gate and the up row against x; h goes to
//            the workspace.  After its items the CTA adds, per assignment, the
//            rows of h it wrote to a counter in the workspace (one release
//            after a barrier).  Then the CTA's output rows n0..n1 of a token:
//            once the counters of the token's k assignments say all of their h
//            exists (a bounded wait on other CTAs), the k vectors h are staged
//            like x, four lanes form each (rank, row) of y into shared memory,
//            and out[t][n] (+)= sum_j w_j y_j, j ascending, is formed in the
//            CTA: no output row is touched by two CTAs.
// The last CTA to finish (a ticket) clears the counters for the next call.
// Every wait is bounded (about a second, then an error bit and NaN output).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "internal.h"
#include "route_warp.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int kItemRows = 8;                    // rows of h per gate/up work item
constexpr int kGroupWarps = kItemRows;          // one warp per row of an item
constexpr int kConsumerWarps = 2 * kGroupWarps;
constexpr int kThreads = 32 * (kConsumerWarps + 2);
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kMaxSlots = 8;
constexpr int kMaxAssign = 32;                  // one routing lane per assignment
constexpr int kUnit = 64;                       // elements per lane unit
constexpr size_t kSmemBudget = 220 * 1024;      // dynamic shared memory (static use stays under 2 KB)

// Control words (the workspace's first 256 bytes): [0] exit ticket, [2] error
// bits (bit 4 copy producer, 8 consumers, 16 wait for other CTAs' h),
// [32 + a] rows of h of assignment a written.
constexpr int kCtlErr = 2, kCtlHrows = 32;

struct GfParams {
    const uint8_t* slots;
    size_t expert_bytes;
    int S, E, H, I, T, k;
    int rb_h, rb_i;             // bytes of a gate/up row (K = H) and of a down row (K = I)
    const uint16_t* x;          // bf16 [T][H]
    const int32_t* ids;         // [T*k] (when logits is null)
    const float* w;             // [T*k]
    const int32_t* slot_of;     // [E]
    const float* logits;        // fp32 [T][E]: routing in the kernel when non-null
    int32_t* r_ids;
    float* r_w;
    int32_t* r_counts;
    int32_t* r_offsets;
    int32_t* r_perm;
    int32_t* r_inv;
    unsigned* ctl;
    uint16_t* h;                // bf16 [T*k][I]
    float* out;                 // fp32 [T][H]
    int accumulate;
};

struct Table {
    const uint8_t* base[kMaxAssign];
    float w[kMaxAssign];
    float sel_v[kMaxAssign];
    int id[kMaxAssign];
};

struct Bars {
    uint64_t full[kMaxSlots];
    uint64_t empty[kMaxSlots];
    uint64_t down_full;
    uint64_t ranked;        // every routing warp has published its tokens' ranks
    uint64_t routed;
    uint64_t assigned[kMaxAssign];
};

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            tc::smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"r"(kConsumers) : "memory"); }

// Wait (bounded) until *ctr >= target, the counter written by other CTAs.
__device__ __forceinline__ bool wait_counter(const unsigned* ctr, unsigned target, volatile uint32_t* err,
                                             uint32_t code) {
    uint64_t t0 = 0;
    for (uint32_t i = 0; i < tc::kWaitLimit; ++i) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if (v >= target) return true;
        if ((i & 15u) == 15u) {
            if (*err) return false;
            const uint64_t t = tc::global_ns();
            if (t0 == 0) t0 = t;
            else if (t - t0 > tc::kWaitNs) break;
        }
        __nanosleep(100);
    }
    atomicOr(const_cast<uint32_t*>(err), code);
    return false;
}

__device__ __forceinline__ float f16lo(uint32_t b) { return __half2float(__ushort_as_half((unsigned short)(b & 0xffffu))); }

// acc0 += w.lo * x.lo, acc1 += w.hi * x.hi (f16 products, exact in fp32).
__device__ __forceinline__ void fma2(float& acc0, float& acc1, uint32_t w2, uint32_t x2) {
    asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
        "mov.b32 {wl, wh}, %2;\n\tmov.b32 {xl, xh}, %3;\n\t"
        "fma.rn.f32.f16 %0, wl, xl, %0;\n\tfma.rn.f32.f16 %1, wh, xh, %1;\n\t}"
        : "+f"(acc0), "+f"(acc1)
        : "r"(w2), "r"(x2));
}

// The 4-bit fields at bits 6..9 and 22..25 of v as the f16 pair 8 + q/2:
// each field placed in mantissa bits 6..9 of f16 8.0 (0x4800), where a unit
// of the field is worth 1/2.  Exact, and a product (8 + q/2) * x is exact in
// fp32; the bias is taken out per sub-block through sum(q x) = 2 sum((8 +
// q/2) x) - 16 sum(x), folded into the Q4_K min term, which holds sum(x)
// already.
__device__ __forceinline__ uint32_t nib2_b8_f16(uint32_t v) {
    uint32_t r;
    asm("lop3.b32 %0, %1, 0x03c003c0, 0x48004800, 0xea;" : "=r"(r) : "r"(v));
    return r;
}

// Two bytes of v (sel: byte indices in nibbles 0 and 2, 4 in nibbles 1 and
// 3), each an int8 biased by 128 (xor 0x80), as exact f16 integers: the byte
// in the low mantissa bits of 1024, then 1152 subtracted.
__device__ __forceinline__ uint32_t s8x2_f16(uint32_t v_biased, uint32_t sel) {
    uint32_t r, o;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(v_biased), "r"(0x64646464u), "r"(sel));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o) : "r"(r), "r"(0x64806480u));
    return o;
}

// Byte i (0..11) of a Q4_K super-block's packed scales and mins (bytes
// 4..15 of the block: the words y, z, w of its first 16 bytes).
__device__ __forceinline__ int packed_byte(const uint4& hdr, int i) {
    const uint32_t v = i < 4 ? hdr.y : (i < 8 ? hdr.z : hdr.w);
    return int((v >> (8 * (i & 3))) & 0xffu);
}

// 6-bit scale and min of sub-block j: 0..3 keep them in the low 6 bits of
// bytes j and j+4; 4..7 keep their low 4 bits in the nibbles of byte j+4 and
// their top 2 bits in the top bits of bytes j-4 (scale) and j (min).
__device__ __forceinline__ void q4k_scale_min(const uint4& hdr, int j, float& sc, float& m) {
    int s, mm;
    if (j < 4) {
        s = packed_byte(hdr, j) & 63;
        mm = packed_byte(hdr, j + 4) & 63;
    } else {
        s = (packed_byte(hdr, j + 4) & 15) | ((packed_byte(hdr, j - 4) >> 6) << 4);
        mm = (packed_byte(hdr, j + 4) >> 4) | ((packed_byte(hdr, j) >> 6) << 4);
    }
    sc = float(s);
    m = float(mm);
}

// A vector staged for the dot products: per unit u of 64 elements eight
// 16-byte chunks of f16 (chunk c of unit u at index c * U + u, so the lanes
// of a warp, each on its own unit, read consecutive chunks), scaled per block
// of 32 by 2^-e; fac[b] = 2^e and sum[b] = the block's fp32 sum.  For Q4_K
// each group of four elements is stored as (0, 2, 1, 3): the pairs that the
// low and high nibble fields of a code word meet.
struct Staged {
    const uint4* chunks;
    const float* fac;
    const float* sum;
    int U;
};

// Block b (elements 32b .. 32b+31) of a vector of U units at src into its
// staged copy (chunks, fac, sum).
template <int FMT>
__device__ __forceinline__ void stage_block(const uint16_t* __restrict__ src, int b, int U, uint4* chunks,
                                            float* fac, float* sum) {
    {
        const uint4* s4 = reinterpret_cast<const uint4*>(src + 32 * b);
        uint32_t v[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 c = __ldcg(s4 + q);
            v[4 * q] = c.x;
            v[4 * q + 1] = c.y;
            v[4 * q + 2] = c.z;
            v[4 * q + 3] = c.w;
        }
        float amax = 0.f, s = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float a = __uint_as_float(v[i] << 16), c = __uint_as_float(v[i] & 0xffff0000u);
            amax = fmaxf(amax, fmaxf(fabsf(a), fabsf(c)));
            s += a;
            s += c;
        }
        const int ef = int((__float_as_uint(amax) >> 23) & 0xffu);
        const int e = (amax == 0.f) ? 0 : (ef == 0 ? -126 - 14 : ef - 127 - 14);
        const float m = ldexpf(1.0f, -e);
        const int u = b >> 1, c0 = (b & 1) * 4;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            // elements 8q .. 8q+7 of the block: words v[4q .. 4q+3] hold pairs (2i, 2i+1)
            float e8[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                e8[2 * i] = __uint_as_float(v[4 * q + i] << 16) * m;
                e8[2 * i + 1] = __uint_as_float(v[4 * q + i] & 0xffff0000u) * m;
            }
            uint32_t o[4];
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                const float* f = e8 + 4 * g;
                __half2 p0, p1;
                if constexpr (FMT == MOE_GGUF_Q4_K) {
                    p0 = __floats2half2_rn(f[0], f[2]);
                    p1 = __floats2half2_rn(f[1], f[3]);
                } else {
                    p0 = __floats2half2_rn(f[0], f[1]);
                    p1 = __floats2half2_rn(f[2], f[3]);
                }
                o[2 * g] = *reinterpret_cast<const uint32_t*>(&p0);
                o[2 * g + 1] = *reinterpret_cast<const uint32_t*>(&p1);
            }
            chunks[(c0 + q) * U + u] = make_uint4(o[0], o[1], o[2], o[3]);
        }
        fac[b] = ldexpf(1.0f, e);
        sum[b] = s;
    }
}

// Contributions of unit u (elements 64u .. 64u+63) of NR GGUF rows to their
// dot products with the staged vector xs, added to acc[r].  The loop runs
// over the unit's four pairs of x chunks without unrolling (the codes and x
// are read from shared memory each pass), so one copy of its body serves all
// passes: the kernel's code stays small enough for the instruction cache.
template <int FMT, int NR>
__device__ __forceinline__ void unit_dots(const uint8_t* const (&rows)[NR], int u, const Staged& xs,
                                          float (&acc)[NR]) {
    const float f0 = xs.fac[2 * u], f1 = xs.fac[2 * u + 1];
    float a0[NR], a1[NR], b0[NR], b1[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) a0[r] = a1[r] = b0[r] = b1[r] = 0.f;
    if constexpr (FMT == MOE_GGUF_Q4_K) {
        const int sb = u >> 2, g = u & 3;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            // code words 2c and 2c+1 (values 8c .. 8c+7 of sub-blocks 2g and
            // 2g+1); x chunks c and 4 + c hold those values of the two blocks
            const uint4 xl = xs.chunks[c * xs.U + u], xh = xs.chunks[(4 + c) * xs.U + u];
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const uint2 wv = *reinterpret_cast<const uint2*>(rows[r] + 144 * sb + 16 + 32 * g + 8 * c);
                // low nibbles of bytes 0 and 2 (bits 0, 16), of bytes 1 and 3
                // (bits 8, 24); high nibbles of bytes 0, 2 (4, 20) and 1, 3
                // (12, 28): each shifted to bits 6 and 22
                fma2(a0[r], a1[r], nib2_b8_f16(wv.x << 6), xl.x);
                fma2(a0[r], a1[r], nib2_b8_f16(wv.x >> 2), xl.y);
                fma2(b0[r], b1[r], nib2_b8_f16(wv.x << 2), xh.x);
                fma2(b0[r], b1[r], nib2_b8_f16(wv.x >> 6), xh.y);
                fma2(a0[r], a1[r], nib2_b8_f16(wv.y << 6), xl.z);
                fma2(a0[r], a1[r], nib2_b8_f16(wv.y >> 2), xl.w);
                fma2(b0[r], b1[r], nib2_b8_f16(wv.y << 2), xh.z);
                fma2(b0[r], b1[r], nib2_b8_f16(wv.y >> 6), xh.w);
            }
        }
        const float x0 = xs.sum[2 * u], x1 = xs.sum[2 * u + 1];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const uint4 hdr = *reinterpret_cast<const uint4*>(rows[r] + 144 * sb);
            float sc0, m0, sc1, m1;
            q4k_scale_min(hdr, 2 * g, sc0, m0);
            q4k_scale_min(hdr, 2 * g + 1, sc1, m1);
            const float d = f16lo(hdr.x), dmin = f16lo(hdr.x >> 16);
            // sum(w x) = d sc sum(q x) - dmin m sum(x), sum(q x) = 2 f sum(b x') - 16 sum(x)
            const float ds0 = d * sc0, ds1 = d * sc1;
            acc[r] += ((2.0f * ds0) * (f0 * (a0[r] + a1[r])) - (16.0f * ds0 + dmin * m0) * x0) +
                      ((2.0f * ds1) * (f1 * (b0[r] + b1[r])) - (16.0f * ds1 + dmin * m1) * x1);
        }
    } else {
        // blocks 2u and 2u + 1: 68 bytes at 68 u (4-byte aligned); block 2u's
        // values 8c .. 8c+7 sit in bytes 2+8c .. 9+8c (words 2c .. 2c+2),
        // block 2u+1's in bytes 36+8c .. 43+8c (words 9+2c, 10+2c)
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            const uint4 xl = xs.chunks[c * xs.U + u], xh = xs.chunks[(4 + c) * xs.U + u];
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const uint32_t* p = reinterpret_cast<const uint32_t*>(rows[r] + 68 * u) + 2 * c;
                const uint32_t w0 = p[0] ^ 0x80808080u, w1 = p[1] ^ 0x80808080u, w2 = p[2] ^ 0x80808080u;
                const uint32_t v0 = p[9] ^ 0x80808080u, v1 = p[10] ^ 0x80808080u;
                fma2(a0[r], a1[r], s8x2_f16(w0, 0x4342u), xl.x);
                fma2(a0[r], a1[r], s8x2_f16(w1, 0x4140u), xl.y);
                fma2(a0[r], a1[r], s8x2_f16(w1, 0x4342u), xl.z);
                fma2(a0[r], a1[r], s8x2_f16(w2, 0x4140u), xl.w);
                fma2(b0[r], b1[r], s8x2_f16(v0, 0x4140u), xh.x);
                fma2(b0[r], b1[r], s8x2_f16(v0, 0x4342u), xh.y);
                fma2(b0[r], b1[r], s8x2_f16(v1, 0x4140u), xh.z);
                fma2(b0[r], b1[r], s8x2_f16(v1, 0x4342u), xh.w);
            }
        }
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const uint32_t* p = reinterpret_cast<const uint32_t*>(rows[r] + 68 * u);
            const float d0 = f16lo(p[0]), d1 = f16lo(p[8] >> 16);
            acc[r] += d0 * (f0 * (a0[r] + a1[r])) + d1 * (f1 * (b0[r] + b1[r]));
        }
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Shared-memory carve-up, in bytes from the dynamic base (all offsets
// multiples of 128).  The staged h of the down phase reuses the ring.  When
// the CTA's down rows do not fit beside a ring of three slots (several
// tokens), they are prefetched into L2 instead and read from there.
struct Carve {
    int x_off, xf_off, xs_off, ring_off, down_off, total;
    int slot_bytes, n_slots;
    int down_smem;
};

__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

template <int FMT, int NU>
__global__ void __launch_bounds__(kThreads, 1) gguf_fused_kernel(GfParams p, Carve cv) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ Table tab;
    __shared__ __align__(8) Bars bars;
    __shared__ int h_ok;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = gridDim.x;
    const int A = p.T * p.k;
    volatile uint32_t* err = p.ctl + kCtlErr;
    const int UX = p.H / kUnit, UH = p.I / kUnit;

    if (threadIdx.x == 0) {
        for (int s = 0; s < cv.n_slots; ++s) {
            tc::mbar_init(&bars.full[s], 1);
            tc::mbar_init(&bars.empty[s], kGroupWarps);
        }
        tc::mbar_init(&bars.down_full, 1);
        tc::mbar_init(&bars.routed, 1);
        tc::mbar_init(&bars.ranked, p.logits != nullptr ? unsigned(min(p.T, 1 + kConsumerWarps)) : 1u);
        for (int a = 0; a < A; ++a) tc::mbar_init(&bars.assigned[a], 1);
        tc::fence_barrier_init();
    }
    __syncthreads();

    // Gate/up rows of h in (assignment, row) order, and down rows in
    // (assignment, output row) order, each cut into one contiguous range per CTA.
    const int ra_tot = A * p.I, pa = (ra_tot + G - 1) / G;
    const int ra0 = min(ra_tot, (int)blockIdx.x * pa), ra1 = min(ra_tot, ra0 + pa);
    const int o_tot = p.T * p.H, po = (o_tot + G - 1) / G;
    const int o0 = min(o_tot, (int)blockIdx.x * po), o1 = min(o_tot, o0 + po);
    uint8_t* ring = smem + cv.ring_off;
    uint8_t* dbuf = smem + cv.down_off;

    // ---- routing: with logits, warp 0 and up to 16 consumer warps each rank
    // their own tokens (t = r, r + R, ...; warp 0 is router 0, warp w >= 2
    // router w - 1), publishing each assignment as soon as its rank is
    // decided; warp 0 weighs every assignment once all routers reported ----
    const int R = (p.logits != nullptr) ? min(p.T, 1 + kConsumerWarps) : 0;
    const int rw = (warp == 0) ? 0 : warp - 1;
    if (p.logits != nullptr && (warp == 0 || (warp >= 2 && rw < R))) {
        auto route_tokens = [&](auto epl_tag) {
            constexpr int EPL = decltype(epl_tag)::value;
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
                        tc::mbar_arrive(&bars.assigned[a]);
                    }
                }
            }
        };
        if (p.E <= 32) route_tokens(std::integral_constant<int, 1>{});
        else if (p.E <= 64) route_tokens(std::integral_constant<int, 2>{});
        else if (p.E <= 128) route_tokens(std::integral_constant<int, 4>{});
        else route_tokens(std::integral_constant<int, 8>{});
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bars.ranked);
    }
    if (warp == 0) {
        if (p.logits != nullptr) {
            // every assignment's weight in one pass (lane a: assignment a)
            const bool ranked = tc::mbar_wait_suspend(&bars.ranked, 0u, err, 8u);
            const float sv = (ranked && lane < A) ? tab.sel_v[lane] : __int_as_float(0x7fc00000);
            const float wv = softmax_assign(sv, p.k, A);
            if (lane < A) tab.w[lane] = wv;
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars.routed);
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
                for (int a = 0; a < A; ++a) tc::mbar_arrive(&bars.assigned[a]);
                tc::mbar_arrive(&bars.routed);
            }
        }
    } else if (warp == 1) {
        // ---- copy producer ----
        if (lane == 0) {
            bool ok = true;
            auto issue_down = [&]() {
                // the down rows n0..n1 of each rank of each token segment; every
                // segment's slots first, so the byte count is known
                uint32_t total = 0;
                for (int o = o0; o < o1 && ok;) {
                    const int t = o / p.H, n1 = min(o1, (t + 1) * p.H) - t * p.H, R = n1 - (o - t * p.H);
                    for (int j = 0; j < p.k && ok; ++j) {
                        const int a = t * p.k + j;
                        if (!tc::mbar_wait_suspend(&bars.assigned[a], 0u, err, 4u)) ok = false;
                        else if (tab.base[a] != nullptr) total += uint32_t(R) * uint32_t(p.rb_i);
                    }
                    o = t * p.H + n1;
                }
                if (!ok) return;
                if (!cv.down_smem) total = 0;
                if (total) tc::mbar_arrive_expect_tx(&bars.down_full, total);
                else tc::mbar_arrive(&bars.down_full);
                int c_rows = 0;
                for (int o = o0; o < o1;) {
                    const int t = o / p.H, n0 = o - t * p.H, n1 = min(o1, (t + 1) * p.H) - t * p.H, R = n1 - n0;
                    for (int j = 0; j < p.k; ++j) {
                        const uint8_t* eb = tab.base[t * p.k + j];
                        if (eb == nullptr) continue;
                        const uint8_t* src = eb + size_t(2) * p.I * p.rb_h + size_t(n0) * p.rb_i;
                        const uint32_t bytes = uint32_t(R) * uint32_t(p.rb_i);
                        if (cv.down_smem)
                            bulk_g2s(dbuf + (size_t(c_rows) * p.k + size_t(j) * R) * p.rb_i, src, bytes,
                                     &bars.down_full);
                        else
                            prefetch_l2(src, bytes);
                    }
                    c_rows += R;
                    o = t * p.H + n1;
                }
            };
            int a = ra0 / max(p.I, 1), r = ra0 - a * p.I, left = ra1 - ra0;
            int slot = 0;
            uint32_t ph = 0;
            while (left > 0 && ok) {
                const int rows = min(kItemRows, min(p.I - r, left));
                if (!tc::mbar_wait_suspend(&bars.empty[slot], ph ^ 1u, err, 4u)) { ok = false; break; }
                if (!tc::mbar_wait_suspend(&bars.assigned[a], 0u, err, 4u)) { ok = false; break; }
                const uint8_t* eb = tab.base[a];
                uint8_t* dst = ring + size_t(slot) * cv.slot_bytes;
                if (eb != nullptr) {
                    const uint32_t part = uint32_t(rows) * uint32_t(p.rb_h);
                    tc::mbar_arrive_expect_tx(&bars.full[slot], 2 * part);
                    bulk_g2s(dst, eb + size_t(r) * p.rb_h, part, &bars.full[slot]);
                    bulk_g2s(dst + size_t(kItemRows) * p.rb_h, eb + size_t(p.I + r) * p.rb_h, part, &bars.full[slot]);
                } else {
                    tc::mbar_arrive(&bars.full[slot]);
                }
                left -= rows;
                if ((r += rows) == p.I) { r = 0; ++a; }
                if (++slot == cv.n_slots) { slot = 0; ph ^= 1u; }
            }
            // the down rows go out after every gate/up row: they are needed
            // only once all of h exists, and would otherwise take HBM time
            // from the gate/up rows still to come
            if (ok) issue_down();
        }
    } else {
        // ---- consumers ----
        const int ct = threadIdx.x - 64;
        const int grp = (warp - 2) / kGroupWarps, wj = (warp - 2) % kGroupWarps;
        // stage every token's x
        uint4* xch = reinterpret_cast<uint4*>(smem + cv.x_off);
        float* xfac = reinterpret_cast<float*>(smem + cv.xf_off);
        float* xsum = reinterpret_cast<float*>(smem + cv.xs_off);
        for (int i = ct; i < p.T * (p.H / 32); i += kConsumers) {
            const int t = i / (p.H / 32), b = i - t * (p.H / 32);
            stage_block<FMT>(p.x + (size_t)t * p.H, b, UX, xch + (size_t)t * UX * 8, xfac + t * (p.H / 32),
                             xsum + t * (p.H / 32));
        }
        consumers_sync();

        // (1) gate/up items: group grp takes items grp, grp + 2, ...
        {
            int a = ra0 / max(p.I, 1), r = ra0 - a * p.I, left = ra1 - ra0;
            int slot = 0, n = 0;
            uint32_t ph = 0;
            while (left > 0) {
                const int rows = min(kItemRows, min(p.I - r, left));
                if ((n & 1) == grp) {
                    const bool got = tc::mbar_wait_suspend(&bars.full[slot], ph, err, 8u);
                    if (wj < rows) {
                        const uint8_t* eb = got ? tab.base[a] : nullptr;
                        float hj = __int_as_float(0x7fc00000);
                        if (eb != nullptr) {
                            const int t = a / p.k;
                            const Staged xs{xch + (size_t)t * UX * 8, xfac + t * (p.H / 32), xsum + t * (p.H / 32), UX};
                            const uint8_t* gr = ring + size_t(slot) * cv.slot_bytes + size_t(wj) * p.rb_h;
                            const uint8_t* const rows2[2] = {gr, gr + size_t(kItemRows) * p.rb_h};
                            float acc2[2] = {0.f, 0.f};
#pragma unroll
                            for (int i = 0; i < NU; ++i) {
                                const int u = lane + 32 * i;
                                if (i < NU - 1 || u < UX) unit_dots<FMT, 2>(rows2, u, xs, acc2);
                            }
                            const float ag = warp_sum(acc2[0]);
                            const float au = warp_sum(acc2[1]);
                            const float silu = __fdividef(ag, 1.0f + __expf(-ag));
                            hj = silu * au;
                        }
                        if (lane == 0) {
                            const __nv_bfloat16 hb = __float2bfloat16_rn(hj);
                            p.h[(size_t)a * p.I + r + wj] = *reinterpret_cast<const uint16_t*>(&hb);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&bars.empty[slot]);
                }
                left -= rows;
                if ((r += rows) == p.I) { r = 0; ++a; }
                if (++slot == cv.n_slots) { slot = 0; ph ^= 1u; }
                ++n;
            }
        }
        consumers_sync();
        if (ct == 0) {
            // publish the rows of h this CTA wrote, per assignment: the
            // barrier orders the writers' stores before this release
            __threadfence();
            for (int r = ra0; r < ra1;) {
                const int a = r / p.I, r1 = min(ra1, (a + 1) * p.I);
                atomicAdd(p.ctl + kCtlHrows + a, unsigned(r1 - r));
                r = r1;
            }
        }

        // (2) the CTA's output rows (token t, rows n0..n1) for all k ranks of
        // the token: h of the k ranks staged side by side in the (now idle)
        // ring, four lanes per (rank, row), y in shared memory, then the
        // rank-order combine
        const bool dgot = (o1 > o0) ? tc::mbar_wait_suspend(&bars.down_full, 0u, err, 8u) : true;
        const bool routed = (o1 > o0) ? tc::mbar_wait_suspend(&bars.routed, 0u, err, 8u) : true;
        const int hstride = p.I * 2 + (p.I / 32) * 8;   // staged h of one rank: chunks, factors, sums
        float* ys = reinterpret_cast<float*>(ring + size_t(p.k) * hstride);
        const int j4 = ct & 3, pr = ct >> 2;
        int c_rows = 0;   // output rows of the earlier segments
        for (int o = o0; o < o1;) {
            const int t = o / p.H, n0 = o - t * p.H, n1 = min(o1, (t + 1) * p.H) - t * p.H, R = n1 - n0;
            consumers_sync();   // the previous segment's staged h and y are no longer read
            if (ct < 32) {
                // lane j waits for assignment t*k + j: the k waits overlap
                bool mine = true;
                for (int j = ct; j < p.k; j += 32)
                    mine = mine && wait_counter(p.ctl + kCtlHrows + t * p.k + j, unsigned(p.I), err, 16u);
                const bool all = __all_sync(0xffffffffu, mine);
                if (ct == 0) h_ok = all ? 1 : 0;
            }
            consumers_sync();
            const bool seg_ok = h_ok && dgot;
            if (seg_ok)
                for (int i = ct; i < p.k * (p.I / 32); i += kConsumers) {
                    const int j = i / (p.I / 32), b = i - j * (p.I / 32);
                    uint8_t* hb = ring + size_t(j) * hstride;
                    float* hf = reinterpret_cast<float*>(hb + size_t(p.I) * 2);
                    stage_block<FMT>(p.h + (size_t)(t * p.k + j) * p.I, b, UH, reinterpret_cast<uint4*>(hb), hf,
                                     hf + p.I / 32);
                }
            consumers_sync();
            for (int q0 = 0; q0 < p.k * R; q0 += kConsumers / 4) {
                const int q = q0 + pr;
                const bool live = q < p.k * R;
                const int j = live ? q / R : 0, n = n0 + (q - j * R);
                const int a = t * p.k + j;
                const uint8_t* eb = live ? tab.base[a] : nullptr;
                float acc = 0.f;
                if (seg_ok && eb != nullptr) {
                    const uint8_t* hb = ring + size_t(j) * hstride;
                    const float* hf = reinterpret_cast<const float*>(hb + size_t(p.I) * 2);
                    const Staged hs{reinterpret_cast<const uint4*>(hb), hf, hf + p.I / 32, UH};
                    const uint8_t* row = cv.down_smem
                                             ? dbuf + (size_t(c_rows) * p.k + size_t(j) * R + (n - n0)) * p.rb_i
                                             : eb + size_t(2) * p.I * p.rb_h + size_t(n) * p.rb_i;
                    const uint8_t* const rows1[1] = {row};
                    float acc1[1] = {0.f};
                    for (int u = j4; u < UH; u += 4) unit_dots<FMT, 1>(rows1, u, hs, acc1);
                    acc = acc1[0];
                }
                acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                if (j4 == 0 && live) ys[q] = (seg_ok && eb != nullptr) ? acc : __int_as_float(0x7fc00000);
            }
            consumers_sync();
            // out[t][n] (+)= sum_j w_j y_j, j ascending, no FMA contraction
            for (int i = ct; i < R; i += kConsumers) {
                float acc = 0.f;
                for (int j = 0; j < p.k; ++j) {
                    const float wv = routed ? tab.w[t * p.k + j] : __int_as_float(0x7fc00000);
                    acc = __fadd_rn(acc, __fmul_rn(wv, ys[j * R + i]));
                }
                float* op = p.out + (size_t)t * p.H + n0 + i;
                *op = p.accumulate ? __fadd_rn(*op, acc) : acc;
            }
            c_rows += R;
            o = t * p.H + n1;
        }
    }

    // ---- exit: the last CTA clears the counters for the next call ----
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned ticket = atomicAdd(p.ctl, 1u);
        if (ticket == unsigned(G - 1)) {
            for (int a = 0; a < A; ++a) p.ctl[kCtlHrows + a] = 0u;
            p.ctl[0] = 0u;
            __threadfence();
        }
    }
}

size_t round_up_sz(size_t v, size_t m) { return (v + m - 1) / m * m; }

bool carve(int fmt, int T, int k, int H, int I, int G, Carve* cv) {
    const int A = T * k;
    const size_t rb_h = gguf_row_bytes(fmt, H), rb_i = gguf_row_bytes(fmt, I);
    if (!rb_h || !rb_i || rb_h % 16 || rb_i % 16 || A > kMaxAssign || A < 1) return false;
    const size_t x_bytes = round_up_sz(size_t(T) * H * 2, 128);
    const size_t f_bytes = round_up_sz(size_t(T) * (H / 32) * 4, 128);
    // a CTA's output rows, and the down rows behind them (k per output row)
    const size_t po = (size_t(T) * H + G - 1) / G;
    const size_t slot = round_up_sz(2 * kItemRows * rb_h, 128);
    // the down phase's staged h of the k ranks and its y, in the ring
    const size_t h_stage = size_t(k) * (size_t(I) * 2 + size_t(I / 32) * 8) + size_t(k) * po * 4;
    // down rows in shared memory when they fit beside three ring slots
    size_t down_bytes = round_up_sz(po * k * rb_i, 128);
    if (x_bytes + 2 * f_bytes + down_bytes + 3 * slot > kSmemBudget) down_bytes = 0;
    const size_t fixed = x_bytes + 2 * f_bytes + down_bytes;
    int n = kMaxSlots;
    while (n >= 2 && fixed + n * slot > kSmemBudget) --n;
    if (n < 2 || n * slot < h_stage) return false;
    cv->down_smem = down_bytes > 0 ? 1 : 0;
    cv->x_off = 0;
    cv->xf_off = int(x_bytes);
    cv->xs_off = int(x_bytes + f_bytes);
    cv->down_off = int(x_bytes + 2 * f_bytes);
    cv->ring_off = int(x_bytes + 2 * f_bytes + down_bytes);
    cv->slot_bytes = int(slot);
    cv->n_slots = n;
    cv->total = int(fixed + n * slot);
    return true;
}

}  // namespace

// Workspace of the GGUF decode calls: a 256-byte control block, bf16 h
// [T*k][I], then fp32 y [T*k][H] (the three-launch path's down outputs).
size_t gguf_h_offset() { return 256; }
size_t gguf_y_offset(int T, int k, int I) { return 256 + round_up_sz(size_t(T) * k * I * 2, 256); }
size_t gguf_workspace_bytes(int T, int k, int H, int I) {
    return gguf_y_offset(T, k, I) + round_up_sz(size_t(T) * k * H * 4, 256);
}

bool gguf_fused_supported(int fmt, int T, int k, int H, int I) {
    DeviceInfo di;
    if (current_device_info(&di) != MOE_OK || di.sms <= 0) return false;
    Carve cv;
    if (!carve(fmt, T, k, H, I, di.sms, &cv)) return false;
    const int nu = (H / kUnit + 31) / 32;
    return nu >= 1 && nu <= 2 && kSmemBudget + 2048 <= di.smem_optin;
}

int launch_gguf_fused(int fmt, const uint8_t* slots, int S, int E, int H, int I, const uint16_t* x, int T, int k,
                      const int32_t* ids, const float* w, const int32_t* slot_of, const RouteOut* ro, void* ws,
                      float* out, bool accumulate, cudaStream_t s) {
    DeviceInfo di;
    int rc = current_device_info(&di);
    if (rc != MOE_OK) return rc;
    Carve cv;
    if (!carve(fmt, T, k, H, I, di.sms, &cv) || kSmemBudget + 2048 > di.smem_optin) return MOE_ERR_UNSUPPORTED;
    if (di.device < 0 || di.device >= 64) return MOE_ERR_UNSUPPORTED;
    const int nu = (H / kUnit + 31) / 32;
    if (nu < 1 || nu > 2) return MOE_ERR_UNSUPPORTED;
    GfParams p;
    p.slots = slots;
    p.expert_bytes = gguf_expert_bytes(fmt, H, I);
    p.S = S;
    p.E = E;
    p.H = H;
    p.I = I;
    p.T = T;
    p.k = k;
    p.rb_h = int(gguf_row_bytes(fmt, H));
    p.rb_i = int(gguf_row_bytes(fmt, I));
    p.x = x;
    p.ids = ids;
    p.w = w;
    p.slot_of = slot_of;
    p.logits = ro ? ro->logits : nullptr;
    p.r_ids = ro ? ro->ids : nullptr;
    p.r_w = ro ? ro->w : nullptr;
    p.r_counts = ro ? ro->counts : nullptr;
    p.r_offsets = ro ? ro->offsets : nullptr;
    p.r_perm = ro ? ro->perm : nullptr;
    p.r_inv = ro ? ro->inv : nullptr;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    p.ctl = reinterpret_cast<unsigned*>(wsb);
    p.h = reinterpret_cast<uint16_t*>(wsb + gguf_h_offset());
    p.out = out;
    p.accumulate = accumulate ? 1 : 0;

    using Kern = void (*)(GfParams, Carve);
    Kern kern = nullptr;
    int vi = 0;
    if (fmt == MOE_GGUF_Q8_0) {
        kern = nu == 1 ? gguf_fused_kernel<MOE_GGUF_Q8_0, 1> : gguf_fused_kernel<MOE_GGUF_Q8_0, 2>;
        vi = nu - 1;
    } else {
        kern = nu == 1 ? gguf_fused_kernel<MOE_GGUF_Q4_K, 1> : gguf_fused_kernel<MOE_GGUF_Q4_K, 2>;
        vi = 2 + nu - 1;
    }
    static DeviceOnce attr_set[4];
    if (!attr_set[vi].done(di.device)) {
        MOE_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBudget)));
        attr_set[vi].mark(di.device);
    }
    // cooperative: every CTA resident at once (the down rows wait for h
    // written by other CTAs)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(di.sms));
    cfg.blockDim = dim3(unsigned(kThreads));
    cfg.dynamicSmemBytes = size_t(cv.total);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, p, cv));
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

}  // namespace moe
