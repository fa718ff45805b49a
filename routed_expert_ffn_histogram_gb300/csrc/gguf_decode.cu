// Decode path on GGUF expert weights (Q8_0 and Q4_K), read in place.
//
// Source: tinyserve README, "How it works" item 2 -- the expert runs on its
// native quantised bytes (the README lists Q4_K, Q5_K, Q6_K and Q8_0), and
// "Supported models", Formats.  The block layouts are the published GGUF /
// ggml ones:
//   Q8_0  per 32 elements 34 bytes: binary16 d (little-endian), 32 int8 q;
//         element = d * q.
//   Q4_K  per 256 elements 144 bytes: binary16 d and dmin, 12 bytes packing
//         eight 6-bit scales and mins, 128 bytes of 4-bit values (sub-blocks
//         2g and 2g+1 in the low and high nibbles of the same 32 bytes);
//         element = d * sc * q - dmin * m.
// Arithmetic is the decode path's: bf16 activations times the exactly
// dequantised weights, fp32 sums, h = bf16(silu(g) * u).  Each block's sum is
// formed in the block's own factors (sum q*x, then times d; for Q4_K
// d*sc*sum(q*x) - dmin*m*sum(x), with sum(x) per 32 shared by every row), so
// only the fp32 rounding order differs from a dequantise-then-multiply
// evaluation.
//
// One expert in a slot is [gate I rows][up I rows][down H rows], each row
// the format's blocks back to back; the slot size is a multiple of 256 bytes.
// Calls of at most 32 assignments whose rows are multiples of 16 bytes run
// as one launch (gguf_fused.cu); the others as three launches:
//   gguf_gateup_kernel  one warp per (assignment, row pair), the gate and up
//                       rows read in one pass: h = bf16(silu(g) u) into the
//                       workspace; x staged once per CTA as fp32.
//   gguf_down_kernel    one group of lanes per (assignment, output row): y.
//   gguf_combine_kernel out[t] (+)= sum_j w_j y_j in rank order (no atomics).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;

__device__ __forceinline__ float f16_bits_to_float(uint32_t b) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(b & 0xffffu)));
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// Elements per unit of work of one lane: two Q8_0 blocks, or two Q4_K
// sub-blocks (the pair sharing 32 value bytes).
template <int FMT>
struct Unit;
template <>
struct Unit<MOE_GGUF_Q8_0> {
    static constexpr int kElems = 64;
    static constexpr int kBlockElems = 32, kBlockBytes = 34;
    __host__ __device__ static size_t row_bytes(int K) { return size_t(K / 32) * 34; }
};
template <>
struct Unit<MOE_GGUF_Q4_K> {
    static constexpr int kElems = 64;
    static constexpr int kBlockElems = 256, kBlockBytes = 144;
    __host__ __device__ static size_t row_bytes(int K) { return size_t(K / 256) * 144; }
};

// Staged vectors keep each unit of 64 elements in 65 floats (element i at
// i + i / 64), so the lanes of a warp, each reading its own unit, fall on
// distinct shared-memory banks.
__host__ __device__ constexpr int staged_len(int n) { return n + n / 64; }

// Partial dot products of this lane's units u = sub + G i of NR rows (K
// elements each, rows[r]) with xs (staged fp32 of K elements) -- xsum (fp32,
// K / 32: the per-32 sums of xs) is used by Q4_K.  The rows' loads of a unit
// are issued together.
template <int FMT, int NR>
__device__ __forceinline__ void row_dot(const uint8_t* const (&rows)[NR], const float* __restrict__ xs,
                                        const float* __restrict__ xsum, int K, int sub, int G, float (&acc)[NR]);

template <int NR>
__device__ __forceinline__ void row_dot_q8_0(const uint8_t* const (&rows)[NR], const float* __restrict__ xs, int K,
                                             int sub, int G, float (&acc)[NR]) {
    // unit u: blocks 2u and 2u + 1, 68 bytes at 68 u (4-byte aligned)
    const int U = K / 64;
    for (int u = sub; u < U; u += G) {
        uint32_t wd[NR][17];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const uint32_t* p = reinterpret_cast<const uint32_t*>(rows[r] + 68 * u);
#pragma unroll
            for (int i = 0; i < 17; ++i) wd[r][i] = __ldg(p + i);
        }
        const float* x = xs + 65 * u;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            // block 2u: d in bytes 0-1, q in bytes 2..33; block 2u + 1: d in
            // bytes 34-35, q in bytes 36..67
            float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int b0 = 2 + i, b1 = 36 + i;
                const int q0 = int(int8_t((wd[r][b0 >> 2] >> (8 * (b0 & 3))) & 0xffu));
                const int q1 = int(int8_t((wd[r][b1 >> 2] >> (8 * (b1 & 3))) & 0xffu));
                s0 = fmaf(float(q0), x[i], s0);
                s1 = fmaf(float(q1), x[32 + i], s1);
            }
            acc[r] = fmaf(f16_bits_to_float(wd[r][0]), s0, acc[r]);
            acc[r] = fmaf(f16_bits_to_float(wd[r][8] >> 16), s1, acc[r]);
        }
    }
}

// Byte i (0..11) of the packed scales and mins: bytes 4..15 of the
// super-block, held in the words y, z, w of its first 16 bytes.
__device__ __forceinline__ int packed_byte(const uint4& hdr, int i) {
    const uint32_t w = i < 4 ? hdr.y : (i < 8 ? hdr.z : hdr.w);
    return int((w >> (8 * (i & 3))) & 0xffu);
}

// 6-bit scale and min of sub-block j of a Q4_K super-block, from its 12
// packed bytes p: sub-blocks 0-3 keep theirs in the low 6 bits of p[j] and
// p[j+4]; 4-7 keep their low 4 bits in the nibbles of p[j+4] and their top 2
// bits in the top bits of p[j-4] (scale) and p[j] (min).

__device__ __forceinline__ void q4k_scale_min(const uint4& hdr, int j, int& sc, int& m) {
    if (j < 4) {
        sc = packed_byte(hdr, j) & 63;
        m = packed_byte(hdr, j + 4) & 63;
    } else {
        sc = (packed_byte(hdr, j + 4) & 15) | ((packed_byte(hdr, j - 4) >> 6) << 4);
        m = (packed_byte(hdr, j + 4) >> 4) | ((packed_byte(hdr, j) >> 6) << 4);
    }
}

template <int NR>
__device__ __forceinline__ void row_dot_q4_k(const uint8_t* const (&rows)[NR], const float* __restrict__ xs,
                                             const float* __restrict__ xsum, int K, int sub, int G,
                                             float (&acc)[NR]) {
    // unit u: super-block u / 4, value bytes 32 g .. 32 g + 31 (g = u % 4),
    // i.e. sub-blocks 2g (low nibbles) and 2g + 1 (high nibbles)
    const int U = (K / 256) * 4;
    for (int u = sub; u < U; u += G) {
        const int sb = u >> 2, g = u & 3;
        uint4 hdr[NR], v0[NR], v1[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const uint8_t* blk = rows[r] + 144 * sb;
            hdr[r] = __ldg(reinterpret_cast<const uint4*>(blk));
            v0[r] = __ldg(reinterpret_cast<const uint4*>(blk + 16 + 32 * g));
            v1[r] = __ldg(reinterpret_cast<const uint4*>(blk + 32 + 32 * g));
        }
        const float* x0 = xs + 65 * u;   // elements 256 sb + 64 g .. + 63
        const float* x1 = x0 + 32;
        const int j0 = 8 * sb + 2 * g;
        const float xs0 = xsum[j0], xs1 = xsum[j0 + 1];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            int sc0, m0, sc1, m1;
            q4k_scale_min(hdr[r], 2 * g, sc0, m0);
            q4k_scale_min(hdr[r], 2 * g + 1, sc1, m1);
            const float d = f16_bits_to_float(hdr[r].x), dmin = f16_bits_to_float(hdr[r].x >> 16);
            const uint32_t w[8] = {v0[r].x, v0[r].y, v0[r].z, v0[r].w, v1[r].x, v1[r].y, v1[r].z, v1[r].w};
            float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
            for (int l = 0; l < 32; ++l) {
                const uint32_t byte = (w[l >> 2] >> (8 * (l & 3))) & 0xffu;
                s0 = fmaf(float(byte & 15u), x0[l], s0);
                s1 = fmaf(float(byte >> 4), x1[l], s1);
            }
            acc[r] += (d * float(sc0)) * s0 - (dmin * float(m0)) * xs0;
            acc[r] += (d * float(sc1)) * s1 - (dmin * float(m1)) * xs1;
        }
    }
}

template <int FMT, int NR>
__device__ __forceinline__ void row_dot(const uint8_t* const (&rows)[NR], const float* __restrict__ xs,
                                        const float* __restrict__ xsum, int K, int sub, int G, float (&acc)[NR]) {
    if constexpr (FMT == MOE_GGUF_Q8_0)
        row_dot_q8_0<NR>(rows, xs, K, sub, G, acc);
    else
        row_dot_q4_k<NR>(rows, xs, xsum, K, sub, G, acc);
}

// Sum over the G lanes of an aligned group (G a power of two, <= 32).
__device__ __forceinline__ float group_sum(float v, int G) {
    for (int off = G >> 1; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// fp32 copy of a bf16 vector of n elements (n a multiple of 64) into shared
// memory in the staged layout, plus its per-32 sums (sums may be null): one
// warp per 32-block, a lane per element, a warp reduction per sum.
__device__ __forceinline__ void stage_bf16(const uint16_t* __restrict__ src, int n, float* dst, float* sums) {
    const int lane = threadIdx.x & 31, warps = blockDim.x >> 5;
    for (int b = threadIdx.x >> 5; b < n / 32; b += warps) {
        const int i = 32 * b + lane;
        const float v = bf16_bits_to_float(src[i]);
        dst[i + (i >> 6)] = v;
        if (sums) {
            float s = v;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
            if (lane == 0) sums[b] = s;
        }
    }
    __syncthreads();
}

struct GgufParams {
    const uint8_t* slots;
    size_t expert_bytes;
    int S, E, H, I, T, k;
    size_t rb_h, rb_i;        // row bytes of a gate/up row (K = H) and of a down row (K = I)
    const uint16_t* x;        // bf16 [T][H]
    const int32_t* ids;       // [T*k]
    const float* w;           // [T*k]
    const int32_t* slot_of;   // [E]
    uint16_t* h;              // bf16 [T*k][I]
    float* y;                 // fp32 [T*k][H]: each assignment's down output
    float* out;               // fp32 [T][H]
    int accumulate;
};

__device__ __forceinline__ const uint8_t* expert_of(const GgufParams& p, int a) {
    const int e = p.ids[a];
    if (e < 0 || e >= p.E) return nullptr;
    const int s = p.slot_of[e];
    if (s < 0 || s >= p.S) return nullptr;
    return p.slots + size_t(s) * p.expert_bytes;
}

// grid (ceil(I / 8), T*k), 8 warps: warp w forms h[a][8 blockIdx.x + w] from
// its gate and up rows, both read in one pass.
template <int FMT>
__global__ void __launch_bounds__(kThreads) gguf_gateup_kernel(GgufParams p) {
    extern __shared__ float sh[];
    float* xs = sh;                            // staged [H]
    float* xsum = sh + staged_len(p.H);        // [H / 32]
    const int a = blockIdx.y;
    const int t = a / p.k;
    stage_bf16(p.x + size_t(t) * p.H, p.H, xs, FMT == MOE_GGUF_Q4_K ? xsum : nullptr);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * kWarps + warp;
    if (r >= p.I) return;
    const uint8_t* eb = expert_of(p, a);
    float hv = __int_as_float(0x7fc00000);
    if (eb != nullptr) {
        const uint8_t* const rows[2] = {eb + size_t(r) * p.rb_h, eb + size_t(p.I + r) * p.rb_h};
        float acc[2] = {0.0f, 0.0f};
        row_dot<FMT, 2>(rows, xs, xsum, p.H, lane, 32, acc);
        const float g = group_sum(acc[0], 32), u = group_sum(acc[1], 32);
        const float s = g / (1.0f + expf(-g));
        hv = s * u;
    }
    if (lane == 0) {
        const __nv_bfloat16 hb = __float2bfloat16_rn(hv);
        p.h[size_t(a) * p.I + r] = *reinterpret_cast<const uint16_t*>(&hb);
    }
}

// grid (ceil(H / rows_per_cta), T*k), 8 warps; each warp serves 32 / G down
// rows of assignment blockIdx.y with lane groups of G lanes: y[a][n].
template <int FMT>
__global__ void __launch_bounds__(kThreads) gguf_down_kernel(GgufParams p, int G) {
    extern __shared__ float sh[];
    const int a = blockIdx.y;
    float* hs = sh;                            // staged [I]
    float* hsum = sh + staged_len(p.I);        // [I / 32]
    stage_bf16(p.h + size_t(a) * p.I, p.I, hs, FMT == MOE_GGUF_Q4_K ? hsum : nullptr);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = (blockIdx.x * kWarps + warp) * (32 / G) + lane / G;
    const uint8_t* eb = expert_of(p, a);
    float acc[1] = {0.0f};
    if (eb != nullptr && n < p.H) {
        const uint8_t* const rows[1] = {eb + size_t(2 * p.I) * p.rb_h + size_t(n) * p.rb_i};
        row_dot<FMT, 1>(rows, hs, hsum, p.I, lane % G, G, acc);
    }
    const float y = group_sum(acc[0], G);
    if (lane % G == 0 && n < p.H) p.y[size_t(a) * p.H + n] = eb != nullptr ? y : __int_as_float(0x7fc00000);
}

// out[t][n] (+)= sum_j w[t][j] * y[t*k+j][n], j ascending, no FMA contraction.
__global__ void gguf_combine_kernel(GgufParams p) {
    const int t = blockIdx.y;
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= p.H) return;
    float acc = 0.0f;
    for (int j = 0; j < p.k; ++j) {
        const int a = t * p.k + j;
        acc = __fadd_rn(acc, __fmul_rn(p.w[a], p.y[size_t(a) * p.H + n]));
    }
    float* o = p.out + size_t(t) * p.H + n;
    *o = p.accumulate ? __fadd_rn(*o, acc) : acc;
}

template <int FMT>
int launch_gguf(const GgufParams& p, cudaStream_t s) {
    const int A = p.T * p.k;
    const size_t sm1 = (size_t(staged_len(p.H)) + p.H / 32) * sizeof(float);
    const size_t sm2 = (size_t(staged_len(p.I)) + p.I / 32) * sizeof(float);
    DeviceInfo di;
    int rc = current_device_info(&di);
    if (rc != MOE_OK) return rc;
    if (sm1 > 48 * 1024 || sm2 > 48 * 1024) return MOE_ERR_UNSUPPORTED;
    gguf_gateup_kernel<FMT><<<dim3((p.I + kWarps - 1) / kWarps, A), kThreads, sm1, s>>>(p);
    MOE_CUDA_TRY(cudaGetLastError());
    // lanes per down row: the units of a row rounded up to a power of two (at most 32)
    const int units = (FMT == MOE_GGUF_Q8_0) ? p.I / 64 : (p.I / 256) * 4;
    int G = 1;
    while (G < units && G < 32) G <<= 1;
    const int rows_per_cta = kWarps * (32 / G);
    gguf_down_kernel<FMT><<<dim3((p.H + rows_per_cta - 1) / rows_per_cta, A), kThreads, sm2, s>>>(p, G);
    MOE_CUDA_TRY(cudaGetLastError());
    gguf_combine_kernel<<<dim3((p.H + 255) / 256, p.T), 256, 0, s>>>(p);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

}  // namespace

// Bytes of one GGUF row of K elements in the formats this path runs (Q8_0
// needs K a multiple of 64 -- two blocks per lane unit -- and Q4_K a
// multiple of 256), or 0.
size_t gguf_row_bytes(int fmt, int K) {
    if (fmt == MOE_GGUF_Q8_0) return (K > 0 && K % 64 == 0) ? Unit<MOE_GGUF_Q8_0>::row_bytes(K) : 0;
    if (fmt == MOE_GGUF_Q4_K) return (K > 0 && K % 256 == 0) ? Unit<MOE_GGUF_Q4_K>::row_bytes(K) : 0;
    return 0;
}

size_t gguf_expert_bytes(int fmt, int H, int I) {
    const size_t rh = gguf_row_bytes(fmt, H), ri = gguf_row_bytes(fmt, I);
    if (!rh || !ri) return 0;
    return round_up(2 * size_t(I) * rh + size_t(H) * ri, 256);
}

int launch_gguf_ffn(int fmt, const uint8_t* slots, int S, int E, int H, int I, const uint16_t* x, int T, int k,
                    const int32_t* ids, const float* w, const int32_t* slot_of, void* ws, float* out,
                    bool accumulate, cudaStream_t s) {
    GgufParams p;
    p.slots = slots;
    p.expert_bytes = gguf_expert_bytes(fmt, H, I);
    p.S = S;
    p.E = E;
    p.H = H;
    p.I = I;
    p.T = T;
    p.k = k;
    p.rb_h = gguf_row_bytes(fmt, H);
    p.rb_i = gguf_row_bytes(fmt, I);
    p.x = x;
    p.ids = ids;
    p.w = w;
    p.slot_of = slot_of;
    p.h = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + gguf_h_offset());
    p.y = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + gguf_y_offset(T, k, I));
    p.out = out;
    p.accumulate = accumulate ? 1 : 0;
    if (T == 0) return MOE_OK;
    // decode-sized calls whose rows suit bulk copies take the single-launch kernel
    if (T * k <= 32 && reinterpret_cast<uintptr_t>(x) % 16 == 0 && gguf_fused_supported(fmt, T, k, H, I))
        return launch_gguf_fused(fmt, slots, S, E, H, I, x, T, k, ids, w, slot_of, nullptr, ws, out, accumulate, s);
    return fmt == MOE_GGUF_Q8_0 ? launch_gguf<MOE_GGUF_Q8_0>(p, s) : launch_gguf<MOE_GGUF_Q4_K>(p, s);
}

}  // namespace moe
