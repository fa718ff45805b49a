// Prefill-side elementwise kernels: MXFP8 quantisation of activations
// (gathered into grouped order) and the weighted combine of grouped expert
// outputs.
//
// MXFP8 rule (OCP Microscaling Formats v1.0, section 6.3): per block of 32
// along the reduction dimension, shared exponent = floor(log2(amax)) - 8
// (8 = largest E4M3 exponent), stored as an E8M0 byte clamped to [0, 254]
// (0 for an all-zero block); elements are E4M3 with round-to-nearest-even
// and saturation of finite overflow to +-448.
//
// Combine: llama.cpp discussion "fixed GPU expert working set with Native
// CPU miss execution", main post -- routed experts' outputs are merged with
// the routing weights; here in ascending rank j, fp32, without fused
// multiply-add so the sum is the plain w*y + acc sequence.
#include "internal.h"

namespace moe {
namespace {

__device__ __forceinline__ uint32_t e8m0_of_amax(float amax) {
    const uint32_t bits = __float_as_uint(amax);
    const int ef = int((bits >> 23) & 0xffu);
    if (amax == 0.0f || ef == 0) return 0u;  // zero or subnormal amax clamps to 0
    return uint32_t(min(max(ef - 8, 0), 254));
}

// 2^(127 - sb) as fp32 (sb in [0, 254]).
__device__ __forceinline__ float inv_scale(uint32_t sb) {
    const int ef = 254 - int(sb);
    return ef > 0 ? __uint_as_float(uint32_t(ef) << 23) : __uint_as_float(0x00400000u);
}

__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// One lane quantises one 32-element block (64 bytes of bf16 in, 32 codes +
// 1 scale out); a warp handles a run of 32 consecutive blocks of one row.
__device__ __forceinline__ void quant_block(const uint16_t* __restrict__ xrow, int b, bool act, uint32_t (&w)[8],
                                            uint32_t& sb) {
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = 0;
    sb = 0;
    if (!act) return;
    const uint4* p = reinterpret_cast<const uint4*>(xrow + (size_t)b * 32);
    uint4 v[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) v[c] = __ldg(p + c);
    float f[32];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t u[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f[c * 8 + 2 * j] = __uint_as_float(u[j] << 16);
            f[c * 8 + 2 * j + 1] = __uint_as_float(u[j] & 0xffff0000u);
        }
    }
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(f[j]));
    sb = e8m0_of_amax(amax);
    const float m = inv_scale(sb);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t a = cvt_e4m3x2(f[4 * j] * m, f[4 * j + 1] * m);
        const uint32_t c = cvt_e4m3x2(f[4 * j + 2] * m, f[4 * j + 3] * m);
        w[j] = a | (c << 16);
    }
}

// Stores a warp's run of quantised blocks (lane l holds block b0 + l) to
// row `out` (already offset to block b0): the warp exchanges halves with
// shuffles so that each store instruction writes 512 contiguous bytes
// (blocks 16i..16i+15 of the run) rather than 16 bytes in each of 32 blocks.
__device__ __forceinline__ void store_run(uint8_t* out, const uint32_t (&w)[8], int nvalid, int lane) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int srcl = 16 * i + (lane >> 1);
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t lo = __shfl_sync(0xffffffffu, w[j], srcl);
            const uint32_t hi = __shfl_sync(0xffffffffu, w[4 + j], srcl);
            o[j] = (lane & 1) ? hi : lo;
        }
        if (srcl < nvalid)
            *reinterpret_cast<uint4*>(out + 512 * i + 16 * lane) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// Gather form: output row r is the quantised x row perm[r] / k (or r when
// perm is null).  Warp w handles blocks 32c..32c+31 of output row r,
// (r, c) = divmod(w, warps_per_row).
__global__ void __launch_bounds__(256) quant_mxfp8_kernel(const uint16_t* __restrict__ x, int K,
                                                          const int32_t* __restrict__ perm, int k, int rows,
                                                          uint8_t* __restrict__ q, uint8_t* __restrict__ scales,
                                                          int scale_stride, int warps_per_row) {
    const int nb = K / 32;
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int row = gw / warps_per_row;               // warp-uniform
    const int b0 = (gw - row * warps_per_row) * 32;
    if (row >= rows) return;                           // whole warp
    const int nvalid = min(32, nb - b0);
    const int src = perm ? perm[row] / k : row;
    uint32_t w[8], sb;
    quant_block(x + (size_t)src * K, b0 + lane, lane < nvalid, w, sb);
    if (lane < nvalid) scales[(size_t)row * scale_stride + b0 + lane] = uint8_t(sb);
    store_run(q + (size_t)row * K + (size_t)b0 * 32, w, nvalid, lane);
}

// Scatter form for the grouped prefill operand: token t's row is read and
// quantised once, then written to the grouped rows inv[t*k + j], j < k.
// (Quantisation does not depend on the expert, and reading each token once
// keeps x from being re-read from DRAM k times in grouped order.)
__global__ void __launch_bounds__(256) quant_mxfp8_scatter_kernel(const uint16_t* __restrict__ x, int K,
                                                                  const int32_t* __restrict__ inv, int k, int T,
                                                                  uint8_t* __restrict__ q,
                                                                  uint8_t* __restrict__ scales, int scale_stride,
                                                                  int warps_per_row) {
    const int nb = K / 32;
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int t = gw / warps_per_row;                 // warp-uniform
    const int b0 = (gw - t * warps_per_row) * 32;
    if (t >= T) return;                                // whole warp
    const int nvalid = min(32, nb - b0);
    uint32_t w[8], sb;
    quant_block(x + (size_t)t * K, b0 + lane, lane < nvalid, w, sb);
    for (int j = 0; j < k; ++j) {
        const int row = inv[(size_t)t * k + j];
        if (lane < nvalid) scales[(size_t)row * scale_stride + b0 + lane] = uint8_t(sb);
        store_run(q + (size_t)row * K + (size_t)b0 * 32, w, nvalid, lane);
    }
}

// out[t][h] = sum_j w[t][j] * y[inv[t*k+j]][h]; one thread per 4 outputs.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y, const float* __restrict__ w,
                                                      const int32_t* __restrict__ inv, int T, int k, int H,
                                                      float* __restrict__ out) {
    const int h4 = H / 4;
    const long total = (long)T * h4;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
        const int t = int(i / h4), c = int(i - (long)t * h4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const float wj = w[(size_t)t * k + j];
            const float4 v = __ldg(reinterpret_cast<const float4*>(y + (size_t)inv[(size_t)t * k + j] * H) + c);
            acc.x = __fadd_rn(acc.x, __fmul_rn(wj, v.x));
            acc.y = __fadd_rn(acc.y, __fmul_rn(wj, v.y));
            acc.z = __fadd_rn(acc.z, __fmul_rn(wj, v.z));
            acc.w = __fadd_rn(acc.w, __fmul_rn(wj, v.w));
        }
        reinterpret_cast<float4*>(out + (size_t)t * H)[c] = acc;
    }
}

__global__ void __launch_bounds__(256) combine_scalar_kernel(const float* __restrict__ y,
                                                             const float* __restrict__ w,
                                                             const int32_t* __restrict__ inv, int T, int k,
                                                             int H, float* __restrict__ out) {
    const long total = (long)T * H;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
        const int t = int(i / H), c = int(i - (long)t * H);
        float acc = 0.0f;
        for (int j = 0; j < k; ++j)
            acc = __fadd_rn(acc, __fmul_rn(w[(size_t)t * k + j], y[(size_t)inv[(size_t)t * k + j] * H + c]));
        out[(size_t)t * H + c] = acc;
    }
}

int grid_for(long work, int threads) {
    DeviceInfo di;
    if (current_device_info(&di) != MOE_OK) return 1;
    long g = (work + threads - 1) / threads;
    const long cap = long(di.sms) * 8;
    return int(g < 1 ? 1 : (g > cap ? cap : g));
}

}  // namespace

// MXFP4 quantisation of bf16 rows (OCP MX v1.0: E2M1 elements, shared
// exponent floor(log2(amax)) - 2, E8M0 byte clamped to [0, 254], RNE with
// finite overflow saturated to +-6), codes packed two per byte with element
// 2i in the low nibble.  One thread per 32-element block: 64 bytes in, 16
// code bytes and one scale byte out.
__global__ void __launch_bounds__(256) quant_mxfp4_kernel(const uint16_t* __restrict__ x, int K, long blocks,
                                                          uint8_t* __restrict__ q, uint8_t* __restrict__ scales,
                                                          int scale_stride) {
    const long g = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= blocks) return;
    const int nb = K / 32;
    const long row = g / nb;
    const int b = int(g - row * nb);
    const uint4* src = reinterpret_cast<const uint4*>(x + row * K + (long)b * 32);
    uint32_t w[16];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint4 v = __ldg(src + c);
        w[4 * c] = v.x;
        w[4 * c + 1] = v.y;
        w[4 * c + 2] = v.z;
        w[4 * c + 3] = v.w;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        amax = fmaxf(amax, fabsf(__uint_as_float(w[i] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(w[i] & 0xffff0000u)));
    }
    const int ef = int((__float_as_uint(amax) >> 23) & 0xffu);
    // floor(log2 amax) = ef - 127 for normal amax; bf16 subnormals land far
    // below the clamp, which gives byte 0 as well
    const int sb = (amax == 0.0f || ef == 0) ? 0 : min(max(ef - 127 - 2 + 127, 0), 254);
    const float mul = ldexpf(1.0f, 127 - sb);
    uint32_t out[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t r;
        // four bytes, each two E2M1 codes: element 2i in the low nibble
        asm("{\n\t.reg .b8 c0, c1, c2, c3;\n\t"
            "cvt.rn.satfinite.e2m1x2.f32 c0, %2, %1;\n\t"
            "cvt.rn.satfinite.e2m1x2.f32 c1, %4, %3;\n\t"
            "cvt.rn.satfinite.e2m1x2.f32 c2, %6, %5;\n\t"
            "cvt.rn.satfinite.e2m1x2.f32 c3, %8, %7;\n\t"
            "mov.b32 %0, {c0, c1, c2, c3};\n\t}"
            : "=r"(r)
            : "f"(__uint_as_float(w[4 * j] << 16) * mul), "f"(__uint_as_float(w[4 * j] & 0xffff0000u) * mul),
              "f"(__uint_as_float(w[4 * j + 1] << 16) * mul), "f"(__uint_as_float(w[4 * j + 1] & 0xffff0000u) * mul),
              "f"(__uint_as_float(w[4 * j + 2] << 16) * mul), "f"(__uint_as_float(w[4 * j + 2] & 0xffff0000u) * mul),
              "f"(__uint_as_float(w[4 * j + 3] << 16) * mul), "f"(__uint_as_float(w[4 * j + 3] & 0xffff0000u) * mul));
        out[j] = r;
    }
    *reinterpret_cast<uint4*>(q + row * (K / 2) + (long)b * 16) = make_uint4(out[0], out[1], out[2], out[3]);
    scales[row * scale_stride + b] = uint8_t(sb);
}

int launch_quant_mxfp4(const uint16_t* x, int K, int rows, uint8_t* q, uint8_t* scales, int scale_stride,
                       cudaStream_t s) {
    const long blocks = (long)rows * (K / 32);
    const long grid = (blocks + 255) / 256;
    if (grid > 0x7fffffffL) return MOE_ERR_UNSUPPORTED;
    if (grid == 0) return MOE_OK;
    quant_mxfp4_kernel<<<(unsigned)grid, 256, 0, s>>>(x, K, blocks, q, scales, scale_stride);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

int launch_quant_mxfp8(const uint16_t* x, int K, const int32_t* perm, int k, int rows, uint8_t* q,
                       uint8_t* scales, int scale_stride, cudaStream_t s) {
    // one warp per 32 blocks of a row: the gather (perm, then x) is a
    // dependent load chain, so memory parallelism comes from many warps
    const int warps_per_row = (K / 32 + 31) / 32;
    const long warps = (long)rows * warps_per_row;
    const long grid = (warps + 7) / 8;
    if (grid > 0x7fffffffL || warps > 0x7fffffffL) return MOE_ERR_UNSUPPORTED;
    if (grid == 0) return MOE_OK;
    quant_mxfp8_kernel<<<(unsigned)grid, 256, 0, s>>>(x, K, perm, k, rows, q, scales, scale_stride, warps_per_row);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

int launch_quant_mxfp8_scatter(const uint16_t* x, int K, const int32_t* inv, int k, int T, uint8_t* q,
                               uint8_t* scales, int scale_stride, cudaStream_t s) {
    const int warps_per_row = (K / 32 + 31) / 32;
    const long warps = (long)T * warps_per_row;
    const long grid = (warps + 7) / 8;
    if (grid > 0x7fffffffL || warps > 0x7fffffffL) return MOE_ERR_UNSUPPORTED;
    if (grid == 0) return MOE_OK;
    quant_mxfp8_scatter_kernel<<<(unsigned)grid, 256, 0, s>>>(x, K, inv, k, T, q, scales, scale_stride,
                                                              warps_per_row);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

int launch_combine(const float* y, const float* w, const int32_t* inv, int T, int k, int H, float* out,
                   cudaStream_t s) {
    const bool vec = (H % 4 == 0) && (reinterpret_cast<uintptr_t>(y) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(out) % 16 == 0);
    if (vec) {
        combine_kernel<<<grid_for((long)T * (H / 4), 256), 256, 0, s>>>(y, w, inv, T, k, H, out);
    } else {
        combine_scalar_kernel<<<grid_for((long)T * H, 256), 256, 0, s>>>(y, w, inv, T, k, H, out);
    }
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

}  // namespace moe
