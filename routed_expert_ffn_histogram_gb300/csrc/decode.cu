// Decode path of the expert FFN: fused MXFP4 dequant + GEMV on CUDA cores.
//
// Source: tinyserve README, "How it works" item 2 -- each expert is a gate,
// an up and a down product computed directly on the quantised bytes, with no
// intermediate BF16 weights; llama.cpp discussion "fixed GPU expert working
// set with Native CPU miss execution", main post -- the routed experts'
// outputs are merged with the routing weights.  Number formats: OCP MX v1.0
// (E2M1 elements, one E8M0 scale per 32 along the reduction dimension).
//
// Arithmetic: bf16 activation x fp32-dequantised fp4, fp32 accumulation;
// SwiGLU h = bf16(silu(g) * u); down product on bf16(h); the combine sums
// w_j * y_j in ascending j.  Each E2M1 x bf16 product is exact in fp32.
//
// Kernels (both HBM-bound: every weight byte is read once per call):
//   gateup: one warp per (assignment, row) item reads the gate row and the up
//           row (they sit 32 rows apart in the native layout), one 16-byte
//           load = 32 codes = exactly one MX block per lane; x is staged in
//           shared memory (bf16, 16-byte chunks XOR-swizzled so a warp's
//           LDS.128 is conflict-free);
//   down:   one warp per output row of a token reads that row of all k
//           experts and applies the routing weights in rank order, so the
//           combine is fused and deterministic.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
    return b ? __uint_as_float(b << 23) : __uint_as_float(0x00400000u);
}

// Index of the 16-byte chunk q (0..3) of 32-element block b in shared memory.
__device__ __forceinline__ int swz(int b, int q) { return b * 4 + (q ^ ((b >> 1) & 3)); }

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ldg_u8(const uint8_t* p) {
    return (uint32_t)__ldg(p);
}

// Eight E2M1 codes (one 32-bit word, element 2i in the low nibble of byte i)
// to fp32.
__device__ __forceinline__ void e2m1x8(uint32_t word, float (&f)[8]) {
    uint32_t h[4];
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(word));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 hh = *reinterpret_cast<__half2*>(&h[i]);
        float2 ff = __half22float2(hh);
        f[2 * i] = ff.x;
        f[2 * i + 1] = ff.y;
    }
}

__device__ __forceinline__ void bf16x8(uint4 v, float (&f)[8]) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(u[i] << 16);
        f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Dot of one MX block (codes c, scale byte s) with the staged block b.
__device__ __forceinline__ float block_dot(const uint4 c, const uint4* __restrict__ xs, int b) {
    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
    float acc = 0.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float wf[8], xf[8];
        e2m1x8(cw[q], wf);
        bf16x8(xs[swz(b, q)], xf);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc = fmaf(wf[i], xf[i], acc);
    }
    return acc;
}

struct DecodeParams {
    const uint8_t* slots;
    size_t expert_bytes;
    int S, E, H, I, k;
    size_t rs_gu, rs_d, d_off;
    const uint16_t* x;
    const int32_t* ids;
    const float* w;
    const int32_t* slot_of;
    uint16_t* h;      // bf16 [T*k][I]
    float* out;       // fp32 [T][H]
    int accumulate;   // out += result
};

__device__ __forceinline__ const uint8_t* expert_base(const DecodeParams& p, int a) {
    const int e = p.ids[a];
    if (e < 0 || e >= p.E) return nullptr;
    const int s = p.slot_of[e];
    if (s < 0 || s >= p.S) return nullptr;
    return p.slots + (size_t)s * p.expert_bytes;
}

// Stage one bf16 row of K elements (K/32 blocks) into swizzled shared memory.
__device__ __forceinline__ void stage_row(const uint16_t* __restrict__ src, int K, uint4* dst) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    for (int c = threadIdx.x; c < K / 8; c += kThreads) dst[swz(c >> 2, c & 3)] = s4[c];
}

template <int NIT>
__global__ void __launch_bounds__(kThreads) decode_gateup_kernel(DecodeParams p) {
    extern __shared__ uint4 xs[];
    const int t = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    stage_row(p.x + (size_t)t * p.H, p.H, xs);
    __syncthreads();
    const int nb = p.H / 32;
    const int items = p.k * p.I;
    for (int item = blockIdx.x * kWarps + warp; item < items; item += gridDim.x * kWarps) {
        const int j = item / p.I, r = item - j * p.I;
        const int a = t * p.k + j;
        const uint8_t* base = expert_base(p, a);
        if (base == nullptr) {
            if (lane == 0) p.h[(size_t)a * p.I + r] = 0x7fc0;  // NaN: routed expert not resident
            continue;
        }
        const uint8_t* g = base + Layout::gate_row(r) * p.rs_gu;
        const uint8_t* u = g + Layout::kChunk * p.rs_gu;
        uint4 cg[NIT], cu[NIT];
        uint32_t sg[NIT], su[NIT];
#pragma unroll
        for (int i = 0; i < NIT; ++i) {
            const int b = lane + 32 * i;
            if (b < nb) {
                cg[i] = ldg_stream(g + 16 * b);
                cu[i] = ldg_stream(u + 16 * b);
                sg[i] = ldg_u8(g + p.H / 2 + b);
                su[i] = ldg_u8(u + p.H / 2 + b);
            }
        }
        float ag = 0.0f, au = 0.0f;
#pragma unroll
        for (int i = 0; i < NIT; ++i) {
            const int b = lane + 32 * i;
            if (b < nb) {
                const uint32_t cwg[4] = {cg[i].x, cg[i].y, cg[i].z, cg[i].w};
                const uint32_t cwu[4] = {cu[i].x, cu[i].y, cu[i].z, cu[i].w};
                float dg = 0.0f, du = 0.0f;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float xf[8], wg[8], wu[8];
                    bf16x8(xs[swz(b, q)], xf);
                    e2m1x8(cwg[q], wg);
                    e2m1x8(cwu[q], wu);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        dg = fmaf(wg[e], xf[e], dg);
                        du = fmaf(wu[e], xf[e], du);
                    }
                }
                ag = fmaf(dg, e8m0_to_f32(sg[i]), ag);
                au = fmaf(du, e8m0_to_f32(su[i]), au);
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
}

// Experts whose rows one warp loads before it computes (bounds registers).
template <int NIT>
struct DownBatch {
    static constexpr int value = NIT >= 3 ? 2 : 4;
};

template <int NIT>
__global__ void __launch_bounds__(kThreads) decode_down_kernel(DecodeParams p) {
    extern __shared__ uint4 hs[];  // k rows of I bf16, each swizzled
    const int t = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nb = p.I / 32;
    for (int j = 0; j < p.k; ++j)
        stage_row(p.h + ((size_t)t * p.k + j) * p.I, p.I, hs + (size_t)j * (p.I / 8));
    __syncthreads();
    constexpr int JB = DownBatch<NIT>::value;
    for (int r = blockIdx.x * kWarps + warp; r < p.H; r += gridDim.x * kWarps) {
        float out = 0.0f;
        bool bad = false;
        for (int j0 = 0; j0 < p.k; j0 += JB) {
            uint4 c[JB][NIT];
            uint32_t sc[JB][NIT];
#pragma unroll
            for (int jj = 0; jj < JB; ++jj) {
                const int j = j0 + jj;
                if (j >= p.k) break;
                const uint8_t* base = expert_base(p, t * p.k + j);
                if (base == nullptr) { bad = true; continue; }
                const uint8_t* row = base + p.d_off + (size_t)r * p.rs_d;
#pragma unroll
                for (int i = 0; i < NIT; ++i) {
                    const int b = lane + 32 * i;
                    if (b < nb) {
                        c[jj][i] = ldg_stream(row + 16 * b);
                        sc[jj][i] = ldg_u8(row + p.I / 2 + b);
                    }
                }
            }
#pragma unroll
            for (int jj = 0; jj < JB; ++jj) {
                const int j = j0 + jj;
                if (j >= p.k) break;
                if (expert_base(p, t * p.k + j) == nullptr) continue;
                const uint4* hj = hs + (size_t)j * (p.I / 8);
                float acc = 0.0f;
#pragma unroll
                for (int i = 0; i < NIT; ++i) {
                    const int b = lane + 32 * i;
                    if (b < nb) acc = fmaf(block_dot(c[jj][i], hj, b), e8m0_to_f32(sc[jj][i]), acc);
                }
                const float y = warp_sum(acc);
                out = __fadd_rn(out, __fmul_rn(p.w[t * p.k + j], y));
            }
        }
        if (lane == 0) {
            float* o = p.out + (size_t)t * p.H + r;
            const float v = bad ? __int_as_float(0x7fc00000) : out;
            *o = p.accumulate ? __fadd_rn(*o, v) : v;
        }
    }
}

// Per-device launch shape of a kernel: occupancy (blocks per SM) for its
// dynamic shared memory, computed once outside any stream capture.
struct LaunchCache {
    int occ[64] = {};
    size_t smem[64] = {};
};

template <typename K>
int occupancy(K kernel, LaunchCache& c, size_t smem, const DeviceInfo& di, int* occ) {
    if (di.device < 0 || di.device >= 64) return MOE_ERR_UNSUPPORTED;
    if (c.occ[di.device] == 0 || c.smem[di.device] < smem) {
        const size_t s = smem < 48 * 1024 ? 48 * 1024 : smem;
        MOE_CUDA_TRY(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s));
        int o = 0;
        MOE_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kernel, kThreads, s));
        c.occ[di.device] = o > 0 ? o : 1;
        c.smem[di.device] = s;
    }
    *occ = c.occ[di.device];
    return MOE_OK;
}

template <int NIT>
int launch_nit(const DecodeParams& p, int T, cudaStream_t s) {
    static LaunchCache cache;
    DeviceInfo di;
    int rc = current_device_info(&di);
    if (rc != MOE_OK) return rc;
    const size_t smem = size_t(p.H) * 2;
    if (smem > di.smem_optin) return MOE_ERR_UNSUPPORTED;
    int occ = 1;
    rc = occupancy(decode_gateup_kernel<NIT>, cache, smem, di, &occ);
    if (rc != MOE_OK) return rc;
    const int items = p.k * p.I;
    int gx = (items + kWarps - 1) / kWarps;
    const int cap = max(1, di.sms * occ / max(T, 1));
    gx = max(1, min(gx, cap));
    decode_gateup_kernel<NIT><<<dim3(gx, T), kThreads, smem, s>>>(p);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

template <int NIT>
int launch_down_nit(const DecodeParams& p, int T, cudaStream_t s) {
    static LaunchCache cache;
    DeviceInfo di;
    int rc = current_device_info(&di);
    if (rc != MOE_OK) return rc;
    const size_t smem = size_t(p.k) * p.I * 2;
    if (smem > di.smem_optin) return MOE_ERR_UNSUPPORTED;
    int occ = 1;
    rc = occupancy(decode_down_kernel<NIT>, cache, smem, di, &occ);
    if (rc != MOE_OK) return rc;
    int gx = (p.H + kWarps - 1) / kWarps;
    const int cap = max(1, di.sms * occ / max(T, 1));
    gx = max(1, min(gx, cap));
    decode_down_kernel<NIT><<<dim3(gx, T), kThreads, smem, s>>>(p);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

}  // namespace

// Decode workspace: [0, 256) control words (zero between calls), then h as
// bf16 [T*k][I] (two-kernel path), then the fp32 [T][H] accumulator of the
// fused kernel (zero between calls).
size_t decode_acc_offset(int T, int k, int I) { return 256 + round_up(size_t(T) * k * I * 2, 256); }

size_t decode_workspace_bytes(int T, int k, int H, int I) {
    return decode_acc_offset(T, k, I) + round_up(size_t(T) * H * 4, 256);
}

int launch_decode_ffn(const FfnArgs& a, void* ws, size_t ws_bytes, cudaStream_t s) {
    const Layout& L = *a.L;
    if (ws_bytes < decode_workspace_bytes(a.T, a.k, L.H, L.I)) return MOE_ERR_INVALID;
    if (L.H > 4096 || L.I > 4096 * 4) return MOE_ERR_UNSUPPORTED;
    if (a.T == 0) return MOE_OK;
    // one kernel per layer when the activations and a work-item ring fit
    // in shared memory; otherwise a gate/up launch and a down launch (which
    // read the row-major down matrix, absent from decode-only staged pools)
    if (decode_fused_smem(a.T, a.k, L.H, L.I) != 0) {
        const int rc = launch_decode_fused(a, ws, s);
        if (rc != MOE_ERR_UNSUPPORTED) return rc;
    }
    if (a.decode_parts_only || a.skip_absent) return MOE_ERR_UNSUPPORTED;
    DecodeParams p;
    p.slots = a.slots;
    p.expert_bytes = a.expert_bytes;
    p.S = a.S;
    p.E = a.E;
    p.H = L.H;
    p.I = L.I;
    p.k = a.k;
    p.rs_gu = L.rs_gu;
    p.rs_d = L.rs_d;
    p.d_off = L.d_off;
    p.x = a.x;
    p.ids = a.ids;
    p.w = a.w;
    p.slot_of = a.slot_of;
    p.h = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + 256);
    p.out = a.out;
    p.accumulate = a.accumulate ? 1 : 0;
    const int nit_gu = (L.H / 32 + 31) / 32;
    int rc;
    switch (nit_gu) {
        case 1: rc = launch_nit<1>(p, a.T, s); break;
        case 2: rc = launch_nit<2>(p, a.T, s); break;
        case 3: rc = launch_nit<3>(p, a.T, s); break;
        case 4: rc = launch_nit<4>(p, a.T, s); break;
        default: return MOE_ERR_UNSUPPORTED;
    }
    if (rc != MOE_OK) return rc;
    const int nit_d = (L.I / 32 + 31) / 32;
    switch (nit_d) {
        case 1: return launch_down_nit<1>(p, a.T, s);
        case 2: return launch_down_nit<2>(p, a.T, s);
        case 3: return launch_down_nit<3>(p, a.T, s);
        case 4: return launch_down_nit<4>(p, a.T, s);
        default: return MOE_ERR_UNSUPPORTED;
    }
}

}  // namespace moe
