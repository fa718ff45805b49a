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
// Shape: one CTA per SM (or as many as fit), 16 warps each, all co-resident
// (cooperative launch).
//   phase 1  every warp takes (token, expert, row) items: the gate row and
//            the up row (64 rows apart in the packed layout), one 16-byte
//            load = one MX block per lane, x staged once per CTA in shared
//            memory as fp32 (XOR-swizzled 16-byte chunks, conflict-free),
//            products accumulated with packed fp32x2 FMAs; lane 0 writes
//            bf16(silu(g) * u).  Meanwhile each CTA asks L2 to prefetch its
//            share of the routed experts' down matrices, so HBM stays busy
//            across the phase boundary and phase 2 reads from L2.
//   barrier  bounded grid barrier (arrival counter zeroed before launch).
//   phase 2  h of a token staged per CTA (bf16, swizzled); every warp takes
//            output rows, reads that row of all k experts, and folds
//            w_j * y_j in rank order.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#include "internal.h"

namespace moe {
namespace {

constexpr int kThreads = 768;
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
__device__ __forceinline__ float block_dot_f16(const uint4 c, const uint4* __restrict__ xs, int b) {
    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 xv = xs[hswz(b, q)];
        uint32_t wv[4];
        e2m1x8_f16(cw[q], wv);
        fma2_f16_f32(a0, a1, wv[0], xv.x);
        fma2_f16_f32(a0, a1, wv[1], xv.y);
        fma2_f16_f32(a0, a1, wv[2], xv.z);
        fma2_f16_f32(a0, a1, wv[3], xv.w);
    }
    return a0 + a1;
}

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
    unsigned* bar;     // [0] arrivals (zeroed before launch), [1] error bits
};

__device__ __forceinline__ const uint8_t* expert_of(const FusedParams& p, int a) {
    const int e = p.ids[a];
    if (e < 0 || e >= p.E) return nullptr;
    const int s = p.slot_of[e];
    if (s < 0 || s >= p.S) return nullptr;
    return p.slots + (size_t)s * p.expert_bytes;
}

__device__ bool grid_barrier(unsigned* bar, unsigned target, int* ok_smem) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(bar, 1u);
        int ok = 1;
        for (uint32_t i = 0;; ++i) {
            unsigned v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(bar) : "memory");
            if (v >= target) break;
            if (i >= kBarrierLimit) {
                atomicOr(bar + 1, 1u);
                ok = 0;
                break;
            }
            __nanosleep(64);
        }
        __threadfence();
        *ok_smem = ok;
    }
    __syncthreads();
    return *ok_smem != 0;
}

template <int NG, int ND>
__global__ void __launch_bounds__(kThreads, 1) decode_fused_kernel(FusedParams p) {
    extern __shared__ uint4 sm4[];
    __shared__ int ok_smem;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = gridDim.x;
    const int A = p.T * p.k;

    // L2 prefetch of this CTA's share of the routed down matrices
    if (threadIdx.x == 0) {
        const size_t dbytes = (size_t)p.H * p.rs_d;
        const size_t total = (size_t)A * dbytes;
        size_t lo = (total * blockIdx.x / G) & ~size_t(15), hi = (total * (blockIdx.x + 1) / G) & ~size_t(15);
        if (blockIdx.x + 1 == (unsigned)G) hi = total;
        while (lo < hi) {
            const int a = int(lo / dbytes);
            const size_t in = lo - (size_t)a * dbytes;
            const size_t n = min(min(hi - lo, dbytes - in), size_t(1) << 16);
            const uint8_t* base = expert_of(p, a);
            if (base != nullptr && n >= 16)
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(base + p.d_off + in),
                             "r"(uint32_t(n & ~size_t(15)))
                             : "memory");
            lo += n;
        }
    }

    // ---- phase 1: gate/up + SwiGLU ----
    const int nbx = p.H / 32;
    {
        uint4* xs = sm4;
        int* xe = reinterpret_cast<int*>(sm4 + (size_t)p.T * nbx * 4);
        for (int c = threadIdx.x; c < p.T * nbx; c += kThreads) {
            const int t = c / nbx, b = c - t * nbx;
            stage_block_f16(p.x + (size_t)t * p.H, xs + (size_t)t * nbx * 4, b, xe + t * nbx);
        }
        __syncthreads();
        const int items = A * p.I;
        for (int item = blockIdx.x * kWarps + warp; item < items; item += G * kWarps) {
            const int a = item / p.I, r = item - a * p.I;
            const int t = a / p.k;
            const uint8_t* eb = expert_of(p, a);
            if (eb == nullptr) {
                if (lane == 0) p.h[(size_t)a * p.I + r] = 0x7fc0;
                continue;
            }
            const uint8_t* g = eb + Layout::gate_row(r) * p.rs_gu;
            const uint8_t* u = g + 64 * p.rs_gu;
            uint4 cg[NG], cu[NG];
            int sg[NG], su[NG];
#pragma unroll
            for (int i = 0; i < NG; ++i) {
                const int b = lane + 32 * i;
                if (b < nbx) {
                    cg[i] = ld_stream(g + 16 * b);
                    cu[i] = ld_stream(u + 16 * b);
                    sg[i] = __ldg(g + p.H / 2 + b);
                    su[i] = __ldg(u + p.H / 2 + b);
                }
            }
            const uint4* xt = xs + (size_t)t * nbx * 4;
            const int* et = xe + t * nbx;
            float ag = 0.0f, au = 0.0f;
#pragma unroll
            for (int i = 0; i < NG; ++i) {
                const int b = lane + 32 * i;
                if (b < nbx) {
                    float dg, du;
                    block_dot2_f16(cg[i], cu[i], xt, b, dg, du);
                    const int e = et[b];
                    ag = fmaf(dg, pow2_biased(sg[i] + e), ag);
                    au = fmaf(du, pow2_biased(su[i] + e), au);
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

    const bool ok = grid_barrier(p.bar, (unsigned)G, &ok_smem);

    // ---- phase 2: down + weighted combine ----
    uint4* hs = sm4;
    const int nbh = p.I / 32;
    int* he = reinterpret_cast<int*>(sm4 + (size_t)p.k * nbh * 4);
    for (int t = 0; t < p.T; ++t) {
        __syncthreads();
        for (int c = threadIdx.x; c < p.k * nbh; c += kThreads) {
            const int j = c / nbh, b = c - j * nbh;
            stage_block_f16(p.h + ((size_t)t * p.k + j) * p.I, hs + (size_t)j * nbh * 4, b, he + j * nbh);
        }
        __syncthreads();
        for (int r = blockIdx.x * kWarps + warp; r < p.H; r += G * kWarps) {
            float out = 0.0f;
            bool bad = !ok;
            for (int j0 = 0; j0 < p.k && !bad; j0 += 2) {
                uint4 c[2][ND];
                int sc[2][ND];
                const uint8_t* rows[2];
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const int j = j0 + jj;
                    rows[jj] = nullptr;
                    if (j < p.k) {
                        const uint8_t* eb = expert_of(p, t * p.k + j);
                        if (eb == nullptr) bad = true;
                        else rows[jj] = eb + p.d_off + (size_t)r * p.rs_d;
                    }
                    if (rows[jj] != nullptr) {
#pragma unroll
                        for (int i = 0; i < ND; ++i) {
                            const int b = lane + 32 * i;
                            if (b < nbh) {
                                c[jj][i] = __ldg(reinterpret_cast<const uint4*>(rows[jj] + 16 * b));
                                sc[jj][i] = __ldg(rows[jj] + p.I / 2 + b);
                            }
                        }
                    }
                }
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    if (rows[jj] == nullptr) continue;
                    const int j = j0 + jj;
                    const uint4* hj = hs + (size_t)j * nbh * 4;
                    const int* ej = he + j * nbh;
                    float acc = 0.0f;
#pragma unroll
                    for (int i = 0; i < ND; ++i) {
                        const int b = lane + 32 * i;
                        if (b < nbh) {
                            acc = fmaf(block_dot_f16(c[jj][i], hj, b), pow2_biased(sc[jj][i] + ej[b]), acc);
                        }
                    }
                    const float y = warp_sum(acc);
                    out = __fadd_rn(out, __fmul_rn(p.w[t * p.k + j], y));
                }
            }
            if (lane == 0) p.out[(size_t)t * p.H + r] = bad ? __int_as_float(0x7fc00000) : out;
        }
    }
}

}  // namespace

// Shared memory the fused kernel needs, or 0 if the shape does not fit it.
size_t decode_fused_smem(int T, int k, int H, int I) {
    const size_t x = size_t(T) * H * 2 + size_t(T) * (H / 32) * 4;
    const size_t h = size_t(k) * I * 2 + size_t(k) * (I / 32) * 4;
    const size_t s = x > h ? x : h;
    return s <= 96 * 1024 ? s : 0;
}

int launch_decode_fused(const FfnArgs& a, void* ws, cudaStream_t s) {
    const Layout& L = *a.L;
    DeviceInfo di;
    int rc = current_device_info(&di);
    if (rc != MOE_OK) return rc;
    const size_t smem = decode_fused_smem(a.T, a.k, L.H, L.I);
    if (smem == 0) return MOE_ERR_UNSUPPORTED;
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
    const int ng = (L.H / 32 + 31) / 32, nd = (L.I / 32 + 31) / 32;
    void (*kern)(FusedParams) = nullptr;
#define MOE_PICK(G_, D_) \
    if (ng == G_ && nd == D_) kern = decode_fused_kernel<G_, D_>;
    MOE_PICK(1, 1) MOE_PICK(1, 2) MOE_PICK(2, 1) MOE_PICK(2, 2) MOE_PICK(3, 3) MOE_PICK(3, 1)
    MOE_PICK(1, 3) MOE_PICK(4, 4) MOE_PICK(2, 4) MOE_PICK(4, 2) MOE_PICK(3, 2) MOE_PICK(2, 3)
#undef MOE_PICK
    if (kern == nullptr) return MOE_ERR_UNSUPPORTED;
    static int occ_cache[64][16] = {};
    const int slot = (ng - 1) * 4 + (nd - 1);
    if (di.device >= 64) return MOE_ERR_UNSUPPORTED;
    if (occ_cache[di.device][slot] == 0) {
        MOE_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024));
        int occ = 0;
        MOE_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, 96 * 1024));
        occ_cache[di.device][slot] = occ > 0 ? occ : -1;
    }
    const int occ = occ_cache[di.device][slot];
    if (occ < 0) return MOE_ERR_UNSUPPORTED;
    MOE_CUDA_TRY(cudaMemsetAsync(p.bar, 0, 8, s));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(di.sms * occ);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, p));
    return MOE_OK;
}

}  // namespace moe
