// Rate probe of the prefill GEMM's tensor-core instruction: one CTA per SM
// issues back-to-back tcgen05.mma.kind::mxf8f6f4.block_scale MMAs (E4M3 A
// tile 128x32, E2M1 B tile 256x32, E8M0 scale factors from tensor memory)
// of exactly the shape, operand layout and descriptors the grouped GEMM
// uses, on operands that stay in shared memory.  Timed by the caller, it
// gives the peak rate of that instruction on this GPU: the denominator of
// the prefill roofline.  No global memory is read; the only global write
// is an error bit when the bounded completion wait runs out.
#include <cuda_runtime.h>

#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int kM = 128, kN = 256, kK = 32, kStageK = 128;
constexpr uint32_t kBytesA = kM * kStageK;   // E4M3, one byte per element
constexpr uint32_t kBytesB = kN * kStageK;   // E2M1 in the 16-byte-aligned unpacked layout
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColSfA = kN, kColSfB = kN + 8;

__global__ void __launch_bounds__(128, 1) mma_probe_kernel(int stages, uint32_t* err) {
    extern __shared__ uint8_t raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    uint8_t* a = base;
    uint8_t* b = base + kBytesA;
    __shared__ __align__(8) uint64_t done;
    __shared__ uint32_t tmem_base;
    const int warp = threadIdx.x >> 5;
    // operands: pseudo-random finite bytes (E4M3 codes with bit 3 and the
    // sign clear never encode NaN), so the tensor pipe multiplies data of
    // ordinary density rather than zeros
    for (uint32_t i = threadIdx.x * 16; i < kBytesA + kBytesB; i += blockDim.x * 16) {
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t h = (i + 4 * j + 1) * 2654435761u;
            h ^= h >> 15;
            w[j] = h & 0x77777777u;
        }
        *reinterpret_cast<uint4*>(base + i) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (warp == 0) tc::tmem_alloc(&tmem_base, kTmemCols);
    if (threadIdx.x == 0) {
        tc::mbar_init(&done, 1);
        tc::fence_barrier_init();
    }
    // shared-memory operands written by ordinary stores, read by the tensor core
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = tmem_base;
    // scale factors 2^0 for every row and K-block, each lane quarter its own copy
    const uint32_t lane_base = tmem + (uint32_t(warp * 32) << 16);
    const uint32_t one = 0x7f7f7f7fu;
    tc::tmem_st_x4(lane_base + kColSfA, one, one, one, one);
    const uint32_t ones[8] = {one, one, one, one, one, one, one, one};
    tc::tmem_st_x8(lane_base + kColSfB, ones);
    tc::tmem_st_wait();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (threadIdx.x == 0) {
        const uint32_t a0 = tc::smem_u32(a), b0 = tc::smem_u32(b);
        for (int s = 0; s < stages; ++s) {
#pragma unroll
            for (int kk = 0; kk < kStageK / kK; ++kk) {
                const uint32_t idesc = tc::idesc_mxf8f6f4(0, 5, kM, kN, kk, kk);
                tc::mma_mxf8f6f4(tmem, tc::smem_desc_sw128(a0 + kk * 32), tc::smem_desc_sw128(b0 + kk * 32), idesc,
                                 tmem + kColSfA, tmem + kColSfB, (s | kk) != 0);
            }
        }
        tc::mma_commit(&done);
        tc::mbar_wait(&done, 0, err, 1u);
    }
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

int launch_mma_probe(int stages, uint32_t* err, int* ctas, cudaStream_t s) {
    static DeviceOnce attr_set;
    DeviceInfo di;
    int rc = current_device_info(&di);
    if (rc != MOE_OK) return rc;
    if (di.cc_major < 10 || di.device < 0 || di.device >= 64) return MOE_ERR_UNSUPPORTED;
    // more than half an SM's shared memory, so no two CTAs share an SM (and
    // its tensor memory); the operands use the first 49 KB
    const size_t smem = 120 * 1024;
    if (smem > di.smem_optin) return MOE_ERR_UNSUPPORTED;
    if (!attr_set.done(di.device)) {
        MOE_CUDA_TRY(cudaFuncSetAttribute(mma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
        attr_set.mark(di.device);
    }
    mma_probe_kernel<<<di.sms, 128, smem, s>>>(stages, err);
    MOE_CUDA_TRY(cudaGetLastError());
    if (ctas) *ctas = di.sms;
    return MOE_OK;
}

}  // namespace moe

extern "C" int moe_probe_mxf8f6f4(int stages, uint32_t* status_dev, int* ctas, moe_stream_t stream) {
    if (stages < 1 || stages > (1 << 16) || status_dev == nullptr) return MOE_ERR_INVALID;
    return moe::launch_mma_probe(stages, status_dev, ctas, static_cast<cudaStream_t>(stream));
}
