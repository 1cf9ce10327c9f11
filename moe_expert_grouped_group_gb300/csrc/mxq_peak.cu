// mxq_peak.cu -- utilities beside the MXFP8 path: the tensor-pipe ceiling
// of this GPU (a yardstick for the grouped GEMMs' roofline) and a self-test
// of the bounded on-chip wait every kernel uses.
//
// One CTA per SM streams block-scaled 128x256x32 tcgen05 MMAs (E4M3 x E4M3,
// E8M0 scales, fp32 accumulation in TMEM) from operands that stay resident
// in shared memory: the instruction mix of the GEMM's MMA loop (three scale
// copies, four MMAs and a commit per 128-deep K block) without the loads,
// the waits between blocks, the tile boundaries or the epilogue. Its rate is
// the most any kernel built from these instructions can reach on this GPU.
// The operands are zeros, or pseudo-random E4M3 bytes with unit scales: the
// tensor pipe's power grows with the bits it multiplies, so a long stream of
// random operands (as a GEMM on real data) meets the board's power limit and
// runs at a lower clock than a stream of zeros.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "mxq_common.cuh"
#include "mxq_peak.h"

namespace mxq {
namespace {

constexpr int kPeakThreads = 128;
constexpr int kOperandBytes = 16384 + 32768;  // A 128x128 and B 256x128 E4M3 tiles
constexpr int kScaleBytes = 1536;             // the K block's scale atoms: A (512), B (2 x 512)
constexpr int kPeakSmem = 160 * 1024;         // more than half an SM: one CTA per SM

__device__ __forceinline__ uint64_t peak_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)(layout & 7u) << 61);
}
// kind::mxf8f6f4, E4M3 x E4M3, K-major both, N = 256, M = 128, UE8M0 scales, scale byte k of each word
__device__ __forceinline__ uint32_t peak_idesc(uint32_t k) {
    return (k << 4) | ((uint32_t)(256 >> 3) << 17) | (1u << 23) | ((uint32_t)(128 >> 4) << 24) | (k << 29);
}

__global__ void __launch_bounds__(kPeakThreads) mma_stream_kernel(int64_t mmas, int random, int32_t* status) {
    extern __shared__ uint8_t peak_raw[];
    uint8_t* smem = smem_align<1024>(peak_raw);
    __shared__ uint32_t s_tmem;
    __shared__ __align__(8) uint64_t s_bar[2];  // [0]: per-K-block commits (never waited on), [1]: all done
    __shared__ int s_abort;
    // random operands: a multiplicative hash of the word index and the SM, each byte's exponent
    // field kept at most 6 (no NaN code; products and sums stay finite); scales 127 (2^0)
    for (int i = threadIdx.x; i < kOperandBytes / 4; i += blockDim.x) {
        uint32_t h = (uint32_t)(i + 1) * 2654435761u ^ ((uint32_t)blockIdx.x << 20);
        h ^= h >> 13;
        h *= 0x5bd1e995u;
        h ^= h >> 15;
        reinterpret_cast<uint32_t*>(smem)[i] = random ? (h & 0xB7B7B7B7u) : 0u;
    }
    for (int i = threadIdx.x; i < kScaleBytes / 4; i += blockDim.x)
        reinterpret_cast<uint32_t*>(smem + kOperandBytes)[i] = random ? 0x7F7F7F7Fu : 0u;
    if (threadIdx.x == 0) {
        s_abort = 0;
        mbar_init(smem_u32(&s_bar[0]), 1);
        mbar_init(smem_u32(&s_bar[1]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the zeros, for the tensor core
    if (threadIdx.x < 32) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = s_tmem;
    if (threadIdx.x == 0 && mmas > 0) {
        const uint32_t base = smem_u32(smem);
        const uint64_t ad = peak_desc(base, 16, 1024, 2), bd = peak_desc(base + 16384, 16, 1024, 2);
        const uint64_t sfd = peak_desc(base + kOperandBytes, 0, 128, 0);
        const uint32_t sfa = tmem + 256, sfb = tmem + 264;
        for (int64_t it = 0; it < mmas; ++it) {
            const uint32_t k = (uint32_t)(it & 3);
            if (k == 0) {
                asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(sfa), "l"(sfd) : "memory");
                asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(sfb), "l"(sfd + 32) : "memory");
                asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(sfb + 4), "l"(sfd + 64)
                             : "memory");
            }
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
                    tmem),
                "l"(ad + 2 * k), "l"(bd + 2 * k), "r"(peak_idesc(k)), "r"((uint32_t)(it != 0)), "r"(sfa), "r"(sfb)
                : "memory");
            if (k == 3)
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                 smem_u32(&s_bar[0]))
                             : "memory");
        }
        // every MMA has completed before the accumulator's columns are freed
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         smem_u32(&s_bar[1]))
                     : "memory");
        if (!mbar_wait(smem_u32(&s_bar[1]), 0, &s_abort)) report_status(status, MXQ_STATUS_WAIT_TIMEOUT);
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (threadIdx.x < 32)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
}

// Self-test of the bounded on-chip wait: lane 0 of warp 0 waits, limit_ns
// long, on an mbarrier that nothing arrives on; lane 0 of warp 1 waits on the
// same barrier with the kernels' own bound. The first wait expires and sets
// the CTA's abort flag, which ends the second; the kernel then reports
// MXQ_STATUS_WAIT_TIMEOUT and returns (no trap, no fault).
__global__ void __launch_bounds__(64) wait_timeout_kernel(unsigned long long limit_ns, int32_t* status) {
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ int s_abort;
    if (threadIdx.x == 0) {
        s_abort = 0;
        mbar_init(smem_u32(&s_bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) {
        if (threadIdx.x == 0) (void)mbar_wait_for(smem_u32(&s_bar), 0, &s_abort, limit_ns);
        else (void)mbar_wait(smem_u32(&s_bar), 0, &s_abort);
    }
    __syncthreads();
    if (threadIdx.x == 0 && s_abort) report_status(status, MXQ_STATUS_WAIT_TIMEOUT);
}

}  // namespace

cudaError_t run_wait_timeout(int64_t limit_ns, int32_t* status, cudaStream_t s) {
    wait_timeout_kernel<<<1, 64, 0, s>>>((unsigned long long)limit_ns, status);
    return cudaGetLastError();
}

cudaError_t run_mma_stream(int64_t mmas_per_sm, int random, int32_t* status, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const cudaError_t attr =
        cudaFuncSetAttribute(mma_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPeakSmem);
    if (attr != cudaSuccess) return attr;
    mma_stream_kernel<<<sms, kPeakThreads, kPeakSmem, s>>>(mmas_per_sm, random, status);
    return cudaGetLastError();
}

}  // namespace mxq
