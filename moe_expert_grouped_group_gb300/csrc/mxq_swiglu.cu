// mxq_swiglu.cu -- SwiGLU between FC1 and FC2 of a fused grouped MoE MLP
// (TransformerEngine PR #3545, "Fix distributed BF16 weights and trim NVFP4
// saved state in the fused grouped MLP": FC1 -> activation -> FC2). The FC1
// output row is [gate | up] (gate first); h = silu(gate) * up.
// Elementwise and HBM-bound: each thread moves 8 bf16 of gate and of up with
// 16-byte loads; fp32 math in the explicit steps of mxq_common.cuh (the same
// steps the fused SwiGLU + quantize kernels use), bf16 RNE outputs.
#include <cuda_bf16.h>

#include <algorithm>

#include "mxq_common.cuh"
#include "mxq_internal.h"

namespace mxq {

__device__ __forceinline__ void unpack8(uint4 w, float* f) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        f[2 * j] = __uint_as_float(ws[j] << 16);
        f[2 * j + 1] = __uint_as_float(ws[j] & 0xFFFF0000u);
    }
}
__device__ __forceinline__ uint4 pack8(const float* f) {
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
        o[j] = *reinterpret_cast<uint32_t*>(&b);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

__global__ void __launch_bounds__(256) swiglu_fwd_kernel(const uint16_t* __restrict__ y, int64_t M, int64_t F,
                                                         uint16_t* __restrict__ h) {
    const int64_t vecs = M * (F / 8);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < vecs; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = i / (F / 8), f = (i % (F / 8)) * 8;
        float g[8], u[8], o[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(y + m * 2 * F + f)), g);
        unpack8(__ldg(reinterpret_cast<const uint4*>(y + m * 2 * F + F + f)), u);
#pragma unroll
        for (int j = 0; j < 8; ++j) o[j] = swiglu_h(g[j], u[j]);
        *reinterpret_cast<uint4*>(h + m * F + f) = pack8(o);
    }
}

__global__ void __launch_bounds__(256) swiglu_bwd_kernel(const uint16_t* __restrict__ dh,
                                                         const uint16_t* __restrict__ y, int64_t M, int64_t F,
                                                         uint16_t* __restrict__ dy) {
    const int64_t vecs = M * (F / 8);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < vecs; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = i / (F / 8), f = (i % (F / 8)) * 8;
        float d[8], g[8], u[8], dg[8], du[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(dh + m * F + f)), d);
        unpack8(__ldg(reinterpret_cast<const uint4*>(y + m * 2 * F + f)), g);
        unpack8(__ldg(reinterpret_cast<const uint4*>(y + m * 2 * F + F + f)), u);
#pragma unroll
        for (int j = 0; j < 8; ++j) swiglu_grads(d[j], g[j], u[j], dg[j], du[j]);
        *reinterpret_cast<uint4*>(dy + m * 2 * F + f) = pack8(dg);
        *reinterpret_cast<uint4*>(dy + m * 2 * F + F + f) = pack8(du);
    }
}

static unsigned grid_for(int64_t vecs) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return (unsigned)std::max<int64_t>(1, std::min<int64_t>((vecs + 255) / 256, (int64_t)sms * 8));
}

cudaError_t run_swiglu_fwd(const void* y, int64_t M, int64_t F, void* h, cudaStream_t s) {
    const int64_t vecs = M * (F / 8);
    if (vecs == 0) return cudaSuccess;
    swiglu_fwd_kernel<<<grid_for(vecs), 256, 0, s>>>((const uint16_t*)y, M, F, (uint16_t*)h);
    return cudaGetLastError();
}

cudaError_t run_swiglu_bwd(const void* dh, const void* y, int64_t M, int64_t F, void* dy, cudaStream_t s) {
    const int64_t vecs = M * (F / 8);
    if (vecs == 0) return cudaSuccess;
    swiglu_bwd_kernel<<<grid_for(vecs), 256, 0, s>>>((const uint16_t*)dh, (const uint16_t*)y, M, F, (uint16_t*)dy);
    return cudaGetLastError();
}

}  // namespace mxq
