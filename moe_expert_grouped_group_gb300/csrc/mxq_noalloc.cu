// mxq_noalloc.cu -- per-expert dbias for callers that cannot allocate device
// memory.
//
// mxq_grouped_dbias needs a caller-provided workspace for its per-tile fp32
// partial sums. Some callers cannot provide one: code that runs where no
// allocator may be called (inside another library's callback, a custom
// allocator's own bookkeeping, a runtime that owns the whole device heap and
// forbids cudaMalloc, or an embedding that has no access to an allocator at
// all). mxq_grouped_dbias_noalloc runs the same two kernels, but its partial
// sums live in a fixed file-scope device array that every GPU loading this
// library holds until the process exits.
//
// Limits and behaviour:
//   - scratch capacity: kScratchFloats fp32 partials, i.e. (M/128) * N must
//     be <= 2,097,152 (8 MiB); larger problems get MXQ_ERR_SCRATCH_LIMIT;
//   - the first call on a device resolves the array's device address with
//     cudaGetSymbolAddress (once per device, with that device current), so
//     make that first call before any stream capture;
//   - every call shares the one array and it keeps the last call's partials;
//     the tile kernel overwrites every partial it later reads, so nothing
//     needs clearing between calls;
//   - calls that overlap on the GPU (other streams, other host threads) race
//     on the array: serialise them.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/mxq.h"
#include "mxq_internal.h"

namespace {

constexpr size_t kScratchFloats = size_t(2) << 20;

static __device__ __align__(256) float g_dbias_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_dbias_scratch on the current device (resolved once).
cudaError_t scratch_on_current_device(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_dbias_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

bool device_ok() {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    return major == 10 && minor == 3;
}

bool on_device(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

}  // namespace

extern "C" int mxq_grouped_dbias_noalloc(const void* dy_bf16, int64_t M, int64_t N, int E,
                                         const int64_t* d_m_splits, float* dbias_out, int32_t* d_status,
                                         mxq_stream_t stream) {
    if ((M != 0 && !dy_bf16) || !dbias_out || !d_m_splits) return MXQ_ERR_NULL;
    if (!device_ok()) return MXQ_ERR_ARCH;
    if (M < 0 || N <= 0 || M % 128 || N % 128 || E < 1 || E > MXQ_MAX_EXPERTS) return MXQ_ERR_SHAPE;
    if (((uintptr_t)dy_bf16 & 15u) || ((uintptr_t)dbias_out & 15u)) return MXQ_ERR_ALIGN;
    if (!on_device(d_m_splits)) return MXQ_ERR_HOST_POINTER;
    if ((size_t)(M / 128) * (size_t)N > kScratchFloats) return MXQ_ERR_SCRATCH_LIMIT;
    float* scratch = nullptr;
    cudaError_t e = scratch_on_current_device(&scratch);
    if (e == cudaSuccess)
        e = mxq::run_grouped_dbias(dy_bf16, M, N, E, d_m_splits, dbias_out, scratch, d_status, (cudaStream_t)stream);
    return e == cudaSuccess ? MXQ_OK : MXQ_ERR_LAUNCH;
}
