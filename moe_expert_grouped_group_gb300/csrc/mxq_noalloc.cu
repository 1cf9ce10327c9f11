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
//   - the array's device address is looked up with cudaGetSymbolAddress, with
//     the device current, on the first call in each CUDA context of a device:
//     the first call of the process on that device, and the first call after
//     the device's context was destroyed and re-created (cudaDeviceReset), in
//     which the module and its array may have moved;
//   - every call shares the one array and it keeps the last call's partials;
//     the tile kernel overwrites every partial it later reads, so nothing
//     needs clearing between calls;
//   - calls that overlap on the GPU (other streams, other host threads) race
//     on the array: serialise them.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/mxq.h"
#include "mxq_internal.h"

namespace {

constexpr size_t kScratchFloats = size_t(2) << 20;

static __device__ __align__(256) float g_dbias_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;

// Driver calls that identify the current context: the unique id of a context
// changes when the device's primary context is destroyed and created again.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct Driver {
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
};

const Driver& driver() {
    static Driver d;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            d.get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            d.get_id = reinterpret_cast<CtxGetIdFn>(f);
    });
    return d;
}

// Id of the calling thread's current context; 0 when there is none.
unsigned long long current_context_id() {
    const Driver& d = driver();
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!d.get_current || !d.get_id || d.get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (d.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

struct Slot {
    unsigned long long ctx_id = 0;
    float* ptr = nullptr;
};
std::mutex g_scratch_mu;
Slot g_slot[kMaxDevices];

// Device address of g_dbias_scratch on the current device, looked up again
// whenever the device's current context is not the one it was looked up in.
cudaError_t scratch_on_current_device(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    Slot& s = g_slot[dev];
    const unsigned long long id = current_context_id();
    if (!s.ptr || id == 0 || id != s.ctx_id) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_dbias_scratch);  // creates the context if there is none yet
        if (e != cudaSuccess) return e;
        s.ptr = static_cast<float*>(p);
        s.ctx_id = current_context_id();
    }
    *out = s.ptr;
    return cudaSuccess;
}

}  // namespace

extern "C" int mxq_grouped_dbias_noalloc(const void* dy_bf16, int64_t M, int64_t N, int E,
                                         const int64_t* d_m_splits, float* dbias_out, int32_t* d_status,
                                         mxq_stream_t stream) {
    if ((M != 0 && !dy_bf16) || !dbias_out) return MXQ_ERR_NULL;
    if (int r = mxq::check_common(M, N, E, d_m_splits, true)) return r;
    if (!mxq::aligned16(dy_bf16) || !mxq::aligned16(dbias_out)) return MXQ_ERR_ALIGN;
    if ((size_t)(M / 128) * (size_t)N > kScratchFloats) return MXQ_ERR_SCRATCH_LIMIT;
    float* scratch = nullptr;
    cudaError_t e = scratch_on_current_device(&scratch);
    if (e == cudaSuccess)
        e = mxq::run_grouped_dbias(dy_bf16, M, N, E, d_m_splits, dbias_out, scratch, d_status, (cudaStream_t)stream);
    return e == cudaSuccess ? MXQ_OK : mxq::fail_cuda(e);
}
