// mxq_api.cu -- extern "C" entry points declared in include/mxq.h: host-side
// validation (pointers, alignment, shapes, device residency of m_splits,
// device architecture, workspace size), then one launch sequence on the
// caller's stream. Nothing here synchronizes except mxq_status_read; nothing
// here allocates.
#include <cuda_runtime.h>

#include <atomic>

#include "../../include/mxq.h"
#include "mxq_internal.h"
#include "mxq_peak.h"

namespace mxq {

thread_local int g_last_cuda = 0;

int fail_cuda(cudaError_t e) {
    g_last_cuda = (int)e;
    return MXQ_ERR_LAUNCH;
}

bool aligned16(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device attribute cache: 1 = sm_103 (GB300), -1 = other, 0 = unknown (atomic: calls may come from
// several host threads).
bool arch_ok() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c) return c > 0;
    }
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    const int ok = (major == 10 && minor == 3) ? 1 : -1;
    if (dev < 64) cache[dev].store(ok, std::memory_order_relaxed);
    return ok > 0;
}

// m_splits must be reachable from the device without a host round trip
// [DI: host m_splits are rejected on the device-init path].
bool device_pointer(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

int check_common(int64_t M, int64_t K, int E, const int64_t* m_splits, bool splits_required, bool padded) {
    if (!arch_ok()) return MXQ_ERR_ARCH;
    if (M < 0 || K <= 0 || (!padded && M % 128) || K % 128) return MXQ_ERR_SHAPE;
    if (padded && !m_splits) return MXQ_ERR_NULL;
    if (E < 1 || E > MXQ_MAX_EXPERTS) return MXQ_ERR_SHAPE;
    if (M > ((int64_t)1 << 31) - 128 || K > ((int64_t)1 << 31) - 128) return MXQ_ERR_SHAPE;
    if (m_splits == nullptr) {
        if (splits_required) return MXQ_ERR_NULL;
        if (M % E || (M / E) % 128) return MXQ_ERR_SHAPE;
    } else if (!device_pointer(m_splits)) {
        return MXQ_ERR_HOST_POINTER;
    }
    return MXQ_OK;
}

}  // namespace mxq

using mxq::aligned16;
using mxq::arch_ok;
using mxq::check_common;
using mxq::device_pointer;
using mxq::fail_cuda;

extern "C" {

int mxq_version(void) { return 100; }

size_t mxq_scale_bytes(int64_t rows, int64_t cols, int colwise) {
    auto up = [](int64_t a, int64_t b) { return (a + b - 1) / b * b; };
    if (rows < 0 || cols < 0) return 0;
    if (!colwise) return (size_t)(up(rows, 128) * up(cols / 32, 4));
    return (size_t)(up(rows / 32, 4) * up(cols, 128));
}

// Rows of the padded scale row space of E experts with M rows in total, at
// most: sum round_up(m_e, 128) <= round_up(M, 128) + 128 E.
static int64_t padded_rows_bound(int64_t M, int E) { return (M + 127) / 128 * 128 + (int64_t)128 * E; }

size_t mxq_scale_bytes_grouped(int64_t rows, int64_t cols, int E, int colwise) {
    if (rows < 0 || cols < 0 || E < 1) return 0;
    return mxq_scale_bytes(padded_rows_bound(rows, E), cols, colwise);
}

size_t mxq_workspace_bytes(int op, int64_t M, int64_t N, int64_t K, int E, int flags) {
    const int64_t Mt = (flags & MXQ_PAD_EXPERTS) ? padded_rows_bound(M, E) : M;
    switch (op) {
        case MXQ_OP_GROUP_QUANTIZE:
        case MXQ_OP_REQUANT_COLWISE: return (size_t)(Mt / 128) * (size_t)K * sizeof(float);
        case MXQ_OP_GROUPED_DBIAS: return (size_t)(M / 128) * (size_t)N * sizeof(float);
        case MXQ_OP_SWIGLU_BWD_QUANTIZE: return (size_t)(M / 128) * (size_t)(2 * K) * sizeof(float);
        case MXQ_OP_SCALED_BIAS:  // column-sum partials (M/128, K) + row-dot partials (M, K/128)
            return 2 * (size_t)(M / 128) * (size_t)K * sizeof(float);
        case MXQ_OP_GEMM_DGRAD_SWIGLU:  // dY1 column sums per 32 rows: (M/32, 2K)
            return (size_t)(M / 32) * (size_t)(2 * K) * sizeof(float);
        default: return 0;
    }
}

int mxq_group_quantize(const void* x_bf16, int64_t M, int64_t K, int E, const int64_t* d_m_splits, int flags,
                       void* row_data, void* row_scale, void* col_data, void* col_scale, float* dbias_out,
                       const int32_t* d_noop, int32_t* d_status, void* ws, size_t ws_bytes, mxq_stream_t stream) {
    if (flags & ~(MXQ_ROWWISE | MXQ_COLWISE | MXQ_SWIZZLE | MXQ_PAD_EXPERTS)) return MXQ_ERR_FLAGS;
    const bool row = flags & MXQ_ROWWISE, col = flags & MXQ_COLWISE, pad = flags & MXQ_PAD_EXPERTS;
    if (!row && !col && !dbias_out) return MXQ_ERR_FLAGS;
    // With M == 0 every data buffer is empty (and may be NULL).
    if (M != 0 && (!x_bf16 || (row && (!row_data || !row_scale)) || (col && (!col_data || !col_scale))))
        return MXQ_ERR_NULL;
    if (int r = check_common(M, K, E, d_m_splits, false, pad)) return r;
    if (!aligned16(x_bf16) || !aligned16(row_data) || !aligned16(row_scale) || !aligned16(col_data) ||
        !aligned16(col_scale) || !aligned16(dbias_out) || !aligned16(ws))
        return MXQ_ERR_ALIGN;
    if (dbias_out && M != 0 && (!ws || ws_bytes < mxq_workspace_bytes(MXQ_OP_GROUP_QUANTIZE, M, 0, K, E, flags)))
        return MXQ_ERR_WORKSPACE;
    mxq::QuantCall c{};
    c.x = x_bf16;
    c.M = M;
    c.K = K;
    c.E = E;
    c.m_splits = d_m_splits;
    c.row_q = row ? row_data : nullptr;
    c.row_s = row ? row_scale : nullptr;
    c.col_q = col ? col_data : nullptr;
    c.col_s = col ? col_scale : nullptr;
    c.dbias = dbias_out;
    c.partials = dbias_out ? static_cast<float*>(ws) : nullptr;
    c.swizzle = (flags & MXQ_SWIZZLE) != 0;
    c.noop = d_noop;
    c.status = d_status;
    cudaError_t e = pad ? mxq::run_group_quantize_padded(c, (cudaStream_t)stream)
                        : mxq::run_group_quantize(c, (cudaStream_t)stream);
    return e == cudaSuccess ? MXQ_OK : fail_cuda(e);
}

int mxq_requant_colwise(const void* row_data, const void* row_scale_compact, int64_t M, int64_t K, int E,
                        const int64_t* d_m_splits, int flags, void* col_data, void* col_scale,
                        void* row_scale_swizzled_out, float* dbias_out, void* dequant_bf16_out,
                        const int32_t* d_noop, int32_t* d_status, void* ws, size_t ws_bytes, mxq_stream_t stream) {
    if (flags & ~(MXQ_ROWWISE | MXQ_COLWISE | MXQ_SWIZZLE | MXQ_DEQUANT_OUT | MXQ_PAD_EXPERTS)) return MXQ_ERR_FLAGS;
    const bool row = flags & MXQ_ROWWISE, col = flags & MXQ_COLWISE, deq = flags & MXQ_DEQUANT_OUT,
               pad = flags & MXQ_PAD_EXPERTS;
    if (!row && !col && !deq && !dbias_out) return MXQ_ERR_FLAGS;
    if (M != 0 && (!row_data || !row_scale_compact || (col && (!col_data || !col_scale)) ||
                   (row && !row_scale_swizzled_out) || (deq && !dequant_bf16_out)))
        return MXQ_ERR_NULL;
    if (int r = check_common(M, K, E, d_m_splits, false, pad)) return r;
    if (!aligned16(row_data) || !aligned16(row_scale_compact) || !aligned16(col_data) || !aligned16(col_scale) ||
        !aligned16(row_scale_swizzled_out) || !aligned16(dbias_out) || !aligned16(dequant_bf16_out) ||
        !aligned16(ws))
        return MXQ_ERR_ALIGN;
    if (dbias_out && M != 0 && (!ws || ws_bytes < mxq_workspace_bytes(MXQ_OP_REQUANT_COLWISE, M, 0, K, E, flags)))
        return MXQ_ERR_WORKSPACE;
    mxq::RequantCall c{};
    c.row_q = row_data;
    c.row_s_compact = row_scale_compact;
    c.M = M;
    c.K = K;
    c.E = E;
    c.m_splits = d_m_splits;
    c.col_q = col ? col_data : nullptr;
    c.col_s = col ? col_scale : nullptr;
    c.row_s_swizzled = row ? row_scale_swizzled_out : nullptr;
    c.dbias = dbias_out;
    c.partials = dbias_out ? static_cast<float*>(ws) : nullptr;
    c.deq_out = deq ? dequant_bf16_out : nullptr;
    c.swizzle = (flags & MXQ_SWIZZLE) != 0;
    c.noop = d_noop;
    c.status = d_status;
    cudaError_t e = pad ? mxq::run_requant_padded(c, (cudaStream_t)stream) : mxq::run_requant(c, (cudaStream_t)stream);
    return e == cudaSuccess ? MXQ_OK : fail_cuda(e);
}

// Checks shared by the two scaled-bias entry points; on success fills the
// workspace split (column-sum partials first, then row-dot partials).
static int scaled_bias_common(int64_t M, int64_t K, int E, const int64_t* d_m_splits, const float* probs,
                              const void* bias, float* dbias_out, float* dprobs_out, void* ws, size_t ws_bytes,
                              float** partials, float** dp_partials) {
    if (!dbias_out && !dprobs_out) return MXQ_ERR_FLAGS;
    if (!bias || (M != 0 && !probs)) return MXQ_ERR_NULL;
    if (int r = check_common(M, K, E, d_m_splits, true)) return r;
    if (!aligned16(probs) || !aligned16(bias) || !aligned16(dbias_out) || !aligned16(dprobs_out) || !aligned16(ws))
        return MXQ_ERR_ALIGN;
    if (M != 0 && (!ws || ws_bytes < mxq_workspace_bytes(MXQ_OP_SCALED_BIAS, M, 0, K, E, 0)))
        return MXQ_ERR_WORKSPACE;
    *partials = static_cast<float*>(ws);
    *dp_partials = ws ? static_cast<float*>(ws) + (M / 128) * K : nullptr;
    return MXQ_OK;
}

int mxq_group_quantize_scaled_bias(const void* x_bf16, int64_t M, int64_t K, int E, const int64_t* d_m_splits,
                                   int flags, void* row_data, void* row_scale, void* col_data, void* col_scale,
                                   const float* probs, const void* bias_bf16, float* dbias_out, float* dprobs_out,
                                   const int32_t* d_noop, int32_t* d_status, void* ws, size_t ws_bytes,
                                   mxq_stream_t stream) {
    if (flags & ~(MXQ_ROWWISE | MXQ_COLWISE | MXQ_SWIZZLE)) return MXQ_ERR_FLAGS;
    const bool row = flags & MXQ_ROWWISE, col = flags & MXQ_COLWISE;
    if (M != 0 && (!x_bf16 || (row && (!row_data || !row_scale)) || (col && (!col_data || !col_scale))))
        return MXQ_ERR_NULL;
    float *partials = nullptr, *dp = nullptr;
    if (int r = scaled_bias_common(M, K, E, d_m_splits, probs, bias_bf16, dbias_out, dprobs_out, ws, ws_bytes,
                                   &partials, &dp))
        return r;
    if (!aligned16(x_bf16) || !aligned16(row_data) || !aligned16(row_scale) || !aligned16(col_data) ||
        !aligned16(col_scale))
        return MXQ_ERR_ALIGN;
    mxq::QuantCall c{};
    c.x = x_bf16;
    c.M = M;
    c.K = K;
    c.E = E;
    c.m_splits = d_m_splits;
    c.row_q = row ? row_data : nullptr;
    c.row_s = row ? row_scale : nullptr;
    c.col_q = col ? col_data : nullptr;
    c.col_s = col ? col_scale : nullptr;
    c.dbias = dbias_out;
    c.partials = partials;
    c.swizzle = (flags & MXQ_SWIZZLE) != 0;
    c.noop = d_noop;
    c.status = d_status;
    c.probs = probs;
    c.bias = bias_bf16;
    c.dprobs = dprobs_out;
    c.dp_partials = dp;
    cudaError_t e = mxq::run_group_quantize(c, (cudaStream_t)stream);
    return e == cudaSuccess ? MXQ_OK : fail_cuda(e);
}

int mxq_requant_colwise_scaled_bias(const void* row_data, const void* row_scale_compact, int64_t M, int64_t K, int E,
                                    const int64_t* d_m_splits, int flags, void* col_data, void* col_scale,
                                    void* row_scale_swizzled_out, const float* probs, const void* bias_bf16,
                                    float* dbias_out, float* dprobs_out, void* dequant_bf16_out,
                                    const int32_t* d_noop, int32_t* d_status, void* ws, size_t ws_bytes,
                                    mxq_stream_t stream) {
    if (flags & ~(MXQ_ROWWISE | MXQ_COLWISE | MXQ_SWIZZLE | MXQ_DEQUANT_OUT)) return MXQ_ERR_FLAGS;
    const bool row = flags & MXQ_ROWWISE, col = flags & MXQ_COLWISE, deq = flags & MXQ_DEQUANT_OUT;
    if (M != 0 && (!row_data || !row_scale_compact || (col && (!col_data || !col_scale)) ||
                   (row && !row_scale_swizzled_out) || (deq && !dequant_bf16_out)))
        return MXQ_ERR_NULL;
    float *partials = nullptr, *dp = nullptr;
    if (int r = scaled_bias_common(M, K, E, d_m_splits, probs, bias_bf16, dbias_out, dprobs_out, ws, ws_bytes,
                                   &partials, &dp))
        return r;
    if (!aligned16(row_data) || !aligned16(row_scale_compact) || !aligned16(col_data) || !aligned16(col_scale) ||
        !aligned16(row_scale_swizzled_out) || !aligned16(dequant_bf16_out))
        return MXQ_ERR_ALIGN;
    mxq::RequantCall c{};
    c.row_q = row_data;
    c.row_s_compact = row_scale_compact;
    c.M = M;
    c.K = K;
    c.E = E;
    c.m_splits = d_m_splits;
    c.col_q = col ? col_data : nullptr;
    c.col_s = col ? col_scale : nullptr;
    c.row_s_swizzled = row ? row_scale_swizzled_out : nullptr;
    c.dbias = dbias_out;
    c.partials = partials;
    c.deq_out = deq ? dequant_bf16_out : nullptr;
    c.swizzle = (flags & MXQ_SWIZZLE) != 0;
    c.noop = d_noop;
    c.status = d_status;
    c.probs = probs;
    c.bias = bias_bf16;
    c.dprobs = dprobs_out;
    c.dp_partials = dp;
    cudaError_t e = mxq::run_requant(c, (cudaStream_t)stream);
    return e == cudaSuccess ? MXQ_OK : fail_cuda(e);
}

int mxq_grouped_dbias(const void* dy_bf16, int64_t M, int64_t N, int E, const int64_t* d_m_splits, float* dbias_out,
                      int32_t* d_status, void* ws, size_t ws_bytes, mxq_stream_t stream) {
    if ((M != 0 && !dy_bf16) || !dbias_out) return MXQ_ERR_NULL;
    if (int r = check_common(M, N, E, d_m_splits, true)) return r;
    if (!aligned16(dy_bf16) || !aligned16(dbias_out) || !aligned16(ws)) return MXQ_ERR_ALIGN;
    if (M != 0 && (!ws || ws_bytes < mxq_workspace_bytes(MXQ_OP_GROUPED_DBIAS, M, N, 0, E, 0))) return MXQ_ERR_WORKSPACE;
    cudaError_t e = mxq::run_grouped_dbias(dy_bf16, M, N, E, d_m_splits, dbias_out, static_cast<float*>(ws), d_status,
                                           (cudaStream_t)stream);
    return e == cudaSuccess ? MXQ_OK : fail_cuda(e);
}

static int gemm_common(int mode, const void* a, const void* as, const void* b, const void* bs, const void* bias,
                       int64_t M, int64_t N, int64_t K, int E, const int64_t* m_splits, void* out, int accumulate,
                       int out_bf16, int32_t* d_status, mxq_stream_t stream, const mxq::GemmExtra* extra = nullptr,
                       bool pad = false) {
    // With M == 0 the token-major operands (and fprop/dgrad outputs) are empty.
    const bool a_empty_ok = (M == 0), b_empty_ok = (M == 0 && mode == mxq::kWgrad);
    const bool out_empty_ok = (M == 0 && mode != mxq::kWgrad) || mode == mxq::kDgradSwiglu;
    if ((!a && !a_empty_ok) || (!as && !a_empty_ok) || (!b && !b_empty_ok) || (!bs && !b_empty_ok) ||
        (!out && !out_empty_ok))
        return MXQ_ERR_NULL;
    if (int r = check_common(M, K, E, m_splits, true, pad)) return r;
    if (pad && E > 512) return MXQ_ERR_SHAPE;  // the padded offset table's shared-memory budget
    if (N <= 0 || N % 128 || N > ((int64_t)1 << 31) / 128) return MXQ_ERR_SHAPE;
    if ((int64_t)E * N > ((int64_t)1 << 31) - 256) return MXQ_ERR_SHAPE;
    const bool fwd = (mode == mxq::kFprop || mode == mxq::kFpropSwiglu);
    if (fwd && N % 256) return MXQ_ERR_SHAPE;
    if (!fwd && K % 256) return MXQ_ERR_SHAPE;
    if (!aligned16(a) || !aligned16(as) || !aligned16(b) || !aligned16(bs) || !aligned16(bias) || !aligned16(out))
        return MXQ_ERR_ALIGN;
    mxq::GemmCall c{};
    c.mode = mode;
    c.a_data = a;
    c.a_scale = as;
    c.b_data = b;
    c.b_scale = bs;
    c.bias = bias;
    c.M = M;
    c.N = N;
    c.K = K;
    c.E = E;
    c.m_splits = m_splits;
    c.out = out;
    c.accumulate = accumulate;
    c.out_bf16 = out_bf16;
    c.status = d_status;
    c.pad = pad;
    if (extra) {
        c.q_row = extra->q_row;
        c.q_row_s = extra->q_row_s;
        c.q_col = extra->q_col;
        c.q_col_s = extra->q_col_s;
        c.swizzle = extra->swizzle;
        c.y1 = extra->y1;
        c.dbias_part = extra->dbias_part;
        c.side_bf16 = extra->side_bf16;
    }
    cudaError_t e = mxq::run_grouped_gemm(c, (cudaStream_t)stream);
    return e == cudaSuccess ? MXQ_OK : fail_cuda(e);
}

int mxq_grouped_gemm_fprop_swiglu(const void* x_data, const void* x_scale, const void* w1_data, const void* w1_scale,
                                  const void* bias_bf16, int64_t M, int64_t K, int64_t F, int E,
                                  const int64_t* d_m_splits, int flags, void* y1_bf16, void* h_row_data,
                                  void* h_row_scale, void* h_col_data, void* h_col_scale, void* h_bf16_out,
                                  int32_t* d_status, void* ws, size_t ws_bytes, mxq_stream_t stream) {
    (void)ws;
    (void)ws_bytes;
    if (flags & ~(MXQ_SWIZZLE | MXQ_DEQUANT_OUT)) return MXQ_ERR_FLAGS;
    const bool side = flags & MXQ_DEQUANT_OUT;
    if (F <= 0 || F % 128 || F > ((int64_t)1 << 30)) return MXQ_ERR_SHAPE;
    if (M != 0 && (!h_row_data || !h_row_scale || !h_col_data || !h_col_scale || (side && !h_bf16_out)))
        return MXQ_ERR_NULL;
    if (!aligned16(h_row_data) || !aligned16(h_row_scale) || !aligned16(h_col_data) || !aligned16(h_col_scale) ||
        !aligned16(h_bf16_out))
        return MXQ_ERR_ALIGN;
    mxq::GemmExtra x{};
    x.q_row = h_row_data;
    x.q_row_s = h_row_scale;
    x.q_col = h_col_data;
    x.q_col_s = h_col_scale;
    x.swizzle = (flags & MXQ_SWIZZLE) != 0;
    x.side_bf16 = side ? h_bf16_out : nullptr;
    return gemm_common(mxq::kFpropSwiglu, x_data, x_scale, w1_data, w1_scale, bias_bf16, M, 2 * F, K, E, d_m_splits,
                       y1_bf16, 0, 1, d_status, stream, &x);
}

int mxq_grouped_gemm_dgrad_swiglu(const void* dy_data, const void* dy_scale, const void* w_col_data,
                                  const void* w_col_scale, const void* y1_bf16, int64_t M, int64_t N, int64_t F,
                                  int E, const int64_t* d_m_splits, int flags, void* dy1_row_data,
                                  void* dy1_row_scale, void* dy1_col_data, void* dy1_col_scale, float* dbias_out,
                                  void* dy1_bf16_out, int32_t* d_status, void* ws, size_t ws_bytes,
                                  mxq_stream_t stream) {
    if (flags & ~(MXQ_SWIZZLE | MXQ_DEQUANT_OUT)) return MXQ_ERR_FLAGS;
    const bool side = flags & MXQ_DEQUANT_OUT;
    if (F <= 0 || F % 256) return MXQ_ERR_SHAPE;
    if (M != 0 &&
        (!y1_bf16 || !dy1_row_data || !dy1_row_scale || !dy1_col_data || !dy1_col_scale || (side && !dy1_bf16_out)))
        return MXQ_ERR_NULL;
    if (!aligned16(y1_bf16) || !aligned16(dy1_row_data) || !aligned16(dy1_row_scale) || !aligned16(dy1_col_data) ||
        !aligned16(dy1_col_scale) || !aligned16(dbias_out) || !aligned16(dy1_bf16_out) || !aligned16(ws))
        return MXQ_ERR_ALIGN;
    if (dbias_out && M != 0 && (!ws || ws_bytes < mxq_workspace_bytes(MXQ_OP_GEMM_DGRAD_SWIGLU, M, N, F, E, 0)))
        return MXQ_ERR_WORKSPACE;
    mxq::GemmExtra x{};
    x.q_row = dy1_row_data;
    x.q_row_s = dy1_row_scale;
    x.q_col = dy1_col_data;
    x.q_col_s = dy1_col_scale;
    x.swizzle = (flags & MXQ_SWIZZLE) != 0;
    x.y1 = y1_bf16;
    x.dbias_part = dbias_out ? static_cast<float*>(ws) : nullptr;
    x.side_bf16 = side ? dy1_bf16_out : nullptr;
    const int r = gemm_common(mxq::kDgradSwiglu, dy_data, dy_scale, w_col_data, w_col_scale, nullptr, M, N, F, E,
                              d_m_splits, nullptr, 0, 1, d_status, stream, &x);
    if (r != MXQ_OK || !dbias_out) return r;
    cudaError_t e = M == 0 ? cudaMemsetAsync(dbias_out, 0, (size_t)E * 2 * F * sizeof(float), (cudaStream_t)stream)
                           : mxq::run_dbias_finalize(static_cast<float*>(ws), M, 2 * F, E, d_m_splits, dbias_out,
                                                     nullptr, (cudaStream_t)stream, 32);
    return e == cudaSuccess ? MXQ_OK : fail_cuda(e);
}

int mxq_grouped_gemm_fprop_ex(const void* x_data, const void* x_scale, const void* w_data, const void* w_scale,
                              const void* bias_bf16, int64_t M, int64_t N, int64_t K, int E,
                              const int64_t* d_m_splits, int flags, void* y_bf16, int32_t* d_status, void* ws,
                              size_t ws_bytes, mxq_stream_t stream) {
    (void)ws;
    (void)ws_bytes;
    if (flags & ~MXQ_PAD_EXPERTS) return MXQ_ERR_FLAGS;
    return gemm_common(mxq::kFprop, x_data, x_scale, w_data, w_scale, bias_bf16, M, N, K, E, d_m_splits, y_bf16, 0, 1,
                       d_status, stream, nullptr, (flags & MXQ_PAD_EXPERTS) != 0);
}

int mxq_grouped_gemm_fprop(const void* x_data, const void* x_scale, const void* w_data, const void* w_scale,
                           const void* bias_bf16, int64_t M, int64_t N, int64_t K, int E,
                           const int64_t* d_m_splits, void* y_bf16, int32_t* d_status, void* ws,
                           size_t ws_bytes, mxq_stream_t stream) {
    return mxq_grouped_gemm_fprop_ex(x_data, x_scale, w_data, w_scale, bias_bf16, M, N, K, E, d_m_splits, 0, y_bf16,
                                     d_status, ws, ws_bytes, stream);
}

int mxq_grouped_gemm_dgrad_ex(const void* dy_data, const void* dy_scale, const void* w_col_data,
                              const void* w_col_scale, int64_t M, int64_t N, int64_t K, int E,
                              const int64_t* d_m_splits, int flags, void* dx_bf16, int32_t* d_status, void* ws,
                              size_t ws_bytes, mxq_stream_t stream) {
    (void)ws;
    (void)ws_bytes;
    if (flags & ~MXQ_PAD_EXPERTS) return MXQ_ERR_FLAGS;
    return gemm_common(mxq::kDgrad, dy_data, dy_scale, w_col_data, w_col_scale, nullptr, M, N, K, E, d_m_splits,
                       dx_bf16, 0, 1, d_status, stream, nullptr, (flags & MXQ_PAD_EXPERTS) != 0);
}

int mxq_grouped_gemm_dgrad(const void* dy_data, const void* dy_scale, const void* w_col_data,
                           const void* w_col_scale, int64_t M, int64_t N, int64_t K, int E,
                           const int64_t* d_m_splits, void* dx_bf16, int32_t* d_status, void* ws,
                           size_t ws_bytes, mxq_stream_t stream) {
    return mxq_grouped_gemm_dgrad_ex(dy_data, dy_scale, w_col_data, w_col_scale, M, N, K, E, d_m_splits, 0, dx_bf16,
                                     d_status, ws, ws_bytes, stream);
}

int mxq_grouped_gemm_wgrad(const void* dy_col_data, const void* dy_col_scale, const void* x_col_data,
                           const void* x_col_scale, int64_t M, int64_t N, int64_t K, int E,
                           const int64_t* d_m_splits, int flags, void* dw, int32_t* d_status, void* ws,
                           size_t ws_bytes, mxq_stream_t stream) {
    (void)ws;
    (void)ws_bytes;
    if (flags & ~(MXQ_ACCUMULATE | MXQ_OUT_BF16 | MXQ_PAD_EXPERTS)) return MXQ_ERR_FLAGS;
    return gemm_common(mxq::kWgrad, dy_col_data, dy_col_scale, x_col_data, x_col_scale, nullptr, M, N, K, E,
                       d_m_splits, dw, (flags & MXQ_ACCUMULATE) != 0, (flags & MXQ_OUT_BF16) != 0, d_status, stream,
                       nullptr, (flags & MXQ_PAD_EXPERTS) != 0);
}

int mxq_probe_mma_stream_ex(int64_t mmas_per_sm, int operands, int32_t* d_status, mxq_stream_t stream) {
    if (operands != MXQ_PROBE_ZEROS && operands != MXQ_PROBE_RANDOM) return MXQ_ERR_FLAGS;
    if (!arch_ok()) return MXQ_ERR_ARCH;
    if (mmas_per_sm < 0 || mmas_per_sm >= ((int64_t)1 << 31)) return MXQ_ERR_SHAPE;
    cudaError_t e = mxq::run_mma_stream(mmas_per_sm, operands == MXQ_PROBE_RANDOM, d_status, (cudaStream_t)stream);
    return e == cudaSuccess ? MXQ_OK : fail_cuda(e);
}

int mxq_probe_mma_stream(int64_t mmas_per_sm, int32_t* d_status, mxq_stream_t stream) {
    return mxq_probe_mma_stream_ex(mmas_per_sm, MXQ_PROBE_ZEROS, d_status, stream);
}

int mxq_selftest_wait_timeout(int64_t limit_ns, int32_t* d_status, mxq_stream_t stream) {
    if (!d_status) return MXQ_ERR_NULL;
    if (!arch_ok()) return MXQ_ERR_ARCH;
    if (limit_ns < 1000 || limit_ns > 10000000000LL) return MXQ_ERR_SHAPE;
    if (!device_pointer(d_status)) return MXQ_ERR_HOST_POINTER;
    cudaError_t e = mxq::run_wait_timeout(limit_ns, d_status, (cudaStream_t)stream);
    return e == cudaSuccess ? MXQ_OK : fail_cuda(e);
}

int mxq_swiglu_fwd(const void* y_bf16, int64_t M, int64_t F, void* h_bf16, mxq_stream_t stream) {
    if (!y_bf16 || !h_bf16) return MXQ_ERR_NULL;
    if (!arch_ok()) return MXQ_ERR_ARCH;
    if (M < 0 || F <= 0 || F % 8) return MXQ_ERR_SHAPE;
    if (!aligned16(y_bf16) || !aligned16(h_bf16)) return MXQ_ERR_ALIGN;
    cudaError_t e = mxq::run_swiglu_fwd(y_bf16, M, F, h_bf16, (cudaStream_t)stream);
    return e == cudaSuccess ? MXQ_OK : fail_cuda(e);
}

int mxq_swiglu_bwd(const void* dh_bf16, const void* y_bf16, int64_t M, int64_t F, void* dy_bf16,
                   mxq_stream_t stream) {
    if (!dh_bf16 || !y_bf16 || !dy_bf16) return MXQ_ERR_NULL;
    if (!arch_ok()) return MXQ_ERR_ARCH;
    if (M < 0 || F <= 0 || F % 8) return MXQ_ERR_SHAPE;
    if (!aligned16(dh_bf16) || !aligned16(y_bf16) || !aligned16(dy_bf16)) return MXQ_ERR_ALIGN;
    cudaError_t e = mxq::run_swiglu_bwd(dh_bf16, y_bf16, M, F, dy_bf16, (cudaStream_t)stream);
    return e == cudaSuccess ? MXQ_OK : fail_cuda(e);
}

static int swiglu_quantize_common(int backward, const void* dh, const void* y, int64_t M, int64_t F, int E,
                                  const int64_t* m_splits, int flags, void* row_data, void* row_scale,
                                  void* col_data, void* col_scale, float* dbias_out, void* bf16_out,
                                  const int32_t* d_noop, int32_t* d_status, void* ws, size_t ws_bytes,
                                  mxq_stream_t stream) {
    if (flags & ~(MXQ_ROWWISE | MXQ_COLWISE | MXQ_SWIZZLE | MXQ_DEQUANT_OUT)) return MXQ_ERR_FLAGS;
    const bool row = flags & MXQ_ROWWISE, col = flags & MXQ_COLWISE, deq = flags & MXQ_DEQUANT_OUT;
    if (!row && !col && !deq && !dbias_out) return MXQ_ERR_FLAGS;
    if (M != 0 && (!y || (backward && !dh) || (row && (!row_data || !row_scale)) ||
                   (col && (!col_data || !col_scale)) || (deq && !bf16_out)))
        return MXQ_ERR_NULL;
    if (int r = check_common(M, F, E, m_splits, true)) return r;
    if (!aligned16(y) || !aligned16(dh) || !aligned16(row_data) || !aligned16(row_scale) || !aligned16(col_data) ||
        !aligned16(col_scale) || !aligned16(dbias_out) || !aligned16(bf16_out) || !aligned16(ws))
        return MXQ_ERR_ALIGN;
    if (dbias_out && M != 0 &&
        (!ws || ws_bytes < mxq_workspace_bytes(MXQ_OP_SWIGLU_BWD_QUANTIZE, M, 0, backward ? F : F / 2, E, 0)))
        return MXQ_ERR_WORKSPACE;
    mxq::SwigluQuantCall c{};
    c.backward = backward;
    c.y = y;
    c.dh = dh;
    c.M = M;
    c.F = F;
    c.E = E;
    c.m_splits = m_splits;
    c.row_q = row ? row_data : nullptr;
    c.row_s = row ? row_scale : nullptr;
    c.col_q = col ? col_data : nullptr;
    c.col_s = col ? col_scale : nullptr;
    c.dbias = dbias_out;
    c.partials = dbias_out ? static_cast<float*>(ws) : nullptr;
    c.bf16_out = deq ? bf16_out : nullptr;
    c.swizzle = (flags & MXQ_SWIZZLE) != 0;
    c.noop = d_noop;
    c.status = d_status;
    cudaError_t e = mxq::run_swiglu_quantize(c, (cudaStream_t)stream);
    return e == cudaSuccess ? MXQ_OK : fail_cuda(e);
}

int mxq_swiglu_quantize(const void* y_bf16, int64_t M, int64_t F, int E, const int64_t* d_m_splits, int flags,
                        void* row_data, void* row_scale, void* col_data, void* col_scale, void* h_bf16_out,
                        const int32_t* d_noop, int32_t* d_status, mxq_stream_t stream) {
    return swiglu_quantize_common(0, nullptr, y_bf16, M, F, E, d_m_splits, flags, row_data, row_scale, col_data,
                                  col_scale, nullptr, h_bf16_out, d_noop, d_status, nullptr, 0, stream);
}

int mxq_swiglu_bwd_quantize(const void* dh_bf16, const void* y_bf16, int64_t M, int64_t F, int E,
                            const int64_t* d_m_splits, int flags, void* row_data, void* row_scale, void* col_data,
                            void* col_scale, float* dbias_out, void* dy_bf16_out, const int32_t* d_noop,
                            int32_t* d_status, void* ws, size_t ws_bytes, mxq_stream_t stream) {
    return swiglu_quantize_common(1, dh_bf16, y_bf16, M, F, E, d_m_splits, flags, row_data, row_scale, col_data,
                                  col_scale, dbias_out, dy_bf16_out, d_noop, d_status, ws, ws_bytes, stream);
}

int mxq_status_read(const int32_t* d_status, int32_t* h_out, mxq_stream_t stream) {
    if (!d_status || !h_out) return MXQ_ERR_NULL;
    cudaError_t e = cudaMemcpyAsync(h_out, d_status, sizeof(int32_t), cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    return e == cudaSuccess ? MXQ_OK : fail_cuda(e);
}

const char* mxq_error_string(int code) {
    switch (code) {
        case MXQ_OK: return "ok";
        case MXQ_ERR_NULL: return "a required pointer is NULL";
        case MXQ_ERR_SHAPE: return "a dimension breaks the shape contract";
        case MXQ_ERR_HOST_POINTER: return "m_splits must be device memory (host m_splits are rejected)";
        case MXQ_ERR_ARCH: return "the current device is not sm_103 (GB300)";
        case MXQ_ERR_WORKSPACE: return "workspace missing or smaller than mxq_workspace_bytes()";
        case MXQ_ERR_LAUNCH: return "a CUDA call failed (see mxq_last_cuda_error)";
        case MXQ_ERR_FLAGS: return "unknown or inconsistent flags";
        case MXQ_ERR_ALIGN: return "a pointer is not 16-byte aligned";
        case MXQ_ERR_SCRATCH_LIMIT:
            return "(M/128)*N exceeds the 2,097,152-float scratch of mxq_grouped_dbias_noalloc";
        default: return "unknown error";
    }
}

int mxq_last_cuda_error(void) { return mxq::g_last_cuda; }

}  // extern "C"
