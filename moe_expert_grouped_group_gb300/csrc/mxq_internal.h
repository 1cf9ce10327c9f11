// mxq_internal.h -- launcher interfaces between the C ABI (mxq_api.cu) and
// the kernel translation units. Not installed; not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mxq {

struct QuantCall {
    const void* x;
    int64_t M, K;
    int E;
    const int64_t* m_splits;
    void *row_q, *row_s, *col_q, *col_s;
    float* dbias;
    float* partials;  // workspace, (M/128)*K fp32, when dbias != nullptr
    int swizzle;
    const int32_t* noop;
    int32_t* status;
    // scaled bias (probs != nullptr): s_m (M), b_e (E, K) bf16; outputs
    // dbias = sum s_m dY_m (uses partials) and dprobs (M) from dp_partials
    // (M, K/128) fp32 of workspace
    const float* probs;
    const void* bias;
    float* dprobs;
    float* dp_partials;
};

struct RequantCall {
    const void* row_q;
    const void* row_s_compact;
    int64_t M, K;
    int E;
    const int64_t* m_splits;
    void *col_q, *col_s, *row_s_swizzled;
    float* dbias;
    float* partials;
    void* deq_out;
    int swizzle;
    const int32_t* noop;
    int32_t* status;
    // scaled bias, as in QuantCall
    const float* probs;
    const void* bias;
    float* dprobs;
    float* dp_partials;
};

// SwiGLU fused with group quantization: forward quantizes h (M, F); backward
// quantizes dY1 = [dg | du] (M, 2F) and reduces its dbias.
struct SwigluQuantCall {
    int backward;
    const void* y;   // FC1 output (M, 2F) bf16, [gate | up]
    const void* dh;  // backward: gradient of h (M, F) bf16
    int64_t M, F;
    int E;
    const int64_t* m_splits;
    void *row_q, *row_s, *col_q, *col_s;
    float* dbias;
    float* partials;  // workspace, (M/128) * Kout fp32, when dbias != nullptr
    void* bf16_out;   // optional h or dY1 in bf16
    int swizzle;
    const int32_t* noop;
    int32_t* status;
};

// kFpropSwiglu: FC1 fprop of a SwiGLU MLP (N = 2F) whose epilogue also
// applies SwiGLU to the bf16 output and quantizes h (rowwise + colwise).
// kDgradSwiglu: FC2 dgrad (output dh, K = F) whose epilogue applies the
// SwiGLU backward with the saved FC1 output and quantizes dY1 = [dg | du]
// (rowwise + colwise) and reduces its dbias partials.
enum GemmMode { kFprop = 0, kDgrad = 1, kWgrad = 2, kFpropSwiglu = 3, kDgradSwiglu = 4 };

struct GemmCall {
    int mode;
    const void *a_data, *a_scale, *b_data, *b_scale;
    const void* bias;  // fprop only
    int64_t M, N, K;
    int E;
    const int64_t* m_splits;
    void* out;
    int accumulate, out_bf16;  // wgrad only
    int32_t* status;
    // kFpropSwiglu: h (M, N/2); kDgradSwiglu: dY1 (M, 2K) -- codes and scales
    void *q_row, *q_row_s, *q_col, *q_col_s;
    int swizzle;
    const void* y1;      // kDgradSwiglu: saved FC1 output (M, 2K) bf16
    float* dbias_part;   // kDgradSwiglu: (M/32, 2K) fp32 column sums per 32 rows, or null
    void* side_bf16;     // SwiGLU modes: optional bf16 copy of h (M, N/2) or dY1 (M, 2K), or null
    int pad;             // fprop/dgrad/wgrad: padded grouping (expert counts not multiples of 128)
};

// The extra operands of the SwiGLU-fused modes, as passed through the C ABI.
struct GemmExtra {
    void *q_row, *q_row_s, *q_col, *q_col_s;
    int swizzle;
    const void* y1;
    float* dbias_part;
    void* side_bf16;
};

// Encodes a 2-D row-major tensor map (rows x cols elements of elem_bytes)
// with a box of box_rows x box_cols. swizzle_bytes: 0 (none), 64 or 128 (the
// 64- or 128-byte shared-memory swizzle; box_cols * elem_bytes must then
// equal it). False on failure.
bool encode_tmap_2d(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int elem_bytes, int box_cols,
                    int box_rows, int swizzle_bytes);

// Host-side checks shared by the entry points (mxq_api.cu).
// Records e as this thread's last CUDA error (mxq_last_cuda_error) and returns MXQ_ERR_LAUNCH.
int fail_cuda(cudaError_t e);
// The current device is sm_103 (cached per device).
bool arch_ok();
bool aligned16(const void* p);
// p is device (or managed) memory, reachable without a host round trip.
bool device_pointer(const void* p);
// Device, shape and m_splits checks of a grouped (M, K) tensor with E experts; MXQ_OK or an error code.
int check_common(int64_t M, int64_t K, int E, const int64_t* m_splits, bool splits_required, bool padded = false);

cudaError_t run_group_quantize(const QuantCall& c, cudaStream_t s);
cudaError_t run_requant(const RequantCall& c, cudaStream_t s);
cudaError_t run_grouped_dbias(const void* dy, int64_t M, int64_t N, int E, const int64_t* m_splits, float* out,
                              float* partials, int32_t* status, cudaStream_t s);
cudaError_t run_grouped_gemm(const GemmCall& c, cudaStream_t s);
// Expert counts that need not be multiples of 128 (per-expert padded scales).
cudaError_t run_group_quantize_padded(const QuantCall& c, cudaStream_t s);
cudaError_t run_requant_padded(const RequantCall& c, cudaStream_t s);
cudaError_t run_swiglu_quantize(const SwigluQuantCall& c, cudaStream_t s);
// out[e, :] = fp64 sum, in order, of expert e's partial rows; each partial row
// covers rows_per_partial consecutive token rows.
cudaError_t run_dbias_finalize(const float* partials, int64_t M, int64_t K, int E, const int64_t* m_splits,
                               float* out, const int32_t* noop, cudaStream_t s, int64_t rows_per_partial = 128);
cudaError_t run_swiglu_fwd(const void* y, int64_t M, int64_t F, void* h, cudaStream_t s);
cudaError_t run_swiglu_bwd(const void* dh, const void* y, int64_t M, int64_t F, void* dy, cudaStream_t s);

}  // namespace mxq
