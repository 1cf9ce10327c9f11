/*
 * mxq.h -- C ABI of the GB300 (sm_103a) MXFP8 grouped-quantization and
 * grouped-GEMM library for mixture-of-experts expert layers.
 *
 * The operations follow three TransformerEngine pull-request pages:
 *   [RQ] PR #3244 "[Pytorch] Add support for row-wise quanted input for
 *        grouped gemm" -- the description (fprop/dgrad read the rowwise
 *        prequantized input directly; wgrad needs a columnwise copy made by
 *        dequantize + columnwise requantize), the review threads on
 *        prepare_prequantized_mxfp8_grouped_input (compact scale shape
 *        (round_up(tokens,128), round_up(cols/32,4)); 128-token per-expert
 *        alignment and hidden % 512 from the dispatch; dense swizzle of the
 *        dispatch's rowwise scales; "group_quantize + swizzle fusion" for the
 *        columnwise scales; compact scales required for dequantization) and
 *        the Greptile flowchart (bias and routing-scale reductions from the
 *        dequantized tensor).
 *   [FM] PR #3545 "Fix distributed BF16 weights and trim NVFP4 saved state
 *        in the fused grouped MLP" -- forward GEMMs read rowwise weights, the
 *        columnwise weight copy exists for dgrad, every wgrad path reads
 *        only columnwise input tiles; FC1 -> activation -> FC2.
 *   [DI] PR #3224 "Improve device-init grouped linear module with single
 *        grouped weight support" -- device-resident int64 m_splits (host
 *        m_splits rejected), one grouped weight (E, out, in) and a 2-D
 *        grouped bias (E, out), group_quantize output= reuse (caller-owned
 *        outputs, stable pointers) and noop_flag for graph replay,
 *        per-member swizzled scale bases in group_quantize_mxfp8, explicit
 *        errors instead of silent fallbacks.
 *
 * Formats. E4M3 data bytes; one E8M0 scale byte (2^(code-127)) per 32
 * contiguous elements: "rowwise" blocks run along the last dimension,
 * "colwise" blocks along tokens (the first dimension) inside one expert.
 * Colwise data bytes keep the (rows, cols) row-major byte order of the
 * source. Shared exponent s = floor(log2(amax)) - 8 (clamped to
 * [-127,127]; all-zero block -> code 0x00); elements are cast with
 * round-to-nearest-even, saturating at +-448, sign kept (OCP MX v1.0).
 *
 * Scale layouts.
 *   compact rowwise (R, C=cols/32) : (round_up(R,128), round_up(C,4)) bytes,
 *                                    row-major, zero padded   [RQ]
 *   compact colwise                : (round_up(R/32,4), round_up(cols,128))
 *   swizzled                       : 128x4 tensor-core atoms (512 B): logical
 *        S[r][c] of an (R, C) matrix lives at byte
 *        ((r/128)*(C/4) + c/4)*512 + (r%32)*16 + ((r%128)/32)*4 + c%4.
 *        Rowwise scales of a grouped tensor are swizzled as one (R, cols/32)
 *        matrix (valid because every m_e % 128 == 0 [RQ]); colwise scales
 *        are swizzled PER EXPERT as the (cols, m_e/32) matrix
 *        S_e[k][i] = scale of token block i of expert e at column k, placed
 *        at byte cols*off_e/32 (off_e = tokens before expert e) [DI].
 *
 * Grouping contract: E >= 1 (<= MXQ_MAX_EXPERTS); every m_e >= 0 and a
 * multiple of 128; sum(m_e) == M. cols (K, N) multiples of 128 for the
 * quantizers; the GEMMs additionally need the output-tile width (the
 * dimension written as 256-column tiles) to be a multiple of 256.
 *
 * Ownership. The caller allocates every input, output and workspace (device
 * memory, 16-byte aligned); the library allocates nothing and keeps no
 * state between calls other than a per-device cache of device attributes.
 * Every call is asynchronous on `stream` and never synchronizes, except
 * mxq_status_read.
 *
 * Errors. Host-detectable faults return a negative mxq error code before
 * anything is launched. Data-dependent faults (m_splits on the device) are
 * OR-ed into the caller's device status word *d_status (may be NULL to
 * skip reporting); the work that depends on the bad data is skipped and its
 * outputs are left untouched.
 */
#ifndef MXQ_H
#define MXQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* mxq_stream_t; /* identical to cudaStream_t */

#if defined(__GNUC__)
#define MXQ_API __attribute__((visibility("default")))
#else
#define MXQ_API
#endif

#define MXQ_MAX_EXPERTS 1024

/* host return codes */
enum {
    MXQ_OK = 0,
    MXQ_ERR_NULL = -1,         /* a required pointer is NULL */
    MXQ_ERR_SHAPE = -2,        /* a dimension breaks the contract above */
    MXQ_ERR_HOST_POINTER = -3, /* m_splits (or data) is not device memory [DI] */
    MXQ_ERR_ARCH = -4,         /* current device is not sm_103 (GB300) */
    MXQ_ERR_WORKSPACE = -5,    /* workspace smaller than mxq_workspace_bytes() */
    MXQ_ERR_LAUNCH = -6,       /* a CUDA call failed (see mxq_last_cuda_error) */
    MXQ_ERR_FLAGS = -7,        /* unknown or inconsistent flags */
    MXQ_ERR_ALIGN = -8,        /* a pointer is not 16-byte aligned */
    MXQ_ERR_SCRATCH_LIMIT = -9 /* problem larger than mxq_grouped_dbias_noalloc's fixed scratch */
};

/* device status word bits (sticky; OR-ed by the kernels) */
enum {
    MXQ_STATUS_SPLIT_UNALIGNED = 1, /* some m_e % 128 != 0 */
    MXQ_STATUS_SPLIT_NEGATIVE = 2,  /* some m_e < 0 */
    MXQ_STATUS_SPLIT_SUM = 4,       /* sum(m_e) != M */
    MXQ_STATUS_WAIT_TIMEOUT = 8     /* a bounded on-chip wait expired (the kernel bailed out) */
};

/* flags */
enum {
    MXQ_ROWWISE = 1,      /* group_quantize: emit the rowwise copy;
                             requant: emit the swizzled copy of the rowwise scales */
    MXQ_COLWISE = 2,      /* emit the colwise copy */
    MXQ_SWIZZLE = 4,      /* scales in the swizzled GEMM layout (else compact) */
    MXQ_DEQUANT_OUT = 8,  /* requant: also write the dequantized bf16 tensor; SwiGLU
                             paths: also write the bf16 values that were quantized */
    MXQ_ACCUMULATE = 16,  /* wgrad: dW += product (else dW = product) */
    MXQ_OUT_BF16 = 32,    /* wgrad: dW in bf16 (else fp32) */
    MXQ_PAD_EXPERTS = 64  /* group_quantize / requant: expert counts need not be
                             multiples of 128; see "Padded grouping" below */
};

/* operation ids for mxq_workspace_bytes */
enum {
    MXQ_OP_GROUP_QUANTIZE = 1,
    MXQ_OP_REQUANT_COLWISE = 2,
    MXQ_OP_GROUPED_DBIAS = 3,
    MXQ_OP_GEMM_FPROP = 4,
    MXQ_OP_GEMM_DGRAD = 5,
    MXQ_OP_GEMM_WGRAD = 6,
    MXQ_OP_SWIGLU_BWD_QUANTIZE = 7,
    MXQ_OP_SCALED_BIAS = 8,
    MXQ_OP_GEMM_DGRAD_SWIGLU = 9
};

/* Library version (major*10000 + minor*100 + patch). */
MXQ_API int mxq_version(void);

/* Bytes of one scale buffer for an (rows, cols) tensor: the padded compact
 * shape of [RQ]; for rows % 128 == 0 and cols % 128 == 0 the swizzled
 * layout has the same size. colwise != 0 selects the colwise shape. */
MXQ_API size_t mxq_scale_bytes(int64_t rows, int64_t cols, int colwise);

/* Padded grouping (flag MXQ_PAD_EXPERTS on mxq_group_quantize and
 * mxq_requant_colwise) [RQ: the review of the grouped swizzle -- a dense
 * swizzle is valid only when each expert's tokens are padded to a multiple
 * of 128; a grouped swizzle handles variable per-expert dims]. Each m_e may
 * be any count >= 0 (M any, d_m_splits required). Every expert is padded,
 * in the scale row space only, to round_up(m_e, 128) rows: expert e's scale
 * rows start at poff_e = sum_{e'<e} round_up(m_e', 128), R = poff_E.
 *   - E4M3 codes (row and col), the compact rowwise scales and the bf16
 *     dequant output keep the dense (M, K) layouts;
 *   - swizzled rowwise scales: the swizzle of the (R, K/32) matrix whose row
 *     poff_e + i holds token row off_e + i (pad rows 0);
 *   - colwise blocks are 32 rows of one expert starting at off_e; the last
 *     block of an expert may hold fewer rows and is scaled by them (as if
 *     the padding were zero rows). Compact colwise scales: (R/32, K), block
 *     i of expert e at row poff_e/32 + i; swizzled: expert e's logical
 *     (K, round_up(m_e,128)/32) matrix at byte K * poff_e / 32; pads 0;
 *   - dbias as usual (workspace: mxq_workspace_bytes with the flag).
 * With 128-aligned counts every output equals the unflagged call's.
 * mxq_scale_bytes_grouped(rows = M, cols = K, E, colwise) is a size that
 * holds the padded scale buffers for any split of M rows into E experts. */
MXQ_API size_t mxq_scale_bytes_grouped(int64_t rows, int64_t cols, int E, int colwise);

/* Workspace bytes `op` needs for these sizes and flags (0 if none). For
 * group_quantize / requant it is nonzero only when dbias is requested:
 * fp32 column partial sums of every 128-row tile, (M/128) * K * 4 bytes. */
MXQ_API size_t mxq_workspace_bytes(int op, int64_t M, int64_t N, int64_t K, int E, int flags);

/* group_quantize [RQ][DI]: bf16 x (M, K) row-major, split into E experts by
 * the device int64 array d_m_splits (NULL: E uniform members of M/E rows,
 * the weight case (E*N, K) -- then M/E must be a multiple of 128) into
 * MXFP8. flags: MXQ_ROWWISE and/or MXQ_COLWISE, optional MXQ_SWIZZLE.
 *   row_data (M,K) E4M3, row_scale mxq_scale_bytes(M,K,0) bytes;
 *   col_data (M,K) E4M3, col_scale mxq_scale_bytes(M,K,1) bytes;
 *   dbias_out (E,K) fp32 or NULL: per-expert column sums of x (needs ws);
 *   d_noop: NULL or a device int32; when it is nonzero the call writes
 *   nothing (graph replay with a skipped step [DI]).
 * Unused outputs may be NULL. Returns MXQ_OK or a negative code. */
MXQ_API int mxq_group_quantize(const void* x_bf16, int64_t M, int64_t K, int E, const int64_t* d_m_splits, int flags,
                       void* row_data, void* row_scale, void* col_data, void* col_scale, float* dbias_out,
                       const int32_t* d_noop, int32_t* d_status, void* ws, size_t ws_bytes, mxq_stream_t stream);

/* requant_colwise [RQ]: from a rowwise-prequantized grouped input (the
 * expert-parallel FP8 dispatch's wire format: row_data (M,K) E4M3 with
 * COMPACT scales row_scale_compact) build the colwise copy wgrad needs by
 * dequantizing (exactly) and quantizing the dequantized values colwise.
 *   flags: MXQ_COLWISE (col_data + col_scale, layout per MXQ_SWIZZLE),
 *          MXQ_ROWWISE (row_scale_swizzled_out: the rowwise scales in the
 *          GEMM layout, for fprop/dgrad on the rowwise data),
 *          MXQ_DEQUANT_OUT (dequant_bf16_out (M,K)).
 *   dbias_out (E,K) fp32 or NULL: per-expert sums of the dequantized
 *   values (the "ordinary dbias" reduced without a wgrad stage; needs ws). */
MXQ_API int mxq_requant_colwise(const void* row_data, const void* row_scale_compact, int64_t M, int64_t K, int E,
                        const int64_t* d_m_splits, int flags, void* col_data, void* col_scale,
                        void* row_scale_swizzled_out, float* dbias_out, void* dequant_bf16_out,
                        const int32_t* d_noop, int32_t* d_status, void* ws, size_t ws_bytes, mxq_stream_t stream);

/* grouped_dbias [RQ]: db[e, n] = sum over expert e's rows of dy[m, n];
 * dy bf16 (M, N); out fp32 (E, N); an empty expert gets 0. Deterministic
 * (fixed-order tree per 128-row tile, fp64 across tiles); needs ws. */
MXQ_API int mxq_grouped_dbias(const void* dy_bf16, int64_t M, int64_t N, int E, const int64_t* d_m_splits, float* dbias_out,
                      int32_t* d_status, void* ws, size_t ws_bytes, mxq_stream_t stream);

/* Scaled bias and routing-scale gradients [RQ: "bias and routing-scale
 * reductions" are taken from the dequantized gradient] (reading: expert e
 * adds its bias scaled by the token's routing scale, y[m,:] = X[m,:] W_e^T
 * + s_m * b_e; the pages print no formula). From the gradient dY (M, K):
 *   dbias_out[e, k] = sum over expert e's rows m of s_m * dY[m, k]  (E, K) fp32
 *   dprobs_out[m]   = sum over k of dY[m, k] * b_e(m)[k]             (M)    fp32
 * fused into the pass that quantizes (bf16 dY) or requantizes (rowwise E4M3
 * wire format, reductions of the exact dequantized values) the gradient.
 * probs: device fp32 (M), the routing scales s_m; bias_bf16: device (E, K).
 * Either output may be NULL, not both; d_m_splits is required. Workspace:
 * mxq_workspace_bytes(MXQ_OP_SCALED_BIAS, M, 0, K, E, 0) bytes. Sums are
 * fp32 in a fixed order per 128x128 tile, then fp64 over tiles: identical
 * run to run. Other arguments, flags and errors as mxq_group_quantize /
 * mxq_requant_colwise; with flags == 0 (and MXQ_DEQUANT_OUT unset) only the
 * two reductions run. */
MXQ_API int mxq_group_quantize_scaled_bias(const void* x_bf16, int64_t M, int64_t K, int E,
                                           const int64_t* d_m_splits, int flags, void* row_data, void* row_scale,
                                           void* col_data, void* col_scale, const float* probs,
                                           const void* bias_bf16, float* dbias_out, float* dprobs_out,
                                           const int32_t* d_noop, int32_t* d_status, void* ws, size_t ws_bytes,
                                           mxq_stream_t stream);
MXQ_API int mxq_requant_colwise_scaled_bias(const void* row_data, const void* row_scale_compact, int64_t M,
                                            int64_t K, int E, const int64_t* d_m_splits, int flags, void* col_data,
                                            void* col_scale, void* row_scale_swizzled_out, const float* probs,
                                            const void* bias_bf16, float* dbias_out, float* dprobs_out,
                                            void* dequant_bf16_out, const int32_t* d_noop, int32_t* d_status,
                                            void* ws, size_t ws_bytes, mxq_stream_t stream);

/* grouped fprop [RQ][DI]: Y[m, :] = X[m, :] . W[e(m)]^T (+ bias[e(m)]),
 * X rowwise (M,K) E4M3 + swizzled rowwise scales; W rowwise (E,N,K) E4M3
 * + swizzled rowwise scales of the (E*N, K) matrix; bias bf16 (E,N) or
 * NULL (added in fp32 before rounding); Y bf16 (M,N). N % 256 == 0. */
MXQ_API int mxq_grouped_gemm_fprop(const void* x_data, const void* x_scale, const void* w_data, const void* w_scale,
                           const void* bias_bf16, int64_t M, int64_t N, int64_t K, int E,
                           const int64_t* d_m_splits, void* y_bf16, int32_t* d_status, void* ws,
                           size_t ws_bytes, mxq_stream_t stream);

/* mxq_grouped_gemm_fprop / _dgrad with flags. MXQ_PAD_EXPERTS: expert
 * counts need not be multiples of 128 (M any, E <= 512); the activation's
 * (X's, or dY's) rowwise scales are in the padded swizzled layout that
 * mxq_group_quantize / mxq_requant_colwise produce with the same flag;
 * rows are processed per expert in 128-row slices and only the expert's
 * rows of the output are written. Without flags these are the plain calls. */
MXQ_API int mxq_grouped_gemm_fprop_ex(const void* x_data, const void* x_scale, const void* w_data,
                                      const void* w_scale, const void* bias_bf16, int64_t M, int64_t N, int64_t K,
                                      int E, const int64_t* d_m_splits, int flags, void* y_bf16, int32_t* d_status,
                                      void* ws, size_t ws_bytes, mxq_stream_t stream);
MXQ_API int mxq_grouped_gemm_dgrad_ex(const void* dy_data, const void* dy_scale, const void* w_col_data,
                                      const void* w_col_scale, int64_t M, int64_t N, int64_t K, int E,
                                      const int64_t* d_m_splits, int flags, void* dx_bf16, int32_t* d_status,
                                      void* ws, size_t ws_bytes, mxq_stream_t stream);

/* grouped fprop of FC1 with SwiGLU and its quantization in the epilogue
 * (the fused grouped MLP's FC1 -> activation [FM]; quantization as
 * mxq_group_quantize [RQ][DI]). x_data (M, K) E4M3 rowwise with swizzled
 * scales; w1_data (E, 2F, K) E4M3 rowwise (rows [0, F) of each expert are
 * the gate, [F, 2F) the up projection) with swizzled scales; bias_bf16
 * (E, 2F) or NULL. Writes:
 *   y1_bf16 (M, 2F): the FC1 output, bit-identical to mxq_grouped_gemm_fprop
 *     (saved for the SwiGLU backward);
 *   h = silu(gate) * up from those bf16 values in the fp32 steps of
 *     mxq_swiglu_fwd, quantized rowwise (h_row_data (M, F), h_row_scale) and
 *     colwise (h_col_data (M, F), h_col_scale) exactly as mxq_swiglu_quantize
 *     would quantize it (flags: MXQ_SWIZZLE selects swizzled scales, else
 *     compact);
 *   with MXQ_DEQUANT_OUT, h_bf16_out (M, F): the bf16 h that was quantized
 *     (else h_bf16_out is ignored and may be NULL).
 * F % 128 == 0, K % 128 == 0. ws may be NULL. */
MXQ_API int mxq_grouped_gemm_fprop_swiglu(const void* x_data, const void* x_scale, const void* w1_data,
                                          const void* w1_scale, const void* bias_bf16, int64_t M, int64_t K,
                                          int64_t F, int E, const int64_t* d_m_splits, int flags, void* y1_bf16,
                                          void* h_row_data, void* h_row_scale, void* h_col_data, void* h_col_scale,
                                          void* h_bf16_out, int32_t* d_status, void* ws, size_t ws_bytes,
                                          mxq_stream_t stream);

/* grouped dgrad [RQ][FM]: dX[m, :] = dY[m, :] . W[e(m)], dY rowwise (M,N)
 * + swizzled rowwise scales; W colwise (E,N,K) E4M3 (W's byte order,
 * blocks along N) + per-expert swizzled colwise scales (expert e: logical
 * (K, N/32) at byte e*K*N/32); dX bf16 (M,K). K % 256 == 0. */
MXQ_API int mxq_grouped_gemm_dgrad(const void* dy_data, const void* dy_scale, const void* w_col_data,
                           const void* w_col_scale, int64_t M, int64_t N, int64_t K, int E,
                           const int64_t* d_m_splits, void* dx_bf16, int32_t* d_status, void* ws,
                           size_t ws_bytes, mxq_stream_t stream);

/* grouped dgrad of FC2 with the SwiGLU backward and the quantization of its
 * result in the epilogue (the fused grouped MLP's activation backward [FM];
 * quantization and dbias as mxq_group_quantize [RQ][DI]). dh = dY2 . W2_e
 * (dy_data (M, N) rowwise with swizzled scales, w_col_data (E, N, F)
 * colwise) never leaves the chip: it is rounded to bf16 as
 * mxq_grouped_gemm_dgrad would write it and, with the saved FC1 output
 * y1_bf16 (M, 2F) = [g | u], turned into dY1 = [dg | du] (M, 2F) in the fp32
 * steps of mxq_swiglu_bwd, rounded to bf16 and quantized rowwise
 * (dy1_row_*) and colwise (dy1_col_*) exactly as mxq_swiglu_bwd_quantize
 * would quantize it (flags: MXQ_SWIZZLE, else compact scales).
 * dbias_out (E, 2F) fp32 or NULL: per-expert column sums of dY1 (fp32 per 32
 * rows in a fixed order, fp64 over blocks; needs ws of
 * mxq_workspace_bytes(MXQ_OP_GEMM_DGRAD_SWIGLU, M, N, F, E, 0) bytes).
 * With MXQ_DEQUANT_OUT, dy1_bf16_out (M, 2F) gets the bf16 dY1 that was
 * quantized (else it is ignored and may be NULL).
 * F % 256 == 0, N % 128 == 0. */
MXQ_API int mxq_grouped_gemm_dgrad_swiglu(const void* dy_data, const void* dy_scale, const void* w_col_data,
                                          const void* w_col_scale, const void* y1_bf16, int64_t M, int64_t N,
                                          int64_t F, int E, const int64_t* d_m_splits, int flags,
                                          void* dy1_row_data, void* dy1_row_scale, void* dy1_col_data,
                                          void* dy1_col_scale, float* dbias_out, void* dy1_bf16_out,
                                          int32_t* d_status, void* ws, size_t ws_bytes, mxq_stream_t stream);

/* grouped wgrad [RQ][FM]: dW[e] = dY_e^T . X_e over expert e's tokens,
 * from the colwise copies only: dY colwise (M,N) + per-expert swizzled
 * colwise scales, X colwise (M,K) + per-expert swizzled colwise scales.
 * dW (E,N,K) fp32 (bf16 with MXQ_OUT_BF16); MXQ_ACCUMULATE adds into dW.
 * An empty expert gets dW[e] = 0 (unchanged with MXQ_ACCUMULATE).
 * MXQ_PAD_EXPERTS: expert counts need not be multiples of 128 (M any,
 * E <= 512), both colwise scale sets in the padded layout; the tokens past
 * an expert in its last 128-token block are cleared on chip before the
 * MMAs. K % 256 == 0. */
MXQ_API int mxq_grouped_gemm_wgrad(const void* dy_col_data, const void* dy_col_scale, const void* x_col_data,
                           const void* x_col_scale, int64_t M, int64_t N, int64_t K, int E,
                           const int64_t* d_m_splits, int flags, void* dw, int32_t* d_status, void* ws,
                           size_t ws_bytes, mxq_stream_t stream);

/* grouped_dbias without any allocation, for callers that cannot allocate
 * device memory (code running where no allocator may be called, or with no
 * access to one). The pages have no counterpart: this is a library
 * convenience. Same result as mxq_grouped_dbias, but the per-tile partial
 * sums live in a fixed 8 MiB file-scope device array that every GPU loading
 * the library holds until the process exits:
 *   - (M/128) * N must be <= 2,097,152, else MXQ_ERR_SCRATCH_LIMIT;
 *   - the first call in each CUDA context of a device (the first call of the
 *     process on that device, and again after cudaDeviceReset) looks up the
 *     array's device address with a host-side symbol query;
 *   - all calls share the array (it keeps the last call's partials, which the
 *     next call overwrites before reading); calls that overlap on the GPU
 *     race, so serialise them. */
MXQ_API int mxq_grouped_dbias_noalloc(const void* dy_bf16, int64_t M, int64_t N, int E, const int64_t* d_m_splits,
                                      float* dbias_out, int32_t* d_status, mxq_stream_t stream);

/* SwiGLU between FC1 and FC2 of the fused grouped MLP [FM] (reading: the
 * first F columns of the FC1 output are the gate):
 *   fwd: y (M, 2F) bf16 -> h (M, F) bf16, h = silu(g) * u;
 *   bwd: dh (M, F), y (M, 2F) -> dy (M, 2F) = [dh*u*silu'(g) | dh*silu(g)].
 * bf16 I/O; the math is fp32: sigmoid(g) = 1 / (1 + 2^(-g log2 e)) with the
 * hardware base-2 exponential and reciprocal (relative errors near 2^-22),
 * h = (g*s)*u, dg = ((dh*u)*s)*(1 + g*(1 - s)), du = dh*(g*s), each result
 * rounded once to bf16: within one bf16 step of the exact value. Every
 * SwiGLU path of this library runs the same steps and agrees bit for bit.
 * F % 8 == 0. */
MXQ_API int mxq_swiglu_fwd(const void* y_bf16, int64_t M, int64_t F, void* h_bf16, mxq_stream_t stream);
MXQ_API int mxq_swiglu_bwd(const void* dh_bf16, const void* y_bf16, int64_t M, int64_t F, void* dy_bf16,
                   mxq_stream_t stream);

/* SwiGLU fused with group_quantize [FM][RQ][DI] (the fused grouped MLP's
 * FC1 -> activation -> FC2, with the activation's output quantized where it
 * is produced). y (M, 2F) bf16 is the FC1 output [gate | up]; h = silu(g)*u
 * is computed in fp32 (the same steps as mxq_swiglu_fwd, so the results
 * agree bit for bit), rounded to bf16 and
 * quantized exactly as mxq_group_quantize would quantize that bf16 h.
 * flags: MXQ_ROWWISE / MXQ_COLWISE / MXQ_SWIZZLE as for group_quantize;
 * MXQ_DEQUANT_OUT also writes h in bf16 to h_bf16_out (M, F). Outputs are
 * (M, F) tensors with their scale buffers. F % 128 == 0. */
MXQ_API int mxq_swiglu_quantize(const void* y_bf16, int64_t M, int64_t F, int E, const int64_t* d_m_splits,
                                int flags, void* row_data, void* row_scale, void* col_data, void* col_scale,
                                void* h_bf16_out, const int32_t* d_noop, int32_t* d_status, mxq_stream_t stream);

/* SwiGLU backward fused with group_quantize and dbias [FM][RQ]: from dh
 * (M, F) and y (M, 2F), dY1 = [dg | du] (M, 2F) is computed in fp32 (the
 * steps of mxq_swiglu_bwd), rounded to bf16 and quantized as
 * mxq_group_quantize would quantize it; dbias_out (E, 2F) fp32 or NULL gets
 * its per-expert column sums (needs ws of mxq_workspace_bytes(
 * MXQ_OP_SWIGLU_BWD_QUANTIZE, M, 0, F, E, 0) bytes); MXQ_DEQUANT_OUT also
 * writes dY1 in bf16 to dy_bf16_out. F % 128 == 0. */
MXQ_API int mxq_swiglu_bwd_quantize(const void* dh_bf16, const void* y_bf16, int64_t M, int64_t F, int E,
                                    const int64_t* d_m_splits, int flags, void* row_data, void* row_scale,
                                    void* col_data, void* col_scale, float* dbias_out, void* dy_bf16_out,
                                    const int32_t* d_noop, int32_t* d_status, void* ws, size_t ws_bytes,
                                    mxq_stream_t stream);

/* Measurement utility beside the MXFP8 path: the tensor-pipe ceiling that
 * bounds the grouped GEMMs on this GPU. Launches one CTA per SM on `stream`;
 * each issues mmas_per_sm block-scaled 128x256x32 tcgen05 MMAs (E4M3 x E4M3,
 * E8M0 scales, fp32 accumulation in TMEM) back to back from operands resident
 * in shared memory, with the scale copies and commit of the grouped GEMM's
 * 128-deep K block but no loads, waits between K blocks, tile boundaries or
 * epilogue. Timed on the stream, 2*128*256*32*mmas_per_sm*SMs / time is the
 * most a kernel built from these instructions can reach. Reads and writes no
 * global memory except *d_status (MXQ_STATUS_WAIT_TIMEOUT; may be NULL).
 * mmas_per_sm in [0, 2^31); MXQ_ERR_SHAPE otherwise. */
MXQ_API int mxq_probe_mma_stream(int64_t mmas_per_sm, int32_t* d_status, mxq_stream_t stream);

/* The same probe with a choice of operands: MXQ_PROBE_ZEROS (as above) or
 * MXQ_PROBE_RANDOM, pseudo-random E4M3 bytes (exponent field <= 6, so no NaN
 * and finite sums) with unit E8M0 scales. The tensor pipe draws more power
 * multiplying random bits than zeros; a stream of random operands long
 * enough to reach the board's power limit (about a second) measures the
 * sustained ceiling a GEMM on real data meets. Any other `operands` value:
 * MXQ_ERR_FLAGS. */
enum { MXQ_PROBE_ZEROS = 0, MXQ_PROBE_RANDOM = 1 };
MXQ_API int mxq_probe_mma_stream_ex(int64_t mmas_per_sm, int operands, int32_t* d_status, mxq_stream_t stream);

/* Self-test of the failure path every kernel shares: one CTA waits, limit_ns
 * long, on an mbarrier that nothing arrives on, with the kernels' bounded wait;
 * the wait expires, the CTA's other waiter is released through the abort flag,
 * MXQ_STATUS_WAIT_TIMEOUT is set in *d_status (required) and the kernel returns,
 * leaving the context usable. limit_ns in [1e3, 1e10]; MXQ_ERR_SHAPE otherwise. */
MXQ_API int mxq_selftest_wait_timeout(int64_t limit_ns, int32_t* d_status, mxq_stream_t stream);

/* Copy the device status word to *h_out after `stream` drains (the only
 * synchronizing call). */
MXQ_API int mxq_status_read(const int32_t* d_status, int32_t* h_out, mxq_stream_t stream);

/* Text for a host return code. */
MXQ_API const char* mxq_error_string(int code);

/* The last CUDA error code seen by the library on this thread (0 if none). */
MXQ_API int mxq_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MXQ_H */
