// mxq_quant.cu -- MXFP8 group quantization, dequant->colwise requantization and
// per-expert dbias for grouped MoE activations on GB300 (sm_103a).
//
// Operations (TransformerEngine PR #3244, "[Pytorch] Add support for row-wise
// quanted input for grouped gemm"; PR #3224, "Improve device-init grouped
// linear module with single grouped weight support"):
//   group_quantize : bf16 (M,K) -> E4M3 rowwise and/or colwise copies with
//                    E8M0 scales, compact or swizzled; per-member swizzled
//                    colwise scale bases for ragged experts (PR #3224,
//                    group_quantize_mxfp8 VARYING_FIRST_DIM / SAME_BOTH_DIMS);
//   requant        : rowwise E4M3 + compact scales (the EP dispatch wire
//                    format) -> exact dequant -> colwise E4M3 + scales, the
//                    swizzled copy of the rowwise scales, optional dbias of
//                    the dequantized values and optional bf16 dequant output
//                    (PR #3244 description and flowchart);
//   dbias          : per-expert column sums (PR #3244, ordinary dbias reduced
//                    directly, without a wgrad stage).
//
// Design (HBM-bound): persistent CTAs (several per SM) stream 128x128 input
// tiles through a TMA-fed shared-memory ring while 4 compute warps quantize;
// lane l of warp w owns columns 4l..4l+3 of rows 32w..32w+31, so every
// warp-wide store is one contiguous stretch of a row. The colwise amax of a
// 32-row block and the dbias column sums are thread-local; the rowwise block
// spans 8 lanes. The E8M0 code depends only on the largest exponent field of the
// block, so rowwise maxima are reduced as packed 8-bit exponents (4 rows per
// word, byte-wise max shuffles). A 128x128 tile produces exactly one
// 512-byte rowwise and one 512-byte colwise scale atom of the swizzled
// layout; both are assembled in shared memory and written with 16-byte
// stores. Because every expert's row count is a multiple of 128, a tile never
// straddles two experts. dbias sums each lane's 32 rows in order, then the
// four row groups in order (fp32 partial per 128-row tile, kept in the
// caller's workspace), then each expert's tiles in order in fp64 --
// deterministic run to run.
#include "mxq_tile.cuh"

namespace mxq {

// Second dbias stage: out[e, c] = sum over expert e's row blocks of the block
// partials (one per `rpp` rows: 128 for the tile kernels, 32 where a warp's
// rows are reduced on their own), in block order, accumulated in fp64.
__global__ void __launch_bounds__(256) dbias_finalize_kernel(const float* __restrict__ partials, int64_t M,
                                                             int64_t K, int E, const int64_t* m_splits,
                                                             float* __restrict__ out, const int32_t* noop,
                                                             int64_t rpp) {
    __shared__ int64_t s_off[MXQ_MAX_EXPERTS + 1];
    if (noop && *noop) return;
    if (load_offsets(m_splits, E, M, s_off)) return;  // reported by the tile kernel
    const int e = blockIdx.y;
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= K) return;
    const int64_t t0 = s_off[e] / rpp, t1 = s_off[e + 1] / rpp;
    double acc = 0.0;
#pragma unroll 8
    for (int64_t t = t0; t < t1; ++t) acc += (double)partials[t * K + c];  // loads run ahead of the adds
    out[(int64_t)e * K + c] = (float)acc;
}

// Second stage of the routing-scale gradient: ds[m] = sum over the K/128
// column tiles of row m's partial dot products, in tile order, in fp64.
__global__ void __launch_bounds__(256) dprobs_finalize_kernel(const float* __restrict__ dp_partials, int64_t M,
                                                              int64_t tilesK, int E, const int64_t* m_splits,
                                                              float* __restrict__ out, const int32_t* noop) {
    __shared__ int64_t s_off[MXQ_MAX_EXPERTS + 1];
    if (noop && *noop) return;
    if (load_offsets(m_splits, E, M, s_off)) return;  // reported by the tile kernel
    const int64_t m = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (m >= M) return;
    double acc = 0.0;
#pragma unroll 8
    for (int64_t t = 0; t < tilesK; ++t) acc += (double)dp_partials[m * tilesK + t];
    out[m] = (float)acc;
}

static cudaError_t launch_finalize(const float* partials, int64_t M, int64_t K, int E, const int64_t* m_splits,
                                   float* out, const int32_t* noop, cudaStream_t s, int64_t rpp = kTile) {
    dim3 grid((unsigned)((K + 255) / 256), (unsigned)E);
    dbias_finalize_kernel<<<grid, 256, 0, s>>>(partials, M, K, E, m_splits, out, noop, rpp);
    return cudaGetLastError();
}

cudaError_t run_dbias_finalize(const float* partials, int64_t M, int64_t K, int E, const int64_t* m_splits,
                               float* out, const int32_t* noop, cudaStream_t s, int64_t rows_per_partial) {
    return launch_finalize(partials, M, K, E, m_splits, out, noop, s, rows_per_partial);
}

// After a scaled-bias tile launch: the per-expert scaled column sums and the
// per-row routing-scale gradients, each finalized only when asked for.
static cudaError_t finish_scaled(const float* partials, const float* dp_partials, int64_t M, int64_t K, int E,
                                 const int64_t* m_splits, float* dbias, float* dprobs, const int32_t* noop,
                                 cudaError_t err, cudaStream_t s) {
    if (err != cudaSuccess || M == 0) return err;
    if (dbias) {
        err = launch_finalize(partials, M, K, E, m_splits, dbias, noop, s);
        if (err != cudaSuccess) return err;
    }
    if (dprobs) {
        dprobs_finalize_kernel<<<(unsigned)((M + 255) / 256), 256, 0, s>>>(dp_partials, M, K / kTile, E, m_splits,
                                                                          dprobs, noop);
        err = cudaGetLastError();
    }
    return err;
}

cudaError_t run_group_quantize(const QuantCall& c, cudaStream_t s) {
    TileArgs a{};
    a.src = c.x;
    a.M = c.M;
    a.K = c.K;
    a.E = c.E;
    a.m_splits = c.m_splits;
    a.row_q = (uint8_t*)c.row_q;
    a.row_s = (uint8_t*)c.row_s;
    a.col_q = (uint8_t*)c.col_q;
    a.col_s = (uint8_t*)c.col_s;
    a.partials = c.partials;
    a.swizzle = c.swizzle;
    a.noop = c.noop;
    a.status = c.status;
    const bool r = c.row_q != nullptr, k = c.col_q != nullptr, b = c.partials != nullptr;
    cudaError_t err;
    if (c.probs) {
        a.probs = c.probs;
        a.bias = static_cast<const __nv_bfloat16*>(c.bias);
        a.dp_partials = c.dp_partials;
        if (r && k) err = launch_tile<false, true, true, true, false, true>(a, s);
        else if (r) err = launch_tile<false, true, false, true, false, true>(a, s);
        else if (k) err = launch_tile<false, false, true, true, false, true>(a, s);
        else err = launch_tile<false, false, false, true, false, true>(a, s);
        return finish_scaled(c.partials, c.dp_partials, c.M, c.K, c.E, c.m_splits, c.dbias, c.dprobs, c.noop, err, s);
    }
    if (r && k && b) err = launch_tile<false, true, true, true, false>(a, s);
    else if (r && k) err = launch_tile<false, true, true, false, false>(a, s);
    else if (r && b) err = launch_tile<false, true, false, true, false>(a, s);
    else if (r) err = launch_tile<false, true, false, false, false>(a, s);
    else if (k && b) err = launch_tile<false, false, true, true, false>(a, s);
    else if (k) err = launch_tile<false, false, true, false, false>(a, s);
    else if (b) err = launch_tile<false, false, false, true, false>(a, s);
    else return cudaSuccess;
    if (err != cudaSuccess || !b) return err;
    return launch_finalize(c.partials, c.M, c.K, c.E, c.m_splits, c.dbias, c.noop, s);
}

cudaError_t run_requant(const RequantCall& c, cudaStream_t s) {
    TileArgs a{};
    a.src = c.row_q;
    a.src_scale = (const uint8_t*)c.row_s_compact;
    a.M = c.M;
    a.K = c.K;
    a.E = c.E;
    a.m_splits = c.m_splits;
    a.row_s = (uint8_t*)c.row_s_swizzled;
    a.col_q = (uint8_t*)c.col_q;
    a.col_s = (uint8_t*)c.col_s;
    a.partials = c.partials;
    a.deq_out = (__nv_bfloat16*)c.deq_out;
    a.swizzle = c.swizzle;
    a.noop = c.noop;
    a.status = c.status;
    const bool r = c.row_s_swizzled != nullptr, k = c.col_q != nullptr, b = c.partials != nullptr,
               d = c.deq_out != nullptr;
    cudaError_t err;
    if (c.probs) {
        a.probs = c.probs;
        a.bias = static_cast<const __nv_bfloat16*>(c.bias);
        a.dp_partials = c.dp_partials;
#define MXQ_RQS(R, K_, D) \
    else if (r == R && k == K_ && d == D) err = launch_tile<true, R, K_, true, D, true>(a, s);
        if (false) err = cudaSuccess;
        MXQ_RQS(true, true, false)
        MXQ_RQS(false, true, false)
        MXQ_RQS(true, false, false)
        MXQ_RQS(false, false, false)
        MXQ_RQS(true, true, true)
        MXQ_RQS(false, true, true)
        MXQ_RQS(true, false, true)
        MXQ_RQS(false, false, true)
#undef MXQ_RQS
        else err = cudaErrorInvalidValue;
        return finish_scaled(c.partials, c.dp_partials, c.M, c.K, c.E, c.m_splits, c.dbias, c.dprobs, c.noop, err, s);
    }
    // The common dispatch shapes get their own instantiation; the rest share
    // the full variant with unused outputs masked by null checks below.
    if (r && k && !b && !d) err = launch_tile<true, true, true, false, false>(a, s);
    else if (r && k && b && !d) err = launch_tile<true, true, true, true, false>(a, s);
    else if (!r && k && !b && !d) err = launch_tile<true, false, true, false, false>(a, s);
    else if (!r && k && b && !d) err = launch_tile<true, false, true, true, false>(a, s);
    else if (r && k && b && d) err = launch_tile<true, true, true, true, true>(a, s);
    else if (r && k && !b && d) err = launch_tile<true, true, true, false, true>(a, s);
    else if (!r && k && !b && d) err = launch_tile<true, false, true, false, true>(a, s);
    else if (!r && k && b && d) err = launch_tile<true, false, true, true, true>(a, s);
    else if (r && !k && !b && !d) err = launch_tile<true, true, false, false, false>(a, s);
    else if (!k && d) err = r ? (b ? launch_tile<true, true, false, true, true>(a, s)
                                   : launch_tile<true, true, false, false, true>(a, s))
                              : (b ? launch_tile<true, false, false, true, true>(a, s)
                                   : launch_tile<true, false, false, false, true>(a, s));
    else if (!k && b) err = r ? launch_tile<true, true, false, true, false>(a, s)
                              : launch_tile<true, false, false, true, false>(a, s);
    else return cudaSuccess;
    if (err != cudaSuccess || !b) return err;
    return launch_finalize(c.partials, c.M, c.K, c.E, c.m_splits, c.dbias, c.noop, s);
}

cudaError_t run_grouped_dbias(const void* dy, int64_t M, int64_t N, int E, const int64_t* m_splits, float* out,
                              float* partials, int32_t* status, cudaStream_t s) {
    TileArgs a{};
    a.src = dy;
    a.M = M;
    a.K = N;
    a.E = E;
    a.m_splits = m_splits;
    a.partials = partials;
    a.status = status;
    cudaError_t err = launch_tile<false, false, false, true, false>(a, s);
    if (err != cudaSuccess) return err;
    return launch_finalize(partials, M, N, E, m_splits, out, nullptr, s);
}

}  // namespace mxq
