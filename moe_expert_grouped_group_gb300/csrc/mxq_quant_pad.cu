// mxq_quant_pad.cu -- group_quantize, requant and dbias for expert counts
// that are not multiples of 128 (per-expert padded scale layouts).
//
// TransformerEngine PR #3244's review notes that swizzling a grouped
// activation as one dense tensor is valid only when every expert's token
// count is padded to a multiple of 128, and that a grouped swizzle handles
// variable per-expert dims. Here each expert's rows are padded (in the scale
// row space only) to a multiple of 128: expert e's scale rows start at
// poff_e = sum_{e' < e} round_up(m_e', 128). The E4M3 codes, the compact
// rowwise scales and the bf16 dequant output stay dense; the swizzled
// scales, the compact colwise scales and the dbias tile partials use the
// padded row space, pad entries 0. A colwise 32-row block that crosses the
// end of an expert covers that expert's rows only (the result is that of
// zero rows in the padding). The tile kernel is mx_tile_kernel<..., kPad>:
// it walks each expert's 128-row slices, loads them from the expert's first
// row (TMA rows need no alignment) and masks the rows past the expert.
#include "mxq_tile.cuh"

namespace mxq {

// out[e, c] = sum, in order and in fp64, of expert e's 128-row tile partials,
// which sit at padded tile rows [poff_e / 128, poff_{e+1} / 128).
__global__ void __launch_bounds__(256) dbias_finalize_padded_kernel(const float* __restrict__ partials, int64_t M,
                                                                    int64_t K, int E, const int64_t* m_splits,
                                                                    float* __restrict__ out, const int32_t* noop) {
    __shared__ int64_t s_off[MXQ_MAX_EXPERTS + 1];
    __shared__ int64_t s_poff[MXQ_MAX_EXPERTS + 1];
    if (noop && *noop) return;
    if (load_offsets_padded(m_splits, E, M, s_off, s_poff)) return;  // reported by the tile kernel
    const int e = blockIdx.y;
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= K) return;
    const int64_t t0 = s_poff[e] / kTile, t1 = s_poff[e + 1] / kTile;
    double acc = 0.0;
#pragma unroll 8
    for (int64_t t = t0; t < t1; ++t) acc += (double)partials[t * K + c];
    out[(int64_t)e * K + c] = (float)acc;
}

static cudaError_t finalize_padded(const float* partials, int64_t M, int64_t K, int E, const int64_t* m_splits,
                                   float* out, const int32_t* noop, cudaStream_t s) {
    if (M == 0) return cudaMemsetAsync(out, 0, (size_t)E * K * sizeof(float), s);
    dim3 grid((unsigned)((K + 255) / 256), (unsigned)E);
    dbias_finalize_padded_kernel<<<grid, 256, 0, s>>>(partials, M, K, E, m_splits, out, noop);
    return cudaGetLastError();
}

cudaError_t run_group_quantize_padded(const QuantCall& c, cudaStream_t s) {
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
    if (r && k && b) err = launch_tile<false, true, true, true, false, false, true>(a, s);
    else if (r && k) err = launch_tile<false, true, true, false, false, false, true>(a, s);
    else if (r && b) err = launch_tile<false, true, false, true, false, false, true>(a, s);
    else if (r) err = launch_tile<false, true, false, false, false, false, true>(a, s);
    else if (k && b) err = launch_tile<false, false, true, true, false, false, true>(a, s);
    else if (k) err = launch_tile<false, false, true, false, false, false, true>(a, s);
    else if (b) err = launch_tile<false, false, false, true, false, false, true>(a, s);
    else return cudaSuccess;
    if (err != cudaSuccess || !b) return err;
    return finalize_padded(c.partials, c.M, c.K, c.E, c.m_splits, c.dbias, c.noop, s);
}

cudaError_t run_requant_padded(const RequantCall& c, cudaStream_t s) {
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
#define MXQ_RQP(R, K_, B, D) \
    else if (r == R && k == K_ && b == B && d == D) err = launch_tile<true, R, K_, B, D, false, true>(a, s);
    if (!r && !k && !b && !d) return cudaSuccess;
    MXQ_RQP(true, true, false, false)
    MXQ_RQP(true, true, true, false)
    MXQ_RQP(false, true, false, false)
    MXQ_RQP(false, true, true, false)
    MXQ_RQP(true, true, false, true)
    MXQ_RQP(true, true, true, true)
    MXQ_RQP(false, true, false, true)
    MXQ_RQP(false, true, true, true)
    MXQ_RQP(true, false, false, false)
    MXQ_RQP(true, false, true, false)
    MXQ_RQP(false, false, true, false)
    MXQ_RQP(true, false, false, true)
    MXQ_RQP(true, false, true, true)
    MXQ_RQP(false, false, false, true)
    MXQ_RQP(false, false, true, true)
#undef MXQ_RQP
    else err = cudaErrorInvalidValue;
    if (err != cudaSuccess || !b) return err;
    return finalize_padded(c.partials, c.M, c.K, c.E, c.m_splits, c.dbias, c.noop, s);
}

}  // namespace mxq
