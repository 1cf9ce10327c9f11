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
// Design (HBM-bound): one CTA of 8 warps handles a 128x128 tile. Warp w owns
// rows 32*(w/2)..+31 and columns 64*(w%2)..+63; lane l owns one row of that
// strip (128 contiguous input bytes). Rowwise amax is thread-local; the
// colwise amax of a 32-row block is one warp-wide redux.sync per column. A
// 128x128 tile produces exactly one 512-byte rowwise scale atom and one
// 512-byte colwise scale atom of the swizzled layout; both are assembled in
// shared memory and written with 16-byte stores. Because every expert's row
// count is a multiple of 128, a tile never straddles two experts. dbias uses
// a fixed-order butterfly over lanes, a fixed-order sum over the four row
// groups (fp32 partial per 128-row tile, kept in the caller's workspace) and
// an fp64 ordered sum over each expert's tiles -- deterministic run to run.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "mxq_common.cuh"
#include "mxq_internal.h"

namespace mxq {

struct TileArgs {
    const void* src;           // bf16 x (M,K), or rowwise E4M3 data (requant)
    const uint8_t* src_scale;  // requant: compact rowwise scales of src
    int64_t M, K;
    int E;
    const int64_t* m_splits;   // device, or nullptr for uniform members
    uint8_t* row_q;            // quantize: rowwise codes
    uint8_t* row_s;            // rowwise scales (requant: swizzled copy of src_scale)
    uint8_t* col_q;
    uint8_t* col_s;
    float* partials;           // (M/128, K) fp32 column sums per tile
    __nv_bfloat16* deq_out;    // requant: bf16 dequantized tensor
    int swizzle;
    const int32_t* noop;
    int32_t* status;
};

__device__ __forceinline__ uint4 ldg_nc(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

template <bool kReq, bool kRow, bool kCol, bool kBias, bool kDeq>
__global__ void __launch_bounds__(256, 2) mx_tile_kernel(TileArgs a) {
    __shared__ int64_t s_off[MXQ_MAX_EXPERTS + 1];
    __shared__ __align__(16) uint8_t s_rs[512];
    __shared__ __align__(16) uint8_t s_cs[512];
    __shared__ float s_red[4][kTile];

    if (a.noop && *a.noop) return;
    const int bad = load_offsets(a.m_splits, a.E, a.M, s_off);
    if (bad) {
        report_status(a.status, bad);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rg = warp >> 1, ch = warp & 1;
    const int64_t K = a.K;
    const int64_t tilesK = K / kTile;
    const int64_t tiles = (a.M / kTile) * tilesK;

    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t mt = t / tilesK, kt = t % tilesK;
        const int64_t row = mt * kTile + rg * 32 + lane;
        const int64_t col = kt * kTile + ch * 64;

        float v[64];
        uint32_t in_code[2] = {0, 0};
        if constexpr (!kReq) {
            const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.src) + row * K + col);
            uint4 w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = ldg_nc(p + i);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t ws[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    v[8 * i + 2 * j] = bf16lo(ws[j]);
                    v[8 * i + 2 * j + 1] = bf16hi(ws[j]);
                }
            }
        } else {
            const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.src) + row * K + col);
            uint4 w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) w[i] = ldg_nc(p + i);
            const uint16_t sc = *reinterpret_cast<const uint16_t*>(a.src_scale + row * (K / 32) + kt * 4 + ch * 2);
            in_code[0] = sc & 0xFF;
            in_code[1] = sc >> 8;
            const float s0 = scale_from_code(in_code[0]), s1 = scale_from_code(in_code[1]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t ws[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 lo = e4m3x2_to_f32((uint16_t)(ws[j] & 0xFFFF));
                    const float2 hi = e4m3x2_to_f32((uint16_t)(ws[j] >> 16));
                    const int c = 16 * i + 4 * j;
                    const float s = (c < 32) ? s0 : s1;
                    v[c] = lo.x * s;
                    v[c + 1] = lo.y * s;
                    v[c + 2] = hi.x * s;
                    v[c + 3] = hi.y * s;
                }
            }
        }

        // ---------------------------------------------------------- rowwise
        if constexpr (kRow && !kReq) {
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                uint32_t amax = 0;
#pragma unroll
                for (int i = 0; i < 32; ++i) amax = max(amax, __float_as_uint(v[32 * b + i]) & 0x7FFFFFFFu);
                const uint32_t code = scale_code_from_f32_absbits(amax);
                const float inv = inv_scale_from_code(code);
                uint32_t q[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t lo = cvt_e4m3x2(v[32 * b + 4 * i] * inv, v[32 * b + 4 * i + 1] * inv);
                    const uint32_t hi = cvt_e4m3x2(v[32 * b + 4 * i + 2] * inv, v[32 * b + 4 * i + 3] * inv);
                    q[i] = lo | (hi << 16);
                }
                uint4* dst = reinterpret_cast<uint4*>(a.row_q + row * K + col + 32 * b);
                dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
                dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
                if (a.swizzle) s_rs[lane * 16 + rg * 4 + ch * 2 + b] = (uint8_t)code;
                else a.row_s[row * (K / 32) + kt * 4 + ch * 2 + b] = (uint8_t)code;
            }
        }
        if constexpr (kRow && kReq) {
            // swizzled copy of the compact rowwise scales of the wire format
            *reinterpret_cast<uint16_t*>(&s_rs[lane * 16 + rg * 4 + ch * 2]) =
                (uint16_t)(in_code[0] | (in_code[1] << 8));
        }

        // ---------------------------------------------------------- colwise
        if constexpr (kCol) {
            uint32_t my_code[2] = {0, 0};
            uint32_t q[16];
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
                const uint32_t m0 = __reduce_max_sync(0xffffffffu, __float_as_uint(v[c]) & 0x7FFFFFFFu);
                const uint32_t m1 = __reduce_max_sync(0xffffffffu, __float_as_uint(v[c + 1]) & 0x7FFFFFFFu);
                const uint32_t c0 = scale_code_from_f32_absbits(m0);
                const uint32_t c1 = scale_code_from_f32_absbits(m1);
                if (lane == (c & 31)) my_code[c >> 5] = c0;
                if (lane == ((c + 1) & 31)) my_code[(c + 1) >> 5] = c1;
                const uint32_t pair = cvt_e4m3x2(v[c] * inv_scale_from_code(c0), v[c + 1] * inv_scale_from_code(c1));
                if ((c & 2) == 0) q[c >> 2] = pair;
                else q[c >> 2] |= pair << 16;
            }
            uint4* dst = reinterpret_cast<uint4*>(a.col_q + row * K + col);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(q[4 * i], q[4 * i + 1], q[4 * i + 2], q[4 * i + 3]);
            if (a.swizzle) {
                s_cs[lane * 16 + (ch * 2) * 4 + rg] = (uint8_t)my_code[0];
                s_cs[lane * 16 + (ch * 2 + 1) * 4 + rg] = (uint8_t)my_code[1];
            } else {
                uint8_t* cs = a.col_s + (mt * 4 + rg) * K + col;
                cs[lane] = (uint8_t)my_code[0];
                cs[32 + lane] = (uint8_t)my_code[1];
            }
        }

        // ------------------------------------------------- dequant output
        if constexpr (kDeq) {
            uint32_t h[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
                h[i] = *reinterpret_cast<uint32_t*>(&b2);
            }
            uint4* dst = reinterpret_cast<uint4*>(a.deq_out + row * K + col);
#pragma unroll
            for (int i = 0; i < 8; ++i) dst[i] = make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
        }

        // ------------------------------------------------- dbias partials
        if constexpr (kBias) {
            // butterfly over lanes: after step `o`, each lane keeps the half
            // of its columns selected by (lane & o); lane l ends with the
            // 32-row sums of columns 2l and 2l+1 of the warp's 64.
            float r[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) r[i] = v[i];
            int n = 64;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                const bool upper = (lane & o) != 0;
                n >>= 1;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    if (i < n) {
                        const float send = upper ? r[i] : r[n + i];
                        const float keep = upper ? r[n + i] : r[i];
                        r[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                    }
                }
            }
            s_red[rg][ch * 64 + 2 * lane] = r[0];
            s_red[rg][ch * 64 + 2 * lane + 1] = r[1];
        }

        if constexpr (kBias || kRow || kCol) __syncthreads();

        if constexpr (kBias) {
            if (threadIdx.x < kTile) {
                const int c = threadIdx.x;
                a.partials[mt * K + kt * kTile + c] = ((s_red[0][c] + s_red[1][c]) + s_red[2][c]) + s_red[3][c];
            }
        }
        if constexpr (kRow) {
            if (a.swizzle || kReq) {
                if (threadIdx.x < 32) {
                    uint4* dst = reinterpret_cast<uint4*>(a.row_s + (mt * tilesK + kt) * 512);
                    dst[threadIdx.x] = reinterpret_cast<const uint4*>(s_rs)[threadIdx.x];
                }
            }
        }
        if constexpr (kCol) {
            if (a.swizzle && threadIdx.x >= 32 && threadIdx.x < 64) {
                const int64_t r0 = mt * kTile;
                const int e = expert_of(s_off, a.E, r0);
                const int64_t off = s_off[e], me = s_off[e + 1] - off;
                const int64_t base = K * off / 32;
                const int64_t atom = kt * (me / kTile) + (r0 - off) / kTile;
                uint4* dst = reinterpret_cast<uint4*>(a.col_s + base + atom * 512);
                dst[threadIdx.x - 32] = reinterpret_cast<const uint4*>(s_cs)[threadIdx.x - 32];
            }
        }
        if constexpr (kBias || kRow || kCol) __syncthreads();
    }
}

// Second dbias stage: out[e, c] = sum over expert e's 128-row tiles of the
// tile partials, in tile order, accumulated in fp64.
__global__ void __launch_bounds__(256) dbias_finalize_kernel(const float* __restrict__ partials, int64_t M,
                                                             int64_t K, int E, const int64_t* m_splits,
                                                             float* __restrict__ out, const int32_t* noop) {
    __shared__ int64_t s_off[MXQ_MAX_EXPERTS + 1];
    if (noop && *noop) return;
    if (load_offsets(m_splits, E, M, s_off)) return;  // reported by the tile kernel
    const int e = blockIdx.y;
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= K) return;
    const int64_t t0 = s_off[e] / kTile, t1 = s_off[e + 1] / kTile;
    double acc = 0.0;
    for (int64_t t = t0; t < t1; ++t) acc += (double)partials[t * K + c];
    out[(int64_t)e * K + c] = (float)acc;
}

static int num_sms() {
    static int n[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && n[dev]) return n[dev];
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (dev < 64) n[dev] = v;
    return v;
}

template <bool kReq, bool kRow, bool kCol, bool kBias, bool kDeq>
static cudaError_t launch_tile(const TileArgs& a, cudaStream_t s) {
    const int64_t tiles = (a.M / kTile) * (a.K / kTile);
    if (tiles == 0) return cudaSuccess;
    const int64_t grid = std::min<int64_t>(tiles, (int64_t)num_sms() * 2);
    mx_tile_kernel<kReq, kRow, kCol, kBias, kDeq><<<(unsigned)grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

static cudaError_t launch_finalize(const float* partials, int64_t M, int64_t K, int E, const int64_t* m_splits,
                                   float* out, const int32_t* noop, cudaStream_t s) {
    dim3 grid((unsigned)((K + 255) / 256), (unsigned)E);
    dbias_finalize_kernel<<<grid, 256, 0, s>>>(partials, M, K, E, m_splits, out, noop);
    return cudaGetLastError();
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
