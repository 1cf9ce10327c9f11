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
// Design (HBM-bound): one CTA of 8 warps handles a 128x128 tile; lane l of
// warp w owns columns 64*(w%2) + 2l, +1 of rows 32*(w/2)..+31, so every
// warp-wide load and store is one contiguous stretch of a row. The colwise
// amax of a 32-row block and the dbias column sums are thread-local; the
// rowwise block spans a half-warp. The E8M0 code depends only on the largest exponent field of the
// block, so rowwise maxima are reduced as packed 8-bit exponents (4 rows per
// word, byte-wise max shuffles). A 128x128 tile produces exactly one
// 512-byte rowwise and one 512-byte colwise scale atom of the swizzled
// layout; both are assembled in shared memory and written with 16-byte
// stores. Because every expert's row count is a multiple of 128, a tile never
// straddles two experts. dbias sums each lane's 32 rows in order, then the
// four row groups in order (fp32 partial per 128-row tile, kept in the
// caller's workspace), then each expert's tiles in order in fp64 --
// deterministic run to run.
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

__device__ __forceinline__ uint2 ldg_nc_v2(const void* p) {
    uint2 r;
    asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}
__device__ __forceinline__ uint32_t ldg_nc_u32(const void* p) {
    uint32_t r;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

// Byte-wise max of 4 packed 8-bit exponents across the 16 lanes of a half-warp.
__device__ __forceinline__ uint32_t group16_max_u8x4(uint32_t v) {
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) v = __vmaxu4(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// One CTA (8 warps) handles a 128x128 tile. Warp w owns rows 32*(w/2)..+31
// and the 64 columns 64*(w%2)..+63; lane l owns columns 2l, 2l+1 of that
// strip in every one of its 32 rows, so each warp-wide load or store is one
// contiguous stretch of a row. The colwise amax of a 32-row block and the
// dbias column sums are thread-local (over the lane's 32 rows); a rowwise
// block of 32 columns spans one half-warp, whose exponents are reduced four
// rows at a time with byte-wise max shuffles (the scale depends only on the
// block's largest exponent field).
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
    const int blk = ch * 2 + (lane >> 4);  // 32-column block of the tile holding this lane's columns
    const int64_t K = a.K;
    const int64_t tilesK = K / kTile;
    const int64_t tiles = (a.M / kTile) * tilesK;

    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t mt = t / tilesK, kt = t % tilesK;
        const int64_t r0 = mt * kTile + rg * 32;             // this warp's first row
        const int64_t col = kt * kTile + ch * 64 + lane * 2;  // this lane's first column

        // ------------------------------------------------------------ load
        uint32_t raw[32];   // bf16x2, or two E4M3 bytes in the low half
        float rsc[kReq ? 32 : 1];
        (void)rsc;
        if constexpr (!kReq) {
            const uint16_t* p = static_cast<const uint16_t*>(a.src) + r0 * K + col;
#pragma unroll
            for (int r = 0; r < 32; ++r) raw[r] = ldg_nc_u32(p + r * K);
        } else {
            const uint8_t* p = static_cast<const uint8_t*>(a.src) + r0 * K + col;
#pragma unroll
            for (int r = 0; r < 32; ++r) raw[r] = __ldg(reinterpret_cast<const unsigned short*>(p + r * K));
            // lane l reads the 4 compact rowwise scale codes of row r0 + l
            const uint32_t sw = ldg_nc_u32(a.src_scale + (r0 + lane) * (K / 32) + kt * 4);
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                const uint32_t word = __shfl_sync(0xffffffffu, sw, r);
                rsc[r] = scale_from_code((word >> (8 * blk)) & 0xFFu);
            }
            if constexpr (kRow) {
                if (ch == 0) *reinterpret_cast<uint32_t*>(&s_rs[lane * 16 + rg * 4]) = sw;
            }
        }
        // values of row r, exact fp32
        auto val2 = [&](int r) -> float2 {
            if constexpr (!kReq) {
                return make_float2(bf16lo(raw[r]), bf16hi(raw[r]));
            } else {
                const float2 f = e4m3x2_to_f32((uint16_t)raw[r]);
                return make_float2(f.x * rsc[r], f.y * rsc[r]);
            }
        };

        // ---------------------------------------------------------- rowwise
        if constexpr (kRow && !kReq) {
#pragma unroll
            for (int r4 = 0; r4 < 32; r4 += 4) {
                uint32_t packed = 0;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t w = raw[r4 + k] & 0x7FFF7FFFu;
                    packed |= (max(w & 0xFFFFu, w >> 16) >> 7) << (8 * k);  // bf16 exponent field
                }
                packed = group16_max_u8x4(packed);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t code = (uint32_t)max((int)((packed >> (8 * k)) & 0xFFu) - 8, 0);
                    const float inv = inv_scale_from_code(code);
                    const float2 v = val2(r4 + k);
                    *reinterpret_cast<uint16_t*>(a.row_q + (r0 + r4 + k) * K + col) =
                        (uint16_t)cvt_e4m3x2(v.x * inv, v.y * inv);
                    if ((lane & 15) == 0) {
                        if (a.swizzle) s_rs[(r4 + k) * 16 + rg * 4 + blk] = (uint8_t)code;
                        else a.row_s[(r0 + r4 + k) * (K / 32) + kt * 4 + blk] = (uint8_t)code;
                    }
                }
            }
        }

        // ---------------------------------------------------------- colwise
        if constexpr (kCol) {
            uint32_t e0, e1;  // largest exponent field of each of the 2 columns
            if constexpr (!kReq) {
                uint32_t m = 0;
#pragma unroll
                for (int r = 0; r < 32; ++r) m = __vmaxu2(m, raw[r] & 0x7FFF7FFFu);
                e0 = (m >> 7) & 0xFFu;
                e1 = (m >> 23) & 0xFFu;
            } else {
                uint32_t m0 = 0, m1 = 0;
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    const float2 v = val2(r);
                    m0 = max(m0, __float_as_uint(v.x) & 0x7FFFFFFFu);
                    m1 = max(m1, __float_as_uint(v.y) & 0x7FFFFFFFu);
                }
                e0 = m0 >> 23;
                e1 = m1 >> 23;
            }
            const uint32_t c0 = (uint32_t)max((int)e0 - 8, 0), c1 = (uint32_t)max((int)e1 - 8, 0);
            const float i0 = inv_scale_from_code(c0), i1 = inv_scale_from_code(c1);
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                const float2 v = val2(r);
                *reinterpret_cast<uint16_t*>(a.col_q + (r0 + r) * K + col) = (uint16_t)cvt_e4m3x2(v.x * i0, v.y * i1);
            }
            if (a.swizzle) {
                const int cc = (2 * lane) & 31, cb = blk;  // both columns share the 32-column block
                s_cs[cc * 16 + cb * 4 + rg] = (uint8_t)c0;
                s_cs[(cc + 1) * 16 + cb * 4 + rg] = (uint8_t)c1;
            } else {
                *reinterpret_cast<uint16_t*>(a.col_s + (mt * 4 + rg) * K + col) = (uint16_t)(c0 | (c1 << 8));
            }
        }

        // ------------------------------------------------- dequant output
        if constexpr (kDeq) {
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                const float2 v = val2(r);
                __nv_bfloat162 b = __floats2bfloat162_rn(v.x, v.y);
                *reinterpret_cast<__nv_bfloat162*>(a.deq_out + (r0 + r) * K + col) = b;
            }
        }

        // ------------------------------------------------- dbias partials
        if constexpr (kBias) {
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                const float2 v = val2(r);
                s0 += v.x;
                s1 += v.y;
            }
            *reinterpret_cast<float2*>(&s_red[rg][ch * 64 + lane * 2]) = make_float2(s0, s1);
        }

        __syncthreads();
        if constexpr (kBias) {
            if (threadIdx.x < kTile) {
                const int c = threadIdx.x;
                a.partials[mt * K + kt * kTile + c] = ((s_red[0][c] + s_red[1][c]) + s_red[2][c]) + s_red[3][c];
            }
        }
        if constexpr (kRow) {
            if ((a.swizzle || kReq) && threadIdx.x < 32) {
                uint4* dst = reinterpret_cast<uint4*>(a.row_s + (mt * tilesK + kt) * 512);
                dst[threadIdx.x] = reinterpret_cast<const uint4*>(s_rs)[threadIdx.x];
            }
        }
        if constexpr (kCol) {
            if (a.swizzle && threadIdx.x >= 32 && threadIdx.x < 64) {
                const int64_t rt0 = mt * kTile;
                const int e = expert_of(s_off, a.E, rt0);
                const int64_t off = s_off[e], me = s_off[e + 1] - off;
                const int64_t base = K * off / 32;
                const int64_t atom = kt * (me / kTile) + (rt0 - off) / kTile;
                uint4* dst = reinterpret_cast<uint4*>(a.col_s + base + atom * 512);
                dst[threadIdx.x - 32] = reinterpret_cast<const uint4*>(s_cs)[threadIdx.x - 32];
            }
        }
        __syncthreads();
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
    const int64_t grid = std::min<int64_t>(tiles, (int64_t)num_sms() * 4);
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
