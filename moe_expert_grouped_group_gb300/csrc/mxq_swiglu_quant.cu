// mxq_swiglu_quant.cu -- SwiGLU fused with MXFP8 group quantization, for the
// grouped MoE MLP FC1 -> SwiGLU -> FC2 (TransformerEngine PR #3545, "Fix
// distributed BF16 weights and trim NVFP4 saved state in the fused grouped
// MLP"; quantization as in PR #3244 / PR #3224, see mxq_quant.cu).
//
//   forward : y = FC1 output (M, 2F) bf16 = [gate | up] -> h = silu(g) * u,
//             rounded to bf16, quantized rowwise (FC2 fprop) and colwise
//             (FC2 wgrad). h itself is written only if asked for.
//   backward: dh (M, F), y (M, 2F) -> dY1 = [dg | du] (M, 2F), rounded to
//             bf16, quantized rowwise (FC1 dgrad) and colwise (FC1 wgrad),
//             with the per-expert FC1 dbias reduced from the same bf16 values.
//
// Persistent CTAs of 8 compute warps + 1 TMA producer warp, 128x128 output
// tiles. A stage holds the 128x128 input tiles a tile needs (g and u; plus
// dh backward). Warp w turns rows 16w..16w+15 into bf16 h (or dg and du),
// written back in place -- the fp32 steps of mxq_common.cuh, two values per
// packed instruction (bit-identical), one bf16 rounding
// -- gathering each column's exponent maximum (and dbias sum) in registers
// on the way. After one exchange of those 16-row statistics through shared
// memory (a 32-row colwise block is two warps), every warp encodes its own
// rows rowwise and colwise (the backward's dg and du rows side by side, two
// independent chains per step): the same codes as "SwiGLU, then
// group_quantize" bit for bit, while h (or dY1) never makes a round trip
// through HBM.
#include <cuda_bf16.h>

#include <algorithm>

#include "mxq_common.cuh"
#include "mxq_internal.h"

namespace mxq {
namespace swq {

constexpr int kWarps = 8;                       // compute warps
constexpr int kThreads = (kWarps + 1) * 32;     // + 1 TMA producer warp
constexpr int kTileBytes = kTile * kTile * 2;   // one 128x128 bf16 tile
constexpr int kPreRows = kTile / kWarps;        // rows per warp
constexpr int kComputeThreads = kWarps * 32;

struct Args {
    int64_t M, F, E;
    const int64_t* m_splits;
    uint8_t *row_q, *row_s, *col_q, *col_s;  // quantized output (M, Kout)
    float* partials;                          // dbias partials (M/128, Kout)
    __nv_bfloat16* bf16_out;                  // optional h / dY1 (M, Kout)
    int swizzle;
    const int32_t* noop;
    int32_t* status;
};

// Per output tile: its two 512-byte scale atoms, each warp's colwise
// exponent maxima over its 16 rows (four bytes per lane) and its 16-row
// dbias sums.
struct Scratch {
    uint8_t rs[512];
    uint8_t cs[512];
    uint32_t xexp[kWarps][32];
    float red[kWarps][kTile];
};

__device__ __forceinline__ void bar_compute() {
    asm volatile("bar.sync 2, %0;" ::"n"(kComputeThreads) : "memory");
}
__device__ __forceinline__ bool bar_compute_any(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 2, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "n"(kComputeThreads)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Colwise exponent statistics of one output tile over a warp's 16 rows,
// gathered as the bf16 results are produced: per column the largest |bits|
// (two columns per word).
struct ColStats {
    uint32_t m[2] = {0u, 0u};
    __device__ __forceinline__ void add(uint2 w) {
        m[0] = __vmaxu2(m[0], w.x & 0x7FFF7FFFu);
        m[1] = __vmaxu2(m[1], w.y & 0x7FFF7FFFu);
    }
    // the four biased exponents, one byte per column
    __device__ __forceinline__ uint32_t exps() const {
        return ((m[0] >> 7) & 0xFFu) | (((m[0] >> 23) & 0xFFu) << 8) | (((m[1] >> 7) & 0xFFu) << 16) |
               (((m[1] >> 23) & 0xFFu) << 24);
    }
};

// Encode the 16 rows of the kN output tiles that warp w produced (h, or dg and du; bf16 in shared
// memory, tile q at rows + q*kTileBytes, row r at + r*256, lane l reading columns 4l..4l+3) into output
// column tiles kt0 + q*kt_step of an (M, Kout) tensor. Each step encodes four rows of every tile, and with
// one tile four rows of each half of the warp's rows, so that the step holds two independent chains for
// the warp's instructions to overlap. The colwise scale of each 32-row block comes from the exponent maxima
// of warps w and w^1 (the two halves of the block); the rowwise scale of each row from the 8 lanes of its
// 32-column block. Swizzled scale bytes are staged in sc[q] for flush_scratch; with kBias the lane's four
// column sums over the 16 rows (fp32, in row order) go to sc[q].red[w].
template <int kN, bool kRow, bool kCol, bool kDeq, bool kBias>
__device__ __forceinline__ void encode_rows(const uint8_t* rows, const Args& a, int64_t mt, int64_t kt0,
                                            int64_t kt_step, int64_t Kout, Scratch* sc, int w, int lane) {
    // chains per step: tile q = c / kG, rows from g * (kPreRows / kG) on, g = c % kG
    constexpr int kG = kN == 1 && !kBias ? 2 : 1;  // the column sums keep row order: one chain per tile
    constexpr int kC = kN * kG, kSpan = kPreRows / kG;
    auto o = [&](int q, int r) { return *reinterpret_cast<const uint2*>(rows + q * kTileBytes + r * (kTile * 2)); };
    const int blk = lane >> 3;
    const int rg = w >> 1;                          // 32-row block of the tile
    const int64_t r0 = mt * kTile + w * kPreRows;   // first row of this warp
    const uint32_t Ku = (uint32_t)Kout;

    uint64_t cinv01[kN], cinv23[kN], bsum01[kN], bsum23[kN];
    uint8_t *rq[kN], *cq[kN];
    __nv_bfloat16* dq[kN];
#pragma unroll
    for (int q = 0; q < kN; ++q) {
        const int64_t kt = kt0 + q * kt_step;
        const int64_t col = kt * kTile + lane * 4;
        uint32_t ccode[4] = {0, 0, 0, 0};
        float cinv[4] = {1.f, 1.f, 1.f, 1.f};
        if constexpr (kCol) {
            const uint32_t e = __vmaxu4(sc[q].xexp[w][lane], sc[q].xexp[w ^ 1][lane]);
            uint32_t packed = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                ccode[j] = (uint32_t)max((int)((e >> (8 * j)) & 0xFFu) - 8, 0);
                cinv[j] = inv_scale_from_code(ccode[j]);
                packed |= ccode[j] << (8 * j);
            }
            if ((w & 1) == 0) {
                if (a.swizzle) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        sc[q].cs[(4 * (lane & 7) + j) * 16 + blk * 4 + rg] = (uint8_t)ccode[j];
                } else {
                    *reinterpret_cast<uint32_t*>(a.col_s + (mt * 4 + rg) * Kout + col) = packed;
                }
            }
        }
        rq[q] = kRow ? a.row_q + r0 * Kout + col : nullptr;
        cq[q] = kCol ? a.col_q + r0 * Kout + col : nullptr;
        dq[q] = kDeq ? a.bf16_out + r0 * Kout + col : nullptr;
        cinv01[q] = f2pack(cinv[0], cinv[1]);
        cinv23[q] = f2pack(cinv[2], cinv[3]);
        bsum01[q] = bsum23[q] = f2splat(0.f);  // column sums, two columns per packed add
    }
#pragma unroll 2
    for (int r4 = 0; r4 < kSpan; r4 += 4) {
        uint2 ow[kC][4];
        uint32_t packed[kC];  // rowwise codes of the chain's four rows, one byte each
#pragma unroll
        for (int c = 0; c < kC; ++c) {
            const int q = c / kG, rb = (c % kG) * kSpan + r4;
#pragma unroll
            for (int k = 0; k < 4; ++k) ow[c][k] = o(q, rb + k);
            packed[c] = 0;
            if constexpr (kRow) {
                uint32_t m[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    m[k] = __vmaxu2(ow[c][k].x & 0x7FFF7FFFu, ow[c][k].y & 0x7FFF7FFFu);
                // |bits| maxima of rows (0, 1) and (2, 3) as 16-bit halves, then their exponent bytes
                const uint32_t v01 = __vmaxu2(__byte_perm(m[0], m[1], 0x5410), __byte_perm(m[0], m[1], 0x7632));
                const uint32_t v23 = __vmaxu2(__byte_perm(m[2], m[3], 0x5410), __byte_perm(m[2], m[3], 0x7632));
                packed[c] = __byte_perm((v01 >> 7) & 0x00FF00FFu, (v23 >> 7) & 0x00FF00FFu, 0x6420);
            }
        }
        if constexpr (kRow) {
#pragma unroll
            for (int s = 4; s >= 1; s >>= 1)
#pragma unroll
                for (int c = 0; c < kC; ++c)
                    packed[c] = __vmaxu4(packed[c], __shfl_xor_sync(0xffffffffu, packed[c], s));
#pragma unroll
            for (int c = 0; c < kC; ++c) packed[c] = __vsubus4(packed[c], 0x08080808u);  // max(exponent - 8, 0)
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
#pragma unroll
            for (int c = 0; c < kC; ++c) {
                const int q = c / kG, r = (c % kG) * kSpan + r4 + k;
                const uint2 u = ow[c][k];
                const uint64_t v01 = f2pack(bf16lo(u.x), bf16hi(u.x)), v23 = f2pack(bf16lo(u.y), bf16hi(u.y));
                if constexpr (kBias) {
                    bsum01[q] = f2add(bsum01[q], v01);
                    bsum23[q] = f2add(bsum23[q], v23);
                }
                if constexpr (kRow) {
                    const uint32_t code = (packed[c] >> (8 * k)) & 0xFFu;
                    const uint64_t inv = f2splat(inv_scale_from_code(code));
                    const float2 s01 = f2unpack(f2mul(v01, inv)), s23 = f2unpack(f2mul(v23, inv));
                    *reinterpret_cast<uint32_t*>(rq[q] + r * Ku) =
                        cvt_e4m3x2(s01.x, s01.y) | (cvt_e4m3x2(s23.x, s23.y) << 16);
                    if ((lane & 7) == 0) {
                        if (a.swizzle) sc[q].rs[((w & 1) * kPreRows + r) * 16 + rg * 4 + blk] = (uint8_t)code;
                        else a.row_s[(r0 + r) * (Kout / 32) + (kt0 + q * kt_step) * 4 + blk] = (uint8_t)code;
                    }
                }
                if constexpr (kCol) {
                    const float2 s01 = f2unpack(f2mul(v01, cinv01[q])), s23 = f2unpack(f2mul(v23, cinv23[q]));
                    *reinterpret_cast<uint32_t*>(cq[q] + r * Ku) =
                        cvt_e4m3x2(s01.x, s01.y) | (cvt_e4m3x2(s23.x, s23.y) << 16);
                }
                if constexpr (kDeq) *reinterpret_cast<uint2*>(dq[q] + (size_t)r * Ku) = u;
            }
        }
    }
    if constexpr (kBias) {
#pragma unroll
        for (int q = 0; q < kN; ++q) {
            const float2 s01 = f2unpack(bsum01[q]), s23 = f2unpack(bsum23[q]);
            *reinterpret_cast<float4*>(&sc[q].red[w][lane * 4]) = make_float4(s01.x, s01.y, s23.x, s23.y);
        }
    }
}

// Write out one tile's scratch: the dbias partial of each of its 128 columns
// (the eight 16-row sums added in warp order) and, for swizzled scales, its
// rowwise atom and its colwise atom (the latter at the expert's base).
// `t` is this thread's index among the 128 threads that flush the tile.
template <bool kRow, bool kCol, bool kBias>
__device__ __forceinline__ void flush_scratch(const Scratch& sc, const Args& a, int64_t mt, int64_t kt, int64_t Kout,
                                              const int64_t* s_off, int t) {
    if constexpr (kBias) {
        float acc = sc.red[0][t];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) acc += sc.red[w][t];
        a.partials[mt * Kout + kt * kTile + t] = acc;
    }
    if constexpr (kRow) {
        if (a.swizzle && t < 32) {
            uint4* dst = reinterpret_cast<uint4*>(a.row_s + (mt * (Kout / kTile) + kt) * 512);
            dst[t] = reinterpret_cast<const uint4*>(sc.rs)[t];
        }
    }
    if constexpr (kCol) {
        if (a.swizzle && t >= 32 && t < 64) {
            const int64_t rt0 = mt * kTile;
            const int e = expert_of(s_off, (int)a.E, rt0);
            const int64_t off = s_off[e], me = s_off[e + 1] - off;
            const int64_t atom = kt * (me / kTile) + (rt0 - off) / kTile;
            uint4* dst = reinterpret_cast<uint4*>(a.col_s + Kout * off / 32 + atom * 512);
            dst[t - 32] = reinterpret_cast<const uint4*>(sc.cs)[t - 32];
        }
    }
}

// Forward: 3 CTAs per SM (64 KB stage); backward: 2 (96 KB stage).
template <bool kBwd, bool kRow, bool kCol, bool kBias, bool kDeq>
__global__ void __launch_bounds__(kThreads, kBwd ? 2 : 3)
    swiglu_quant_kernel(const __grid_constant__ CUtensorMap tm_y, const __grid_constant__ CUtensorMap tm_dh, Args a) {
    constexpr int kIn = kBwd ? 3 : 2;   // stage: [g][u] or [g][u][dh]
    constexpr int kOut = kBwd ? 2 : 1;  // output tiles per stage: h, or dg and du
    constexpr uint32_t kStageTx = kIn * kTileBytes;
    extern __shared__ uint8_t sq_raw[];
    __shared__ __align__(16) Scratch s_sc[kOut];
    __shared__ int s_abort;

    uint8_t* stage = smem_align<128>(sq_raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(stage + kIn * kTileBytes);
    int64_t* s_off = reinterpret_cast<int64_t*>(bars + 2);

    if (a.noop && *a.noop) return;
    const int bad = load_offsets(a.m_splits, (int)a.E, a.M, s_off);
    if (bad) {
        report_status(a.status, bad);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tilesF = a.F / kTile;
    const int64_t tiles = (a.M / kTile) * tilesF;
    const uint32_t full = smem_u32(bars), empty = smem_u32(bars + 1);
    volatile int* abort_flag = &s_abort;
    if (threadIdx.x == 0) {
        s_abort = 0;
        mbar_init(full, 1);
        mbar_init(empty, kWarps);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == kWarps) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0) {
            uint32_t phase = 0;
            for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
                if (!mbar_wait(empty, phase ^ 1, abort_flag)) break;
                const int x = (int)((t % tilesF) * kTile), y = (int)((t / tilesF) * kTile);
                mbar_expect_tx(full, kStageTx);
                tma_load_2d(smem_u32(stage), &tm_y, full, x, y);                              // gate
                tma_load_2d(smem_u32(stage + kTileBytes), &tm_y, full, x + (int)a.F, y);    // up
                if constexpr (kBwd) tma_load_2d(smem_u32(stage + 2 * kTileBytes), &tm_dh, full, x, y);
                phase ^= 1;
            }
        }
        return;
    }

    // Warp w owns rows 16w..16w+15 of every output tile, lane l columns
    // 4l..4l+3. Backward: the first 128 compute threads flush dg's scratch,
    // the other 128 du's; forward: the first 128 flush h's.
    const int fgrp = threadIdx.x >> 7;
    const int ft_tid = threadIdx.x & 127;
    uint32_t phase = 0;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t mt = t / tilesF, ft = t % tilesF;
        const bool ok = mbar_wait(full, phase, abort_flag);
        if (bar_compute_any(!ok)) break;
        phase ^= 1;

        // SwiGLU of this warp's 16 rows, rounded to bf16 and written back in
        // place (h or dg over the gate tile, du over the up tile), with the
        // colwise statistics of each output tile
        ColStats cs[kOut];
        uint8_t* g_row = stage + (warp * kPreRows) * (kTile * 2) + lane * 8;
        uint8_t* u_row = g_row + kTileBytes;
#pragma unroll 8
        for (int r = 0; r < kPreRows; ++r) {
            uint2* gp = reinterpret_cast<uint2*>(g_row + r * (kTile * 2));
            uint2* up = reinterpret_cast<uint2*>(u_row + r * (kTile * 2));
            const uint2 gw = *gp, uw = *up;
            const float g[4] = {bf16lo(gw.x), bf16hi(gw.x), bf16lo(gw.y), bf16hi(gw.y)};
            const float u[4] = {bf16lo(uw.x), bf16hi(uw.x), bf16lo(uw.y), bf16hi(uw.y)};
            if constexpr (!kBwd) {
                float h[4];
#pragma unroll
                for (int j = 0; j < 4; j += 2) {
                    const float2 h2 = swiglu_h_x2(make_float2(g[j], g[j + 1]), make_float2(u[j], u[j + 1]));
                    h[j] = h2.x;
                    h[j + 1] = h2.y;
                }
                const uint2 hw = make_uint2(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]));
                *gp = hw;
                if (kCol) cs[0].add(hw);
            } else {
                const uint2 dw = *reinterpret_cast<const uint2*>(g_row + 2 * kTileBytes + r * (kTile * 2));
                const float d[4] = {bf16lo(dw.x), bf16hi(dw.x), bf16lo(dw.y), bf16hi(dw.y)};
                float dg[4], du[4];
#pragma unroll
                for (int j = 0; j < 4; j += 2) {
                    float2 dg2, du2;
                    swiglu_grads_x2(make_float2(d[j], d[j + 1]), make_float2(g[j], g[j + 1]),
                                    make_float2(u[j], u[j + 1]), dg2, du2);
                    dg[j] = dg2.x;
                    dg[j + 1] = dg2.y;
                    du[j] = du2.x;
                    du[j + 1] = du2.y;
                }
                const uint2 gw2 = make_uint2(pack_bf16x2(dg[0], dg[1]), pack_bf16x2(dg[2], dg[3]));
                const uint2 uw2 = make_uint2(pack_bf16x2(du[0], du[1]), pack_bf16x2(du[2], du[3]));
                *gp = gw2;
                *up = uw2;
                if (kCol) {
                    cs[0].add(gw2);
                    cs[kOut - 1].add(uw2);
                }
            }
        }
#pragma unroll
        for (int q = 0; q < kOut; ++q)
            if constexpr (kCol) s_sc[q].xexp[warp][lane] = cs[q].exps();
        bar_compute();  // every warp's colwise statistics are in

        const int64_t Kout = kBwd ? 2 * a.F : a.F;
        encode_rows<kOut, kRow, kCol, kDeq, kBias>(g_row, a, mt, ft, tilesF, Kout, s_sc, warp, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty);  // this warp is done with the stage
        bar_compute();                      // scratch complete
        if (fgrp < kOut)
            flush_scratch<kRow, kCol, kBias>(s_sc[fgrp], a, mt, fgrp ? tilesF + ft : ft, Kout, s_off, ft_tid);
        // the next tile's first barrier orders these reads before any new
        // write to the scratch
    }
    if (threadIdx.x == 0 && s_abort && a.status) atomicOr(a.status, MXQ_STATUS_WAIT_TIMEOUT);
}

static int num_sms() {
    int dev = 0, v = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    return v;
}

template <bool kBwd, bool kRow, bool kCol, bool kBias, bool kDeq>
static cudaError_t launch(const Args& a, const void* y, const void* dh, cudaStream_t s) {
    const int64_t tiles = (a.M / kTile) * (a.F / kTile);
    if (tiles == 0) return cudaSuccess;
    constexpr int kIn = kBwd ? 3 : 2;
    const int smem = 128 + kIn * kTileBytes + 16 + (int)(a.E + 1) * 8;
    auto kern = swiglu_quant_kernel<kBwd, kRow, kCol, kBias, kDeq>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    CUtensorMap ty, td;
    if (!encode_tmap_2d(&ty, y, a.M, 2 * a.F, 2, kTile, kTile, 0)) return cudaErrorInvalidValue;
    if (kBwd) {
        if (!encode_tmap_2d(&td, dh, a.M, a.F, 2, kTile, kTile, 0)) return cudaErrorInvalidValue;
    } else {
        td = ty;  // unused
    }
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    const int64_t grid = std::min<int64_t>(tiles, (int64_t)num_sms() * std::max(per_sm, 1));
    kern<<<(unsigned)grid, kThreads, smem, s>>>(ty, td, a);
    return cudaGetLastError();
}

template <bool kBwd>
static cudaError_t dispatch(const Args& a, bool row, bool col, bool bias, bool deq, const void* y, const void* dh,
                            cudaStream_t s) {
#define MXQ_SWQ(R, C, B, D) \
    if (row == R && col == C && bias == B && deq == D) return launch<kBwd, R, C, B, D>(a, y, dh, s);
    MXQ_SWQ(true, true, false, false)
    MXQ_SWQ(true, true, true, false)
    MXQ_SWQ(true, true, false, true)
    MXQ_SWQ(true, true, true, true)
    MXQ_SWQ(true, false, false, false)
    MXQ_SWQ(true, false, true, false)
    MXQ_SWQ(true, false, false, true)
    MXQ_SWQ(true, false, true, true)
    MXQ_SWQ(false, true, false, false)
    MXQ_SWQ(false, true, true, false)
    MXQ_SWQ(false, true, false, true)
    MXQ_SWQ(false, true, true, true)
    MXQ_SWQ(false, false, true, false)
    MXQ_SWQ(false, false, false, true)
    MXQ_SWQ(false, false, true, true)
#undef MXQ_SWQ
    return cudaSuccess;  // nothing requested
}

}  // namespace swq

cudaError_t run_swiglu_quantize(const SwigluQuantCall& c, cudaStream_t s) {
    swq::Args a{};
    a.M = c.M;
    a.F = c.F;
    a.E = c.E;
    a.m_splits = c.m_splits;
    a.row_q = (uint8_t*)c.row_q;
    a.row_s = (uint8_t*)c.row_s;
    a.col_q = (uint8_t*)c.col_q;
    a.col_s = (uint8_t*)c.col_s;
    a.partials = c.partials;
    a.bf16_out = (__nv_bfloat16*)c.bf16_out;
    a.swizzle = c.swizzle;
    a.noop = c.noop;
    a.status = c.status;
    const bool row = c.row_q != nullptr, col = c.col_q != nullptr, bias = c.partials != nullptr,
               deq = c.bf16_out != nullptr;
    cudaError_t e = c.backward ? swq::dispatch<true>(a, row, col, bias, deq, c.y, c.dh, s)
                               : swq::dispatch<false>(a, row, col, bias, deq, c.y, nullptr, s);
    if (e != cudaSuccess || !bias) return e;
    return run_dbias_finalize(c.partials, c.M, c.backward ? 2 * c.F : c.F, c.E, c.m_splits, c.dbias, c.noop, s);
}

}  // namespace mxq
