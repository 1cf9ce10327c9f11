// mxq_tile.cuh -- the persistent 128x128-tile MXFP8 quantization kernel
// shared by mxq_quant.cu (expert counts that are multiples of 128) and
// mxq_quant_pad.cu (any expert counts, per-expert padded scale layouts).
// See mxq_quant.cu for the operations and their sources.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <type_traits>

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
    const float* probs;        // scaled bias: routing scale s_m per row (M)
    const __nv_bfloat16* bias; // scaled bias: b_e (E, K)
    float* dp_partials;        // scaled bias: (M, K/128) fp32 per-tile sums of dY[m,:] . b_e
    int swizzle;
    const int32_t* noop;
    int32_t* status;
};

// Packed half-precision steps of the requant fast path (each f16 lane rounds
// to nearest even, subnormals kept).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v16) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)v16));
    return h;
}
__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t f16x2_max(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
// Two f16 (low, high lane) -> two E4M3 bytes (low, high), RNE, saturating finite.
__device__ __forceinline__ uint32_t f16x2_to_e4m3x2(uint32_t h) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h));
    return (uint32_t)r;
}

// Byte-wise max of 4 packed 8-bit exponents across the 8 lanes of a group.
__device__ __forceinline__ uint32_t group8_max_u8x4(uint32_t v) {
#pragma unroll
    for (int o = 4; o >= 1; o >>= 1) v = __vmaxu4(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Persistent CTAs, several per SM: warp 4 is a TMA producer that keeps the
// next 128x128 input tiles in flight in a small shared-memory ring; warps 0..3
// compute. Warp w owns rows 32w..32w+31 of a tile and lane l owns its columns
// 4l..4l+3, so shared-memory reads are conflict-free and every global store
// of a warp is one contiguous stretch of a row. The tile is read from shared
// memory twice: pass 1 takes the colwise amax (thread-local over the lane's
// 32 rows) and the dbias column sums, pass 2 encodes. A rowwise block of 32
// columns spans 8 lanes, whose exponents are reduced four rows at a time as
// packed bytes (the E8M0 code depends only on the block's largest exponent).
// Ring depth per CTA. The kernel is bound by issue and latency of its compute
// warps, so more resident CTAs (shallower rings) beat deeper prefetch: on the
// 16k-token workload quantize ran 51 us with 1 stage, 64 us with 2, 79 us
// with 3; requant (E4M3 in) 27.8 / 29.8 / 31.7 us with 1 / 2 / 3 stages.
#ifndef MXQ_QUANT_STAGES_BF16
#define MXQ_QUANT_STAGES_BF16 1  // 32 KB bf16 tile in flight per CTA
#endif
#ifndef MXQ_QUANT_STAGES_E4M3
#define MXQ_QUANT_STAGES_E4M3 1  // 16 KB E4M3 tile in flight per CTA
#endif

template <bool kReq>
struct TileShape {
    static constexpr int kInBytes = kReq ? 1 : 2;          // input element size
    static constexpr int kRowBytes = kTile * kInBytes;     // one tile row in shared memory
    static constexpr int kStageBytes = kTile * kRowBytes;  // 16 KB (E4M3) or 32 KB (bf16)
    static constexpr int kStages = kReq ? MXQ_QUANT_STAGES_E4M3 : MXQ_QUANT_STAGES_BF16;
    static constexpr int kSmem = kStages * kStageBytes + 2 * kStages * 8 + 128;
};
constexpr int kComputeWarps = 4;
constexpr int kTileThreads = (kComputeWarps + 1) * 32;

__device__ __forceinline__ void compute_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(kComputeWarps * 32) : "memory");
}
// Barrier over the compute warps that also ORs a predicate across them, so
// that they all take the same exit decision.
__device__ __forceinline__ bool compute_bar_any(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "n"(kComputeWarps * 32)
        : "memory");
    return r != 0;
}

// Sum of v[r] over the 32 lanes for every r, by five exchange-and-add rounds
// that halve the rows each lane keeps: afterwards lane l holds row l's total
// in v[0]. Fixed order, so the result is the same run to run.
__device__ __forceinline__ float transpose_reduce32(float (&v)[32], int lane) {
#pragma unroll
    for (int off = 16, n = 32; off >= 1; off >>= 1, n >>= 1) {
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float keep = up ? v[i + n / 2] : v[i];
            const float send = up ? v[i] : v[i + n / 2];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    return v[0];
}

// Where tile t of the schedule lies. Aligned grouping: tile row 128*mt of the
// dense matrix. Padded grouping (kPad, expert counts that need not be
// multiples of 128): the 128-row slices of each expert in turn (slice j of
// expert e starts at token row off_e + 128 j and at scale-space row
// poff_e + 128 j); the last slice of an expert may hold fewer than 128 of its
// rows, the rest belong to the next expert or lie beyond M and are masked.
struct TileGeom {
    int64_t row0;   // first token row of the tile
    int64_t prow0;  // first row of the tile in the scale row space
    int64_t off_p;  // kPad: first scale-space row of the tile's expert
    int64_t me_p;   // kPad: scale-space rows of the tile's expert (a multiple of 128)
    int vr;         // rows of the tile that belong to its expert
    int e;          // kPad: the tile's expert
};
template <bool kPad>
__device__ __forceinline__ TileGeom tile_geom(int64_t mt, const int64_t* s_off, const int64_t* s_poff, int E) {
    TileGeom g;
    if constexpr (!kPad) {
        g.row0 = g.prow0 = mt * kTile;
        g.off_p = g.me_p = 0;
        g.vr = kTile;
        g.e = -1;
    } else {
        const int e = expert_of(s_poff, E, mt * kTile);
        const int64_t j = mt - s_poff[e] / kTile;
        g.e = e;
        g.off_p = s_poff[e];
        g.me_p = s_poff[e + 1] - s_poff[e];
        g.row0 = s_off[e] + j * kTile;
        g.prow0 = s_poff[e] + j * kTile;
        const int64_t left = (s_off[e + 1] - s_off[e]) - j * kTile;
        g.vr = (int)(left < kTile ? left : kTile);
    }
    return g;
}

// kScaled (scaled bias, with kBias): the column sums weight row m by its
// routing scale s_m, and each row's dot product with its expert's bias is
// reduced per tile into dp_partials. kPad: padded grouping (TileGeom).
template <bool kReq, bool kRow, bool kCol, bool kBias, bool kDeq, bool kScaled = false, bool kPad = false>
__global__ void __launch_bounds__(kTileThreads)
    mx_tile_kernel(const __grid_constant__ CUtensorMap tm_in, TileArgs a) {
    static_assert(!kScaled || kBias, "the scaled-bias reductions ride on the dbias pass");
    using Sh = TileShape<kReq>;
    extern __shared__ uint8_t q_smem_raw[];
    __shared__ __align__(16) uint8_t s_rs[512];
    __shared__ __align__(16) uint8_t s_cs[512];
    __shared__ __align__(16) float s_red[4][kTile];
    __shared__ int s_abort;

    // dynamic shared memory: [input stages][full/empty barriers][expert offsets (E+1)]
    //                        [kPad: padded expert offsets (E+1)]
    uint8_t* q_smem = smem_align<128>(q_smem_raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(q_smem + Sh::kStages * Sh::kStageBytes);
    int64_t* s_off = reinterpret_cast<int64_t*>(bars + 2 * Sh::kStages);
    int64_t* s_poff = s_off + (a.E + 1);

    if (a.noop && *a.noop) return;
    const int bad = kPad ? load_offsets_padded(a.m_splits, a.E, a.M, s_off, s_poff)
                         : load_offsets(a.m_splits, a.E, a.M, s_off);
    if (bad) {
        report_status(a.status, bad);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t K = a.K;
    const int64_t tilesK = K / kTile;
    const int64_t tiles = (kPad ? s_poff[a.E] / kTile : a.M / kTile) * tilesK;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + Sh::kStages);
    volatile int* abort_flag = &s_abort;
    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int st = 0; st < Sh::kStages; ++st) {
            mbar_init(full0 + 8 * st, 1);
            mbar_init(empty0 + 8 * st, kComputeWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tm_in) : "memory");
    }
    __syncthreads();

    if (warp == kComputeWarps) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
                if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag)) break;
                const uint32_t fb = full0 + 8 * stage;
                mbar_expect_tx(fb, Sh::kStageBytes);
                const TileGeom g = tile_geom<kPad>(t / tilesK, s_off, s_poff, a.E);
                tma_load_2d(smem_u32(q_smem + stage * Sh::kStageBytes), &tm_in, fb, (int)((t % tilesK) * kTile),
                            (int)g.row0);  // rows past M read as zeros
                if (++stage == Sh::kStages) { stage = 0; phase ^= 1; }
            }
        }
        return;
    }

    const int rg = warp;         // 32-row group of the tile
    const int blk = lane >> 3;   // 32-column block of the tile holding this lane's 4 columns
    const uint32_t sel_blk = 0x4440u | (uint32_t)blk;  // byte_perm selector: byte blk, zero-extended
    const uint32_t Ku = (uint32_t)K;
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t mt = t / tilesK, kt = t % tilesK;
        const TileGeom g = tile_geom<kPad>(mt, s_off, s_poff, a.E);
        const int64_t r0 = g.row0 + rg * 32;             // this warp's first row
        const int64_t col = kt * kTile + lane * 4;       // this lane's first column
        const int vb = kPad ? max(0, min(32, g.vr - rg * 32)) : 32;  // this warp's rows inside the expert

        // requant: lane l reads the 4 compact rowwise scale codes of row r0 + l
        uint32_t sw = 0;
        if constexpr (kReq) {
            if (!kPad || lane < vb)
                sw = __ldg(reinterpret_cast<const unsigned int*>(a.src_scale + (r0 + lane) * (K / 32) + kt * 4));
        }
        // requant: the largest and smallest rowwise scale code of this lane's 32-column block over the
        // warp's 32 rows (the fast paths below need their spread)
        [[maybe_unused]] uint32_t R = 0, Rmin = 0;
        if constexpr (kReq) {
            uint32_t mx = sw, mn = sw;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                mx = __vmaxu4(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                mn = __vminu4(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            }
            R = __byte_perm(mx, 0u, sel_blk);
            Rmin = __byte_perm(mn, 0u, sel_blk);
        }
        // scaled bias: lane l reads s of row r0 + l and b_e of its 4 columns
        float pw = 0.f, bv[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (kScaled) {
            if (!kPad || lane < vb) pw = __ldg(a.probs + r0 + lane);
            const int e = kPad ? g.e : expert_of(s_off, a.E, mt * kTile);
            const uint2 b2 = __ldg(reinterpret_cast<const uint2*>(a.bias + (int64_t)e * K + col));
            bv[0] = bf16lo(b2.x);
            bv[1] = bf16hi(b2.x);
            bv[2] = bf16lo(b2.y);
            bv[3] = bf16hi(b2.y);
        }

        const bool ok = mbar_wait(full0 + 8 * stage, phase, abort_flag);
        if (compute_bar_any(!ok)) break;
        const uint8_t* src = q_smem + stage * Sh::kStageBytes + (rg * 32) * Sh::kRowBytes + lane * 4 * Sh::kInBytes;

        // raw bits of row r: bf16 x4 (two words) or E4M3 x4 (one word)
        auto ld_row = [&](int r) -> uint2 {
            if constexpr (!kReq) return *reinterpret_cast<const uint2*>(src + r * Sh::kRowBytes);
            else return make_uint2(*reinterpret_cast<const uint32_t*>(src + r * Sh::kRowBytes), 0u);
        };
        // exact fp32 values of row r
        auto vals = [&](int r, uint2 u, float* v) {
            if constexpr (!kReq) {
                v[0] = bf16lo(u.x);
                v[1] = bf16hi(u.x);
                v[2] = bf16lo(u.y);
                v[3] = bf16hi(u.y);
            } else {
                // byte blk of row r's four codes; 2^(code - 127) from the code placed in
                // the exponent field, code 0 -> 2^-127 (the subnormal 0x00400000)
                const uint32_t code = __byte_perm(__shfl_sync(0xffffffffu, sw, r), 0u, sel_blk);
                const float sc = __uint_as_float(max(code << 23, 0x00400000u));
                const float2 lo = e4m3x2_to_f32((uint16_t)(u.x & 0xFFFFu));
                const float2 hi = e4m3x2_to_f32((uint16_t)(u.x >> 16));
                v[0] = lo.x * sc;
                v[1] = lo.y * sc;
                v[2] = hi.x * sc;
                v[3] = hi.y * sc;
            }
        };

        // ------------------------------------ pass 1: colwise amax, dbias
        uint32_t ccode[4] = {0, 0, 0, 0};
        float cinv[4] = {1.f, 1.f, 1.f, 1.f};
        // Both passes; kMask (padded grouping, a warp whose 32 rows reach past its
        // expert) skips the rows past the expert. Whole warps choose one form.
        auto passes = [&](auto mask_t) {
            [[maybe_unused]] constexpr bool kMask = decltype(mask_t)::value;
            // Requant fast path, pass 1 (whole warps of 32 rows inside the expert): when every row scale
            // code of the block is within 5 of the largest, R, |val| 2^(rs - R) is an exact normal f16 for
            // every nonzero E4M3 val (|val| >= 2^-9), so the colwise maxima can be taken in f16x2.
            [[maybe_unused]] constexpr bool kFast1 = kReq && kCol && !kBias && !kScaled && !kMask;
            [[maybe_unused]] constexpr bool kFast2 = kReq && kCol && !kDeq && !kMask;
            [[maybe_unused]] bool fast1 = false;
            if constexpr (kFast1) fast1 = __all_sync(0xffffffffu, R - Rmin <= 5u);
            [[maybe_unused]] uint32_t m16[2] = {0u, 0u};  // fast pass 1: f16x2 maxima of |val| 2^(rs - R)
            [[maybe_unused]] uint32_t nz = 0u;            // requant: bit j set when column j holds a nonzero
            if constexpr (kCol || kBias) {
                [[maybe_unused]] uint32_t m[4] = {0, 0, 0, 0};  // packed bf16 |x| bits (bf16 input, no dbias)
                [[maybe_unused]] float mf[4] = {0.f, 0.f, 0.f, 0.f};  // |v| maxima (every other case)
                [[maybe_unused]] float sum[4] = {0.f, 0.f, 0.f, 0.f};
                if constexpr (kScaled) {
                    float dp[32];  // this lane's 4-column share of each row's dot product with b_e
    #pragma unroll
                    for (int r = 0; r < 32; ++r) {
                        float v[4];
                        vals(r, ld_row(r), v);
                        const float s_r = __shfl_sync(0xffffffffu, pw, r);
                        if (kMask && r >= vb) {
                            dp[r] = 0.f;
                            continue;
                        }
                        dp[r] = v[0] * bv[0] + v[1] * bv[1] + v[2] * bv[2] + v[3] * bv[3];
    #pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            mf[j] = fmaxf(mf[j], fabsf(v[j]));
                            sum[j] += s_r * v[j];
                        }
                    }
                    const float dsum = transpose_reduce32(dp, lane);
                    if (!kMask || lane < vb) a.dp_partials[(r0 + lane) * tilesK + kt] = dsum;
                } else if (kFast1 && fast1) {
    #pragma unroll 8
                    for (int r = 0; r < 32; ++r) {
                        const uint32_t u = ld_row(r).x;
                        const uint32_t code = __byte_perm(__shfl_sync(0xffffffffu, sw, r), 0u, sel_blk);
                        const uint32_t s2 = (code + 15u - R) * 0x04000400u;  // 2^(code - R) in both f16 lanes
                        m16[0] = f16x2_max(m16[0], f16x2_mul(e4m3x2_to_f16x2(u & 0xFFFFu), s2) & 0x7FFF7FFFu);
                        m16[1] = f16x2_max(m16[1], f16x2_mul(e4m3x2_to_f16x2(u >> 16), s2) & 0x7FFF7FFFu);
                    }
                } else {
    #pragma unroll 8
                    for (int r = 0; r < 32; ++r) {
                        if (kMask && r >= vb) continue;
                        const uint2 u = ld_row(r);
                        if constexpr (!kReq && !kBias) {
                            m[0] = __vmaxu2(m[0], u.x & 0x7FFF7FFFu);
                            m[1] = __vmaxu2(m[1], u.y & 0x7FFF7FFFu);
                        } else {
                            float v[4];
                            vals(r, u, v);
    #pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                mf[j] = fmaxf(mf[j], fabsf(v[j]));
                                if constexpr (kBias) sum[j] += v[j];
                            }
                        }
                    }
                }
                if constexpr (kCol) {
                    uint32_t e[4];
                    if constexpr (!kReq && !kBias) {
                        e[0] = (m[0] >> 7) & 0xFFu;
                        e[1] = (m[0] >> 23) & 0xFFu;
                        e[2] = (m[1] >> 7) & 0xFFu;
                        e[3] = (m[1] >> 23) & 0xFFu;
                    } else {
    #pragma unroll
                        for (int j = 0; j < 4; ++j) e[j] = __float_as_uint(mf[j]) >> 23;
                    }
    #pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (kFast1 && fast1) {
                            // the column's largest |value| is m16_j 2^(R - 127), whose floor(log2) is
                            // (ef_j - 15) + (R - 127) for the f16 exponent field ef_j
                            const uint32_t hb = (m16[j >> 1] >> (16 * (j & 1))) & 0x7FFFu;
                            ccode[j] = hb ? (uint32_t)max((int)((hb >> 10) + R) - 23, 0) : 0u;
                            nz |= (uint32_t)(hb != 0u) << j;
                        } else {
                            ccode[j] = (uint32_t)max((int)e[j] - 8, 0);
                            if constexpr (kReq) nz |= (uint32_t)(mf[j] > 0.f) << j;
                        }
                        cinv[j] = inv_scale_from_code(ccode[j]);
                    }
                    if (a.swizzle) {
    #pragma unroll
                        for (int j = 0; j < 4; ++j) s_cs[(4 * (lane & 7) + j) * 16 + blk * 4 + rg] = (uint8_t)ccode[j];
                    } else {
                        *reinterpret_cast<uint32_t*>(a.col_s + (g.prow0 / 32 + rg) * K + col) =
                            ccode[0] | (ccode[1] << 8) | (ccode[2] << 16) | (ccode[3] << 24);
                    }
                }
                if constexpr (kBias) *reinterpret_cast<float4*>(&s_red[rg][lane * 4]) = make_float4(sum[0], sum[1], sum[2], sum[3]);
            }
            if constexpr (kReq && kRow) *reinterpret_cast<uint32_t*>(&s_rs[lane * 16 + rg * 4]) = sw;

            // ------------------------------------------------- pass 2: encode
            if constexpr (kFast2) {
                // Requant fast path, pass 2: when every rs_r - cs_j lies in [-14, 15] (an all-zero column's
                // scale taken as R), 2^(rs_r - cs_j) is a normal f16 and val 2^(rs_r - cs_j) is exact in f16
                // wherever it is at least 2^-14; below that it and the exact value both encode to a signed
                // zero. One f16x2 product per pair of values then gives the codes of the fp32 steps.
                uint32_t csm[4];
                bool ok = true;
    #pragma unroll
                for (int j = 0; j < 4; ++j) {
                    csm[j] = ((nz >> j) & 1u) ? ccode[j] : R;
                    ok = ok && (R <= csm[j] + 15u) && (Rmin + 14u >= csm[j]);
                }
                if (__all_sync(0xffffffffu, ok)) {
                    // f16 bits of 2^(rs - cs) for two columns: rs * 0x04000400 plus these, mod 2^32
                    const uint32_t k01 = (15u - csm[0]) * 1024u + (15u - csm[1]) * 67108864u;
                    const uint32_t k23 = (15u - csm[2]) * 1024u + (15u - csm[3]) * 67108864u;
                    uint8_t* cq = a.col_q + r0 * K + col;
    #pragma unroll 8
                    for (int r = 0; r < 32; ++r) {
                        const uint32_t u = ld_row(r).x;
                        const uint32_t rs2 = __byte_perm(__shfl_sync(0xffffffffu, sw, r), 0u, sel_blk) * 0x04000400u;
                        const uint32_t lo = f16x2_to_e4m3x2(f16x2_mul(e4m3x2_to_f16x2(u & 0xFFFFu), rs2 + k01));
                        const uint32_t hi = f16x2_to_e4m3x2(f16x2_mul(e4m3x2_to_f16x2(u >> 16), rs2 + k23));
                        *reinterpret_cast<uint32_t*>(cq + r * Ku) = lo | (hi << 16);
                    }
                    return;
                }
            }
            if constexpr ((kRow && !kReq) || kCol || kDeq) {
                [[maybe_unused]] uint8_t* rq = kRow && !kReq ? a.row_q + r0 * K + col : nullptr;
                [[maybe_unused]] uint8_t* cq = kCol ? a.col_q + r0 * K + col : nullptr;
                [[maybe_unused]] __nv_bfloat16* dq = kDeq ? a.deq_out + r0 * K + col : nullptr;
    #pragma unroll 1
                for (int r8 = 0; r8 < 32; r8 += 8) {
                    // eight rows in flight: the loads of both four-row groups before any store (the stores
                    // go through pointers the compiler cannot tell apart from the shared tile)
                    uint2 u[8];
    #pragma unroll
                    for (int k = 0; k < 8; ++k) u[k] = ld_row(r8 + k);
                    [[maybe_unused]] uint32_t packed[2] = {0u, 0u};  // rowwise codes, one byte per row
                    if constexpr (kRow && !kReq) {
    #pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint32_t m[4];
    #pragma unroll
                            for (int k = 0; k < 4; ++k)
                                m[k] = __vmaxu2(u[4 * h + k].x & 0x7FFF7FFFu, u[4 * h + k].y & 0x7FFF7FFFu);
                            // |bits| maxima of rows (0, 1) and (2, 3) as 16-bit halves, then their bf16
                            // exponent fields, one byte per row
                            const uint32_t v01 =
                                __vmaxu2(__byte_perm(m[0], m[1], 0x5410), __byte_perm(m[0], m[1], 0x7632));
                            const uint32_t v23 =
                                __vmaxu2(__byte_perm(m[2], m[3], 0x5410), __byte_perm(m[2], m[3], 0x7632));
                            packed[h] = __byte_perm((v01 >> 7) & 0x00FF00FFu, (v23 >> 7) & 0x00FF00FFu, 0x6420);
                        }
    #pragma unroll
                        for (int o = 4; o >= 1; o >>= 1)
    #pragma unroll
                            for (int h = 0; h < 2; ++h)
                                packed[h] = __vmaxu4(packed[h], __shfl_xor_sync(0xffffffffu, packed[h], o));
    #pragma unroll
                        for (int h = 0; h < 2; ++h) packed[h] = __vsubus4(packed[h], 0x08080808u);  // max(e - 8, 0)
                    }
                    [[maybe_unused]] const uint64_t cinv01 = f2pack(cinv[0], cinv[1]), cinv23 = f2pack(cinv[2], cinv[3]);
    #pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int r = r8 + k;
                        const bool valid = !kMask || r < vb;  // kPad: rows past the expert are not written
                        float v[4];
                        vals(r, u[k], v);
                        const uint64_t v01 = f2pack(v[0], v[1]), v23 = f2pack(v[2], v[3]);
                        if constexpr (kRow && !kReq) {
                            const uint32_t code = (packed[k >> 2] >> (8 * (k & 3))) & 0xFFu;
                            const uint64_t inv = f2splat(inv_scale_from_code(code));
                            const float2 s01 = f2unpack(f2mul(v01, inv)), s23 = f2unpack(f2mul(v23, inv));
                            if (valid)
                                *reinterpret_cast<uint32_t*>(rq + r * Ku) =
                                    cvt_e4m3x2(s01.x, s01.y) | (cvt_e4m3x2(s23.x, s23.y) << 16);
                            if ((lane & 7) == 0) {
                                if (a.swizzle) s_rs[r * 16 + rg * 4 + blk] = valid ? (uint8_t)code : (uint8_t)0;
                                else if (valid) a.row_s[(r0 + r) * (K / 32) + kt * 4 + blk] = (uint8_t)code;
                            }
                        }
                        if (!valid) continue;
                        if constexpr (kCol) {
                            const float2 s01 = f2unpack(f2mul(v01, cinv01)), s23 = f2unpack(f2mul(v23, cinv23));
                            *reinterpret_cast<uint32_t*>(cq + r * Ku) =
                                cvt_e4m3x2(s01.x, s01.y) | (cvt_e4m3x2(s23.x, s23.y) << 16);
                        }
                        if constexpr (kDeq) {
                            __nv_bfloat162 b0 = __floats2bfloat162_rn(v[0], v[1]);
                            __nv_bfloat162 b1 = __floats2bfloat162_rn(v[2], v[3]);
                            uint2 o;
                            o.x = *reinterpret_cast<uint32_t*>(&b0);
                            o.y = *reinterpret_cast<uint32_t*>(&b1);
                            *reinterpret_cast<uint2*>(dq + (size_t)r * Ku) = o;
                        }
                    }
                }
            }
        };
        if constexpr (kPad) {
            if (vb < 32) passes(std::true_type{});
            else passes(std::false_type{});
        } else {
            passes(std::false_type{});
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * stage);  // this warp is done with the stage
        if (++stage == Sh::kStages) { stage = 0; phase ^= 1; }

        compute_bar();
        if constexpr (kBias) {
            const int c = threadIdx.x;  // 0..127
            a.partials[(g.prow0 / kTile) * K + kt * kTile + c] =
                ((s_red[0][c] + s_red[1][c]) + s_red[2][c]) + s_red[3][c];
        }
        if constexpr (kRow) {
            if ((a.swizzle || kReq) && threadIdx.x < 32) {
                uint4* dst = reinterpret_cast<uint4*>(a.row_s + ((g.prow0 / kTile) * tilesK + kt) * 512);
                dst[threadIdx.x] = reinterpret_cast<const uint4*>(s_rs)[threadIdx.x];
            }
        }
        if constexpr (kCol) {
            if (a.swizzle && threadIdx.x >= 32 && threadIdx.x < 64) {
                // the expert's (K, rows/32) colwise scales at byte K * first_row / 32 of the scale row
                // space (padded rows with kPad)
                const int64_t rt0 = g.prow0;
                int64_t off, me;
                if constexpr (kPad) {
                    off = g.off_p;
                    me = g.me_p;
                } else {
                    const int e = expert_of(s_off, a.E, rt0);
                    off = s_off[e];
                    me = s_off[e + 1] - off;
                }
                const int64_t base = K * off / 32;
                const int64_t atom = kt * (me / kTile) + (rt0 - off) / kTile;
                uint4* dst = reinterpret_cast<uint4*>(a.col_s + base + atom * 512);
                dst[threadIdx.x - 32] = reinterpret_cast<const uint4*>(s_cs)[threadIdx.x - 32];
            }
        }
        compute_bar();
    }
    if (threadIdx.x == 0 && s_abort && a.status) atomicOr(a.status, MXQ_STATUS_WAIT_TIMEOUT);
}

// SM count per device, cached (atomic: launches may come from several host threads).
static int num_sms() {
    static std::atomic<int> n[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64) {
        const int c = n[dev].load(std::memory_order_relaxed);
        if (c) return c;
    }
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (dev < 64) n[dev].store(v, std::memory_order_relaxed);
    return v;
}

template <bool kReq, bool kRow, bool kCol, bool kBias, bool kDeq, bool kScaled = false, bool kPad = false>
static cudaError_t launch_tile(const TileArgs& a, cudaStream_t s) {
    using Sh = TileShape<kReq>;
    auto kern = mx_tile_kernel<kReq, kRow, kCol, kBias, kDeq, kScaled, kPad>;
    // kPad: the padded row count is only known on the device; size the grid
    // for its bound (round_up(M, 128) + 128 E rows)
    const int64_t rows = kPad ? ((a.M + 127) / 128 * 128 + (int64_t)kTile * a.E) : a.M;
    const int64_t tiles = a.M == 0 ? 0 : (rows / kTile) * (a.K / kTile);
    if (tiles == 0) return cudaSuccess;
    const int smem = Sh::kSmem + (kPad ? 2 : 1) * (a.E + 1) * 8;
    const cudaError_t attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (attr != cudaSuccess) return attr;
    CUtensorMap tm;
    if (!encode_tmap_2d(&tm, a.src, a.M, a.K, Sh::kInBytes, kTile, kTile, 0)) return cudaErrorInvalidValue;
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kTileThreads, smem);
    const int64_t grid = std::min<int64_t>(tiles, (int64_t)num_sms() * std::max(per_sm, 1));
    kern<<<(unsigned)grid, kTileThreads, smem, s>>>(tm, a);
    return cudaGetLastError();
}

}  // namespace mxq
