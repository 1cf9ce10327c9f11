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
    const float* probs;        // scaled bias: routing scale s_m per row (M)
    const __nv_bfloat16* bias; // scaled bias: b_e (E, K)
    float* dp_partials;        // scaled bias: (M, K/128) fp32 per-tile sums of dY[m,:] . b_e
    int swizzle;
    const int32_t* noop;
    int32_t* status;
};

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
// 16k-token workload 1 stage ran 51 us, 2 stages 64 us, 3 stages 79 us.
#ifndef MXQ_QUANT_STAGES_BF16
#define MXQ_QUANT_STAGES_BF16 1  // 32 KB bf16 tiles in flight per CTA
#endif
#ifndef MXQ_QUANT_STAGES_E4M3
#define MXQ_QUANT_STAGES_E4M3 3  // 16 KB E4M3 tiles in flight per CTA
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

// kScaled (scaled bias, with kBias): the column sums weight row m by its
// routing scale s_m, and each row's dot product with its expert's bias is
// reduced per tile into dp_partials.
template <bool kReq, bool kRow, bool kCol, bool kBias, bool kDeq, bool kScaled = false>
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
    uint8_t* q_smem = smem_align<128>(q_smem_raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(q_smem + Sh::kStages * Sh::kStageBytes);
    int64_t* s_off = reinterpret_cast<int64_t*>(bars + 2 * Sh::kStages);

    if (a.noop && *a.noop) return;
    const int bad = load_offsets(a.m_splits, a.E, a.M, s_off);
    if (bad) {
        report_status(a.status, bad);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t K = a.K;
    const int64_t tilesK = K / kTile;
    const int64_t tiles = (a.M / kTile) * tilesK;
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
                tma_load_2d(smem_u32(q_smem + stage * Sh::kStageBytes), &tm_in, fb, (int)((t % tilesK) * kTile),
                            (int)((t / tilesK) * kTile));
                if (++stage == Sh::kStages) { stage = 0; phase ^= 1; }
            }
        }
        return;
    }

    const int rg = warp;         // 32-row group of the tile
    const int blk = lane >> 3;   // 32-column block of the tile holding this lane's 4 columns
    const uint32_t Ku = (uint32_t)K;
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t mt = t / tilesK, kt = t % tilesK;
        const int64_t r0 = mt * kTile + rg * 32;        // this warp's first row
        const int64_t col = kt * kTile + lane * 4;       // this lane's first column

        // requant: lane l reads the 4 compact rowwise scale codes of row r0 + l
        uint32_t sw = 0;
        if constexpr (kReq) sw = __ldg(reinterpret_cast<const unsigned int*>(a.src_scale + (r0 + lane) * (K / 32) + kt * 4));
        // scaled bias: lane l reads s of row r0 + l and b_e of its 4 columns
        float pw = 0.f, bv[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (kScaled) {
            pw = __ldg(a.probs + r0 + lane);
            const int e = expert_of(s_off, a.E, mt * kTile);
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
                const float sc = scale_from_code((__shfl_sync(0xffffffffu, sw, r) >> (8 * blk)) & 0xFFu);
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
        if constexpr (kCol || kBias) {
            uint32_t m[4] = {0, 0, 0, 0};
            float sum[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (kScaled) {
                float dp[32];  // this lane's 4-column share of each row's dot product with b_e
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    float v[4];
                    vals(r, ld_row(r), v);
                    const float s_r = __shfl_sync(0xffffffffu, pw, r);
                    dp[r] = v[0] * bv[0] + v[1] * bv[1] + v[2] * bv[2] + v[3] * bv[3];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        m[j] = max(m[j], __float_as_uint(v[j]) & 0x7FFFFFFFu);
                        sum[j] += s_r * v[j];
                    }
                }
                a.dp_partials[(r0 + lane) * tilesK + kt] = transpose_reduce32(dp, lane);
            } else {
#pragma unroll 8
                for (int r = 0; r < 32; ++r) {
                    const uint2 u = ld_row(r);
                    if constexpr (!kReq && !kBias) {
                        m[0] = __vmaxu2(m[0], u.x & 0x7FFF7FFFu);
                        m[1] = __vmaxu2(m[1], u.y & 0x7FFF7FFFu);
                    } else {
                        float v[4];
                        vals(r, u, v);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            m[j] = max(m[j], __float_as_uint(v[j]) & 0x7FFFFFFFu);
                            sum[j] += v[j];
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
                    for (int j = 0; j < 4; ++j) e[j] = m[j] >> 23;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    ccode[j] = (uint32_t)max((int)e[j] - 8, 0);
                    cinv[j] = inv_scale_from_code(ccode[j]);
                }
                if (a.swizzle) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) s_cs[(4 * (lane & 7) + j) * 16 + blk * 4 + rg] = (uint8_t)ccode[j];
                } else {
                    *reinterpret_cast<uint32_t*>(a.col_s + (mt * 4 + rg) * K + col) =
                        ccode[0] | (ccode[1] << 8) | (ccode[2] << 16) | (ccode[3] << 24);
                }
            }
            if constexpr (kBias) *reinterpret_cast<float4*>(&s_red[rg][lane * 4]) = make_float4(sum[0], sum[1], sum[2], sum[3]);
        }
        if constexpr (kReq && kRow) *reinterpret_cast<uint32_t*>(&s_rs[lane * 16 + rg * 4]) = sw;

        // ------------------------------------------------- pass 2: encode
        if constexpr ((kRow && !kReq) || kCol || kDeq) {
            uint8_t* rq = kRow && !kReq ? a.row_q + r0 * K + col : nullptr;
            uint8_t* cq = kCol ? a.col_q + r0 * K + col : nullptr;
            __nv_bfloat16* dq = kDeq ? a.deq_out + r0 * K + col : nullptr;
#pragma unroll 2
            for (int r4 = 0; r4 < 32; r4 += 4) {
                uint2 u[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) u[k] = ld_row(r4 + k);
                uint32_t packed = 0;
                if constexpr (kRow && !kReq) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t w2 = __vmaxu2(u[k].x & 0x7FFF7FFFu, u[k].y & 0x7FFF7FFFu);
                        packed |= (max(w2 & 0xFFFFu, w2 >> 16) >> 7) << (8 * k);  // bf16 exponent field
                    }
                    packed = group8_max_u8x4(packed);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int r = r4 + k;
                    float v[4];
                    vals(r, u[k], v);
                    if constexpr (kRow && !kReq) {
                        const uint32_t code = (uint32_t)max((int)((packed >> (8 * k)) & 0xFFu) - 8, 0);
                        const float inv = inv_scale_from_code(code);
                        *reinterpret_cast<uint32_t*>(rq + r * Ku) =
                            cvt_e4m3x2(v[0] * inv, v[1] * inv) | (cvt_e4m3x2(v[2] * inv, v[3] * inv) << 16);
                        if ((lane & 7) == 0) {
                            if (a.swizzle) s_rs[r * 16 + rg * 4 + blk] = (uint8_t)code;
                            else a.row_s[(r0 + r) * (K / 32) + kt * 4 + blk] = (uint8_t)code;
                        }
                    }
                    if constexpr (kCol) {
                        *reinterpret_cast<uint32_t*>(cq + r * Ku) = cvt_e4m3x2(v[0] * cinv[0], v[1] * cinv[1]) |
                                                                    (cvt_e4m3x2(v[2] * cinv[2], v[3] * cinv[3]) << 16);
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
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * stage);  // this warp is done with the stage
        if (++stage == Sh::kStages) { stage = 0; phase ^= 1; }

        compute_bar();
        if constexpr (kBias) {
            const int c = threadIdx.x;  // 0..127
            a.partials[mt * K + kt * kTile + c] = ((s_red[0][c] + s_red[1][c]) + s_red[2][c]) + s_red[3][c];
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
        compute_bar();
    }
    if (threadIdx.x == 0 && s_abort && a.status) atomicOr(a.status, MXQ_STATUS_WAIT_TIMEOUT);
}

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

template <bool kReq, bool kRow, bool kCol, bool kBias, bool kDeq, bool kScaled = false>
static cudaError_t launch_tile(const TileArgs& a, cudaStream_t s) {
    using Sh = TileShape<kReq>;
    auto kern = mx_tile_kernel<kReq, kRow, kCol, kBias, kDeq, kScaled>;
    const int64_t tiles = (a.M / kTile) * (a.K / kTile);
    if (tiles == 0) return cudaSuccess;
    const int smem = Sh::kSmem + (a.E + 1) * 8;
    const cudaError_t attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (attr != cudaSuccess) return attr;
    CUtensorMap tm;
    if (!encode_tmap_2d(&tm, a.src, a.M, a.K, Sh::kInBytes, kTile, kTile, false)) return cudaErrorInvalidValue;
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kTileThreads, smem);
    const int64_t grid = std::min<int64_t>(tiles, (int64_t)num_sms() * std::max(per_sm, 1));
    kern<<<(unsigned)grid, kTileThreads, smem, s>>>(tm, a);
    return cudaGetLastError();
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
