// mxq_gemm.cu -- grouped MXFP8 GEMMs of an MoE expert layer on GB300 (sm_103a):
//   fprop  Y[m,:]  = X[m,:]  . W[e(m)]^T (+ b[e(m)])   rowwise X, rowwise W
//   dgrad  dX[m,:] = dY[m,:] . W[e(m)]                 rowwise dY, colwise W
//   wgrad  dW[e]   = dY_e^T . X_e                      colwise dY, colwise X
// (TransformerEngine PR #3244, "[Pytorch] Add support for row-wise quanted
// input for grouped gemm": fprop/dgrad on the rowwise copy, wgrad on the
// columnwise copy; PR #3545, "Fix distributed BF16 weights and trim NVFP4
// saved state in the fused grouped MLP": the columnwise weight copy exists for
// dgrad, wgrad reads only columnwise tiles; PR #3224, "Improve device-init
// grouped linear module with single grouped weight support": device m_splits
// read without a host sync, one grouped weight (E,out,in), 2-D grouped bias.)
//
// Two kernels. The plain fprop, dgrad and wgrad on 128-aligned experts, and
// FC1 with the SwiGLU epilogue, run on two-SM pair tiles (namespace pair
// below: tcgen05 cta_group::2, 256 x 256 tiles). The one-SM kernel described
// here serves padded grouping, the FC2 dgrad with the SwiGLU-backward
// epilogue, more than 512 experts and wgrad with N not a multiple of 256.
//
// One-SM kernel: persistent, one CTA (320 threads) per SM, warp-specialised.
//   warp 0      TMA producer: 128x128-byte E4M3 boxes (128B swizzle) for A and
//               two for B per 128-deep K block, plus the 512-byte scale atoms
//               (already in the tensor-core 128x4 layout) by bulk copy;
//   warp 1      owns TMEM (512 columns) and, from one lane, issues
//               tcgen05.cp (scales -> TMEM) and tcgen05.mma
//               .kind::mxf8f6f4.block_scale (M=128, N=256, K=32, fp32 accum);
//   warps 2..9  epilogue: two warps per TMEM lane quarter each pull a 32x128
//               slice of the 128x256 fp32 accumulator into registers
//               (tcgen05.ld), release the accumulator, then add bias,
//               convert and store to global.
// A 4-stage shared-memory ring (mbarrier full/empty) feeds the tensor core;
// because the accumulator is released as soon as it sits in registers, the
// next tile's MMAs overlap the conversion and the global stores.
//
// Operand majorness: K-major (A of fprop/dgrad, B of fprop) and MN-major (B of
// dgrad, A and B of wgrad: the columnwise copies keep the source's byte
// order, so their contiguous dimension is the MMA's M or N). Both use the
// 128-byte swizzle; MN-major tiles are read straight from the un-transposed
// colwise copy.
//
// Tile schedule: fprop/dgrad are a dense grid of 128-row x 256-col tiles over
// the M routed rows (a 128-row tile never straddles two experts because every
// m_e % 128 == 0; its expert comes from an on-chip prefix sum of the device
// m_splits). wgrad tiles are (expert, 128 rows of N, 256 cols of K) with a
// K loop of m_e/128 blocks; they are ordered heaviest expert first and dealt
// to CTAs in a serpentine so that per-CTA work is balanced.
//
// Every wait on an mbarrier is bounded (about 2 s of wall time); on expiry the
// kernel sets MXQ_STATUS_WAIT_TIMEOUT, stops issuing work, frees its TMEM and
// returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "mxq_common.cuh"
#include "mxq_internal.h"

namespace mxq {
namespace gemm {

constexpr int BM = 128;               // MMA M (rows of A per tile)
constexpr int BN = 256;               // MMA N (cols of the output tile)
constexpr int BK = 128;               // K elements (bytes) per pipeline stage
constexpr int UMMA_K = 32;            // K per tcgen05.mma for 8-bit operands
constexpr int STAGES = 4;
constexpr int EPI_WARPS = 8;
constexpr int A_BYTES = BM * BK;      // 16 KB
constexpr int B_BYTES = BN * BK;      // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 48 KB: every stage stays 1024-aligned
constexpr int SF_STAGE_BYTES = 1536;            // scale atoms of a stage: A (512), B (2 x 512)
constexpr uint32_t STAGE_TX = A_BYTES + B_BYTES + 512 + 1024;
constexpr int NUM_THREADS = 320;      // producer, MMA, 8 epilogue warps
constexpr int TMEM_COLS = 512;
constexpr int TMEM_SFA = 256;         // scale columns after the accumulator
constexpr int TMEM_SFB = 264;
constexpr int EPI_STAGE_BYTES = 2048;           // per epilogue warp: one 32-row output box
// dynamic shared memory: [A/B stages][scale atoms][barriers][epilogue staging][expert tables]
constexpr int SF_REGION = STAGES * STAGE_BYTES;
constexpr int BAR_REGION = SF_REGION + STAGES * SF_STAGE_BYTES;
constexpr int EPI_REGION = (BAR_REGION + 256 + 511) / 512 * 512;  // 512-aligned: the 64-byte swizzle's period
constexpr int TABLE_REGION = EPI_REGION + EPI_WARPS * EPI_STAGE_BYTES;
__host__ __device__ constexpr int smem_bytes(int E) { return 1024 + TABLE_REGION + 8 * (E + 1) + 2 * E; }
// padded grouping keeps a second (E+1)-entry offset table
__host__ __device__ constexpr int smem_bytes_padded(int E) { return smem_bytes(E) + 8 * (E + 1); }
constexpr int MAX_EXPERTS_PADDED = 512;  // smem_bytes_padded(512) fits the 227 KB per-block limit
static_assert(smem_bytes(MXQ_MAX_EXPERTS) <= 232448, "shared memory over the per-block limit");
static_assert(smem_bytes_padded(MAX_EXPERTS_PADDED) <= 232448, "shared memory over the per-block limit");
static_assert(EPI_REGION % 512 == 0, "the 64-byte swizzle of the staging boxes repeats every 512 bytes");

struct Params {
    int mode;
    int64_t M, N, K;
    int E;
    const int64_t* m_splits;
    const uint8_t* sfa;  // scale base of A
    const uint8_t* sfb;  // scale base of B
    const __nv_bfloat16* bias;
    void* out;
    int accumulate, out_bf16;
    int tma_store;  // 1: outputs leave through TMA bulk-tensor stores of staged boxes
    int32_t* status;
    // kFpropSwiglu: quantized h (M, N/2); kDgradSwiglu: quantized dY1 (M, 2K)
    uint8_t *q_row, *q_row_s, *q_col, *q_col_s;
    int swizzle;
    const __nv_bfloat16* y1;  // kDgradSwiglu: saved FC1 output (M, 2K)
    float* dbias_part;        // kDgradSwiglu: (M/32, 2K) per-32-row column sums, or null
    __nv_bfloat16* side;      // optional bf16 copy of what is quantized: h (M, N/2) or dY1 (M, 2K)
};

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05): start>>4 [0,14), LBO>>4 [16,30),
// SBO>>4 [32,46), version 1 [46,48), layout [61,64) (2 = 128B swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)(layout & 7u) << 61;
    return d;
}

// Instruction descriptor for kind::mxf8f6f4 (E4M3 x E4M3, fp32 accum,
// UE8M0 scales): b_sf_id [4,6), a_fmt [7,10)=0, b_fmt [10,13)=0,
// a_major [15], b_major [16], N>>3 [17,23), scale type UE8M0 [23],
// M>>4 [24,29), a_sf_id [29,31).
__device__ __forceinline__ uint32_t idesc(uint32_t a_mn, uint32_t b_mn, uint32_t sf_id) {
    return (sf_id << 4) | (a_mn << 15) | (b_mn << 16) | ((uint32_t)(BN >> 3) << 17) | (1u << 23) |
           ((uint32_t)(BM >> 4) << 24) | (sf_id << 29);
}

__device__ __forceinline__ void mma_mxf8(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t sfa,
                                         uint32_t sfb, uint32_t accum) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a), "l"(b), "r"(id), "r"(accum), "r"(sfa), "r"(sfb)
        : "memory");
}
__device__ __forceinline__ void tmem_cp_sf(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

#define TMEM_LD32(taddr, r)                                                                                     \
    asm volatile(                                                                                              \
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17," \
        "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"                                      \
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),         \
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), \
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),           \
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),           \
          "=r"(r[30]), "=r"(r[31])                                                                              \
        : "r"(taddr))

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------ tile schedule
struct Tile {
    int64_t a_row;   // fprop/dgrad: first token row; wgrad: first N row
    int64_t b_col;   // first output column (N for fprop, K for dgrad/wgrad)
    int e;
    int64_t off, me; // expert token offset / count
    int nk;          // number of 128-deep K blocks
    bool valid;
    // padded grouping (expert counts not multiples of 128; the aligned values otherwise)
    int64_t pa_row;  // fprop/dgrad: the tile's first row in the padded scale row space
    int vr;          // fprop/dgrad: rows of the tile inside its expert
    int64_t poff, mp;// the expert's padded first row / padded row count
    int vk;          // wgrad: tokens of the expert in its last 128-deep K block
};

struct Sched {
    int mode;
    int64_t M, N, K;
    int E;
    const int64_t* off;     // shared: exclusive offsets
    const int16_t* order;   // shared (wgrad): experts sorted by load, heaviest first
    const int64_t* poff;    // shared (padded grouping): padded offsets, each expert rounded up to 128 rows
    bool pad;
    int64_t tiles_n;        // fprop/dgrad: output col tiles; wgrad: tiles per expert
    int64_t total;

    __device__ void init(int mode_, int64_t M_, int64_t N_, int64_t K_, int E_, const int64_t* off_,
                         const int16_t* order_, const int64_t* poff_ = nullptr, bool pad_ = false) {
        mode = mode_; M = M_; N = N_; K = K_; E = E_; off = off_; order = order_; poff = poff_; pad = pad_;
        const int64_t row_tiles = (pad ? poff[E] : M) / BM;  // padded grouping: each expert's 128-row slices
        if (mode == kFprop || mode == kFpropSwiglu) { tiles_n = N / BN; total = row_tiles * tiles_n; }
        else if (mode == kDgrad || mode == kDgradSwiglu) { tiles_n = K / BN; total = row_tiles * tiles_n; }
        else { tiles_n = (N / BM) * (K / BN); total = (int64_t)E * tiles_n; }
    }
    // i-th tile of CTA `cta` among `ncta` (serpentine deal over the ordered list)
    __device__ int64_t pick(int64_t i, int cta, int ncta) const {
        const int64_t round = i, base = round * ncta;
        return (round & 1) ? base + (ncta - 1 - cta) : base + cta;
    }
    __device__ Tile get(int64_t t) const {
        Tile T;
        T.valid = t < total;
        if (!T.valid) return T;
        if (mode != kWgrad) {
            const int64_t mt = t / tiles_n, nt = t % tiles_n;
            // kFpropSwiglu: tile nt covers gate columns [128 nt, +128) and the
            // matching up columns [N/2 + 128 nt, +128)
            T.b_col = nt * (mode == kFpropSwiglu ? BN / 2 : BN);
            if (!pad) {
                T.a_row = T.pa_row = mt * BM;
                T.e = expert_of(off, E, T.a_row);
                T.off = T.poff = off[T.e];
                T.me = T.mp = off[T.e + 1] - T.off;
                T.vr = BM;
            } else {
                // slice j of expert e: token rows off_e + 128 j .., scale rows poff_e + 128 j ..
                T.e = expert_of(poff, E, mt * BM);
                const int64_t j = mt - poff[T.e] / BM;
                T.off = off[T.e];
                T.me = off[T.e + 1] - T.off;
                T.poff = poff[T.e];
                T.mp = poff[T.e + 1] - T.poff;
                T.a_row = T.off + j * BM;
                T.pa_row = T.poff + j * BM;
                const int64_t left = T.me - j * BM;
                T.vr = (int)(left < BM ? left : BM);
            }
            T.nk = (int)((mode == kDgrad || mode == kDgradSwiglu ? N : K) / BK);
            T.vk = BK;
        } else {
            const int64_t ei = t / tiles_n, r = t % tiles_n;
            const int64_t kt = K / BN;
            T.e = order[ei];
            T.a_row = T.pa_row = (r / kt) * BM;
            T.b_col = (r % kt) * BN;
            T.off = off[T.e];
            T.me = off[T.e + 1] - T.off;
            T.poff = pad ? poff[T.e] : T.off;
            T.mp = pad ? poff[T.e + 1] - T.poff : T.me;
            T.nk = (int)(T.mp / BK);  // padded grouping: the last block may hold fewer tokens
            T.vk = (int)(T.me - (int64_t)(T.nk > 0 ? T.nk - 1 : 0) * BK);
            T.vr = BM;
        }
        return T;
    }
};

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
    __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&b2);
}

// Sum of v[i] over the 32 lanes for every i: five exchange-and-add rounds
// halve the values each lane keeps; afterwards lane l holds i = l in v[0].
// Fixed order, so the sums are the same run to run.
__device__ __forceinline__ float lane_transpose_sum32(float (&v)[32], int lane) {
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

// MXFP8-quantize one 32-column block of a warp's 32 rows of an (M, W) bf16
// tensor, as group_quantize does: w holds this lane's row (lane = row
// rb0 + lane) at columns col0 .. col0+31 as bf16 pairs. Rowwise: one block
// per lane. Colwise: per column the largest exponent across the lanes (the
// 32-row block rb0 .. rb0+31, inside expert T.e). Codes go to p.q_row /
// p.q_col, E8M0 scales to p.q_row_s / p.q_col_s (swizzled per p.swizzle).
// With p.dbias_part, the block's 32 column sums go to row rb0/32 of it.
__device__ __forceinline__ void quant_block32(const uint32_t (&w)[16], const Params& p, const Tile& T, int64_t W,
                                              int64_t rb0, int64_t col0, int lane) {
    const int64_t row = rb0 + lane;
    // rowwise
    {
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) m = __vmaxu2(m, w[i] & 0x7FFF7FFFu);
        const uint32_t code = (uint32_t)max((int)(max(m & 0xFFFFu, m >> 16) >> 7) - 8, 0);
        const uint64_t inv = f2splat(inv_scale_from_code(code));
        uint32_t o[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t w0 = w[2 * k], w1 = w[2 * k + 1];
            const float2 a = f2unpack(f2mul(f2pack(bf16lo(w0), bf16hi(w0)), inv));
            const float2 b = f2unpack(f2mul(f2pack(bf16lo(w1), bf16hi(w1)), inv));
            o[k] = cvt_e4m3x2(a.x, a.y) | (cvt_e4m3x2(b.x, b.y) << 16);
        }
        uint4* d = reinterpret_cast<uint4*>(p.q_row + row * W + col0);
        d[0] = make_uint4(o[0], o[1], o[2], o[3]);
        d[1] = make_uint4(o[4], o[5], o[6], o[7]);
        const int64_t c = col0 / 32;
        if (p.swizzle)
            p.q_row_s[((row / 128) * (W / 128) + c / 4) * 512 + (row % 32) * 16 + ((row % 128) / 32) * 4 + c % 4] =
                (uint8_t)code;
        else
            p.q_row_s[row * (W / 32) + c] = (uint8_t)code;
    }
    // colwise
    uint32_t e4[8];  // four columns per word, one exponent byte each
#pragma unroll
    for (int i = 0; i < 8; ++i)  // the exponent fields of both halves of two words: bytes 0 and 2 of each
        e4[i] = __byte_perm((w[2 * i] >> 7) & 0x00FF00FFu, (w[2 * i + 1] >> 7) & 0x00FF00FFu, 0x6420);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
        for (int i = 0; i < 8; ++i) e4[i] = __vmaxu4(e4[i], __shfl_xor_sync(0xffffffffu, e4[i], off));
#pragma unroll
    for (int i = 0; i < 8; ++i) e4[i] = __vsub4(__vmaxu4(e4[i], 0x08080808u), 0x08080808u);  // max(e - 8, 0)
#pragma unroll
    for (int v = 0; v < 2; ++v) {
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t cw = e4[4 * v + k];
            const uint32_t w0 = w[8 * v + 2 * k], w1 = w[8 * v + 2 * k + 1];
            const float2 a = f2unpack(f2mul(f2pack(bf16lo(w0), bf16hi(w0)),
                                            f2pack(inv_scale_from_code(cw & 0xFFu),
                                                   inv_scale_from_code((cw >> 8) & 0xFFu))));
            const float2 b = f2unpack(f2mul(f2pack(bf16lo(w1), bf16hi(w1)),
                                            f2pack(inv_scale_from_code((cw >> 16) & 0xFFu),
                                                   inv_scale_from_code(cw >> 24))));
            o[k] = cvt_e4m3x2(a.x, a.y) | (cvt_e4m3x2(b.x, b.y) << 16);
        }
        *reinterpret_cast<uint4*>(p.q_col + row * W + col0 + 16 * v) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    uint32_t mine = 0;  // lane l < 8 writes the scales of columns col0 + 4l .. +3
#pragma unroll
    for (int i = 0; i < 8; ++i) mine = (lane == i) ? e4[i] : mine;
    if (lane < 8) {
        const int64_t k0 = col0 + 4 * lane;
        if (p.swizzle) {
            // per expert: logical (W, m_e/32) at byte W * off_e / 32
            const int64_t i = (rb0 - T.off) / 32, C4 = T.me / 128;
            uint8_t* base = p.q_col_s + W * T.off / 32;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t k = k0 + j;
                base[((k / 128) * C4 + i / 4) * 512 + (k % 32) * 16 + ((k % 128) / 32) * 4 + i % 4] =
                    (uint8_t)(mine >> (8 * j));
            }
        } else {
            *reinterpret_cast<uint32_t*>(p.q_col_s + (rb0 / 32) * W + k0) = mine;
        }
    }
    if (p.dbias_part) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            v[2 * j] = bf16lo(w[j]);
            v[2 * j + 1] = bf16hi(w[j]);
        }
        p.dbias_part[(rb0 / 32) * W + col0 + lane] = lane_transpose_sum32(v, lane);
    }
}

// Epilogue of the SwiGLU-fused FC2 dgrad (kDgradSwiglu) for one tile: the
// accumulator holds dh for 128 rows x 256 columns of F. Warp (q, half) takes
// rows 32q..32q+31 (lane = row) and columns T.b_col + 128 half + [0, 128),
// in four 32-column chunks: dh rounded to bf16 as the plain dgrad writes
// it, g and u from the saved FC1 output, dg and du in the fp32 steps of
// mxq_common.cuh, each rounded to bf16 and quantized into dY1 (columns f and
// F + f) with its dbias partials. This epilogue does about twice the
// arithmetic of the forward one on the same 8 warps per SM, so on the
// 64-expert workload it outlasts the dgrad mainloop (736 us against 440 us
// for dgrad followed by the standalone 16-warp-per-SM swiglu_bwd_quantize).
__device__ __forceinline__ void swiglu_bwd_tile_epilogue(const Params& p, const Tile& T, uint32_t tmem, int q,
                                                         int half, int lane, uint32_t acc_empty) {
    const int64_t F = p.K, W = 2 * p.K;
    uint32_t r[BN / 2];
    const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + 128 * half;
    TMEM_LD32(tbase + 0, (r + 0));
    TMEM_LD32(tbase + 32, (r + 32));
    TMEM_LD32(tbase + 64, (r + 64));
    TMEM_LD32(tbase + 96, (r + 96));
    tmem_wait_ld();
    fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(acc_empty);  // the MMA warp may start the next tile
    uint32_t dh2[BN / 4];  // dh rounded to bf16 as the plain dgrad writes it, as pairs
#pragma unroll
    for (int j = 0; j < BN / 4; ++j) dh2[j] = bf16x2_bits(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));

    const int64_t f0 = T.b_col + 128 * half;
    const int64_t rb0 = T.a_row + 32 * q;
    const __nv_bfloat16* yr = p.y1 + (rb0 + lane) * W;
    // The chunk loop stays rolled (an unrolled body would not fit the
    // instruction cache); dh2 is shifted down one chunk per pass so that the
    // body only ever reads dh2[0..15] and the array stays in registers.
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        const int64_t fc = f0 + 32 * c;
        uint32_t gw[16], uw[16];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const uint4 g4 = __ldg(reinterpret_cast<const uint4*>(yr + fc) + v);
            const uint4 u4 = __ldg(reinterpret_cast<const uint4*>(yr + F + fc) + v);
            gw[4 * v] = g4.x; gw[4 * v + 1] = g4.y; gw[4 * v + 2] = g4.z; gw[4 * v + 3] = g4.w;
            uw[4 * v] = u4.x; uw[4 * v + 1] = u4.y; uw[4 * v + 2] = u4.z; uw[4 * v + 3] = u4.w;
        }
        uint32_t dgw[16], duw[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const uint32_t dw = dh2[j];
            float dg0, du0, dg1, du1;
            swiglu_grads(bf16lo(dw), bf16lo(gw[j]), bf16lo(uw[j]), dg0, du0);
            swiglu_grads(bf16hi(dw), bf16hi(gw[j]), bf16hi(uw[j]), dg1, du1);
            dgw[j] = bf16x2_bits(dg0, dg1);
            duw[j] = bf16x2_bits(du0, du1);
        }
        if (p.side) {
            uint4* dg_out = reinterpret_cast<uint4*>(p.side + (rb0 + lane) * W + fc);
            uint4* du_out = reinterpret_cast<uint4*>(p.side + (rb0 + lane) * W + F + fc);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                dg_out[v] = make_uint4(dgw[4 * v], dgw[4 * v + 1], dgw[4 * v + 2], dgw[4 * v + 3]);
                du_out[v] = make_uint4(duw[4 * v], duw[4 * v + 1], duw[4 * v + 2], duw[4 * v + 3]);
            }
        }
        quant_block32(dgw, p, T, W, rb0, fc, lane);
        quant_block32(duw, p, T, W, rb0, F + fc, lane);
#pragma unroll
        for (int j = 0; j < BN / 4 - 16; ++j) dh2[j] = dh2[j + 16];
    }
}

// Epilogue of the SwiGLU-fused FC1 fprop (kFpropSwiglu) for one tile: the
// accumulator holds gate columns [T.b_col, +128) in TMEM columns 0..127 and
// the matching up columns in 128..255. Warp (q, half) takes rows 32q..32q+31
// (lane = row) and the 64 columns T.b_col + 64 half + [0, 64) of both halves.
// It writes y1 = bf16(acc + bias) as the plain fprop epilogue does (the
// saved FC1 output), then h = silu(g) * u from those bf16 values in the fp32
// steps of mxq_common.cuh, and quantizes h as group_quantize does: rowwise
// over the lane's two 32-column blocks, colwise over the warp's 32 rows (a
// byte-wise max of exponents across the lanes), E4M3 by the same cast.
// `release(lane)` hands the accumulator back once this warp's slice is in registers; with
// store == false (the duplicate half of a pair tile) nothing is written.
template <class Release>
__device__ __forceinline__ void swiglu_tile_epilogue(const Params& p, const Tile& T, uint32_t tmem, int q, int half,
                                                     int lane, uint8_t* epi_buf, Release release,
                                                     const CUtensorMap* tmOut, bool store = true) {
    const int64_t F = p.N / 2;
    uint32_t r[BN / 2];
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16) + 64 * half;
    TMEM_LD32(tq + 0, (r + 0));     // gate
    TMEM_LD32(tq + 32, (r + 32));
    TMEM_LD32(tq + 128, (r + 64));  // up
    TMEM_LD32(tq + 160, (r + 96));
    tmem_wait_ld();
    fence_before();
    __syncwarp();
    release(lane);  // the MMA warp may start the next tile
    if (!store) return;

    const int64_t f0 = T.b_col + 64 * half;  // first gate (and h) column of this warp

    // y1 = bf16(acc + bias): y[0, 32) gate pairs, y[32, 64) up pairs
    uint32_t y[64];
#pragma unroll
    for (int hp = 0; hp < 2; ++hp) {
        const __nv_bfloat16* bias = p.bias ? p.bias + (int64_t)T.e * p.N + hp * F + f0 : nullptr;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            uint64_t f2[4];  // accumulator pairs, plus the bias pairs in one packed add each
#pragma unroll
            for (int j = 0; j < 4; ++j)
                f2[j] = f2pack(__uint_as_float(r[64 * hp + 8 * v + 2 * j]), __uint_as_float(r[64 * hp + 8 * v + 2 * j + 1]));
            if (bias) {
                const uint4 bw = __ldg(reinterpret_cast<const uint4*>(bias) + v);
                const uint32_t ws[4] = {bw.x, bw.y, bw.z, bw.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) f2[j] = f2add(f2[j], f2pack(bf16lo(ws[j]), bf16hi(ws[j])));
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 f = f2unpack(f2[j]);
                y[32 * hp + 4 * v + j] = bf16x2_bits(f.x, f.y);
            }
        }
    }
    // y1 through four staged 32x32 boxes: gate f0, f0+32; up F+f0, F+f0+32
    const int out_row0 = (int)(T.a_row + q * 32);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        __syncwarp();
        uint4* dst = reinterpret_cast<uint4*>(epi_buf + lane * 64);
#pragma unroll
        for (int v = 0; v < 4; ++v)
            dst[v ^ ((lane >> 1) & 3)] =
                make_uint4(y[16 * b + 4 * v], y[16 * b + 4 * v + 1], y[16 * b + 4 * v + 2], y[16 * b + 4 * v + 3]);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
            const int col = (int)(b < 2 ? f0 + 32 * b : F + f0 + 32 * (b - 2));
            asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                             (uint64_t)tmOut),
                         "r"(col), "r"(out_row0), "r"(smem_u32(epi_buf))
                         : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
    }

    // h = silu(g) * u, rounded to bf16
    uint32_t hw[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float2 h2 = swiglu_h_x2(make_float2(bf16lo(y[i]), bf16hi(y[i])),
                                      make_float2(bf16lo(y[32 + i]), bf16hi(y[32 + i])));
        hw[i] = bf16x2_bits(h2.x, h2.y);
    }

    if (p.side) {
        uint4* h_out = reinterpret_cast<uint4*>(p.side + (T.a_row + q * 32 + lane) * F + f0);
#pragma unroll
        for (int v = 0; v < 8; ++v) h_out[v] = make_uint4(hw[4 * v], hw[4 * v + 1], hw[4 * v + 2], hw[4 * v + 3]);
    }

    // rowwise and colwise codes of h, two 32-column blocks
    uint32_t w0[16], w1[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        w0[i] = hw[i];
        w1[i] = hw[16 + i];
    }
    quant_block32(w0, p, T, F, T.a_row + q * 32, f0, lane);
    quant_block32(w1, p, T, F, T.a_row + q * 32, f0 + 32, lane);
}

// kPad: padded grouping (expert counts need not be multiples of 128; A's
// rowwise scales, or wgrad's colwise scales, in the per-expert padded layout).
template <int kMode, bool kPad = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmOut, Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align<1024>(smem_raw);
    // tables: offsets (E+1) [kPad: padded offsets (E+1)] expert order (E)
    int64_t* s_off = reinterpret_cast<int64_t*>(smem + TABLE_REGION);
    int64_t* s_poff = s_off + p.E + 1;
    int16_t* s_order = reinterpret_cast<int16_t*>(kPad ? s_poff + p.E + 1 : s_off + p.E + 1);
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bad = kPad ? load_offsets_padded(p.m_splits, p.E, p.M, s_off, s_poff)
                         : load_offsets(p.m_splits, p.E, p.M, s_off);
    if (bad) {
        report_status(p.status, bad);
        return;
    }
    if (kMode == kWgrad) {
        // rank experts by token count, heaviest first (ties: lower index first)
        for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
            const int64_t me = s_off[e + 1] - s_off[e];
            int rank = 0;
            for (int f = 0; f < p.E; ++f) {
                const int64_t mf = s_off[f + 1] - s_off[f];
                rank += (mf > me) || (mf == me && f < e);
            }
            s_order[rank] = (int16_t)e;
        }
    }

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_REGION);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
    const uint32_t acc_full = smem_u32(bars + 2 * STAGES), acc_empty = smem_u32(bars + 2 * STAGES + 1);
    volatile int* abort_flag = &s_abort;

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, EPI_WARPS);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmA) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmB) : "memory");
        if (p.tma_store) asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmOut) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = s_tmem;

    Sched S;
    S.init(kMode, p.M, p.N, p.K, p.E, s_off, s_order, s_poff, kPad);
    const int ncta = gridDim.x, cta = blockIdx.x;
    constexpr bool kFwd = (kMode == kFprop || kMode == kFpropSwiglu);
    const uint32_t a_mn = (kMode == kWgrad) ? 1u : 0u;
    const uint32_t b_mn = kFwd ? 0u : 1u;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            for (int64_t i = 0;; ++i) {
                const Tile T = S.get(S.pick(i, cta, ncta));
                if (!T.valid) break;
                // Per tile: first-block coordinates and scale-atom addresses; each
                // 128-deep K block then advances them by fixed strides.
                int ax, ay, bx, by, adx, ady, bdx, bdy;
                const uint8_t *sfa, *sfb0, *sfb1;  // atoms of K block 0; +512 B per block
                if (kFwd) {
                    const int64_t kbs = p.K / BK, wrow = (int64_t)T.e * p.N + T.b_col;
                    ax = 0; ay = (int)T.a_row; adx = BK; ady = 0;
                    bx = 0; by = (int)wrow; bdx = BK; bdy = 0;
                    sfa = p.sfa + (T.pa_row / 128) * kbs * 512;
                    sfb0 = p.sfb + (wrow / 128) * kbs * 512;
                    // second B box: the next 128 rows, or (SwiGLU) the up rows F further
                    sfb1 = sfb0 + (kMode == kFpropSwiglu ? (p.N / 2) / 128 : 1) * kbs * 512;
                } else if (kMode == kDgrad || kMode == kDgradSwiglu) {
                    const int64_t kbs = p.N / BK;
                    const uint8_t* wb = p.sfb + (int64_t)T.e * p.K * (p.N / 32);
                    ax = 0; ay = (int)T.a_row; adx = BK; ady = 0;
                    bx = (int)T.b_col; by = (int)((int64_t)T.e * p.N); bdx = 0; bdy = BK;
                    sfa = p.sfa + (T.pa_row / 128) * kbs * 512;
                    sfb0 = wb + (T.b_col / 128) * kbs * 512;
                    sfb1 = sfb0 + kbs * 512;
                } else {
                    const int64_t kbs = T.mp / BK;
                    const uint8_t* ab = p.sfa + p.N * T.poff / 32;
                    const uint8_t* bb = p.sfb + p.K * T.poff / 32;
                    ax = (int)T.a_row; ay = (int)T.off; adx = 0; ady = BK;
                    bx = (int)T.b_col; by = (int)T.off; bdx = 0; bdy = BK;
                    sfa = ab + (T.a_row / 128) * kbs * 512;
                    sfb0 = bb + (T.b_col / 128) * kbs * 512;
                    sfb1 = sfb0 + kbs * 512;
                }
                // the second B box: 128 rows further (K-major B) or 128 columns further (MN-major B)
                const int b2x = kFwd ? 0 : 128, b2y = kFwd ? (kMode == kFpropSwiglu ? (int)(p.N / 2) : 128) : 0;
                for (int kb = 0; kb < T.nk; ++kb) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag)) goto done_producer;
                    const uint32_t sb = smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t fb = full0 + 8 * stage;
                    mbar_expect_tx(fb, STAGE_TX);
                    tma_load_2d(sb, &tmA, fb, ax, ay);
                    tma_load_2d(sb + A_BYTES, &tmB, fb, bx, by);  // kFprop: all 256 rows
                    if (kMode != kFprop) tma_load_2d(sb + A_BYTES + 16384, &tmB, fb, bx + b2x, by + b2y);
                    const uint32_t sfs = smem_u32(smem + SF_REGION + stage * SF_STAGE_BYTES);
                    bulk_load(sfs, sfa, 512, fb);
                    bulk_load(sfs + 512, sfb0, 512, fb);
                    bulk_load(sfs + 1024, sfb1, 512, fb);
                    ax += adx; ay += ady; bx += bdx; by += bdy;
                    sfa += 512; sfb0 += 512; sfb1 += 512;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
        done_producer:;
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        // Padded wgrad: the expert's last 128-token block may hold fewer
        // tokens; the rows past them (the next expert's tokens, or zeros past
        // M) are cleared in the A tile and both B boxes by the whole warp
        // before the MMAs read the stage. Elsewhere one lane runs the loop.
        constexpr bool kClear = kPad && kMode == kWgrad;
        if (kClear || lane == 0) {
            const bool leader = (lane == 0);
            int stage = 0;
            uint32_t phase = 0, aphase = 0;
            // Descriptors of stage 0 / k-step 0; every other (stage, k) differs only in
            // the start-address field (bits 0..13, in 16-byte units), which never
            // carries because shared memory addresses stay below 256 KB.
            // K-major k-steps advance 32 bytes, MN-major k-steps 32 rows (4 KB).
            const uint32_t base = smem_u32(smem);
            const uint64_t a_desc0 = a_mn ? smem_desc(base, BK * 128, 1024, 2) : smem_desc(base, 16, 1024, 2);
            const uint64_t b_desc0 =
                b_mn ? smem_desc(base + A_BYTES, BK * 128, 1024, 2) : smem_desc(base + A_BYTES, 16, 1024, 2);
            const uint64_t sf_desc0 = smem_desc(smem_u32(smem + SF_REGION), 0, 128, 0);
            const uint32_t a_step16 = a_mn ? 4096u / 16 : 32u / 16, b_step16 = b_mn ? 4096u / 16 : 32u / 16;
            uint32_t id[BK / UMMA_K];
#pragma unroll
            for (int k = 0; k < BK / UMMA_K; ++k) id[k] = idesc(a_mn, b_mn, (uint32_t)k);
            for (int64_t i = 0;; ++i) {
                const Tile T = S.get(S.pick(i, cta, ncta));
                if (!T.valid) break;
                if (!mbar_wait(acc_empty, aphase ^ 1, abort_flag)) break;
                fence_after();
                if (T.nk == 0) {
                    if (leader) mbar_arrive(acc_full);
                } else {
                    for (int kb = 0; kb < T.nk; ++kb) {
                        if (!mbar_wait(full0 + 8 * stage, phase, abort_flag)) goto done_mma;
                        fence_after();
                        if constexpr (kClear) {
                            if (kb == T.nk - 1 && T.vk < BK) {
                                // token r of each 16 KB tile is its 128-byte row r (the swizzle stays inside a row)
                                uint8_t* st = smem + stage * STAGE_BYTES;
                                const int n16 = (BK - T.vk) * 128 / 16;
                                for (int t3 = 0; t3 < 3; ++t3) {
                                    uint4* z = reinterpret_cast<uint4*>(st + t3 * 16384 + T.vk * 128);
                                    for (int j = lane; j < n16; j += 32) z[j] = make_uint4(0u, 0u, 0u, 0u);
                                }
                                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                            }
                            __syncwarp();
                        }
                        if (leader) {
                            const uint64_t sfd = sf_desc0 + (uint64_t)(stage * (SF_STAGE_BYTES / 16));
                            tmem_cp_sf(tmem + TMEM_SFA, sfd);
                            tmem_cp_sf(tmem + TMEM_SFB, sfd + 512 / 16);
                            tmem_cp_sf(tmem + TMEM_SFB + 4, sfd + 1024 / 16);
                            const uint64_t ad = a_desc0 + (uint64_t)(stage * (STAGE_BYTES / 16));
                            const uint64_t bd = b_desc0 + (uint64_t)(stage * (STAGE_BYTES / 16));
#pragma unroll
                            for (int k = 0; k < BK / UMMA_K; ++k)
                                mma_mxf8(tmem, ad + k * a_step16, bd + k * b_step16, id[k], tmem + TMEM_SFA,
                                         tmem + TMEM_SFB, (kb | k) != 0);
                            mma_commit(empty0 + 8 * stage);
                        }
                        if (++stage == STAGES) { stage = 0; phase ^= 1; }
                    }
                    if (leader) mma_commit(acc_full);
                }
                aphase ^= 1;
            }
        done_mma:;
        }
    } else {
        // ------------------------------------------------------ epilogue
        // Warp w may read TMEM lanes 32*(w%4)..+31 (its quarter of the 128
        // accumulator rows); the two warps of a quarter split the 256 columns.
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        const int row_in_tile = q * 32 + lane;
        const int col0 = half * (BN / 2);
        uint8_t* epi_buf = smem + EPI_REGION + (warp - 2) * EPI_STAGE_BYTES;
        uint32_t aphase = 0;
        for (int64_t i = 0;; ++i) {
            const Tile T = S.get(S.pick(i, cta, ncta));
            if (!T.valid) break;
            const bool ok = mbar_wait(acc_full, aphase, abort_flag);
            __syncwarp();
            if (!ok || *abort_flag) break;
            fence_after();
            if constexpr (kMode == kFpropSwiglu) {
                swiglu_tile_epilogue(p, T, tmem, q, half, lane, epi_buf,
                                     [&](int l) { if (l == 0) mbar_arrive(acc_empty); }, &tmOut);
                aphase ^= 1;
                continue;
            }
            if constexpr (kMode == kDgradSwiglu) {
                swiglu_bwd_tile_epilogue(p, T, tmem, q, half, lane, acc_empty);
                aphase ^= 1;
                continue;
            }
            // Pull this warp's 32 x 128 slice of the accumulator into registers,
            // then hand the accumulator back to the MMA warp before storing.
            uint32_t r[BN / 2];
            const bool zero = (kMode == kWgrad && T.nk == 0);
            if (!zero) {
                const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + col0;
                TMEM_LD32(tbase + 0, (r + 0));
                TMEM_LD32(tbase + 32, (r + 32));
                TMEM_LD32(tbase + 64, (r + 64));
                TMEM_LD32(tbase + 96, (r + 96));
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int j = 0; j < BN / 2; ++j) r[j] = 0u;
            }
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);

            const int64_t row = T.a_row + row_in_tile;
            // padded grouping: a 32-row box that reaches past the expert is written row by row
            const bool box_full = !kPad || kMode == kWgrad || T.vr >= q * 32 + 32;
            if (p.tma_store && box_full) {
                // Stage 32-row boxes in this warp's buffer and write each with one
                // TMA store: a box is 32 columns (bf16) or 16 columns (fp32).
                const bool f32 = (kMode == kWgrad && !p.out_bf16);
                const int box_cols = f32 ? 16 : 32;
                const int out_row0 = (int)((kMode == kWgrad ? (int64_t)T.e * p.N : 0) + T.a_row + q * 32);
                const __nv_bfloat16* bias =
                    (kMode == kFprop && p.bias) ? p.bias + (int64_t)T.e * p.N + T.b_col + col0 : nullptr;
#pragma unroll
                for (int c = 0; c < BN / 2; c += 16) {
                    if (!f32 && (c & 31)) continue;
                    uint32_t w16[16];
                    if (f32) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) w16[j] = r[c + j];
                    } else {
                        float f[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(r[(c + j) & (BN / 2 - 1)]);
                        if (bias) {
#pragma unroll
                            for (int v = 0; v < 4; ++v) {
                                const uint4 bw = __ldg(reinterpret_cast<const uint4*>(bias + c) + v);
                                const uint32_t ws[4] = {bw.x, bw.y, bw.z, bw.w};
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    f[8 * v + 2 * j] += __uint_as_float(ws[j] << 16);
                                    f[8 * v + 2 * j + 1] += __uint_as_float(ws[j] & 0xFFFF0000u);
                                }
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            __nv_bfloat162 b2 = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
                            w16[j] = *reinterpret_cast<uint32_t*>(&b2);
                        }
                    }
                    // the previous box of this buffer must have been read out
                    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                    __syncwarp();
                    // row `lane` of the box; 16-byte chunk v sits at v ^ (row bits 1..2) (64-byte swizzle)
                    uint4* dst = reinterpret_cast<uint4*>(epi_buf + lane * 64);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v ^ ((lane >> 1) & 3)] = make_uint4(w16[4 * v], w16[4 * v + 1], w16[4 * v + 2], w16[4 * v + 3]);
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {
                        asm volatile(
                            "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                                (uint64_t)&tmOut),
                            "r"((int)(T.b_col + col0 + c)), "r"(out_row0), "r"(smem_u32(epi_buf))
                            : "memory");
                        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                    }
                    (void)box_cols;
                }
            } else if (kMode != kWgrad) {
                if (kPad && row_in_tile >= T.vr) {
                    aphase ^= 1;
                    continue;  // past the expert: nothing to write
                }
                const int64_t ldo = (kMode == kFprop) ? p.N : p.K;
                __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + row * ldo + T.b_col + col0;
                const __nv_bfloat16* bias =
                    (kMode == kFprop && p.bias) ? p.bias + (int64_t)T.e * p.N + T.b_col + col0 : nullptr;
#pragma unroll
                for (int c = 0; c < BN / 2; c += 8) {
                    float f[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) f[j] = __uint_as_float(r[c + j]);
                    if (bias) {
                        const uint4 bw = __ldg(reinterpret_cast<const uint4*>(bias + c));
                        const uint32_t ws[4] = {bw.x, bw.y, bw.z, bw.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            f[2 * j] += __uint_as_float(ws[j] << 16);
                            f[2 * j + 1] += __uint_as_float(ws[j] & 0xFFFF0000u);
                        }
                    }
                    uint32_t h[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        __nv_bfloat162 b2 = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
                        h[j] = *reinterpret_cast<uint32_t*>(&b2);
                    }
                    *reinterpret_cast<uint4*>(out + c) = make_uint4(h[0], h[1], h[2], h[3]);
                }
            } else if (!(zero && p.accumulate)) {
                // accumulate into dW: read-modify-write with plain loads and stores
                const int64_t base = ((int64_t)T.e * p.N + row) * p.K + T.b_col + col0;
                if (p.out_bf16) {
                    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + base;
#pragma unroll
                    for (int c = 0; c < BN / 2; c += 8) {
                        float f[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) f[j] = __uint_as_float(r[c + j]);
                        uint4* dst = reinterpret_cast<uint4*>(out + c);
                        if (p.accumulate) {
                            const uint4 o = *dst;
                            const uint32_t ws[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                f[2 * j] += __uint_as_float(ws[j] << 16);
                                f[2 * j + 1] += __uint_as_float(ws[j] & 0xFFFF0000u);
                            }
                        }
                        uint32_t h[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            __nv_bfloat162 b2 = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
                            h[j] = *reinterpret_cast<uint32_t*>(&b2);
                        }
                        *dst = make_uint4(h[0], h[1], h[2], h[3]);
                    }
                } else {
                    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + base);
#pragma unroll
                    for (int v = 0; v < BN / 8; ++v) {
                        float4 o = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                               __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
                        if (p.accumulate) {
                            const float4 old = dst[v];
                            o.x += old.x;
                            o.y += old.y;
                            o.z += old.z;
                            o.w += old.w;
                        }
                        dst[v] = o;
                    }
                }
            }
            aphase ^= 1;
        }
        if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        __syncwarp();
    }

    fence_before();
    __syncthreads();
    if (s_abort && threadIdx.x == 0 && p.status) atomicOr(p.status, MXQ_STATUS_WAIT_TIMEOUT);
    if (warp == 1) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

// ============================================================ two-SM tiles
// The plain fprop / dgrad / wgrad (128-aligned experts) run on CTA pairs:
// a cluster of two CTAs on two SMs computes one 256 x 256 output tile with
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 32). Each CTA stages its own
// 128 rows of A and its own 128-wide half of B (plain TMA loads into its own
// shared memory, completing on the leader CTA's stage barrier), so a
// 32 KB stage covers as many MMA cycles as a 48 KB stage of the one-SM tile
// and the ring is six stages deep. The leader (cluster rank 0) issues the
// scale copies and MMAs for both SMs; every CTA holds the accumulator of its
// own 128 rows (all 256 columns) in its TMEM and drains it with its own eight
// epilogue warps. Semantics used (PTX ISA, tcgen05 with .cta_group::2):
// one warp in each CTA allocates the 512 TMEM columns collectively (both
// get the same address); a tcgen05.cp issued by the leader copies each CTA's
// shared memory into that CTA's TMEM at the same addresses; each CTA's TMEM
// holds the scale factors of its own 128 A rows and of all 256 B columns;
// tcgen05.commit with .multicast::cluster arrives on the barrier at the same
// offset in both CTAs.
//
// Row tiles of fprop / dgrad pair 256 rows of one expert (both halves use
// the same expert's weights); when an expert holds an odd number of 128-row
// blocks, its last pair tile's second CTA recomputes the first CTA's rows and
// does not store them. wgrad tiles pair 256 rows of N with 256 columns of K
// of one expert.
//
// Clusters take tiles in rounds of one tile each, serpentine within a round.
// wgrad's tiles are listed heaviest expert first, and the rounds are walked
// alternately from the two ends of that list (first, last, second, second
// last, ...): every cluster then interleaves light tiles, whose time is their
// dW stores, with heavy tiles, whose time is their MMAs.
namespace pair {

constexpr int PSTAGES = 6;
constexpr int PSTAGE_BYTES = 32768;               // A 16 KB + B half 16 KB
constexpr int PSF_BYTES = 1536;                   // scale atoms: A (512), B both halves (2 x 512)
constexpr uint32_t PTX_CTA = PSTAGE_BYTES + PSF_BYTES;
constexpr int PSF_REGION = PSTAGES * PSTAGE_BYTES;
constexpr int PBAR_REGION = PSF_REGION + PSTAGES * PSF_BYTES;
constexpr int PEPI_REGION = (PBAR_REGION + 256 + 511) / 512 * 512;
constexpr int PTABLE_REGION = PEPI_REGION + EPI_WARPS * EPI_STAGE_BYTES;
constexpr int MAX_EXPERTS = 512;
// producer, MMA, 8 epilogue warps, and one warp that writes the zero dW tiles of empty experts
constexpr int PAIR_THREADS = NUM_THREADS + 32;
__host__ __device__ constexpr int smem_bytes(int E) { return 1024 + PTABLE_REGION + 8 * (E + 1) + 4 * (E + 1); }
static_assert(smem_bytes(MAX_EXPERTS) <= 232448, "shared memory over the per-block limit");
static_assert(PEPI_REGION % 512 == 0, "the 64-byte swizzle of the staging boxes repeats every 512 bytes");

__device__ __forceinline__ uint32_t cta_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// shared::cluster address of the variable at shared::cta address `a` in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
// Arrive on a barrier of the other CTA without a cluster-scope release: the callers only need
// the arrive to follow their completed tcgen05.ld (tcgen05.wait::ld), which it does in program
// order. A release at cluster scope costs about 1.5k cycles here, a relaxed arrive about 65.
__device__ __forceinline__ void arrive_remote_relaxed(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}
// TMA tile load into this CTA's shared memory, completing on the leader's barrier
__device__ __forceinline__ void tma_load_pair(uint32_t dst, const CUtensorMap* map, uint32_t lead_bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
        "%4}], [%2];" ::"r"(dst),
        "l"((uint64_t)map), "r"(lead_bar), "r"(x), "r"(y)
        : "memory");
}
// Non-blocking test of two barrier phases at once: both test_waits issue before either result is
// used, so a pair of ready stages costs the issuing thread one barrier latency, not two.
__device__ __forceinline__ bool mbar_test2(uint32_t a, uint32_t pa, uint32_t b, uint32_t pb) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q, [%3], %4;\n\t"
        "and.pred p, p, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(a), "r"(pa), "r"(b), "r"(pb)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint32_t idesc_pair(uint32_t a_mn, uint32_t b_mn, uint32_t sf_id) {
    return (sf_id << 4) | (a_mn << 15) | (b_mn << 16) | ((uint32_t)(256 >> 3) << 17) | (1u << 23) |
           ((uint32_t)(256 >> 4) << 24) | (sf_id << 29);
}
__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t sfa,
                                         uint32_t sfb, uint32_t accum) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a), "l"(b), "r"(id), "r"(accum), "r"(sfa), "r"(sfb)
        : "memory");
}
__device__ __forceinline__ void cp_sf_pair(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// arrive on the barrier at this offset in both CTAs once the leader's prior tcgen05 work completes
__device__ __forceinline__ void commit_pair(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                     bar),
                 "h"((uint16_t)3)
                 : "memory");
}

// One pair tile as seen by CTA `rank`.
struct PTile {
    bool valid;
    int e;
    int64_t off, me;
    int nk;           // 128-deep K blocks
    int64_t a0;       // fprop/dgrad: this CTA's first A (token) row; wgrad: its first N row
    int64_t out_row;  // first output row of this CTA (dW: e*N + N row)
    int64_t c0;       // first output column of the tile (256 wide)
    bool store;       // this CTA writes its rows (false: the duplicate half of an odd row block)
};

struct PSched {
    int mode;
    int64_t M, N, K;
    int E;
    const int64_t* off;   // token offsets (E+1)
    const int32_t* aux;   // fprop/dgrad: pair row-tile offsets (E+1); wgrad: experts heaviest first (E)
    int64_t tiles_n, total;
    uint32_t rank;

    __device__ int64_t pick(int64_t i, int c, int nc) const {
        const int64_t base = i * nc;
        return (i & 1) ? base + (nc - 1 - c) : base + c;
    }
    // wgrad walk: step i takes round i/2 of the heaviest-first list when i is even, round
    // rounds-1-i/2 when odd (a round's slot past the last tile is invalid and skipped)
    __device__ int64_t pick_alt(int64_t i, int c, int nc, int64_t rounds) const {
        return pick((i & 1) ? rounds - 1 - (i >> 1) : (i >> 1), c, nc);
    }
    __device__ PTile get(int64_t t) const {
        PTile T;
        T.valid = t < total;
        if (!T.valid) return T;
        if (mode != kWgrad) {
            const int64_t prt = t / tiles_n, nt = t % tiles_n;
            int lo = 0, hi = E - 1;  // first e with aux[e + 1] > prt
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (aux[mid + 1] > prt) hi = mid;
                else lo = mid + 1;
            }
            T.e = lo;
            T.off = off[lo];
            T.me = off[lo + 1] - T.off;
            const int64_t r0 = T.off + 256 * (prt - aux[lo]);
            const int64_t left = T.off + T.me - r0;  // rows of the expert from r0 on (128 or >= 256)
            T.store = left > 128 * (int64_t)rank;
            T.a0 = T.store ? r0 + 128 * rank : r0;
            T.out_row = T.a0;
            T.c0 = nt * (mode == kFpropSwiglu ? 128 : 256);  // SwiGLU: 128 gate columns (and their up columns)
            T.nk = (int)((mode == kDgrad ? N : K) / BK);
        } else {
            const int64_t ei = t / tiles_n, r = t % tiles_n;
            // consecutive tiles of an expert share the block of the wider operand and step through
            // the narrower one, so the wider colwise copy (dY's N or X's K columns) is read once
            const int64_t nt = N / 256, kt = K / 256;
            const int64_t nb = N <= K ? r % nt : r / kt, kb = N <= K ? r / nt : r % kt;
            T.e = aux[ei];
            T.off = off[T.e];
            T.me = off[T.e + 1] - T.off;
            T.a0 = nb * 256 + 128 * rank;
            T.out_row = (int64_t)T.e * N + T.a0;
            T.c0 = kb * 256;
            T.nk = (int)(T.me / BK);
            T.store = true;
        }
        return T;
    }
};

template <int kMode>
__global__ void __launch_bounds__(PAIR_THREADS, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                             const __grid_constant__ CUtensorMap tmOut, Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align<1024>(smem_raw);
    int64_t* s_off = reinterpret_cast<int64_t*>(smem + PTABLE_REGION);
    int32_t* s_aux = reinterpret_cast<int32_t*>(s_off + p.E + 1);
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cta_rank();
    const bool leader = rank == 0;
    // every CTA validates the same m_splits; a bad split stops both CTAs of every pair before any
    // cluster-wide step
    const int bad = load_offsets(p.m_splits, p.E, p.M, s_off);
    if (bad) {
        report_status(p.status, bad);
        return;
    }
    if (kMode == kWgrad) {
        for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
            const int64_t me = s_off[e + 1] - s_off[e];
            int rk = 0;
            for (int f = 0; f < p.E; ++f) {
                const int64_t mf = s_off[f + 1] - s_off[f];
                rk += (mf > me) || (mf == me && f < e);
            }
            s_aux[rk] = e;
        }
    } else if (threadIdx.x < 32) {
        // exclusive prefix of ceil(m_e / 256), the pair row tiles of each expert
        const int per = (p.E + 31) / 32;
        const int lo = min(p.E, lane * per), hi = min(p.E, lo + per);
        int32_t local = 0;
        for (int e = lo; e < hi; ++e) local += (int32_t)((s_off[e + 1] - s_off[e] + 255) / 256);
        int32_t incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        int32_t run = incl - local;
        for (int e = lo; e < hi; ++e) {
            s_aux[e] = run;
            run += (int32_t)((s_off[e + 1] - s_off[e] + 255) / 256);
        }
        if (lane == 31) s_aux[p.E] = incl;
    }

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + PBAR_REGION);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + PSTAGES);
    const uint32_t acc_full = smem_u32(bars + 2 * PSTAGES), acc_empty = smem_u32(bars + 2 * PSTAGES + 1);
    volatile int* abort_flag = &s_abort;
    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int st = 0; st < PSTAGES; ++st) {
            mbar_init(full0 + 8 * st, 1);
            mbar_init(empty0 + 8 * st, 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 2 * EPI_WARPS);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmA) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmB) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmSA) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmSB) : "memory");
        if (p.tma_store) asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmOut) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers exist before any load completes on the leader's
    fence_after();
    const uint32_t tmem = s_tmem;

    PSched S;
    S.mode = kMode; S.M = p.M; S.N = p.N; S.K = p.K; S.E = p.E; S.off = s_off; S.aux = s_aux; S.rank = rank;
    if (kMode == kFprop || kMode == kFpropSwiglu) { S.tiles_n = p.N / 256; S.total = (int64_t)s_aux[p.E] * S.tiles_n; }
    else if (kMode == kDgrad) { S.tiles_n = p.K / 256; S.total = (int64_t)s_aux[p.E] * S.tiles_n; }
    else { S.tiles_n = (p.N / 256) * (p.K / 256); S.total = (int64_t)p.E * S.tiles_n; }
    const int ncl = gridDim.x / 2, cl = blockIdx.x / 2;
    constexpr bool kAlt = kMode == kWgrad;
    const int64_t rounds = (S.total + ncl - 1) / ncl;
    // the i-th tile of this cluster's walk (invalid: none in that slot)
    auto walk = [&](int64_t i) -> PTile { return S.get(kAlt ? S.pick_alt(i, cl, ncl, rounds) : S.pick(i, cl, ncl)); };
    const uint32_t a_mn = (kMode == kWgrad) ? 1u : 0u;
    const uint32_t b_mn = (kMode == kFprop || kMode == kFpropSwiglu) ? 0u : 1u;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            for (int64_t i = 0;; ++i) {
                if (kAlt && i >= rounds) break;
                const PTile T = walk(i);
                if (!T.valid) {
                    if (kAlt) continue;
                    break;
                }
                int ax, ay, bx, by, adx, ady, bdx, bdy;
                int sa, sb0, sb1;  // scale atom rows (512 B each) of K block 0; +1 per block
                if (kMode == kFprop) {
                    const int64_t kbs = p.K / BK, wrow = (int64_t)T.e * p.N + T.c0;
                    ax = 0; ay = (int)T.a0; adx = BK; ady = 0;
                    bx = 0; by = (int)(wrow + 128 * rank); bdx = BK; bdy = 0;
                    sa = (int)((T.a0 / 128) * kbs);
                    sb0 = (int)((wrow / 128) * kbs);
                    sb1 = sb0 + (int)kbs;
                } else if (kMode == kFpropSwiglu) {
                    // CTA 0 stages 128 gate rows of W1, CTA 1 the matching up rows F further: the
                    // accumulator's columns 0..127 are gate, 128..255 up, for the same 128 columns of F
                    const int64_t kbs = p.K / BK, grow = (int64_t)T.e * p.N + T.c0, urow = grow + p.N / 2;
                    ax = 0; ay = (int)T.a0; adx = BK; ady = 0;
                    bx = 0; by = (int)(rank ? urow : grow); bdx = BK; bdy = 0;
                    sa = (int)((T.a0 / 128) * kbs);
                    sb0 = (int)((grow / 128) * kbs);
                    sb1 = (int)((urow / 128) * kbs);
                } else if (kMode == kDgrad) {
                    const int64_t kbs = p.N / BK;
                    const int64_t wb = (int64_t)T.e * (p.K / 128) * kbs;  // expert e's colwise atoms
                    ax = 0; ay = (int)T.a0; adx = BK; ady = 0;
                    bx = (int)(T.c0 + 128 * rank); by = (int)((int64_t)T.e * p.N); bdx = 0; bdy = BK;
                    sa = (int)((T.a0 / 128) * kbs);
                    sb0 = (int)(wb + (T.c0 / 128) * kbs);
                    sb1 = sb0 + (int)kbs;
                } else {
                    const int64_t kbs = T.me / BK;
                    const int64_t ab = (p.N / 128) * (T.off / 128), bb = (p.K / 128) * (T.off / 128);
                    ax = (int)T.a0; ay = (int)T.off; adx = 0; ady = BK;
                    bx = (int)(T.c0 + 128 * rank); by = (int)T.off; bdx = 0; bdy = BK;
                    sa = (int)(ab + (T.a0 / 128) * kbs);
                    sb0 = (int)(bb + (T.c0 / 128) * kbs);
                    sb1 = sb0 + (int)kbs;
                }
                for (int kb = 0; kb < T.nk; ++kb) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag)) goto done_producer;
                    const uint32_t sbuf = smem_u32(smem + stage * PSTAGE_BYTES);
                    const uint32_t fb = full0 + 8 * stage;
                    if (leader) mbar_expect_tx(fb, 2 * PTX_CTA);
                    const uint32_t lead = mapa(fb, 0);
                    tma_load_pair(sbuf, &tmA, lead, ax, ay);
                    tma_load_pair(sbuf + 16384, &tmB, lead, bx, by);
                    const uint32_t sfs = smem_u32(smem + PSF_REGION + stage * PSF_BYTES);
                    tma_load_pair(sfs, &tmSA, lead, 0, sa + kb);
                    tma_load_pair(sfs + 512, &tmSB, lead, 0, sb0 + kb);
                    tma_load_pair(sfs + 1024, &tmSB, lead, 0, sb1 + kb);
                    ax += adx; ay += ady; bx += bdx; by += bdy;
                    if (++stage == PSTAGES) { stage = 0; phase ^= 1; }
                }
            }
        done_producer:;
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer (leader only)
        if (leader && lane == 0) {
            int stage = 0;
            uint32_t phase = 0, aphase = 0;
            const uint32_t base = smem_u32(smem);
            const uint64_t a_desc0 = a_mn ? smem_desc(base, BK * 128, 1024, 2) : smem_desc(base, 16, 1024, 2);
            const uint64_t b_desc0 =
                b_mn ? smem_desc(base + 16384, BK * 128, 1024, 2) : smem_desc(base + 16384, 16, 1024, 2);
            const uint64_t sf_desc0 = smem_desc(smem_u32(smem + PSF_REGION), 0, 128, 0);
            const uint32_t a_step16 = a_mn ? 4096u / 16 : 32u / 16, b_step16 = b_mn ? 4096u / 16 : 32u / 16;
            uint32_t id[BK / UMMA_K];
#pragma unroll
            for (int k = 0; k < BK / UMMA_K; ++k) id[k] = idesc_pair(a_mn, b_mn, (uint32_t)k);
            for (int64_t i = 0;; ++i) {
                if (kAlt && i >= rounds) break;
                const PTile T = walk(i);
                if (!T.valid) {
                    if (kAlt) continue;
                    break;
                }
                if (T.nk == 0) continue;  // empty wgrad expert: the epilogues write zeros without the accumulator
                if (!mbar_wait(acc_empty, aphase ^ 1, abort_flag)) break;
                fence_after();
                // K blocks in pairs: one barrier test per two stages (eight MMAs). Any wait on
                // this thread between MMAs idles the tensor pipe for about its latency.
                for (int kb = 0; kb < T.nk; kb += 2) {
                    const int n2 = (kb + 1 < T.nk) ? 2 : 1;
                    const int st1 = (stage + 1 == PSTAGES) ? 0 : stage + 1;
                    const uint32_t ph1 = (st1 == 0) ? (phase ^ 1) : phase;
                    const bool ready = n2 == 2 ? mbar_test2(full0 + 8 * stage, phase, full0 + 8 * st1, ph1)
                                               : mbar_try(full0 + 8 * stage, phase);
                    if (!ready) {
                        if (!mbar_wait(full0 + 8 * stage, phase, abort_flag)) goto done_mma;
                        if (n2 == 2 && !mbar_wait(full0 + 8 * st1, ph1, abort_flag)) goto done_mma;
                    }
                    fence_after();
                    for (int h = 0; h < n2; ++h) {
                        const uint64_t sfd = sf_desc0 + (uint64_t)(stage * (PSF_BYTES / 16));
                        cp_sf_pair(tmem + TMEM_SFA, sfd);
                        cp_sf_pair(tmem + TMEM_SFB, sfd + 512 / 16);
                        cp_sf_pair(tmem + TMEM_SFB + 4, sfd + 1024 / 16);
                        const uint64_t ad = a_desc0 + (uint64_t)(stage * (PSTAGE_BYTES / 16));
                        const uint64_t bd = b_desc0 + (uint64_t)(stage * (PSTAGE_BYTES / 16));
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k)
                            mma_pair(tmem, ad + k * a_step16, bd + k * b_step16, id[k], tmem + TMEM_SFA,
                                     tmem + TMEM_SFB, ((kb + h) | k) != 0);
                        commit_pair(empty0 + 8 * stage);
                        if (++stage == PSTAGES) { stage = 0; phase ^= 1; }
                    }
                }
                commit_pair(acc_full);
                aphase ^= 1;
            }
        done_mma:;
        }
    } else if (warp == 2 + EPI_WARPS) {
        // ------------------------------------------------------ zero dW of empty experts (wgrad)
        // Plain coalesced stores, independent of the accumulator pipeline, so that these writes
        // overlap the MMAs of the heavy experts' tiles instead of queueing behind their epilogues.
        if (kMode == kWgrad && !p.accumulate) {
            const int64_t esz = p.out_bf16 ? 2 : 4;
            const int64_t row_bytes = 256 * esz, vec_per_row = row_bytes / 16;
            uint8_t* out = static_cast<uint8_t*>(p.out);
            for (int64_t i = 0;; ++i) {
                if (kAlt && i >= rounds) break;
                const PTile T = walk(i);
                if (!T.valid) {
                    if (kAlt) continue;
                    break;
                }
                if (T.nk != 0) continue;
                uint8_t* base = out + (T.out_row * p.K + T.c0) * esz;
                for (int64_t v = lane; v < 128 * vec_per_row; v += 32) {
                    const int64_t rr = v / vec_per_row, cc = v % vec_per_row;
                    *reinterpret_cast<uint4*>(base + rr * p.K * esz + cc * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
        }
    } else {
        // ------------------------------------------------------ epilogue (both CTAs, own 128 rows)
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        const int col0 = half * (BN / 2);
        uint8_t* epi_buf = smem + PEPI_REGION + (warp - 2) * EPI_STAGE_BYTES;
        const uint32_t lead_acc_empty = mapa(acc_empty, 0);
        uint32_t aphase = 0;
        for (int64_t i = 0;; ++i) {
            if (kAlt && i >= rounds) break;
            const PTile T = walk(i);
            if (!T.valid) {
                if (kAlt) continue;
                break;
            }
            if constexpr (kMode == kFpropSwiglu) {
                const bool ok = mbar_wait(acc_full, aphase, abort_flag);
                __syncwarp();
                if (!ok || *abort_flag) break;
                fence_after();
                Tile ST;
                ST.a_row = T.out_row;
                ST.b_col = T.c0;
                ST.e = T.e;
                ST.off = T.off;
                ST.me = T.me;
                swiglu_tile_epilogue(p, ST, tmem, q, half, lane, epi_buf,
                                     [&](int l) {
                                         if (l == 0) {
                                             if (leader) mbar_arrive(acc_empty);
                                             else arrive_remote_relaxed(lead_acc_empty);
                                         }
                                     },
                                     &tmOut, T.store);
                aphase ^= 1;
                continue;
            }
            uint32_t r[BN / 2];
            if (kMode == kWgrad && T.nk == 0) continue;  // an empty expert: written by the zero warp
            {
                const bool ok = mbar_wait(acc_full, aphase, abort_flag);
                __syncwarp();
                if (!ok || *abort_flag) break;
                fence_after();
                const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + col0;
                TMEM_LD32(tbase + 0, (r + 0));
                TMEM_LD32(tbase + 32, (r + 32));
                TMEM_LD32(tbase + 64, (r + 64));
                TMEM_LD32(tbase + 96, (r + 96));
                tmem_wait_ld();
                fence_before();
                __syncwarp();
                // this warp's slice is in registers: the leader may overwrite the accumulator
                if (lane == 0) {
                    if (leader) mbar_arrive(acc_empty);
                    else arrive_remote_relaxed(lead_acc_empty);
                }
                aphase ^= 1;
            }
            if (!T.store) continue;
            const int64_t row = T.out_row + q * 32 + lane;
            if (p.tma_store) {
                const bool f32 = (kMode == kWgrad && !p.out_bf16);
                const int out_row0 = (int)(T.out_row + q * 32);
                const __nv_bfloat16* bias =
                    (kMode == kFprop && p.bias) ? p.bias + (int64_t)T.e * p.N + T.c0 + col0 : nullptr;
#pragma unroll
                for (int c = 0; c < BN / 2; c += 16) {
                    if (!f32 && (c & 31)) continue;
                    uint32_t w16[16];
                    if (f32) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) w16[j] = r[c + j];
                    } else {
                        float f[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(r[(c + j) & (BN / 2 - 1)]);
                        if (bias) {
#pragma unroll
                            for (int v = 0; v < 4; ++v) {
                                const uint4 bw = __ldg(reinterpret_cast<const uint4*>(bias + c) + v);
                                const uint32_t ws[4] = {bw.x, bw.y, bw.z, bw.w};
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    f[8 * v + 2 * j] += __uint_as_float(ws[j] << 16);
                                    f[8 * v + 2 * j + 1] += __uint_as_float(ws[j] & 0xFFFF0000u);
                                }
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) w16[j] = bf16x2_bits(f[2 * j], f[2 * j + 1]);
                    }
                    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                    __syncwarp();
                    uint4* dst = reinterpret_cast<uint4*>(epi_buf + lane * 64);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v ^ ((lane >> 1) & 3)] = make_uint4(w16[4 * v], w16[4 * v + 1], w16[4 * v + 2], w16[4 * v + 3]);
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {
                        asm volatile(
                            "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                                (uint64_t)&tmOut),
                            "r"((int)(T.c0 + col0 + c)), "r"(out_row0), "r"(smem_u32(epi_buf))
                            : "memory");
                        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                    }
                }
            } else if (kMode == kWgrad) {
                // accumulate into dW: read-modify-write with plain loads and stores
                const int64_t base = row * p.K + T.c0 + col0;
                if (p.out_bf16) {
                    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + base;
#pragma unroll
                    for (int c = 0; c < BN / 2; c += 8) {
                        float f[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) f[j] = __uint_as_float(r[c + j]);
                        uint4* dst = reinterpret_cast<uint4*>(out + c);
                        const uint4 o = *dst;
                        const uint32_t ws[4] = {o.x, o.y, o.z, o.w};
                        uint32_t h[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            h[j] = bf16x2_bits(f[2 * j] + __uint_as_float(ws[j] << 16),
                                               f[2 * j + 1] + __uint_as_float(ws[j] & 0xFFFF0000u));
                        *dst = make_uint4(h[0], h[1], h[2], h[3]);
                    }
                } else {
                    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + base);
#pragma unroll
                    for (int v = 0; v < BN / 8; ++v) {
                        const float4 old = dst[v];
                        dst[v] = make_float4(__uint_as_float(r[4 * v]) + old.x, __uint_as_float(r[4 * v + 1]) + old.y,
                                             __uint_as_float(r[4 * v + 2]) + old.z,
                                             __uint_as_float(r[4 * v + 3]) + old.w);
                    }
                }
            }
        }
        if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        __syncwarp();
    }

    fence_before();
    __syncthreads();
    if (s_abort && threadIdx.x == 0 && p.status) atomicOr(p.status, MXQ_STATUS_WAIT_TIMEOUT);
    cluster_sync();  // the leader's MMAs have read this CTA's shared memory for the last time
    if (warp == 1) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

}  // namespace pair

// ------------------------------------------------------------------ host side
// 2-D uint8 tensor (outer rows x inner cols, row-major), box 128 x 128, 128B swizzle.
static bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols) {
    return encode_tmap_2d(m, base, rows, cols, 1, 128, 128, 128);
}

}  // namespace gemm

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

bool encode_tmap_2d(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int elem_bytes, int box_cols,
                    int box_rows, int swizzle_bytes) {
    EncodeTiledFn enc = get_encode();
    if (!enc || !base) return false;
    if (swizzle_bytes != 0 && swizzle_bytes != 64 && swizzle_bytes != 128) return false;
    if (swizzle_bytes && box_cols * elem_bytes != swizzle_bytes) return false;
    const CUtensorMapSwizzle sw = swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                        : CU_TENSOR_MAP_SWIZZLE_NONE;
    const CUtensorMapDataType dt = elem_bytes == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_UINT32;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(cols * elem_bytes)};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               sw,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace gemm {

static int sm_count() {
    int dev = 0, v = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    return v;
}

}  // namespace gemm

namespace gemm {

// The plain fprop / dgrad / wgrad on 128-aligned experts run on CTA pairs when the shapes allow:
// 256-wide output tiles along N (fprop, wgrad) and K (dgrad, wgrad), at most pair::MAX_EXPERTS
// experts (the offset tables' shared-memory budget).
static bool pair_eligible(const GemmCall& c) {
    if (c.pad || c.E > pair::MAX_EXPERTS) return false;
    if (c.mode == kFprop || c.mode == kFpropSwiglu) return c.N % 256 == 0;
    if (c.mode == kDgrad) return c.K % 256 == 0;
    if (c.mode == kWgrad) return c.N % 256 == 0 && c.K % 256 == 0;
    return false;
}

// 2-D uint32 view of a swizzled scale buffer: one 512-byte atom (128 words) per row, box = one atom.
static bool make_atom_map(CUtensorMap* m, const void* base, int64_t bytes) {
    return encode_tmap_2d(m, base, bytes / 512, 128, 4, 128, 1, 0);
}

// Largest number of co-resident CTA pairs of the pair kernel for `mode` on the current device.
template <int kMode>
static int max_pairs() {
    static std::atomic<int> cache[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64) {
        const int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2 * (sm_count() / 2), 1, 1);
    cfg.blockDim = dim3(pair::PAIR_THREADS, 1, 1);
    cfg.dynamicSmemBytes = pair::smem_bytes(pair::MAX_EXPERTS);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (void*)pair::grouped_gemm_pair_kernel<kMode>, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = sm_count() / 2;
    }
    if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

template <int kMode>
static cudaError_t launch_pair(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa,
                               const CUtensorMap& tsb, const CUtensorMap& to, const Params& p, int64_t tiles,
                               cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(pair::grouped_gemm_pair_kernel<kMode>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         pair::smem_bytes(pair::MAX_EXPERTS));
    if (e != cudaSuccess) return e;
    const int pairs = (int)std::min<int64_t>(tiles, max_pairs<kMode>());
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.blockDim = dim3(pair::PAIR_THREADS, 1, 1);
    cfg.dynamicSmemBytes = pair::smem_bytes(p.E);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, pair::grouped_gemm_pair_kernel<kMode>, ta, tb, tsa, tsb, to, p);
}

static cudaError_t run_pair(const GemmCall& c, const Params& p, const CUtensorMap& to, cudaStream_t s) {
    // pair tiles, an upper bound of the device-side count (row tiles per expert are rounded up)
    int64_t tiles;
    if (c.mode == kFprop || c.mode == kFpropSwiglu) tiles = (c.M / 256 + c.E) * (c.N / 256);
    else if (c.mode == kDgrad) tiles = (c.M / 256 + c.E) * (c.K / 256);
    else tiles = (int64_t)c.E * (c.N / 256) * (c.K / 256);
    CUtensorMap ta, tb, tsa, tsb;
    bool ok;
    if (c.mode == kFprop || c.mode == kFpropSwiglu)
        ok = make_map(&ta, c.a_data, c.M, c.K) && make_map(&tb, c.b_data, (int64_t)c.E * c.N, c.K) &&
             make_atom_map(&tsa, c.a_scale, c.M * c.K / 32) && make_atom_map(&tsb, c.b_scale, (int64_t)c.E * c.N * c.K / 32);
    else if (c.mode == kDgrad)
        ok = make_map(&ta, c.a_data, c.M, c.N) && make_map(&tb, c.b_data, (int64_t)c.E * c.N, c.K) &&
             make_atom_map(&tsa, c.a_scale, c.M * c.N / 32) && make_atom_map(&tsb, c.b_scale, (int64_t)c.E * c.N * c.K / 32);
    else
        ok = make_map(&ta, c.a_data, c.M, c.N) && make_map(&tb, c.b_data, c.M, c.K) &&
             make_atom_map(&tsa, c.a_scale, c.M * c.N / 32) && make_atom_map(&tsb, c.b_scale, c.M * c.K / 32);
    if (!ok) return cudaErrorInvalidValue;
    if (c.mode == kFprop) return launch_pair<kFprop>(ta, tb, tsa, tsb, to, p, tiles, s);
    if (c.mode == kFpropSwiglu) return launch_pair<kFpropSwiglu>(ta, tb, tsa, tsb, to, p, tiles, s);
    if (c.mode == kDgrad) return launch_pair<kDgrad>(ta, tb, tsa, tsb, to, p, tiles, s);
    return launch_pair<kWgrad>(ta, tb, tsa, tsb, to, p, tiles, s);
}

}  // namespace gemm

cudaError_t run_grouped_gemm(const GemmCall& c, cudaStream_t s) {
    using namespace gemm;
    cudaError_t attr_err;
    if (c.mode == kFpropSwiglu)
        attr_err = cudaFuncSetAttribute(grouped_gemm_kernel<kFpropSwiglu>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes(MXQ_MAX_EXPERTS));
    else if (c.mode == kDgradSwiglu)
        attr_err = cudaFuncSetAttribute(grouped_gemm_kernel<kDgradSwiglu>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes(MXQ_MAX_EXPERTS));
    else if (c.mode == kFprop)
        attr_err = cudaFuncSetAttribute(grouped_gemm_kernel<kFprop>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        smem_bytes(MXQ_MAX_EXPERTS));
    else if (c.mode == kDgrad)
        attr_err = cudaFuncSetAttribute(grouped_gemm_kernel<kDgrad>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        smem_bytes(MXQ_MAX_EXPERTS));
    else
        attr_err = cudaFuncSetAttribute(grouped_gemm_kernel<kWgrad>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        smem_bytes(MXQ_MAX_EXPERTS));
    if (attr_err != cudaSuccess) return attr_err;
    if (c.pad) {
        const int sm = smem_bytes_padded(MAX_EXPERTS_PADDED);
        attr_err = c.mode == kFprop   ? cudaFuncSetAttribute(grouped_gemm_kernel<kFprop, true>,
                                                             cudaFuncAttributeMaxDynamicSharedMemorySize, sm)
                   : c.mode == kDgrad ? cudaFuncSetAttribute(grouped_gemm_kernel<kDgrad, true>,
                                                             cudaFuncAttributeMaxDynamicSharedMemorySize, sm)
                                      : cudaFuncSetAttribute(grouped_gemm_kernel<kWgrad, true>,
                                                             cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
        if (attr_err != cudaSuccess) return attr_err;
    }

    // padded grouping: the row-tile count is known on the device only; the
    // grid is sized for its bound round_up(M, 128) / 128 + E
    const int64_t row_tiles = c.pad ? (c.M + BM - 1) / BM + c.E : c.M / BM;
    int64_t tiles;
    if (c.mode == kFprop || c.mode == kFpropSwiglu) tiles = (c.M == 0 ? 0 : row_tiles) * (c.N / BN);
    else if (c.mode == kDgrad || c.mode == kDgradSwiglu) tiles = (c.M == 0 ? 0 : row_tiles) * (c.K / BN);
    else tiles = (int64_t)c.E * (c.N / BM) * (c.K / BN);
    if (tiles == 0) return cudaSuccess;
    if (c.mode == kWgrad && c.M == 0) {
        // no tokens: every expert is empty, dW = 0 (unchanged when accumulating)
        if (c.accumulate) return cudaSuccess;
        return cudaMemsetAsync(c.out, 0, (size_t)c.E * c.N * c.K * (c.out_bf16 ? 2 : 4), s);
    }

    CUtensorMap ta, tb;
    bool ok;
    if (c.mode == kFprop || c.mode == kFpropSwiglu) {
        // fprop: B's 256 K-major rows in one box (one TMA operation per stage fewer); the SwiGLU
        // variant loads its gate and up rows as two 128-row boxes
        ok = make_map(&ta, c.a_data, c.M, c.K) &&
             (c.mode == kFprop ? encode_tmap_2d(&tb, c.b_data, (int64_t)c.E * c.N, c.K, 1, 128, 256, 128)
                               : make_map(&tb, c.b_data, (int64_t)c.E * c.N, c.K));
    } else if (c.mode == kDgrad || c.mode == kDgradSwiglu) {
        ok = make_map(&ta, c.a_data, c.M, c.N) && make_map(&tb, c.b_data, (int64_t)c.E * c.N, c.K);
    } else {
        ok = make_map(&ta, c.a_data, c.M, c.N) && make_map(&tb, c.b_data, c.M, c.K);
    }
    if (!ok) return cudaErrorInvalidValue;

    // Output boxes for the TMA-store epilogue (not used when accumulating).
    CUtensorMap to;
    memset(&to, 0, sizeof(to));
    const int tma_store = !c.accumulate && c.mode != kDgradSwiglu;  // dh never leaves the chip there
    if (tma_store) {
        // 64-byte boxes rows, 64-byte swizzle: the epilogue's staging writes are bank-conflict free
        if (c.mode == kFprop || c.mode == kFpropSwiglu) ok = encode_tmap_2d(&to, c.out, c.M, c.N, 2, 32, 32, 64);
        else if (c.mode == kDgrad) ok = encode_tmap_2d(&to, c.out, c.M, c.K, 2, 32, 32, 64);
        else if (c.out_bf16) ok = encode_tmap_2d(&to, c.out, (int64_t)c.E * c.N, c.K, 2, 32, 32, 64);
        else ok = encode_tmap_2d(&to, c.out, (int64_t)c.E * c.N, c.K, 4, 16, 32, 64);
        if (!ok) return cudaErrorInvalidValue;
    }

    const bool use_pair = pair_eligible(c);

    Params p{};
    p.mode = c.mode;
    p.M = c.M;
    p.N = c.N;
    p.K = c.K;
    p.E = c.E;
    p.m_splits = c.m_splits;
    p.sfa = static_cast<const uint8_t*>(c.a_scale);
    p.sfb = static_cast<const uint8_t*>(c.b_scale);
    p.bias = static_cast<const __nv_bfloat16*>(c.bias);
    p.out = c.out;
    p.accumulate = c.accumulate;
    p.out_bf16 = c.out_bf16;
    p.tma_store = tma_store;
    p.status = c.status;
    p.q_row = static_cast<uint8_t*>(c.q_row);
    p.q_row_s = static_cast<uint8_t*>(c.q_row_s);
    p.q_col = static_cast<uint8_t*>(c.q_col);
    p.q_col_s = static_cast<uint8_t*>(c.q_col_s);
    p.swizzle = c.swizzle;
    p.y1 = static_cast<const __nv_bfloat16*>(c.y1);
    p.dbias_part = c.dbias_part;
    p.side = static_cast<__nv_bfloat16*>(c.side_bf16);

    if (use_pair) return run_pair(c, p, to, s);

    const int grid = (int)std::min<int64_t>(tiles, sm_count());
    if (c.pad) {
        const int sm = smem_bytes_padded(c.E);
        if (c.mode == kFprop) grouped_gemm_kernel<kFprop, true><<<grid, NUM_THREADS, sm, s>>>(ta, tb, to, p);
        else if (c.mode == kDgrad) grouped_gemm_kernel<kDgrad, true><<<grid, NUM_THREADS, sm, s>>>(ta, tb, to, p);
        else grouped_gemm_kernel<kWgrad, true><<<grid, NUM_THREADS, sm, s>>>(ta, tb, to, p);
    } else if (c.mode == kFpropSwiglu)
        grouped_gemm_kernel<kFpropSwiglu><<<grid, NUM_THREADS, smem_bytes(c.E), s>>>(ta, tb, to, p);
    else if (c.mode == kDgradSwiglu)
        grouped_gemm_kernel<kDgradSwiglu><<<grid, NUM_THREADS, smem_bytes(c.E), s>>>(ta, tb, to, p);
    else if (c.mode == kFprop) grouped_gemm_kernel<kFprop><<<grid, NUM_THREADS, smem_bytes(c.E), s>>>(ta, tb, to, p);
    else if (c.mode == kDgrad) grouped_gemm_kernel<kDgrad><<<grid, NUM_THREADS, smem_bytes(c.E), s>>>(ta, tb, to, p);
    else grouped_gemm_kernel<kWgrad><<<grid, NUM_THREADS, smem_bytes(c.E), s>>>(ta, tb, to, p);
    return cudaGetLastError();
}

}  // namespace mxq
