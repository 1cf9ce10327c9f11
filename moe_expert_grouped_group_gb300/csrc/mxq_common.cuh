// mxq_common.cuh -- device helpers shared by the MXFP8 kernels of this library.
//
// MX conventions (OCP MX v1.0, E4M3 elements, E8M0 scales; the pages name
// MXFP8 E4M3 with one scale per 32 elements -- TransformerEngine PR #3244,
// "[Pytorch] Add support for row-wise quanted input for grouped gemm",
// review on the compact scale shape `cols // 32`):
//   shared exponent s = floor(log2(amax)) - 8, clamped to [-127, 127];
//   all-zero block -> code 0; code = s + 127;
//   element = cvt.rn.satfinite.e4m3(x * 2^-s) (RNE, saturating, sign kept).
// The exponent is read from the bits of amax: for a finite non-negative
// IEEE value with biased exponent field F (bias 127), floor(log2) = F - 127
// for normals and < -126 for subnormals, so code = max(F - 8, 0) for both
// bf16 (F = bits >> 7) and fp32 (F = bits >> 23).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mxq.h"

namespace mxq {

constexpr int kTile = 128;  // rows x cols of one quantization tile

__device__ __forceinline__ uint32_t scale_code_from_bf16_absbits(uint32_t absbits) {
    int f = (int)(absbits >> 7);
    return (uint32_t)max(f - 8, 0);
}
__device__ __forceinline__ uint32_t scale_code_from_f32_absbits(uint32_t absbits) {
    int f = (int)(absbits >> 23);
    return (uint32_t)max(f - 8, 0);
}
// 2^-s as an fp32 for code = s + 127 in [0, 246]: exponent field 254 - code.
__device__ __forceinline__ float inv_scale_from_code(uint32_t code) {
    return __uint_as_float((254u - code) << 23);
}
// 2^s as an fp32 for any code in [0, 254] (code 0 -> 2^-127, an fp32 subnormal).
__device__ __forceinline__ float scale_from_code(uint32_t code) {
    return __uint_as_float(code ? (code << 23) : 0x00400000u);
}

// Two fp32 -> two E4M3 bytes (lo = a, hi = b), RNE, saturating finite.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float a, float b) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
    return (uint32_t)r;
}
// Two E4M3 bytes (lo, hi of v) -> two fp32, exact.
__device__ __forceinline__ float2 e4m3x2_to_f32(uint16_t v) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
    __half2 h = *reinterpret_cast<__half2*>(&h2);
    return __half22float2(h);
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Per-CTA view of the grouping: exclusive token offsets off[0..E] in shared
// memory. d_m_splits == nullptr means E uniform members of M/E rows.
// Validates the contract (m_e >= 0, m_e % 128 == 0, sum == M) and returns a
// status bit mask (0 = valid). Must be called by all threads of the block.
__device__ __forceinline__ int load_offsets(const int64_t* __restrict__ d_m_splits, int E, int64_t M,
                                            int64_t* s_off) {
    __shared__ int s_bad;
    const int tid = threadIdx.x;
    if (tid < 32) {
        const int lane = tid;
        const int per = (E + 31) / 32;
        const int lo = min(E, lane * per), hi = min(E, lo + per);
        int64_t local = 0;
        int bad = 0;
        for (int e = lo; e < hi; ++e) {
            int64_t v = d_m_splits ? d_m_splits[e] : M / E;
            if (v < 0) bad |= MXQ_STATUS_SPLIT_NEGATIVE;
            if (v % 128) bad |= MXQ_STATUS_SPLIT_UNALIGNED;
            local += v;
        }
        int64_t incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int64_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        int64_t run = incl - local;
        for (int e = lo; e < hi; ++e) {
            s_off[e] = run;
            run += d_m_splits ? d_m_splits[e] : M / E;
        }
        int64_t total = __shfl_sync(0xffffffffu, incl, 31);
        bad = __reduce_or_sync(0xffffffffu, bad);
        if (lane == 0) {
            s_off[E] = total;
            if (total != M) bad |= MXQ_STATUS_SPLIT_SUM;
            s_bad = bad;
        }
    }
    __syncthreads();
    return s_bad;
}

// The same view for expert counts that need not be multiples of 128: token
// offsets off[0..E] and padded offsets poff[0..E] (each expert rounded up to
// 128 rows, the row space of per-expert padded scale layouts). Validates
// m_e >= 0 and sum == M. Must be called by all threads of the block.
__device__ __forceinline__ int load_offsets_padded(const int64_t* __restrict__ d_m_splits, int E, int64_t M,
                                                   int64_t* s_off, int64_t* s_poff) {
    __shared__ int s_bad;
    const int tid = threadIdx.x;
    if (tid < 32) {
        const int lane = tid;
        const int per = (E + 31) / 32;
        const int lo = min(E, lane * per), hi = min(E, lo + per);
        int64_t local = 0, plocal = 0;
        int bad = 0;
        for (int e = lo; e < hi; ++e) {
            const int64_t v = d_m_splits[e];
            if (v < 0) bad |= MXQ_STATUS_SPLIT_NEGATIVE;
            local += v;
            plocal += (v + 127) / 128 * 128;
        }
        int64_t incl = local, pincl = plocal;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t t = __shfl_up_sync(0xffffffffu, incl, o);
            const int64_t pt = __shfl_up_sync(0xffffffffu, pincl, o);
            if (lane >= o) {
                incl += t;
                pincl += pt;
            }
        }
        int64_t run = incl - local, prun = pincl - plocal;
        for (int e = lo; e < hi; ++e) {
            const int64_t v = d_m_splits[e];
            s_off[e] = run;
            s_poff[e] = prun;
            run += v;
            prun += (v + 127) / 128 * 128;
        }
        const int64_t total = __shfl_sync(0xffffffffu, incl, 31);
        const int64_t ptotal = __shfl_sync(0xffffffffu, pincl, 31);
        bad = __reduce_or_sync(0xffffffffu, bad);
        if (lane == 0) {
            s_off[E] = total;
            s_poff[E] = ptotal;
            if (total != M) bad |= MXQ_STATUS_SPLIT_SUM;
            s_bad = bad;
        }
    }
    __syncthreads();
    return s_bad;
}

// Expert owning row `row` (0 <= row < M): the e with off[e] <= row < off[e+1].
__device__ __forceinline__ int expert_of(const int64_t* s_off, int E, int64_t row) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {  // first e with off[e+1] > row
        int mid = (lo + hi) >> 1;
        if (s_off[mid + 1] > row) hi = mid;
        else lo = mid + 1;
    }
    return lo;
}

__device__ __forceinline__ void report_status(int32_t* d_status, int bits) {
    if (d_status && bits && blockIdx.x == 0 && threadIdx.x == 0) atomicOr(d_status, bits);
}

// ------------------------------------------------ SwiGLU in fp32
// SwiGLU between FC1 and FC2 of a fused grouped MoE MLP (TransformerEngine
// PR #3545, "Fix distributed BF16 weights and trim NVFP4 saved state in the
// fused grouped MLP": FC1 -> activation -> FC2; gate = first half of FC1's
// output). The sigmoid is 1 / (1 + 2^(-g log2 e)) with the hardware base-2
// exponential and reciprocal (ex2.approx, rcp.approx; relative errors near
// 2^-22), the products are single IEEE fp32 roundings (__f*_rn, never
// contracted). Every fp32 step errs far below half a bf16 ulp (2^-9), so the
// bf16-rounded h, dg and du sit within one bf16 step of the exact values.
// All SwiGLU paths (unfused, fused with quantization, both GEMM epilogues)
// run these same steps and agree bit for bit. Below g = -88.7 the
// exponential overflows to +inf and the sigmoid is 0 (its exact value is
// under 2^-127 there).
// The hardware approximations with subnormal inputs and results flushed to
// zero (.ftz), which spares their subnormal handling. In the sigmoid below
// this changes nothing but s for g below about -87.3, where the exact
// sigmoid is under 2^-126: s is then 0 instead of a subnormal. (A subnormal
// ex2 result is absorbed by 1 + x either way.)
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr float kNegLog2e = -1.44269504088896341f;  // -log2(e), rounded to fp32
__device__ __forceinline__ float sigmoid_f32(float g) {
    return rcp_approx(__fadd_rn(1.0f, ex2_approx(__fmul_rn(g, kNegLog2e))));
}
// h = (g * s) * u
__device__ __forceinline__ float swiglu_h(float g, float u) {
    return __fmul_rn(__fmul_rn(g, sigmoid_f32(g)), u);
}
// dg = ((dh * u) * s) * (1 + g * (1 - s)), the factor by one fused multiply-add; du = dh * (g * s)
__device__ __forceinline__ void swiglu_grads(float d, float g, float u, float& dg, float& du) {
    const float s = sigmoid_f32(g);
    const float fac = __fmaf_rn(g, __fsub_rn(1.0f, s), 1.0f);
    dg = __fmul_rn(__fmul_rn(__fmul_rn(d, u), s), fac);
    du = __fmul_rn(d, __fmul_rn(g, s));
}

// The fp32 SwiGLU steps of mxq_common.cuh on two values at once. Each packed
// instruction (add / sub / mul .rn.f32x2) rounds each lane to nearest even
// without flushing subnormals, exactly as the scalar instruction of the same
// step does, so every result is bit-identical to swiglu_h / swiglu_grads.
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float2 f2unpack(uint64_t v) {
    float2 o;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(v));
    return o;
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t f2sub(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2splat(float a) { return f2pack(a, a); }

// sigmoid_f32 on two lanes: the product and the sum packed, the exponential and reciprocal per lane
__device__ __forceinline__ uint64_t sigmoid_x2(float2 g) {
    const float2 t = f2unpack(f2mul(f2pack(g.x, g.y), f2splat(kNegLog2e)));
    const float2 d = f2unpack(f2add(f2splat(1.0f), f2pack(ex2_approx(t.x), ex2_approx(t.y))));
    return f2pack(rcp_approx(d.x), rcp_approx(d.y));
}
// swiglu_h on two lanes: (g * s) * u
__device__ __forceinline__ float2 swiglu_h_x2(float2 g, float2 u) {
    return f2unpack(f2mul(f2mul(f2pack(g.x, g.y), sigmoid_x2(g)), f2pack(u.x, u.y)));
}
// swiglu_grads on two lanes: dg = ((d * u) * s) * fma(g, 1 - s, 1), du = d * (g * s)
__device__ __forceinline__ void swiglu_grads_x2(float2 d, float2 g, float2 u, float2& dg, float2& du) {
    const uint64_t s = sigmoid_x2(g);
    const uint64_t gp = f2pack(g.x, g.y), dp = f2pack(d.x, d.y), one = f2splat(1.0f);
    const uint64_t fac = f2fma(gp, f2sub(one, s), one);
    dg = f2unpack(f2mul(f2mul(f2mul(dp, f2pack(u.x, u.y)), s), fac));
    du = f2unpack(f2mul(dp, f2mul(gp, s)));
}

// ------------------------------------------ mbarrier and TMA wrappers (PTX)
constexpr unsigned long long kWaitNs = 2000000000ull;  // bound on any on-chip wait

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
// First A-byte-aligned address at or after p, a pointer into dynamic shared
// memory. Offsetting p itself (rather than casting an aligned integer back to
// a pointer) lets the compiler keep the shared address space, so accesses
// through the result are shared-memory loads and stores, not generic ones.
template <uint32_t A>
__device__ __forceinline__ uint8_t* smem_align(uint8_t* p) {
    return p + ((A - (smem_u32(p) & (A - 1))) & (A - 1));
}
__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: true when the phase with `parity` completed; false after
// limit_ns (sets *abort_flag) or once another role has set *abort_flag.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              unsigned long long limit_ns) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 0;; ++i) {
        if (mbar_try(bar, parity)) return true;
        if ((i & 63) == 63) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > limit_ns) {
                *abort_flag = 1;
                return false;
            }
        }
    }
}
// The kernels' wait: bounded by kWaitNs (about 2 s).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    return mbar_wait_for(bar, parity, abort_flag, kWaitNs);
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
        "[%2];" ::"r"(dst),
        "l"((uint64_t)map), "r"(bar), "r"(x), "r"(y)
        : "memory");
}
}  // namespace mxq
