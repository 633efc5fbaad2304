// epilogue.cuh -- the fused epilogue shared by every GEMM kernel.
//
// For each output element the accumulator `acc` (fp32) becomes
//     z = alpha*acc + beta*C_in + bias[j];  y = GELU(z) (bias+GELU only);
//     y += R[i][j] (post-activation residual, extended calls only);
//     C[i][j] = round_to_nearest_even(y) in the output type
// applied in registers before the single store ("Case Study: Steel's
// BlockMMA", the paragraph on store_result / apply_epilogue; "Case Study: The
// Tiled GEMM", the fused alpha*AB + beta*C store).  beta == 0 never reads C.
//
// Two store paths, as the masked write-back of "X3: Metal GEMM" section 5
// separates them: a fast path that moves 32 consecutive outputs of one row
// with 16-byte vector accesses, and a safe path that checks every column
// against N and touches only in-range elements (tiles that straddle the N
// edge, or buffers whose alignment rules out vectors).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "kernel_args.h"
#include "sm103_ptx.cuh"

namespace gb300 {

template <int DT> struct Elem;
template <> struct Elem<kDtF32> {
    using T = float;
    static __device__ __forceinline__ float load(const T *p) { return *p; }
    static __device__ __forceinline__ T cvt(float x) { return x; }
};
template <> struct Elem<kDtF16> {
    using T = __half;
    static __device__ __forceinline__ float load(const T *p) { return __half2float(*p); }
    static __device__ __forceinline__ T cvt(float x) { return __float2half_rn(x); }
};
template <> struct Elem<kDtBF16> {
    using T = __nv_bfloat16;
    static __device__ __forceinline__ float load(const T *p) { return __bfloat162float(*p); }
    static __device__ __forceinline__ T cvt(float x) { return __float2bfloat16_rn(x); }
};
template <> struct Elem<kDtE4M3> {
    using T = __nv_fp8_e4m3;
    static __device__ __forceinline__ float load(const T *p) { return static_cast<float>(*p); }
    // Round to nearest even, saturating to +-448 (OCP E4M3 "fn" has no infinity).
    static __device__ __forceinline__ T cvt(float x) {
        T r;
        r.__x = __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
        return r;
    }
};

// GELU, erf form: 0.5*z*(1 + erf(z/sqrt(2))), with erf from the rational
// approximation of Abramowitz & Stegun, Handbook of Mathematical Functions,
// formula 7.1.26 (Hastings): for x >= 0,
//     erfc(x) = (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-x^2) + e(x),
//     t = 1 / (1 + p x),  |e(x)| <= 1.5e-7,
// p = 0.3275911, a1..a5 = 0.254829592, -0.284496736, 1.421413741,
// -1.453152027, 1.061405429.  With x = |z|/sqrt(2) and q = erfc(x):
//     erf(z/sqrt(2)) = copysign(1 - q, z),   GELU(z) = (z/2) * (1 + erf).
// For z < 0 the sum 1 + erf is exact (Sterbenz) but inherits the rounding
// of 1 - q (<= 2^-25), so the absolute error stays below 3e-8 |z| -- far
// inside the normalised tolerances, whose scale is at least |z|.  The
// reciprocal and 2^x are the hardware approximations (rcp.approx, ex2.approx,
// relative error ~2^-22).  gelu_erf and gelu_erf2 perform the same operations
// in the same order, so a value gets the same result from either.
namespace gelu_c {
constexpr float kRsqrt2 = 0.70710678118654752440f;
constexpr float kP = 0.3275911f;
constexpr float kA1 = 0.254829592f, kA2 = -0.284496736f, kA3 = 1.421413741f, kA4 = -1.453152027f,
                kA5 = 1.061405429f;
constexpr float kNegLog2e = -1.44269504088896340736f;
}  // namespace gelu_c

__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float gelu_erf(float z) {
    using namespace gelu_c;
    const float x = fabsf(z) * kRsqrt2;
    const float t = rcp_approx(fmaf(kP, x, 1.0f));
    float poly = fmaf(kA5, t, kA4);
    poly = fmaf(poly, t, kA3);
    poly = fmaf(poly, t, kA2);
    poly = fmaf(poly, t, kA1);
    const float q = (poly * t) * ex2_approx((x * x) * kNegLog2e);
    const float e = copysignf(fmaf(q, -1.0f, 1.0f), z);
    return (0.5f * z) * (e + 1.0f);
}

// --- two fp32 lanes per instruction (Blackwell f32x2 arithmetic) -----------
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_splat(float c) { return f2_pack(c, c); }

// v[i .. i+3] += b, two lanes per instruction.
__device__ __forceinline__ void add4_f2(float (&v)[32], int i, const float4 &b) {
    f2_unpack(f2_add(f2_pack(v[i], v[i + 1]), f2_pack(b.x, b.y)), v[i], v[i + 1]);
    f2_unpack(f2_add(f2_pack(v[i + 2], v[i + 3]), f2_pack(b.z, b.w)), v[i + 2], v[i + 3]);
}

// GELU of two values at once; same operations as gelu_erf, lane by lane.
__device__ __forceinline__ void gelu_erf2(float &z0, float &z1) {
    using namespace gelu_c;
    const uint64_t z = f2_pack(z0, z1);
    const uint64_t x = f2_mul(z & 0x7FFFFFFF7FFFFFFFull, f2_splat(kRsqrt2));
    const uint64_t d = f2_fma(f2_splat(kP), x, f2_splat(1.0f));
    float d0, d1;
    f2_unpack(d, d0, d1);
    const uint64_t t = f2_pack(rcp_approx(d0), rcp_approx(d1));
    uint64_t poly = f2_fma(f2_splat(kA5), t, f2_splat(kA4));
    poly = f2_fma(poly, t, f2_splat(kA3));
    poly = f2_fma(poly, t, f2_splat(kA2));
    poly = f2_fma(poly, t, f2_splat(kA1));
    const uint64_t u = f2_mul(f2_mul(x, x), f2_splat(kNegLog2e));
    float u0, u1;
    f2_unpack(u, u0, u1);
    const uint64_t q = f2_mul(f2_mul(poly, t), f2_pack(ex2_approx(u0), ex2_approx(u1)));
    const uint64_t omq = f2_fma(q, f2_splat(-1.0f), f2_splat(1.0f));
    const uint64_t e = omq | (z & 0x8000000080000000ull);  // copysign(1 - q, z); 1 - q >= 0
    const uint64_t y = f2_mul(f2_mul(f2_splat(0.5f), z), f2_add(e, f2_splat(1.0f)));
    f2_unpack(y, z0, z1);
}

// --- the other activations -------------------------------------------------
// tanh(u) = sign(u) * (1 - 2 / (1 + e^(2|u|))): the hardware 2^x and
// reciprocal keep the absolute error near 1e-7 (no cancellation for large
// |u|; for small |u| the absolute error is what matters, since the result is
// multiplied by z/2).  e^(2|u|) overflows to +inf for large |u|, giving 1.
__device__ __forceinline__ float tanh_approx_abs(float u) {
    constexpr float kTwoLog2e = 2.88539008177792681472f;  // 2 / ln 2
    const float t = fmaf(-2.0f, rcp_approx(ex2_approx(fabsf(u) * kTwoLog2e) + 1.0f), 1.0f);
    return copysignf(t, u);
}

// GELU, tanh form: 0.5*z*(1 + tanh(sqrt(2/pi)*(z + 0.044715*z^3))).
__device__ __forceinline__ float gelu_tanh(float z) {
    constexpr float kSqrt2OverPi = 0.79788456080286535588f;
    const float u = kSqrt2OverPi * fmaf(0.044715f * z, z * z, z);
    return (0.5f * z) * (1.0f + tanh_approx_abs(u));
}

// SiLU: z * sigmoid(z) = z / (1 + e^-z); e^-z overflows to +inf for very
// negative z, and z * rcp(inf) = -0.
__device__ __forceinline__ float silu(float z) {
    return z * rcp_approx(1.0f + ex2_approx(z * gelu_c::kNegLog2e));
}

// ReLU: max(z, 0), NaN kept.
__device__ __forceinline__ float relu(float z) { return z < 0.0f ? 0.0f : z; }

// --- cheaper forms for 16-bit outputs -----------------------------------------
// A 16-bit output rounds to 2^-9 (bf16) or 2^-12 (fp16) of its value, and its
// tolerance is 2e-3 of the error scale D >= |z|; the forms below stay within
// 4e-4 |z| of the exact activation (about a tenth of the output's unit in the
// last place, relative to |z|) and cost no more than one special-function
// operation per element (the accurate forms above cost two).  They serve F16
// and BF16 outputs only, and not when the call keeps an amax (a reduction held
// to the fp32 tolerance): fp32 and E4M3 outputs and amax calls take the
// accurate forms.  Every instruction per element shows in the fused cost even
// where the epilogue overlaps the next tile's main loop (its warps share the
// issue slots of the MMA and TMA warps), so each form also has a two-lane
// variant that runs its multiply-adds as f32x2.
//
// GELU (erf form) for F16 outputs: Phi(z) - 1/2 = z P(z^2) on |z| <= 4 (z clamped beyond;
// Phi(4) = 1 - 3.2e-5), P of degree 6 with the coefficients of a near-minimax
// fit of the absolute error in Phi (fit_gelu_poly.py beside the package's
// sources: least squares in the Chebyshev basis, reweighted towards the
// largest errors).  Largest error 1.1e-4 in Phi in float32, so at most
// 1.1e-4 |z| in GELU(z) = z Phi(z) -- a twentieth of a bf16 output's own
// rounding; multiply-adds only (measured on GB300, degree 8 at 2.8e-5 cost
// 1.2 points more of fused cost at M = 2048, N = K = 4096).
namespace gelu_p {
constexpr float kZmax = 4.0f;
constexpr float kC0 = 0.3985269069671631f, kC1 = -0.06538835167884827f, kC2 = 0.0091129494830966f,
                kC3 = -0.0008789804996922612f, kC4 = 5.419035005616024e-05f, kC5 = -1.8918872228823602e-06f,
                kC6 = 2.8160954457234766e-08f;
}  // namespace gelu_p

__device__ __forceinline__ float gelu_erf_poly(float z) {
    using namespace gelu_p;
    const float zc = fminf(fmaxf(z, -kZmax), kZmax);
    const float s = zc * zc;
    float p = fmaf(kC6, s, kC5);
    p = fmaf(p, s, kC4);
    p = fmaf(p, s, kC3);
    p = fmaf(p, s, kC2);
    p = fmaf(p, s, kC1);
    p = fmaf(p, s, kC0);
    const float h = zc * p;              // Phi(z) - 1/2
    return fmaf(z, h, 0.5f * z);         // z (1/2 + h)
}

// The same operations on two values, two lanes per instruction.
__device__ __forceinline__ void gelu_erf_poly2(float &z0, float &z1) {
    using namespace gelu_p;
    const uint64_t zc = f2_pack(fminf(fmaxf(z0, -kZmax), kZmax), fminf(fmaxf(z1, -kZmax), kZmax));
    const uint64_t s = f2_mul(zc, zc);
    uint64_t p = f2_fma(f2_splat(kC6), s, f2_splat(kC5));
    p = f2_fma(p, s, f2_splat(kC4));
    p = f2_fma(p, s, f2_splat(kC3));
    p = f2_fma(p, s, f2_splat(kC2));
    p = f2_fma(p, s, f2_splat(kC1));
    p = f2_fma(p, s, f2_splat(kC0));
    const uint64_t h = f2_mul(zc, p);
    const uint64_t z = f2_pack(z0, z1);
    f2_unpack(f2_fma(z, h, f2_mul(f2_splat(0.5f), z)), z0, z1);
}

// The hardware tanh (tanh.approx.f32, relative error about 2^-11).
__device__ __forceinline__ float tanh_hw(float u) {
    float r;
    asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(u));
    return r;
}

// erf-GELU for BF16 outputs: Phi(z) ~ 1/2 + tanh(z (t1 + t3 z^2)) / 2, the
// two coefficients minimax in the absolute error of Phi (1.4e-4; printed by
// fit_gelu_poly.py beside the package's sources), with the hardware tanh
// (at most 2.5e-4 more): at most 3.9e-4 |z| in GELU, a tenth of a bf16
// output's unit in the last place relative to |z|.  No clamp is needed (tanh
// saturates), so it costs half the instructions of the polynomial, which
// F16 outputs keep for their three extra bits.
namespace gelu_t {
constexpr float kT1 = 0.7988014221191406f, kT3 = 0.03528204932808876f;
}  // namespace gelu_t

__device__ __forceinline__ float gelu_erf_tanh(float z) {
    const float s = z * z;
    const float u = z * fmaf(gelu_t::kT3, s, gelu_t::kT1);
    const float hz = 0.5f * z;
    return fmaf(hz, tanh_hw(u), hz);
}

// The same operations on two values, two lanes per instruction.
__device__ __forceinline__ void gelu_erf_tanh2(float &z0, float &z1) {
    const uint64_t z = f2_pack(z0, z1);
    const uint64_t s = f2_mul(z, z);
    float u0, u1;
    f2_unpack(f2_mul(z, f2_fma(f2_splat(gelu_t::kT3), s, f2_splat(gelu_t::kT1))), u0, u1);
    const uint64_t hz = f2_mul(f2_splat(0.5f), z);
    f2_unpack(f2_fma(hz, f2_pack(tanh_hw(u0), tanh_hw(u1)), hz), z0, z1);
}

// GELU (tanh form) with the hardware tanh: error up to 0.5 |z| 2^-11.
__device__ __forceinline__ float gelu_tanh_hw(float z) {
    constexpr float kSqrt2OverPi = 0.79788456080286535588f;
    const float u = kSqrt2OverPi * fmaf(0.044715f * z, z * z, z);
    const float hz = 0.5f * z;
    return fmaf(hz, tanh_hw(u), hz);
}

// The same operations on two values, two lanes per instruction.
__device__ __forceinline__ void gelu_tanh_hw2(float &z0, float &z1) {
    constexpr float kSqrt2OverPi = 0.79788456080286535588f;
    const uint64_t z = f2_pack(z0, z1);
    const uint64_t w = f2_fma(f2_mul(f2_splat(0.044715f), z), f2_mul(z, z), z);
    float u0, u1;
    f2_unpack(f2_mul(f2_splat(kSqrt2OverPi), w), u0, u1);
    const uint64_t hz = f2_mul(f2_splat(0.5f), z);
    f2_unpack(f2_fma(hz, f2_pack(tanh_hw(u0), tanh_hw(u1)), hz), z0, z1);
}

// SiLU as z sigmoid(z) = (z/2) (1 + tanh(z/2)) with the hardware tanh.
__device__ __forceinline__ float silu_hw(float z) {
    const float hz = 0.5f * z;
    return fmaf(hz, tanh_hw(hz), hz);
}

// The same operations on two values, two lanes per instruction.
__device__ __forceinline__ void silu_hw2(float &z0, float &z1) {
    const uint64_t hz = f2_mul(f2_splat(0.5f), f2_pack(z0, z1));
    float h0, h1;
    f2_unpack(hz, h0, h1);
    f2_unpack(f2_fma(hz, f2_pack(tanh_hw(h0), tanh_hw(h1)), hz), z0, z1);
}

// Whether output type OUT may take the cheaper forms.
template <int OUT>
constexpr bool kCheapActivation = OUT == kDtF16 || OUT == kDtBF16;

// The epilogue's activation of z (identity for kEpiNone / kEpiBias): the
// cheaper forms above for 16-bit outputs unless `precise`, else the accurate
// ones.
template <int OUT>
__device__ __forceinline__ float activate_one(float z, int epi, bool precise) {
    const bool kLow = kCheapActivation<OUT> && !precise;
    switch (epi) {
    case kEpiBiasGelu: return kLow ? (OUT == kDtBF16 ? gelu_erf_tanh(z) : gelu_erf_poly(z)) : gelu_erf(z);
    case kEpiBiasGeluTanh: return kLow ? gelu_tanh_hw(z) : gelu_tanh(z);
    case kEpiBiasSilu: return kLow ? silu_hw(z) : silu(z);
    case kEpiBiasRelu: return relu(z);
    default: return z;
    }
}

// The activation of v[off] .. v[off + CNT - 1] (CNT even): one branch on the
// epilogue for the whole run, then the chosen activation straight through --
// a branch per element (indirect, for a switch) cost more than ReLU itself.
// Values get exactly what activate_one gives them.
template <int OUT, int CNT>
__device__ __forceinline__ void activate_run(float (&v)[32], int off, int epi, bool precise) {
    const bool kLow = kCheapActivation<OUT> && !precise;
    if (epi == kEpiBiasGelu) {
        if (kLow) {
            if constexpr (OUT == kDtBF16) {
#pragma unroll
                for (int j = 0; j < CNT; j += 2) gelu_erf_tanh2(v[off + j], v[off + j + 1]);
            } else {
#pragma unroll
                for (int j = 0; j < CNT; j += 2) gelu_erf_poly2(v[off + j], v[off + j + 1]);
            }
        } else {
#pragma unroll
            for (int j = 0; j < CNT; j += 2) gelu_erf2(v[off + j], v[off + j + 1]);
        }
    } else if (epi == kEpiBiasRelu) {
#pragma unroll
        for (int j = 0; j < CNT; ++j) v[off + j] = relu(v[off + j]);
    } else if (epi == kEpiBiasSilu) {
        if (kLow) {
#pragma unroll
            for (int j = 0; j < CNT; j += 2) silu_hw2(v[off + j], v[off + j + 1]);
        } else {
#pragma unroll
            for (int j = 0; j < CNT; ++j) v[off + j] = silu(v[off + j]);
        }
    } else if (epi == kEpiBiasGeluTanh) {
        if (kLow) {
#pragma unroll
            for (int j = 0; j < CNT; j += 2) gelu_tanh_hw2(v[off + j], v[off + j + 1]);
        } else {
#pragma unroll
            for (int j = 0; j < CNT; ++j) v[off + j] = gelu_tanh(v[off + j]);
        }
    }
}

// Product scale of output (row, col) beyond alpha: alpha_scale[0] * row_scale[row]
// * col_scale[col], each factor 1 when absent (1 without any: e.scaled == 0).
__device__ __forceinline__ float product_scale(const EpiParams &e, int row, int col) {
    if (!e.scaled) return 1.0f;
    float f = e.alpha_scale ? *e.alpha_scale : 1.0f;
    if (e.row_scale) f *= e.row_scale[row];
    if (e.col_scale) f *= e.col_scale[col];
    return f;
}

// The same product scale over one chunk of 32 accumulators: the thread's fixed
// index is `lane_idx`, accumulator j has running index run0 + j.  Untransposed
// they are the output row and columns; transposed (the kernel computed C^T)
// the output column and rows.  Running indices at or past the matrix's end
// (masked outputs) keep factor 1.  SC = false compiles it out: kernels built
// for calls without scales keep the registers the scaled path needs.
template <bool SC = true>
__device__ __forceinline__ void product_scale_chunk(float (&v)[32], const EpiParams &e, int lane_idx, int run0,
                                                    bool transposed) {
    if constexpr (!SC) return;
    if (!e.scaled) return;
    const float *lane_vec = transposed ? e.col_scale : e.row_scale;
    const float *run_vec = transposed ? e.row_scale : e.col_scale;
    const int lane_ext = transposed ? e.N : e.M, run_ext = transposed ? e.M : e.N;
    float f = e.alpha_scale ? *e.alpha_scale : 1.0f;
    if (lane_vec && lane_idx < lane_ext) f *= lane_vec[lane_idx];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float r = (run_vec && run0 + j < run_ext) ? run_vec[run0 + j] : 1.0f;
        v[j] *= f * r;
    }
}

// Raise *amax to the largest `local` (>= 0) of the calling threads: one atomic
// per group of converged lanes (non-negative floats order like their bits).
__device__ __forceinline__ void amax_push(float local, float *amax) {
    const unsigned mask = __activemask();
    const unsigned v = __reduce_max_sync(mask, __float_as_uint(local));
    if ((threadIdx.x & 31) == static_cast<unsigned>(__ffs(mask) - 1))
        atomicMax(reinterpret_cast<unsigned int *>(amax), v);
}

// Residual row `row` of the output (NULL without a residual).
template <int OUT>
__device__ __forceinline__ const typename Elem<OUT>::T *residual_row(const EpiParams &e, int row) {
    return e.residual ? reinterpret_cast<const typename Elem<OUT>::T *>(e.residual) + (long long)row * e.ldr
                      : nullptr;
}

// Scalar epilogue of one element (used by the safe path and the SIMT kernel);
// `r` is the element's residual (NULL: none).  Returns the activated value
// (plus the residual) before any output scaling (for amax).
template <int OUT>
__device__ __forceinline__ float epilogue_store_one(float acc, typename Elem<OUT>::T *c, float bias_j,
                                                    const EpiParams &e,
                                                    const typename Elem<OUT>::T *r = nullptr) {
    float z = e.alpha * acc;
    if constexpr (OUT != kDtE4M3) {
        if (e.beta != 0.0f) z = fmaf(e.beta, Elem<OUT>::load(c), z);  // E4M3 outputs are written only
    }
    if (e.epilogue != kEpiNone) z += bias_j;
    z = activate_one<OUT>(z, e.epilogue, e.amax != nullptr);
    if (r != nullptr) z += Elem<OUT>::load(r);
    if constexpr (OUT == kDtE4M3)
        *c = Elem<OUT>::cvt(e.out_scale ? z / *e.out_scale : z);
    else
        *c = Elem<OUT>::cvt(z);
    return z;
}

// --- 16-byte packing helpers for the fast path -----------------------------

template <int OUT> struct Vec16;
template <> struct Vec16<kDtF32> {
    static constexpr int kPerVec = 4;
    static __device__ __forceinline__ void unpack(const uint4 &u, float *f) {
        f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
    }
    static __device__ __forceinline__ uint4 pack(const float *f) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
};
template <> struct Vec16<kDtF16> {
    static constexpr int kPerVec = 8;
    static __device__ __forceinline__ void unpack(const uint4 &u, float *f) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
            float2 t = __half22float2(h);
            f[2 * i] = t.x; f[2 * i + 1] = t.y;
        }
    }
    static __device__ __forceinline__ uint4 pack(const float *f) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};
template <> struct Vec16<kDtBF16> {
    static constexpr int kPerVec = 8;
    static __device__ __forceinline__ void unpack(const uint4 &u, float *f) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162 *>(&w[i]);
            float2 t = __bfloat1622float2(h);
            f[2 * i] = t.x; f[2 * i + 1] = t.y;
        }
    }
    static __device__ __forceinline__ uint4 pack(const float *f) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

template <> struct Vec16<kDtE4M3> {
    static constexpr int kPerVec = 16;
    static __device__ __forceinline__ void unpack(const uint4 &u, float *f) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const __nv_fp8x2_storage_t two = static_cast<__nv_fp8x2_storage_t>(w[i / 2] >> (16 * (i % 2)));
            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(two, __NV_E4M3);
            const float2 t = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
            f[2 * i] = t.x; f[2 * i + 1] = t.y;
        }
    }
    static __device__ __forceinline__ uint4 pack(const float *f) {
        uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t two = __nv_cvt_float2_to_fp8x2(make_float2(f[2 * i], f[2 * i + 1]), __NV_SATFINITE,
                                                          __NV_E4M3);
            w[i / 2] |= (two & 0xFFFFu) << (16 * (i % 2));
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// Add the residual of 32 in-range columns (rchunk: their first element).
template <int OUT>
__device__ __forceinline__ void add_residual32(float (&v)[32], const typename Elem<OUT>::T *rchunk,
                                               const EpiParams &e) {
    constexpr int PV = Vec16<OUT>::kPerVec;
    if (e.r_vec) {
        const uint4 *src = reinterpret_cast<const uint4 *>(rchunk);
#pragma unroll
        for (int q = 0; q < 32 / PV; ++q) {
            float r[PV];
            Vec16<OUT>::unpack(__ldg(src + q), r);
#pragma unroll
            for (int t = 0; t < PV; ++t) v[q * PV + t] += r[t];
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += Elem<OUT>::load(rchunk + j);
    }
}

// Fast path: 32 in-range columns of one row, C and bias 16-byte aligned.
// `bias_chunk` may point to global or shared memory (generic loads).  With SC,
// also the residual (rchunk: R at the chunk's first column, or NULL), the amax
// reduction and (E4M3 output) the output scale.
template <int OUT, bool SC = true>
__device__ __forceinline__ void epilogue_chunk32_fast(float (&v)[32], typename Elem<OUT>::T *crow,
                                                      const float *bias_chunk, const EpiParams &e,
                                                      const typename Elem<OUT>::T *rchunk = nullptr) {
    constexpr int PV = Vec16<OUT>::kPerVec;
    constexpr int NV = 32 / PV;
    const uint64_t alpha2 = f2_splat(e.alpha);
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const uint64_t r = f2_mul(f2_pack(v[j], v[j + 1]), alpha2);
        f2_unpack(r, v[j], v[j + 1]);
    }
    if (e.beta != 0.0f) {
        const uint4 *src = reinterpret_cast<const uint4 *>(crow);
#pragma unroll
        for (int q = 0; q < NV; ++q) {
            float c[PV];
            Vec16<OUT>::unpack(src[q], c);
#pragma unroll
            for (int t = 0; t < PV; ++t) v[q * PV + t] = fmaf(e.beta, c[t], v[q * PV + t]);
        }
    }
    if (e.epilogue != kEpiNone) {
        const float4 *b4 = reinterpret_cast<const float4 *>(bias_chunk);
#pragma unroll
        for (int q = 0; q < 8; ++q) add4_f2(v, 4 * q, b4[q]);
        if (e.epilogue >= kEpiBiasGelu) activate_run<OUT, 32>(v, 0, e.epilogue, SC && e.amax != nullptr);
    }
    if constexpr (SC) {
        if (rchunk != nullptr) add_residual32<OUT>(v, rchunk, e);
        if (e.amax) {
            float m = 0.0f;
#pragma unroll
            for (int j = 0; j < 32; ++j) m = fmaxf(m, fabsf(v[j]));
            amax_push(m, e.amax);
        }
    }
    if constexpr (OUT == kDtE4M3) {
        if (e.out_scale) {
            const float inv = 1.0f / *e.out_scale;
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] *= inv;
        }
    }
    uint4 *dst = reinterpret_cast<uint4 *>(crow);
#pragma unroll
    for (int q = 0; q < NV; ++q) dst[q] = Vec16<OUT>::pack(&v[q * PV]);
}

// Safe path: columns col0 .. col0+31, of which only those < N are touched
// (rchunk: the residual at column col0, or NULL).
template <int OUT, bool SC = true>
__device__ __forceinline__ void epilogue_chunk32_safe(const float (&v)[32], typename Elem<OUT>::T *crow, int col0,
                                                      const EpiParams &e,
                                                      const typename Elem<OUT>::T *rchunk = nullptr) {
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        if (col0 + j < e.N) {
            const float b = (e.epilogue != kEpiNone) ? e.bias[col0 + j] : 0.0f;
            const typename Elem<OUT>::T *r = (SC && rchunk != nullptr) ? rchunk + j : nullptr;
            m = fmaxf(m, fabsf(epilogue_store_one<OUT>(v[j], crow + j, b, e, r)));
        }
    }
    if constexpr (SC) {
        if (e.amax) amax_push(m, e.amax);
    }
}

// One thread's share of a tile's epilogue: row `row` (its TMEM lane), chunks
// 0 .. nvalid-1 of 32 columns starting at TMEM column address t_base and
// output column col_base; bias_base[c] is the bias of column col_base + c (in
// global memory, or staged in shared memory).  The TMEM load of chunk i+1 is
// in flight while chunk i is processed.  Warp-collective (every lane calls it
// with the same t_base, col_base and nvalid); nvalid <= MAXC.
template <int OUT, int MAXC, bool SC = true>
__device__ __forceinline__ void epilogue_row_chunks(uint32_t t_base, int col_base, int nvalid, int row, bool row_ok,
                                                    const float *bias_base, const EpiParams &e) {
    using OutT = typename Elem<OUT>::T;
    if (nvalid <= 0) return;
    OutT *crow = reinterpret_cast<OutT *>(e.C) + (long long)(row_ok ? row : 0) * e.ldc;
    const OutT *rrow = (SC && row_ok) ? residual_row<OUT>(e, row) : nullptr;
    uint32_t ra[32], rb[32];
    __syncwarp();
    tmem_ld_issue(t_base, ra);
    tmem_ld_wait(ra);
#pragma unroll
    for (int i = 0; i < MAXC; ++i) {
        if (i >= nvalid) break;  // warp-uniform
        uint32_t(&cur)[32] = (i & 1) ? rb : ra;
        uint32_t(&nxt)[32] = (i & 1) ? ra : rb;
        const bool more = i + 1 < nvalid;
        if (more) tmem_ld_issue(t_base + (i + 1) * 32, nxt);
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(cur[j]);
        const int col0 = col_base + i * 32;
        product_scale_chunk<SC>(v, e, row, col0, false);
        if (row_ok) {
            const OutT *rchunk = rrow != nullptr ? rrow + col0 : nullptr;
            if (e.c_vec && col0 + 32 <= e.N)
                epilogue_chunk32_fast<OUT, SC>(v, crow + col0, bias_base + i * 32, e, rchunk);
            else
                epilogue_chunk32_safe<OUT, SC>(v, crow + col0, col0, e, rchunk);
        }
        __syncwarp();  // reconverge after the per-row store before the collective wait
        if (more) tmem_ld_wait(nxt);
    }
}

// ------------------------------------------- staged epilogue (C by TMA) --
// With one row per thread, direct loads and stores touch 32 rows per warp
// instruction.  The staged form moves C as 32-row x 64-byte boxes between
// global memory and a per-warp 2 KB shared-memory buffer with TMA (coalesced,
// no L1 traffic), and the threads only read and write their own row of the
// buffer.  The box uses the 64-byte TMA swizzle: 16-byte unit q of row r sits
// at unit q ^ ((r >> 1) & 3) of that row, so the eight rows of a quarter-warp
// fall in eight different bank groups.  Elements of a box outside the matrix
// (ragged M or N, the ldc padding) are zero on load and never stored.

constexpr int kStageBoxBytes = 32 * 64;  // one warp's staged box

__device__ __forceinline__ uint32_t sw64_offset(int r, int q) {
    return static_cast<uint32_t>(r * 64 + ((q ^ ((r >> 1) & 3)) << 4));
}

// Columns h*PER .. h*PER+PER-1 of one 32-column chunk (PER = 64 bytes of
// output): beta*C with C read from this thread's row of the staged box,
// bias, GELU, the residual (SC: read from global memory, output row `row`,
// columns x ..), and the result packed back into the same row of the box.
// v holds alpha*acc on entry.
template <int OUT, bool SC = true>
__device__ __forceinline__ void box_math(float (&v)[32], int h, unsigned char *box, const float *bias_chunk,
                                         const EpiParams &e, int row, int x) {
    constexpr int PER = 64 / static_cast<int>(sizeof(typename Elem<OUT>::T));
    constexpr int PV = Vec16<OUT>::kPerVec;
    const int lane = threadIdx.x & 31;
    if (e.beta != 0.0f) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float c[PV];
            Vec16<OUT>::unpack(*reinterpret_cast<const uint4 *>(box + sw64_offset(lane, q)), c);
#pragma unroll
            for (int t = 0; t < PV; ++t) v[h * PER + q * PV + t] = fmaf(e.beta, c[t], v[h * PER + q * PV + t]);
        }
    }
    if (e.epilogue != kEpiNone) {
        const float4 *b4 = reinterpret_cast<const float4 *>(bias_chunk + h * PER);
#pragma unroll
        for (int q = 0; q < PER / 4; ++q) add4_f2(v, h * PER + 4 * q, b4[q]);
        if (e.epilogue >= kEpiBiasGelu) activate_run<OUT, PER>(v, h * PER, e.epilogue, SC && e.amax != nullptr);
    }
    if constexpr (SC) {
        if (e.residual != nullptr && row < e.M) {
            // only columns inside the matrix: the box may reach past N (and R past its allocation)
            const typename Elem<OUT>::T *rr = residual_row<OUT>(e, row) + x;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int c0 = x + q * PV;
                if (e.r_vec && c0 + PV <= e.N) {
                    float r[PV];
                    Vec16<OUT>::unpack(__ldg(reinterpret_cast<const uint4 *>(rr + q * PV)), r);
#pragma unroll
                    for (int t = 0; t < PV; ++t) v[h * PER + q * PV + t] += r[t];
                } else {
#pragma unroll
                    for (int t = 0; t < PV; ++t)
                        if (c0 + t < e.N) v[h * PER + q * PV + t] += Elem<OUT>::load(rr + q * PV + t);
                }
            }
        }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4 *>(box + sw64_offset(lane, q)) = Vec16<OUT>::pack(&v[h * PER + q * PV]);
}

__device__ __forceinline__ void scale_alpha(float (&v)[32], float alpha) {
    const uint64_t alpha2 = f2_splat(alpha);
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const uint64_t r = f2_mul(f2_pack(v[j], v[j + 1]), alpha2);
        f2_unpack(r, v[j], v[j + 1]);
    }
}

// ------------------------------------------------ transposed accumulators --
// When the kernel computes C^T = B^T A^T (so that an N-contiguous B becomes
// the MMA's A operand), TMEM lane l of a warp holds output column n0 + l and
// its 32 accumulator columns are output rows m0 .. m0+31: the warp holds the
// 32 x 32 block C[m0.., n0..] transposed.  The staged box is still C's own
// 32-row x 64-byte box (16-bit output only): lanes 2p and 2p+1 trade values
// with one shuffle per row pair so that each writes whole 32-bit words
// (columns 2p, 2p+1) of alternate rows, two rows per warp instruction.

// Byte offset of a 32-bit word inside a 64-byte-swizzled box.
__device__ __forceinline__ uint32_t sw64_word(uint32_t byte) { return byte ^ (((byte >> 7) & 3u) << 4); }

template <int OUT>
__device__ __forceinline__ uint32_t pack2_out(float lo, float hi) {
    uint32_t w;
    if constexpr (OUT == kDtF16) {
        __half2 h = __floats2half2_rn(lo, hi);
        w = *reinterpret_cast<uint32_t *>(&h);
    } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        w = *reinterpret_cast<uint32_t *>(&h);
    }
    return w;
}

template <int OUT>
__device__ __forceinline__ float2 unpack2_out(uint32_t w) {
    if constexpr (OUT == kDtF16) {
        return __half22float2(*reinterpret_cast<const __half2 *>(&w));
    } else {
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
    }
}

// Transposed counterpart of box_math for one whole chunk (v = alpha*acc of
// output column n0+lane, rows m0 .. m0+31): beta*C from the box, the column's
// bias, GELU, the residual (SC; a warp-wide load per row reads 32 consecutive
// columns), and the result written back into the box.
template <int OUT, bool SC = true>
__device__ __forceinline__ void box_math_t(float (&v)[32], unsigned char *box, float bias_lane, const EpiParams &e,
                                           int n0, int m0) {
    static_assert(OUT == kDtF16 || OUT == kDtBF16, "transposed staging is for 16-bit outputs");
    const int lane = threadIdx.x & 31;
    const uint32_t odd = lane & 1u;
    const uint32_t col_bytes = (lane >> 1) * 4u;
    if (e.beta != 0.0f) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t own = *reinterpret_cast<const uint32_t *>(box + sw64_word((2 * i + odd) * 64u + col_bytes));
            const uint32_t other = __shfl_xor_sync(0xffffffffu, own, 1);
            const float2 a = unpack2_out<OUT>(own), b = unpack2_out<OUT>(other);
            // even lane: own word is row 2i, partner's row 2i+1, low halves are its column
            const float c_even = odd ? b.y : a.x;  // row 2i
            const float c_odd = odd ? a.y : b.x;   // row 2i+1
            v[2 * i] = fmaf(e.beta, c_even, v[2 * i]);
            v[2 * i + 1] = fmaf(e.beta, c_odd, v[2 * i + 1]);
        }
    }
    if (e.epilogue != kEpiNone) {
        const uint64_t b2 = f2_splat(bias_lane);
#pragma unroll
        for (int j = 0; j < 32; j += 2) f2_unpack(f2_add(f2_pack(v[j], v[j + 1]), b2), v[j], v[j + 1]);
        if (e.epilogue >= kEpiBiasGelu) activate_run<OUT, 32>(v, 0, e.epilogue, SC && e.amax != nullptr);
    }
    if constexpr (SC) {
        const int n = n0 + lane;
        if (e.residual != nullptr && n < e.N) {
            const typename Elem<OUT>::T *rc = reinterpret_cast<const typename Elem<OUT>::T *>(e.residual) + n;
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (m0 + j < e.M) v[j] += Elem<OUT>::load(rc + (long long)(m0 + j) * e.ldr);
        }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        // send the row the partner writes, keep the row this lane writes; each
        // lane then stores one 32-bit word (columns 2p, 2p+1) of its row, and a
        // warp's 32 words fill two rows of the box without a bank conflict
        // (2-byte stores of one row measured ~0.7 conflicts per instruction)
        const float send = odd ? v[2 * i] : v[2 * i + 1];
        const float keep = odd ? v[2 * i + 1] : v[2 * i];
        const float got = __shfl_xor_sync(0xffffffffu, send, 1);
        const uint32_t w = odd ? pack2_out<OUT>(got, keep) : pack2_out<OUT>(keep, got);
        *reinterpret_cast<uint32_t *>(box + sw64_word((2 * i + odd) * 64u + col_bytes)) = w;
    }
}

// Epilogue of one 32-column chunk of the warp's 32 rows (this thread: row
// row0 + lane, accumulators v), output columns col0 .. col0+31, bias of those
// columns at bias_chunk (16-byte aligned, shared memory), through the warp's
// one staged box.  Warp-collective; row0 < M and col0 < N.  Stores stay in
// flight when it returns; the box is reused only after the previous store has
// read it.  Returns false if a wait for C gave up.
// With e.swap the accumulators are transposed (TMEM lanes are output columns
// row0 + lane, chunk columns are output rows col0 ..; bias_lane is the
// lane's column bias); see box_math_t.
template <int OUT, bool SC = true>
__device__ __forceinline__ bool epilogue_chunk32_tma(float (&v)[32], int col0, int row0, const float *bias_chunk,
                                                     float bias_lane, const EpiParams &e, const CUtensorMap *tmC,
                                                     unsigned char *buf, uint64_t *cbar, uint32_t &cphase,
                                                     volatile int *abort_flag, unsigned int *status) {
    constexpr int PER = 64 / static_cast<int>(sizeof(typename Elem<OUT>::T));
    constexpr int NSUB = 32 / PER;
    const int lane = threadIdx.x & 31;
    scale_alpha(v, e.alpha);
    product_scale_chunk<SC>(v, e, row0 + lane, col0, e.swap != 0);
    if constexpr (OUT != kDtF32) {
        if (e.swap) {
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
            if (e.beta != 0.0f) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(cbar, kStageBoxBytes);
                    tma_load_2d_hint(buf, tmC, cbar, row0, col0, l2_policy_evict_first());
                }
                const bool got = mbar_wait_bounded(cbar, cphase, abort_flag, status);
                if (!__all_sync(0xffffffffu, got)) return false;
                cphase ^= 1u;
            }
            box_math_t<OUT, SC>(v, buf, bias_lane, e, row0, col0);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_2d_hint(tmC, buf, row0, col0, l2_policy_evict_first());
                bulk_commit();
            }
            return true;
        }
    }
#pragma unroll
    for (int h = 0; h < NSUB; ++h) {
        const int x = col0 + h * PER;
        if (x >= e.N) break;  // warp-uniform
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
        if (e.beta != 0.0f) {
            if (lane == 0) {
                mbar_arrive_expect_tx(cbar, kStageBoxBytes);
                tma_load_2d_hint(buf, tmC, cbar, x, row0, l2_policy_evict_first());
            }
            const bool got = mbar_wait_bounded(cbar, cphase, abort_flag, status);
            if (!__all_sync(0xffffffffu, got)) return false;
            cphase ^= 1u;
        }
        box_math<OUT, SC>(v, h, buf, bias_chunk, e, row0 + lane, x);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d_hint(tmC, buf, x, row0, l2_policy_evict_first());
            bulk_commit();
        }
    }
    return true;
}

// Staged epilogue of one warp's rows row0 .. row0+31 and chunks 0 .. nvalid-1
// of 32 columns from TMEM column address t_base / output column col_base,
// through the warp's one box.  Warp-collective.
template <int OUT, bool SC = true>
__device__ __forceinline__ bool epilogue_rows_tma(uint32_t t_base, int col_base, int nvalid, int row0,
                                                  const float *bias_base, float bias_lane, const EpiParams &e,
                                                  const CUtensorMap *tmC, unsigned char *buf, uint64_t *cbar,
                                                  uint32_t &cphase, volatile int *abort_flag, unsigned int *status) {
    bool ok = true;
#pragma unroll 1
    for (int i = 0; i < nvalid; ++i) {
        uint32_t raw[32];
        __syncwarp();
        tmem_ld_issue(t_base + i * 32, raw);
        tmem_ld_wait(raw);
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(raw[j]);
        if (ok)
            ok = epilogue_chunk32_tma<OUT, SC>(v, col_base + i * 32, row0, bias_base + i * 32, bias_lane, e, tmC, buf,
                                           cbar, cphase, abort_flag, status);
    }
    __syncwarp();
    return ok;
}

// The same for a CTA's last tile, when its operand ring is idle: every box of
// the warp gets its own slot in `area` (box b of chunk i, part h at slot
// i*NSUB + h), all C boxes are requested at once and no store waits for a
// slot to be read, so the tail of the kernel is not a chain of round trips.
template <int OUT, bool SC = true>
__device__ __forceinline__ bool epilogue_rows_tma_burst(uint32_t t_base, int col_base, int nvalid, int row0,
                                                        const float *bias_base, float bias_lane, const EpiParams &e,
                                                        const CUtensorMap *tmC, unsigned char *area, uint64_t *cbar,
                                                        uint32_t &cphase, volatile int *abort_flag,
                                                        unsigned int *status) {
    constexpr int PER = 64 / static_cast<int>(sizeof(typename Elem<OUT>::T));
    constexpr int NSUB = 32 / PER;
    const int lane = threadIdx.x & 31;
    if (nvalid <= 0) return true;
    if constexpr (OUT != kDtF32) {
        if (e.swap) {
            // transposed: chunk i is the box at (x = row0, y = col_base + 32 i), slot i
            if (e.beta != 0.0f) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(cbar, static_cast<uint32_t>(nvalid) * kStageBoxBytes);
                    for (int i = 0; i < nvalid; ++i)
                        tma_load_2d_hint(area + i * kStageBoxBytes, tmC, cbar, row0, col_base + i * 32,
                                         l2_policy_evict_first());
                }
                const bool got = mbar_wait_bounded(cbar, cphase, abort_flag, status);
                if (!__all_sync(0xffffffffu, got)) return false;
                cphase ^= 1u;
            }
#pragma unroll 1
            for (int i = 0; i < nvalid; ++i) {
                uint32_t raw[32];
                __syncwarp();
                tmem_ld_issue(t_base + i * 32, raw);
                tmem_ld_wait(raw);
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(raw[j]);
                scale_alpha(v, e.alpha);
                product_scale_chunk<SC>(v, e, row0 + lane, col_base + i * 32, true);
                box_math_t<OUT, SC>(v, area + i * kStageBoxBytes, bias_lane, e, row0, col_base + i * 32);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d_hint(tmC, area + i * kStageBoxBytes, row0, col_base + i * 32,
                                      l2_policy_evict_first());
                    bulk_commit();
                }
            }
            __syncwarp();
            return true;
        }
    }
    if (e.beta != 0.0f) {
        if (lane == 0) {
            uint32_t nbox = 0;
            for (int i = 0; i < nvalid; ++i)
                for (int h = 0; h < NSUB; ++h)
                    if (col_base + i * 32 + h * PER < e.N) ++nbox;
            mbar_arrive_expect_tx(cbar, nbox * kStageBoxBytes);
            for (int i = 0; i < nvalid; ++i)
                for (int h = 0; h < NSUB; ++h) {
                    const int x = col_base + i * 32 + h * PER;
                    if (x < e.N)
                        tma_load_2d_hint(area + (i * NSUB + h) * kStageBoxBytes, tmC, cbar, x, row0,
                                         l2_policy_evict_first());
                }
        }
        const bool got = mbar_wait_bounded(cbar, cphase, abort_flag, status);
        if (!__all_sync(0xffffffffu, got)) return false;
        cphase ^= 1u;
    }
#pragma unroll 1
    for (int i = 0; i < nvalid; ++i) {
        uint32_t raw[32];
        __syncwarp();
        tmem_ld_issue(t_base + i * 32, raw);
        tmem_ld_wait(raw);
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(raw[j]);
        scale_alpha(v, e.alpha);
        product_scale_chunk<SC>(v, e, row0 + lane, col_base + i * 32, false);
#pragma unroll
        for (int h = 0; h < NSUB; ++h) {
            const int x = col_base + i * 32 + h * PER;
            if (x < e.N)
                box_math<OUT, SC>(v, h, area + (i * NSUB + h) * kStageBoxBytes, bias_base + i * 32, e, row0 + lane, x);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < NSUB; ++h) {
                const int x = col_base + i * 32 + h * PER;
                if (x < e.N)
                    tma_store_2d_hint(tmC, area + (i * NSUB + h) * kStageBoxBytes, x, row0, l2_policy_evict_first());
            }
            bulk_commit();
        }
    }
    __syncwarp();
    return true;
}

// Transposed counterpart of epilogue_prefetch: the warp's block of the
// output is rows col_base .. col_base + 32*nchunk - 1 (within M) by columns
// row0 .. row0+31 (within N); each of those rows' 64 bytes of a residual,
// and of C when `with_c` and beta != 0, is prefetched into L2.  Returns this
// lane's column bias.  Warp-collective.
// Callers ask for C only on a CTA's last tile, whose epilogue nothing
// overlaps: for every other tile the TMA-staged C boxes arrive while the next
// tile's main loop runs anyway, and prefetching their C a main loop ahead
// pushed operand panels out of L2 (8 MB more HBM reads at 4096^3).
template <int OUT>
__device__ __forceinline__ float epilogue_prefetch_t(int col_base, int nchunk, int row0, const EpiParams &e,
                                                     bool with_c) {
    using OutT = typename Elem<OUT>::T;
    const int lane = threadIdx.x & 31;
    const int n = row0 + lane;
    const float b = (e.epilogue != kEpiNone && n < e.N) ? e.bias[n] : 0.0f;
    if (with_c && e.beta != 0.0f && row0 < e.N) {
        const int m_end = min(col_base + nchunk * 32, e.M);
        for (int m = col_base + lane; m < m_end; m += 32) {
            const OutT *p = reinterpret_cast<const OutT *>(e.C) + (long long)m * e.ldc + row0;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
        }
    }
    if (e.residual != nullptr && row0 < e.N) {
        const int m_end = min(col_base + nchunk * 32, e.M);
        for (int m = col_base + lane; m < m_end; m += 32)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(residual_row<OUT>(e, m) + row0));
    }
    __syncwarp();
    return b;
}

// Epilogue inputs of one warp's columns, fetched before the accumulator is
// ready so their latency overlaps the main loop: the 32*nchunk bias values
// go to shared memory (bias_s, 16-byte aligned), and this thread's row of a
// residual, and of C when `with_c` and beta != 0 (see epilogue_prefetch_t),
// is prefetched into L2.  Warp-collective.
template <int OUT>
__device__ __forceinline__ void epilogue_prefetch(float *bias_s, int col_base, int nchunk, int row, bool row_ok,
                                                  const EpiParams &e, bool with_c) {
    using OutT = typename Elem<OUT>::T;
    const int lane = threadIdx.x & 31;
    if (e.epilogue != kEpiNone) {
        for (int c = lane; c < nchunk * 32; c += 32) {
            const int col = col_base + c;
            bias_s[c] = col < e.N ? e.bias[col] : 0.0f;
        }
    }
    const int ncols = min(nchunk * 32, e.N - col_base);  // only columns inside the matrix
    if (with_c && e.beta != 0.0f && row_ok && ncols > 0) {
        const OutT *crow = reinterpret_cast<const OutT *>(e.C) + (long long)row * e.ldc + col_base;
        const int bytes = ncols * static_cast<int>(sizeof(OutT));
        const char *p = reinterpret_cast<const char *>(crow);
        for (int off = 0; off < bytes; off += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(p + off));
    }
    if (e.residual != nullptr && row_ok && ncols > 0) {
        const char *p = reinterpret_cast<const char *>(residual_row<OUT>(e, row) + col_base);
        const int bytes = ncols * static_cast<int>(sizeof(OutT));
        for (int off = 0; off < bytes; off += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(p + off));
    }
    __syncwarp();
}

}  // namespace gb300
