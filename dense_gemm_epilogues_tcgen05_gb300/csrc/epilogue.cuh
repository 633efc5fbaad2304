// epilogue.cuh -- the fused epilogue shared by every GEMM kernel.
//
// For each output element the accumulator `acc` (fp32) becomes
//     z = alpha*acc + beta*C_in + bias[j];  y = GELU(z) (bias+GELU only);
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
};

// GELU, exact erf form: 0.5*z*(1 + erf(z/sqrt(2))).
__device__ __forceinline__ float gelu_erf(float z) {
    return 0.5f * z * (1.0f + erff(z * 0.70710678118654752440f));
}

// Scalar epilogue of one element (used by the safe path and the SIMT kernel).
template <int OUT>
__device__ __forceinline__ void epilogue_store_one(float acc, typename Elem<OUT>::T *c, float bias_j,
                                                   const EpiParams &e) {
    float z = e.alpha * acc;
    if (e.beta != 0.0f) z = fmaf(e.beta, Elem<OUT>::load(c), z);
    if (e.epilogue != kEpiNone) z += bias_j;
    if (e.epilogue == kEpiBiasGelu) z = gelu_erf(z);
    *c = Elem<OUT>::cvt(z);
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

// Fast path: 32 in-range columns of one row, C and bias 16-byte aligned.
template <int OUT>
__device__ __forceinline__ void epilogue_chunk32_fast(float (&v)[32], typename Elem<OUT>::T *crow,
                                                      const float *bias_chunk, const EpiParams &e) {
    constexpr int PV = Vec16<OUT>::kPerVec;
    constexpr int NV = 32 / PV;
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] *= e.alpha;
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
        for (int q = 0; q < 8; ++q) {
            const float4 b = __ldg(b4 + q);
            v[4 * q] += b.x; v[4 * q + 1] += b.y; v[4 * q + 2] += b.z; v[4 * q + 3] += b.w;
        }
        if (e.epilogue == kEpiBiasGelu) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = gelu_erf(v[j]);
        }
    }
    uint4 *dst = reinterpret_cast<uint4 *>(crow);
#pragma unroll
    for (int q = 0; q < NV; ++q) dst[q] = Vec16<OUT>::pack(&v[q * PV]);
}

// Safe path: columns col0 .. col0+31, of which only those < N are touched.
template <int OUT>
__device__ __forceinline__ void epilogue_chunk32_safe(const float (&v)[32], typename Elem<OUT>::T *crow, int col0,
                                                      const EpiParams &e) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        if (col0 + j < e.N) {
            const float b = (e.epilogue != kEpiNone) ? e.bias[col0 + j] : 0.0f;
            epilogue_store_one<OUT>(v[j], crow + j, b, e);
        }
    }
}

}  // namespace gb300
