// gemm_q4.cu -- matrix products with 4-bit group-quantized weights.
//
// "X3: Metal GEMM" section 7 names quantized matmul as the main LLM workload
// on Apple GPUs: a memory-bound GEMV when decoding (a few rows of x against
// the whole weight matrix) and a GEMM when filling the prompt, with the
// dequantisation fused into the multiply-accumulate.  The pages give no
// format; the one used here is affine with groups of 64 along K:
//
//     W[n][k] = s[n][k/64] * q[n][k] + b[n][k/64],   q in 0..15,
//
// codes packed eight to a 32-bit word (code k%8 in bits 4*(k%8)), scale and
// bias binary16, and the product is the library's operation with W^T as B:
// C[m][n] = cast(act(alpha * sum_k x[m][k] W[n][k] + beta*C[m][n] + bias[n])).
//
// q4_gemv_kernel (decode, M <= 8 rows of x): HBM-bound, so every weight byte
// is read once, by 16-byte loads that a warp keeps in flight one step ahead.
// A block takes 4 consecutive rows n (2 for more than two rows of x) and its 8
// warps split K: a step is 1024 consecutive k, 32 per lane (16 bytes of codes
// per row), and warp w takes steps w, w + 8, ...; the warps' partial sums meet
// in shared memory before the epilogue.  Within a
// lane's 32 k the group is fixed, so sum_k x (s q + b) = s * sum_k x q + b *
// sum_k x: one multiply-add per code and row of x (two at a time in f32x2
// arithmetic), x's sum shared by the rows.  Codes become exact floats by a
// byte permute into the mantissa of 2^23 and one f32x2 subtraction per pair,
// unpacked once and used for every row of x.
//
// q4_dequantize_kernel (prefill): W to fp16 / bf16, row-major N x K, one word
// (8 codes, 16 output bytes) per thread; the caller then runs gemm() on it.
#include "epilogue.cuh"
#include "kernel_args.h"

namespace gb300 {

namespace {

constexpr int kQ4Warps = 8;  // warps per block

// Weight rows per block: each x value a lane loads serves every row, so more
// rows cut the x traffic; the per-row, per-x-row partial sums bound it.
template <int MM>
constexpr int q4_rows() { return MM <= 2 ? 4 : 2; }

__device__ __forceinline__ uint4 ldg_stream(const uint4 *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Codes p and p + 4 of `word` as floats (exact; the dequantisation pass).
__device__ __forceinline__ float2 code_pair(uint32_t word, int p) {
    const uint32_t h = ((word >> (4 * p)) & 0x000F000Fu) | 0x64006400u;  // binary16 1024 + code, twice
    __half2 v = __hsub2(*reinterpret_cast<const __half2 *>(&h), __half2(__float2half(1024.0f), __float2half(1024.0f)));
    return __half22float2(v);
}

// Codes 2i and 2i + 1 of `word` as an f32x2 pair (exact): the even codes sit in
// the low nibbles of lo's bytes, the odd ones in hi's; a byte permute puts code
// c into the mantissa of 2^23 (0x4B0000cc) and one f32x2 add removes the 2^23.
__device__ __forceinline__ uint64_t code_pair_f2(uint32_t lo, uint32_t hi, int i) {
    const uint32_t e = __byte_perm(lo, 0x4B000000u, 0x7540u + i);
    const uint32_t o = __byte_perm(hi, 0x4B000000u, 0x7540u + i);
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(e), "r"(o));
    return f2_add(r, 0xCB000000CB000000ull);  // + (-2^23, -2^23)
}

// x values 2i and 2i + 1 of an 8-value chunk as an f32x2 pair.
template <int XT>
__device__ __forceinline__ uint64_t x_pair_f2(uint32_t two) {
    if constexpr (XT == kDtF16) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&two));
        return f2_pack(f.x, f.y);
    } else {
        return f2_pack(__uint_as_float(two << 16), __uint_as_float(two & 0xFFFF0000u));
    }
}

template <int XT>
__device__ __forceinline__ void load_x8(const typename Elem<XT>::T *p, float (&x)[8]) {
    const uint4 v = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (XT == kDtF16) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        } else {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
}

template <int XT, int OUT, int MM>
__global__ void __launch_bounds__(kQ4Warps * 32) q4_gemv_kernel(const Q4Args a) {
    using XInT = typename Elem<XT>::T;
    using OutT = typename Elem<OUT>::T;
    constexpr int R = q4_rows<MM>();
    __shared__ float part[kQ4Warps][R * MM];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int M = a.e.M, N = a.e.N, K = a.K;
    const long long wpr = K / 8;   // words per weight row
    const long long gpr = K / 64;  // groups per weight row
    const XInT *X = static_cast<const XInT *>(a.X);
    const int n0 = blockIdx.x * R;
    const int nsteps = (K + 1023) / 1024;  // a step: 1024 consecutive k, 32 per lane

    // Rows past N re-read row n0 (in range) and are never stored.
    const uint4 *wrow[R];
    const uint32_t *sbrow[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const long long n = n0 + r < N ? n0 + r : n0;
        wrow[r] = reinterpret_cast<const uint4 *>(a.Wq + n * wpr);
        sbrow[r] = a.SB + n * gpr;
    }
    float acc[R][MM];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MM; ++m) acc[r][m] = 0.0f;

    // The block's warps split the steps: warp w takes steps w, w + 8, ...
    int step = warp;
    uint4 wv[R];
    uint32_t sbv[R];
    auto fetch = [&](int st) {
        const int k = st * 1024 + lane * 32;
        if (st < nsteps && k < K) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                wv[r] = ldg_stream(wrow[r] + k / 32);
                sbv[r] = __ldg(sbrow[r] + k / 64);
            }
        }
    };
    fetch(step);
    for (; step < nsteps; step += kQ4Warps) {
        const int kc = step * 1024 + lane * 32;
        // This step's codes are in registers; fetch the warp's next step now.
        uint4 cur[R];
        uint32_t csb[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            cur[r] = wv[r];
            csb[r] = sbv[r];
        }
        fetch(step + kQ4Warps);
        if (kc >= K) continue;
        // Partial sums in f32x2 pairs: the low half sums even k, the high half odd k.
        uint64_t dot[R][MM], xsum[MM];
#pragma unroll
        for (int m = 0; m < MM; ++m) {
            xsum[m] = 0;
#pragma unroll
            for (int r = 0; r < R; ++r) dot[r][m] = 0;
        }
#pragma unroll
        for (int w = 0; w < 4; ++w) {  // word w: k = kc + 8w .. kc + 8w + 7
            // x values of this word for every row of x, as f32x2 pairs (k even, k odd)
            uint64_t x2[MM][4];
#pragma unroll
            for (int m = 0; m < MM; ++m) {
                if (m < M) {
                    const uint4 xv = *reinterpret_cast<const uint4 *>(X + (long long)m * a.ldx + kc + 8 * w);
                    x2[m][0] = x_pair_f2<XT>(xv.x);
                    x2[m][1] = x_pair_f2<XT>(xv.y);
                    x2[m][2] = x_pair_f2<XT>(xv.z);
                    x2[m][3] = x_pair_f2<XT>(xv.w);
                } else {
                    x2[m][0] = x2[m][1] = x2[m][2] = x2[m][3] = 0;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) xsum[m] = f2_add(xsum[m], x2[m][i]);
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t word = w == 0 ? cur[r].x : w == 1 ? cur[r].y : w == 2 ? cur[r].z : cur[r].w;
                const uint32_t lo = word & 0x0F0F0F0Fu, hi = (word >> 4) & 0x0F0F0F0Fu;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint64_t q = code_pair_f2(lo, hi, i);
#pragma unroll
                    for (int m = 0; m < MM; ++m) dot[r][m] = f2_fma(q, x2[m][i], dot[r][m]);
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MM; ++m) {
            float s0, s1;
            f2_unpack(xsum[m], s0, s1);
            const float xs = s0 + s1;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float2 sb = __half22float2(*reinterpret_cast<const __half2 *>(&csb[r]));
                float d0, d1;
                f2_unpack(dot[r][m], d0, d1);
                acc[r][m] += sb.x * (d0 + d1) + sb.y * xs;
            }
        }
    }

    // Sum over each warp's lanes, then over the block's warps (in warp order).
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MM; ++m) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc[r][m] += __shfl_xor_sync(0xffffffffu, acc[r][m], off);
            if (lane == 0) part[warp][r * MM + m] = acc[r][m];
        }
    __syncthreads();
    if (threadIdx.x < R * MM) {
        const int r = threadIdx.x / MM, m = threadIdx.x % MM, n = n0 + r;
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < kQ4Warps; ++w) v += part[w][threadIdx.x];
        if (n < N && m < M) {
            const float b = (a.e.epilogue != kEpiNone) ? a.e.bias[n] : 0.0f;
            epilogue_store_one<OUT>(v, static_cast<OutT *>(a.e.C) + (long long)m * a.e.ldc + n, b, a.e);
        }
    }
}

template <int OUT>
__global__ void q4_dequantize_kernel(long long N, long long K, const uint32_t *__restrict__ Wq,
                                     const uint32_t *__restrict__ SB, typename Elem<OUT>::T *__restrict__ W) {
    using OutT = typename Elem<OUT>::T;
    const long long words = N * (K / 8);
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < words;
         i += (long long)gridDim.x * blockDim.x) {
        const long long n = i / (K / 8), k0 = (i - n * (K / 8)) * 8;
        const uint32_t word = Wq[i];
        const uint32_t sbw = SB[n * (K / 64) + k0 / 64];
        const float2 sb = __half22float2(*reinterpret_cast<const __half2 *>(&sbw));
        alignas(16) OutT out[8];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const float2 q = code_pair(word, p);
            out[p] = Elem<OUT>::cvt(fmaf(sb.x, q.x, sb.y));
            out[p + 4] = Elem<OUT>::cvt(fmaf(sb.x, q.y, sb.y));
        }
        *reinterpret_cast<uint4 *>(W + n * K + k0) = *reinterpret_cast<const uint4 *>(out);
    }
}

// One block per q4_rows<MM>() weight rows: blocks are small and many, so the
// last wave is a small part of the run.
template <int XT, int OUT, int MM>
cudaError_t launch_gemv_mm(const Q4Args &a, cudaStream_t s) {
    const long long blocks = (static_cast<long long>(a.e.N) + q4_rows<MM>() - 1) / q4_rows<MM>();
    if (blocks > 2147483647LL) return cudaErrorInvalidConfiguration;
    q4_gemv_kernel<XT, OUT, MM><<<static_cast<unsigned>(blocks), kQ4Warps * 32, 0, s>>>(a);
    return cudaGetLastError();
}

template <int XT, int OUT>
cudaError_t launch_gemv_rows(const Q4Args &a, cudaStream_t s) {
    const int M = a.e.M;
    if (M <= 1) return launch_gemv_mm<XT, OUT, 1>(a, s);
    if (M <= 2) return launch_gemv_mm<XT, OUT, 2>(a, s);
    if (M <= 4) return launch_gemv_mm<XT, OUT, 4>(a, s);
    return launch_gemv_mm<XT, OUT, 8>(a, s);
}

}  // namespace

cudaError_t launch_q4_gemv(int x_dtype, int out, const Q4Args &a, cudaStream_t s) {
    if (a.e.M < 1 || a.e.M > kQ4MaxRows) return cudaErrorInvalidValue;
    switch (x_dtype * 4 + out) {
    case kDtF16 * 4 + kDtF16: return launch_gemv_rows<kDtF16, kDtF16>(a, s);
    case kDtF16 * 4 + kDtBF16: return launch_gemv_rows<kDtF16, kDtBF16>(a, s);
    case kDtF16 * 4 + kDtF32: return launch_gemv_rows<kDtF16, kDtF32>(a, s);
    case kDtBF16 * 4 + kDtF16: return launch_gemv_rows<kDtBF16, kDtF16>(a, s);
    case kDtBF16 * 4 + kDtBF16: return launch_gemv_rows<kDtBF16, kDtBF16>(a, s);
    case kDtBF16 * 4 + kDtF32: return launch_gemv_rows<kDtBF16, kDtF32>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_q4_dequantize(int out, long long N, long long K, const uint32_t *Wq, const uint32_t *SB, void *W,
                                 cudaStream_t s) {
    const long long words = N * (K / 8);
    long long blocks = (words + 255) / 256;
    if (blocks > 152LL * 32) blocks = 152LL * 32;  // grid-stride beyond a few waves
    if (blocks < 1) blocks = 1;
    if (out == kDtF16)
        q4_dequantize_kernel<kDtF16><<<static_cast<unsigned>(blocks), 256, 0, s>>>(N, K, Wq, SB,
                                                                                  static_cast<__half *>(W));
    else if (out == kDtBF16)
        q4_dequantize_kernel<kDtBF16><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
            N, K, Wq, SB, static_cast<__nv_bfloat16 *>(W));
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace gb300
