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

// ---------------------------------------------------------------------------
// q4_mma_kernel (decode on the tensor cores, M <= 8 rows of x).
//
// The codes (one 2-D TMA box of the block's rows per stage) and x (one bulk
// copy per row) reach shared memory on an mbarrier ring that one producer
// warp keeps full, so each SM holds tens of KB of HBM reads in flight without
// spending registers on them.  Four consumer warps
// turn the codes into exact 16-bit integers and multiply them with x by
// mma.sync.m16n8k16: the instruction's 16 rows are weight rows and its 8
// columns the rows of x, so one x fragment serves all of a warp's weight rows.
//
// A block owns kQmRows weight rows.  A stage holds kQmChunk consecutive k of
// those rows and of every row of x; consumer warp w takes group w (64 k) of
// every stage.  The weight box is 160 bytes wide although a stage uses 128:
// rows then sit 160 bytes apart in shared memory, where the consumers' reads
// meet no bank conflicts, and the extra 32 bytes (the next stage's first
// codes) come again from L2, not from HBM.  Scale and bias are fixed within a group, so
// sum_k x (s q + b) = s * (sum_k x q) + b * (sum_k x): the MMA sums x q over
// the group in fp32, and s and b are applied once per group.
//
// The sum over k does not depend on the order of the k, so the MMA's k
// positions are matched to memory by a permutation both operands share: the
// thread that supplies k-pair (2t, 2t+1) of a weight row supplies codes j and
// j + 4 of one 32-bit word, which one mask-and-or puts in the two halves of a
// 16-bit pair (exponent of 1024 for fp16 or 128 for bf16, then that constant
// subtracted: exact), and the x fragment is permuted alike by byte permutes.
constexpr int kQmRows = 32;                              // weight rows per block (two 16-row MMA tiles)
constexpr int kQmChunk = 256;                            // k per stage (four groups)
constexpr int kQmWPitch = 160;                           // weight box width in bytes (128 of this stage's codes)
constexpr int kQmXPitch = 528;                           // bytes per x row in a stage (512 of values)
constexpr int kQmConsumers = 4;                          // one per group of a stage
constexpr int kQmThreads = (kQmConsumers + 1) * 32;      // + the producer warp

template <int MM>
struct QmCfg {
    static constexpr int STAGES = MM == 8 ? 5 : 6;
    static constexpr int W_BYTES = kQmRows * kQmWPitch;
    static constexpr int STAGE_BYTES = (W_BYTES + MM * kQmXPitch + 127) / 128 * 128;  // boxes 128-byte aligned
    static constexpr int PART_OFF = STAGES * STAGE_BYTES;                  // per-warp partial sums
    static constexpr int BAR_OFF = PART_OFF + kQmConsumers * kQmRows * 8 * 4;
    static constexpr int SMEM = BAR_OFF + 2 * STAGES * 8 + 16 + 128;       // + the abort flag, + alignment slack
};
// Pitches: the weight rows' 8-byte reads of a half-warp and the x rows'
// 16-byte reads of a quarter-warp each fall in distinct banks.
static_assert(kQmWPitch % 16 == 0 && kQmXPitch % 16 == 0, "bulk copy destinations are 16-byte aligned");
static_assert(QmCfg<8>::SMEM * 4 + 4 * 1024 <= 228 * 1024, "four blocks of the widest build fit on an SM");

// Nibbles at bits 0-3 and 16-19 of w as an exact 16-bit pair of type XT.
template <int XT>
__device__ __forceinline__ uint32_t code_pair_16(uint32_t w) {
    uint32_t r;
    if constexpr (XT == kDtF16) {
        const uint32_t h = (w & 0x000F000Fu) | 0x64006400u;  // 1024 + code, twice
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64006400u));
    } else {
        const uint32_t h = (w & 0x000F000Fu) | 0x43004300u;  // 128 + code, twice
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x43004300u));
    }
    return r;
}

template <int XT>
__device__ __forceinline__ void mma_m16n8k16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if constexpr (XT == kDtF16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int XT, int OUT, int MM>
__global__ void __launch_bounds__(kQmThreads, 4)
    q4_mma_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ Q4Args a) {
    using Cfg = QmCfg<MM>;
    using OutT = typename Elem<OUT>::T;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::BAR_OFF);
    uint64_t *empty = full + Cfg::STAGES;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + Cfg::STAGES);
    float *part = reinterpret_cast<float *>(smem + Cfg::PART_OFF);  // [warp][row][column of x]

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int M = a.e.M, N = a.e.N, K = a.K;
    const int n0 = blockIdx.x * kQmRows;
    const int nvalid = min(kQmRows, N - n0);
    const int nchunks = (K + kQmChunk - 1) / kQmChunk;
    const int wp = a.w_pitch;  // bytes per weight row in a stage: the box width, min(160, K / 2)

    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmW);
        for (int st = 0; st < Cfg::STAGES; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], kQmConsumers);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kQmConsumers) {
        // Producer: lane 0 loads the weight box (rows past N and bytes past K / 2
        // read as zero), lanes below M copy the rows of x.
        const uint8_t *xg = static_cast<const uint8_t *>(a.X);
        const long long xrow = a.ldx * 2;  // bytes per row of x
        int issued = 0;
        for (int i = 0; i < nchunks; ++i) {
            const int st = i % Cfg::STAGES;
            if (i >= Cfg::STAGES) {
                const bool ok = mbar_wait_bounded(&empty[st], ((i / Cfg::STAGES) & 1) ^ 1, abort_flag, a.status);
                if (!__all_sync(0xffffffffu, ok)) break;
            }
            const int kc = min(kQmChunk, K - i * kQmChunk);
            const uint32_t xb = kc * 2;
            uint8_t *stage = smem + st * Cfg::STAGE_BYTES;
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[st], kQmRows * wp + M * xb);
                tma_load_2d(stage, &tmW, &full[st], i * (kQmChunk / 2), n0);
            }
            __syncwarp();
            if (lane < M)
                bulk_load_1d(stage + Cfg::W_BYTES + lane * kQmXPitch,
                             xg + (long long)lane * xrow + (long long)i * (kQmChunk * 2), xb, &full[st]);
            issued = i + 1;
        }
        // After an abort, let the copies already issued land before the block exits.
        if (*abort_flag && lane == 0)
            for (int j = max(0, issued - Cfg::STAGES); j < issued; ++j)
                mbar_drain_wait(&full[j % Cfg::STAGES], (j / Cfg::STAGES) & 1, kWaitLimitNs);
    } else {
        const int w = warp, g = lane >> 2, t = lane & 3;
        const long long gpr = K / 64;  // groups per weight row
        // This thread's rows: 16R + g (j = 2R) and 16R + g + 8 (j = 2R + 1).
        const uint32_t *sbrow[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int r = (j >> 1) * 16 + (j & 1) * 8 + g;
            sbrow[j] = a.SB + (long long)(n0 + (r < nvalid ? r : 0)) * gpr;
        }
        // Scale and bias of group w of a chunk, two chunks ahead.
        uint32_t sbc[4], sbn[4];
        auto load_sb = [&](int i, uint32_t (&d)[4]) {
            const long long G = 4LL * i + w;
#pragma unroll
            for (int j = 0; j < 4; ++j) d[j] = (i < nchunks && G < gpr) ? __ldg(sbrow[j] + G) : 0u;
        };
        load_sb(0, sbc);
        load_sb(1, sbn);
        float tot[2][4];
#pragma unroll
        for (int R = 0; R < 2; ++R)
#pragma unroll
            for (int c = 0; c < 4; ++c) tot[R][c] = 0.0f;

        for (int i = 0; i < nchunks; ++i) {
            const int st = i % Cfg::STAGES;
            const bool ok = mbar_wait_bounded(&full[st], (i / Cfg::STAGES) & 1, abort_flag, a.status);
            if (!__all_sync(0xffffffffu, ok)) break;
            const int ngroups = min(kQmChunk, K - i * kQmChunk) / 64;
            if (w < ngroups) {
                const uint8_t *stage = smem + st * Cfg::STAGE_BYTES;
                // x row g, k 16t .. 16t + 15 of group w (zero for rows past M)
                uint32_t v[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) v[q] = 0u;
                if (g < M) {
                    const uint8_t *xp = stage + Cfg::W_BYTES + g * kQmXPitch + 128 * w + 32 * t;
                    const uint4 p0 = *reinterpret_cast<const uint4 *>(xp);
                    const uint4 p1 = *reinterpret_cast<const uint4 *>(xp + 16);
                    v[0] = p0.x; v[1] = p0.y; v[2] = p0.z; v[3] = p0.w;
                    v[4] = p1.x; v[5] = p1.y; v[6] = p1.z; v[7] = p1.w;
                }
                // sum over the group of x row g (fp32), then the sums of rows 2t and 2t + 1
                uint64_t s2 = 0;
#pragma unroll
                for (int q = 0; q < 8; ++q) s2 = f2_add(s2, x_pair_f2<XT>(v[q]));
                float xs0, xs1;
                f2_unpack(s2, xs0, xs1);
                float xs = xs0 + xs1;
                xs += __shfl_xor_sync(0xffffffffu, xs, 1);
                xs += __shfl_xor_sync(0xffffffffu, xs, 2);
                const float xc0 = __shfl_sync(0xffffffffu, xs, 8 * t);
                const float xc1 = __shfl_sync(0xffffffffu, xs, 8 * t + 4);
                // B fragments of MMA h: (x_p, x_p+4) and (x_p+1, x_p+5), p = 8 (h / 2) + 2 (h % 2)
                uint32_t bf[4][2];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const uint32_t lo = v[4 * (h >> 1) + (h & 1)], hi = v[4 * (h >> 1) + (h & 1) + 2];
                    bf[h][0] = __byte_perm(lo, hi, 0x5410);
                    bf[h][1] = __byte_perm(lo, hi, 0x7632);
                }
#pragma unroll
                for (int R = 0; R < 2; ++R) {
                    const uint8_t *wrow = stage + (16 * R + g) * wp + 32 * w + 8 * t;
                    const uint2 wa = *reinterpret_cast<const uint2 *>(wrow);           // row 16R + g
                    const uint2 wb = *reinterpret_cast<const uint2 *>(wrow + 8 * wp);  // row 16R + g + 8
                    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const uint32_t ua = h < 2 ? wa.x : wa.y, ub = h < 2 ? wb.x : wb.y;
                        const int sh = (h & 1) * 8;
                        const uint32_t af[4] = {code_pair_16<XT>(ua >> sh), code_pair_16<XT>(ub >> sh),
                                                code_pair_16<XT>(ua >> (sh + 4)), code_pair_16<XT>(ub >> (sh + 4))};
                        mma_m16n8k16<XT>(d, af, bf[h][0], bf[h][1]);
                    }
                    const float2 sb0 = __half22float2(*reinterpret_cast<const __half2 *>(&sbc[2 * R]));
                    const float2 sb1 = __half22float2(*reinterpret_cast<const __half2 *>(&sbc[2 * R + 1]));
                    tot[R][0] = fmaf(sb0.x, d[0], fmaf(sb0.y, xc0, tot[R][0]));
                    tot[R][1] = fmaf(sb0.x, d[1], fmaf(sb0.y, xc1, tot[R][1]));
                    tot[R][2] = fmaf(sb1.x, d[2], fmaf(sb1.y, xc0, tot[R][2]));
                    tot[R][3] = fmaf(sb1.x, d[3], fmaf(sb1.y, xc1, tot[R][3]));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
#pragma unroll
            for (int j = 0; j < 4; ++j) sbc[j] = sbn[j];
            load_sb(i + 2, sbn);
        }
        // D fragment: (row g, x rows 2t, 2t + 1) and (row g + 8, same)
#pragma unroll
        for (int R = 0; R < 2; ++R) {
            float *p0 = part + (w * kQmRows + 16 * R + g) * 8 + 2 * t;
            p0[0] = tot[R][0];
            p0[1] = tot[R][1];
            p0[8 * 8] = tot[R][2];
            p0[8 * 8 + 1] = tot[R][3];
        }
    }
    __syncthreads();
    if (*abort_flag) return;
    // Sum the warps' partials in warp order; consecutive threads take consecutive n.
    for (int idx = threadIdx.x; idx < kQmRows * M; idx += blockDim.x) {
        const int r = idx % kQmRows, m = idx / kQmRows;
        if (r >= nvalid) continue;
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < kQmConsumers; ++w) v += part[(w * kQmRows + r) * 8 + m];
        const int n = n0 + r;
        const float b = (a.e.epilogue != kEpiNone) ? a.e.bias[n] : 0.0f;
        epilogue_store_one<OUT>(v, static_cast<OutT *>(a.e.C) + (long long)m * a.e.ldc + n, b, a.e);
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

// One block per kQmRows weight rows; the smallest x staging that holds M rows.
template <int XT, int OUT, int MM>
cudaError_t launch_mma_mm(const CUtensorMap &tmW, const Q4Args &a, cudaStream_t s) {
    using Cfg = QmCfg<MM>;
    auto kern = q4_mma_kernel<XT, OUT, MM>;
    const cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (err != cudaSuccess) return err;
    const long long blocks = (static_cast<long long>(a.e.N) + kQmRows - 1) / kQmRows;
    if (blocks > 2147483647LL) return cudaErrorInvalidConfiguration;
    kern<<<static_cast<unsigned>(blocks), kQmThreads, Cfg::SMEM, s>>>(tmW, a);
    return cudaGetLastError();
}

template <int XT, int OUT>
cudaError_t launch_rows(const CUtensorMap *tmW, const Q4Args &a, cudaStream_t s) {
    const int M = a.e.M;
    if (tmW != nullptr) {
        if (M <= 1) return launch_mma_mm<XT, OUT, 1>(*tmW, a, s);
        if (M <= 2) return launch_mma_mm<XT, OUT, 2>(*tmW, a, s);
        if (M <= 4) return launch_mma_mm<XT, OUT, 4>(*tmW, a, s);
        return launch_mma_mm<XT, OUT, 8>(*tmW, a, s);
    }
    return launch_gemv_rows<XT, OUT>(a, s);
}

}  // namespace

cudaError_t launch_q4_gemv(int x_dtype, int out, const CUtensorMap *tmW, const Q4Args &a, cudaStream_t s) {
    if (a.e.M < 1 || a.e.M > kQ4MaxRows) return cudaErrorInvalidValue;
    switch (x_dtype * 4 + out) {
    case kDtF16 * 4 + kDtF16: return launch_rows<kDtF16, kDtF16>(tmW, a, s);
    case kDtF16 * 4 + kDtBF16: return launch_rows<kDtF16, kDtBF16>(tmW, a, s);
    case kDtF16 * 4 + kDtF32: return launch_rows<kDtF16, kDtF32>(tmW, a, s);
    case kDtBF16 * 4 + kDtF16: return launch_rows<kDtBF16, kDtF16>(tmW, a, s);
    case kDtBF16 * 4 + kDtBF16: return launch_rows<kDtBF16, kDtBF16>(tmW, a, s);
    case kDtBF16 * 4 + kDtF32: return launch_rows<kDtBF16, kDtF32>(tmW, a, s);
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
