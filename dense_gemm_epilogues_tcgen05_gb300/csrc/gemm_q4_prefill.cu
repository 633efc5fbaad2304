// gemm_q4_prefill.cu -- the 4-bit group-quantized product for many rows of x
// (prefill), with the dequantisation fused into the tensor-core product.
//
// "X3: Metal GEMM" section 7 names quantized matmul as the main LLM workload,
// a GEMM with the dequantisation fused into the multiply-accumulate when the
// prompt is filled.  With W = s*q + b per group of 64 k (gemm_gb300.h), the
// kernel computes the transposed product C^T = W x^T on the tensor cores:
//
//   warp 0 (one lane)  TMA loads, per stage of one 64-k group: 128 rows of x
//                      (the MMA's B operand, 128-byte swizzle, zero fill past
//                      M and K) and the 4-bit codes of 128 rows of W (32 bytes
//                      a row, zero fill past N);
//   warps 2-9          converters: two warps per 32 rows of W, one thread per
//                      row and half-group, 32 codes to 32 16-bit values
//                      round(s*q + b) (exact q, one rounding), stored straight
//                      into tensor memory with tcgen05.st -- the MMA's A
//                      operand, so dequantised W never touches shared memory
//                      or HBM (one warp per 32 rows measured latency-bound:
//                      a stage took three times its MMAs);
//   warp 1 (one lane)  tcgen05.mma kind::f16 with A from tensor memory (W) and
//                      B from shared memory (x) into one of two fp32
//                      accumulators (TMEM lanes = rows of W = output columns);
//   warps 10-13        epilogue: alpha, beta*C, bias, activation, cast; each
//                      thread holds one output column, 32 rows at a time, and a
//                      warp's stores of one row are 32 consecutive columns.
//
// The product in each accumulator is sum_k W[n][k] x[m][k] in fp32 over the
// rounded 16-bit W, the same rounding gemm_q4_dequantize applies.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "epilogue.cuh"
#include "gemm_tcgen05.cuh"
#include "kernel_args.h"
#include "sm103_ptx.cuh"

namespace gb300 {

template <int STAGES_>
struct Q4PConfig {
    static constexpr int BW = 128;                     // rows of W per tile (TMEM lanes)
    static constexpr int BX = 128;                     // rows of x per tile (MMA N)
    static constexpr int GROUP = 64;                   // k per stage: one quantisation group
    static constexpr int STAGES = STAGES_;
    static constexpr int X_BYTES = BX * GROUP * 2;     // 16 KB: 128 rows x 128 bytes
    static constexpr int CODE_BYTES = BW * GROUP / 2;  // 4 KB: 128 rows x 32 bytes
    static constexpr int STAGE_BYTES = X_BYTES + CODE_BYTES;
    static constexpr int ACC_COLS = 2 * BX;            // two fp32 accumulators
    static constexpr int W_SLOT_COLS = GROUP / 2;      // a stage's W: two 16-bit values a column
    static constexpr int TMEM_COLS = 512;
    static constexpr int CONV_WARPS = 8, EPI_WARPS = 4;  // converters: two per TMEM lane quadrant
    static constexpr int THREADS = 64 + 32 * (CONV_WARPS + EPI_WARPS);
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
    static_assert(STAGE_BYTES % 1024 == 0, "stages stay 1024-byte aligned (128-byte swizzle atoms)");
    static_assert(ACC_COLS + STAGES * W_SLOT_COLS <= TMEM_COLS, "W slots fit beside the accumulators");
    static_assert((3 * STAGES + 5) * 8 + 8 <= BAR_BYTES, "barriers fit their slot");
    static_assert(SMEM_BYTES <= 232448, "fits the 227 KB opt-in shared memory");
    static_assert(SMEM_BYTES > 232448 / 2, "one CTA per SM: it allocates all 512 TMEM columns");
};

// Two codes (low nibble: even k, high nibble: odd k) of byte j of `w`, scaled
// and offset: the packed pair (round(s*q_even + b), round(s*q_odd + b)) in the
// element type of x.
template <int XT>
__device__ __forceinline__ uint32_t dequant_pair(uint32_t w, int j, float s, float b, __half2 s2, __half2 b2) {
    if constexpr (XT == kDtF16) {
        // byte j into bytes 0 and 2; its low nibble as the low half's low
        // mantissa bits and its high nibble as the high half's bits 4-7, over
        // the exponent of 1024: (1024 + q_even, 1024 + 16 q_odd), exact; one
        // multiply-add recovers (q_even, q_odd) exactly, one more gives
        // s*q + b rounded once to fp16.
        const uint32_t u = __byte_perm(w, 0u, static_cast<uint32_t>(0x4040 | (j << 8) | j));
        const uint32_t h = (u & 0x00F0000Fu) | 0x64006400u;
        const __half2 q = __hfma2(*reinterpret_cast<const __half2 *>(&h), __halves2half2(__float2half(1.0f), __float2half(0.0625f)),
                                  __halves2half2(__float2half(-1024.0f), __float2half(-64.0f)));
        const __half2 r = __hfma2(q, s2, b2);
        return *reinterpret_cast<const uint32_t *>(&r);
    } else {
        // q as fp32 (2^23 + q minus 2^23, exact), s*q + b by one fused
        // multiply-add (exact for these formats), then rounded once to bf16.
        const uint32_t byte = (w >> (8 * j)) & 0xFFu;
        const float q0 = __uint_as_float(0x4B000000u | (byte & 0xFu)) - 8388608.0f;
        const float q1 = __uint_as_float(0x4B000000u | (byte >> 4)) - 8388608.0f;
        const __nv_bfloat162 r = __floats2bfloat162_rn(fmaf(s, q0, b), fmaf(s, q1, b));
        return *reinterpret_cast<const uint32_t *>(&r);
    }
}

template <int XT, int OUT, int STAGES>
__global__ void __launch_bounds__(Q4PConfig<STAGES>::THREADS, 1)
    q4_prefill_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                      const __grid_constant__ Q4Args args) {
    using Cfg = Q4PConfig<STAGES>;
    constexpr int BW = Cfg::BW, BX = Cfg::BX;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * Cfg::STAGE_BYTES);
    uint64_t *wready = full + STAGES;
    uint64_t *empty = wready + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *mma_done = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const EpiParams &e = args.e;
    const int M = e.M, N = e.N;
    const int num_kb = args.K / Cfg::GROUP;
    const int tiles_w = (N + BW - 1) / BW, tiles_x = (M + BX - 1) / BX;
    const int num_tiles = tiles_w * tiles_x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&wready[s], Cfg::CONV_WARPS);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], Cfg::EPI_WARPS);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ----------------------------------------------------- producer --
            uint32_t stage = 0, phase = 0, armed = 0, armed_parity = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                int tw, tx;
                tile_coords(tile, tiles_w, tiles_x, 8, tw, tx);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], Cfg::STAGE_BYTES);
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    unsigned char *sX = smem + stage * Cfg::STAGE_BYTES;
                    tma_load_2d(sX, &tmX, &full[stage], kb * Cfg::GROUP, tx * BX);
                    tma_load_2d(sX + Cfg::X_BYTES, &tmW, &full[stage], kb * (Cfg::GROUP / 2), tw * BW);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (*abort_flag) {
                for (int s = 0; s < STAGES; ++s)
                    if (armed & (1u << s)) mbar_drain_wait(&full[s], (armed_parity >> s) & 1u, 100000000ull);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // --------------------------------------------------- MMA issuer --
            constexpr uint32_t kIdesc = mma_idesc(TcTraits<XT>::kFmt, TcTraits<XT>::kFmt, BW, BX);
            uint32_t stage = 0, phase = 0;
            bool ok = true, issued = false;
            int local = 0;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++local) {
                const uint32_t acc = local & 1, acc_phase = (local >> 1) & 1;
                if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, args.status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BX;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait_bounded(&full[stage], phase, abort_flag, args.status) ||
                        !mbar_wait_bounded(&wready[stage], phase, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t x_addr = smem_u32(smem + stage * Cfg::STAGE_BYTES);
                    const uint32_t w_tmem = tmem_base + Cfg::ACC_COLS + stage * Cfg::W_SLOT_COLS;
#pragma unroll
                    for (int ks = 0; ks < Cfg::GROUP / 16; ++ks) {
                        // 16 k a step: 8 columns of W, 32 bytes of each x row
                        const uint64_t bd = sw128_desc(x_addr + ks * 32, 16u, 1024u);
                        tc_mma_f16_tmem_a(d_tmem, w_tmem + ks * 8, bd, kIdesc, (kb | ks) != 0 ? 1u : 0u);
                    }
                    issued = true;
                    tc_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) tc_commit(&tfull[acc]);
            }
            if (*abort_flag && issued) {
                tc_commit(mma_done);
                mbar_drain_wait(mma_done, 0, 100000000ull);
            }
        }
    } else if (warp < 2 + Cfg::CONV_WARPS) {
        // ----------------------------------------------------- converters --
        // TMEM lanes 32*(warp%4) .. +31 are this warp's; its thread r holds row
        // r of the tile's W, half `hk` of each group (k 32 hk .. 32 hk + 31).
        const int quad = warp & 3;
        const int hk = (warp - 2) >> 2;
        const int r = quad * 32 + lane;
        const int words_per_row = args.K / Cfg::GROUP;  // (scale, bias) words of one row of W
        uint32_t stage = 0, phase = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            int tw, tx;
            tile_coords(tile, tiles_w, tiles_x, 8, tw, tx);
            const int n = tw * BW + r;
            const uint32_t *sb_row = args.SB + static_cast<long long>(n < N ? n : 0) * words_per_row;
            uint32_t sb_next = n < N ? __ldg(sb_row) : 0u;
            bool ok = true;
            for (int kb = 0; kb < num_kb; ++kb) {
                const uint32_t sb = sb_next;
                if (kb + 1 < num_kb) sb_next = n < N ? __ldg(sb_row + kb + 1) : 0u;  // next group's, early
                const bool got = mbar_wait_bounded(&full[stage], phase, abort_flag, args.status);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const __half2 sb2 = *reinterpret_cast<const __half2 *>(&sb);
                const float s = __low2float(sb2), b = __high2float(sb2);
                const __half2 s2 = __low2half2(sb2), b2 = __high2half2(sb2);
                const uint4 c = *reinterpret_cast<const uint4 *>(smem + stage * Cfg::STAGE_BYTES + Cfg::X_BYTES +
                                                                 r * 32 + hk * 16);
                const uint32_t w4[4] = {c.x, c.y, c.z, c.w};
                uint32_t out[16];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) out[4 * i + j] = dequant_pair<XT>(w4[i], j, s, b, s2, b2);
                const uint32_t slot = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + Cfg::ACC_COLS +
                                      stage * Cfg::W_SLOT_COLS + hk * 16;
                tmem_st_x16(slot, out);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&wready[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
        }
    } else {
        // ------------------------------------------------------- epilogue --
        using OutT = typename Elem<OUT>::T;
        const int quad = warp & 3;
        OutT *C = static_cast<OutT *>(e.C);
        int local = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
            const uint32_t acc = local & 1, acc_phase = (local >> 1) & 1;
            int tw, tx;
            tile_coords(tile, tiles_w, tiles_x, 8, tw, tx);
            const bool got = mbar_wait_bounded(&tfull[acc], acc_phase, abort_flag, args.status);
            if (__any_sync(0xffffffffu, !got)) break;
            tc_fence_after();
            const int n = tw * BW + quad * 32 + lane;  // this thread's output column
            const bool n_ok = n < N;
            const float bias_n = (e.epilogue != kEpiNone && n_ok) ? e.bias[n] : 0.0f;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BX;
#pragma unroll 1
            for (int c = 0; c < BX / 32; ++c) {
                const int m0 = tx * BX + c * 32;
                if (m0 >= M) break;  // warp-uniform
                uint32_t raw[32];
                __syncwarp();
                tmem_ld_issue(t_row + c * 32, raw);
                tmem_ld_wait(raw);
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = e.alpha * __uint_as_float(raw[j]);
                if (e.beta != 0.0f) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (n_ok && m0 + j < M)
                            v[j] = fmaf(e.beta, Elem<OUT>::load(C + static_cast<long long>(m0 + j) * e.ldc + n), v[j]);
                }
                if (e.epilogue != kEpiNone) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] += bias_n;
                    if (e.epilogue >= kEpiBiasGelu) activate_run<OUT, 32>(v, 0, e.epilogue, false);
                }
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (n_ok && m0 + j < M) C[static_cast<long long>(m0 + j) * e.ldc + n] = Elem<OUT>::cvt(v[j]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

template <int XT, int OUT>
cudaError_t launch_q4p_cfg(const CUtensorMap &tmX, const CUtensorMap &tmW, const Q4Args &args, int grid,
                           cudaStream_t stream) {
    constexpr int STAGES = 8;
    using Cfg = Q4PConfig<STAGES>;
    auto kern = q4_prefill_kernel<XT, OUT, STAGES>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    kern<<<grid, Cfg::THREADS, Cfg::SMEM_BYTES, stream>>>(tmX, tmW, args);
    return cudaGetLastError();
}

cudaError_t launch_q4_prefill(int x_dtype, int out, const CUtensorMap &tmX, const CUtensorMap &tmW, const Q4Args &args,
                              int grid, cudaStream_t stream) {
    if (x_dtype == kDtF16) {
        if (out == kDtF32) return launch_q4p_cfg<kDtF16, kDtF32>(tmX, tmW, args, grid, stream);
        if (out == kDtF16) return launch_q4p_cfg<kDtF16, kDtF16>(tmX, tmW, args, grid, stream);
        if (out == kDtBF16) return launch_q4p_cfg<kDtF16, kDtBF16>(tmX, tmW, args, grid, stream);
    } else if (x_dtype == kDtBF16) {
        if (out == kDtF32) return launch_q4p_cfg<kDtBF16, kDtF32>(tmX, tmW, args, grid, stream);
        if (out == kDtF16) return launch_q4p_cfg<kDtBF16, kDtF16>(tmX, tmW, args, grid, stream);
        if (out == kDtBF16) return launch_q4p_cfg<kDtBF16, kDtBF16>(tmX, tmW, args, grid, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gb300
