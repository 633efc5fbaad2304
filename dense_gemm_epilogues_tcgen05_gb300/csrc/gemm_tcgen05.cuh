// gemm_tcgen05.cuh -- persistent, warp-specialised GEMM on the sm_103a tensor
// cores with the epilogue fused before a single store.
//
// The pages' kernels stage A/B tiles in threadgroup memory, multiply 8x8
// fragments from registers and keep fp32 accumulators in registers for the
// whole K march ("X3: Metal GEMM" sections 3-4; "Case Study: Steel's
// BlockMMA", the mma() K-march and the Ctile with AccumType = float; "Case
// Study: The Tiled GEMM", the K-loop).  On this GPU the same roles map to:
//
//   warp 0 (one lane)   producer: TMA 2-D tiled loads of A and B k-blocks into
//                       a STAGES-deep shared-memory ring (128-byte swizzle),
//                       completion counted in bytes on full[s]; out-of-range
//                       rows / columns / k are zero-filled by the TMA unit
//                       (the zero fill of "X3" section 2).
//   warp 1 (one lane)   MMA issuer: tcgen05.mma 128 x BN x K_instr from shared
//                       memory descriptors into an fp32 accumulator in tensor
//                       memory; tcgen05.commit frees the stage (empty[s]) and,
//                       at the end of a tile, publishes the accumulator.
//   warps 2-5           epilogue: tcgen05.ld one TMEM lane (= one output row)
//                       per thread, 32 columns at a time; alpha / beta*C /
//                       bias / GELU / cast in registers, then one store (fast
//                       vector path or masked safe path).
//
// Transposition is carried by strides only (the A_str_m / A_str_k constants
// of Steel's BlockMMA): the host builds each operand's tensor map along its
// contiguous dimension, and the kernel flips the K-major / MN-major bit of the
// MMA instruction descriptor and the matching smem descriptor strides.
//
// The TMEM accumulator is double-buffered (2 x BN fp32 columns) so the
// epilogue of tile t overlaps the main loop of tile t+1.  CTAs walk output
// tiles t = blockIdx.x, blockIdx.x + gridDim.x, ... in a grouped order
// (group_m tile-rows at a time) so concurrently running CTAs share A row
// panels and B column panels in L2.
#pragma once

#include "epilogue.cuh"
#include "kernel_args.h"
#include "sm103_ptx.cuh"

namespace gb300 {

template <int AB> struct TcTraits;
template <> struct TcTraits<kDtF16> {
    static constexpr int kBytes = 2, kUmmaK = 16, kKind = kKindF16;
    static constexpr uint32_t kFmt = 0;
};
template <> struct TcTraits<kDtBF16> {
    static constexpr int kBytes = 2, kUmmaK = 16, kKind = kKindF16;
    static constexpr uint32_t kFmt = 1;
};
template <> struct TcTraits<kDtE4M3> {
    static constexpr int kBytes = 1, kUmmaK = 32, kKind = kKindF8F6F4;
    static constexpr uint32_t kFmt = 0;
};
template <> struct TcTraits<kDtTF32x3> {
    static constexpr int kBytes = 4, kUmmaK = 8, kKind = kKindTF32;
    static constexpr uint32_t kFmt = 2;
};

template <int AB, int BN_, int STAGES_>
struct TcConfig {
    static constexpr int BM = 128;
    static constexpr int BN = BN_;
    static constexpr int STAGES = STAGES_;
    static constexpr int ES = TcTraits<AB>::kBytes;
    static constexpr int SWZ = 128 / ES;           // elements in one 128-byte swizzle row
    static constexpr int BK = SWZ;                 // a k-block is one swizzle row of K
    static constexpr int UMMA_K = TcTraits<AB>::kUmmaK;
    static constexpr int KSTEPS = BK / UMMA_K;
    static constexpr int A_BYTES = BM * BK * ES;
    static constexpr int B_BYTES = BN * BK * ES;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int EPI_WARPS = 4;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "MMA N for M=128 is a multiple of 16 up to 256");
    static_assert(KSTEPS * UMMA_K == BK, "k-block holds whole MMAs");
    static_assert((TMEM_COLS & (TMEM_COLS - 1)) == 0 && TMEM_COLS >= 32 && TMEM_COLS <= 512, "TMEM cols");
    static_assert(BN % SWZ == 0 && BM % SWZ == 0, "MN-major tiles are whole swizzle atoms");
    static_assert(SMEM_BYTES <= 232448, "fits the 227 KB opt-in shared memory");
    // One CTA per SM, so TMEM allocation never waits on a co-resident CTA.
    static_assert(SMEM_BYTES > 232448 / 2 || TMEM_COLS <= 256, "co-resident CTAs must fit TMEM");
};

__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int group_m, int &tm, int &tn) {
    const int per_group = group_m * tiles_n;
    const int g = tile / per_group;
    const int first_m = g * group_m;
    const int gsize = min(tiles_m - first_m, group_m);
    const int r = tile - g * per_group;
    tm = first_m + r % gsize;
    tn = r / gsize;
}

template <int AB, int OUT, int BN, int STAGES>
__global__ void __launch_bounds__(TcConfig<AB, BN, STAGES>::THREADS, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const TcArgs args) {
    using Cfg = TcConfig<AB, BN, STAGES>;
    constexpr int BM = Cfg::BM, BK = Cfg::BK, SWZ = Cfg::SWZ;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * Cfg::STAGE_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *mma_done = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], Cfg::EPI_WARPS);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int M = args.e.M, N = args.e.N;
    const int num_kb = args.num_kb;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer --
            uint32_t stage = 0, phase = 0;
            uint32_t armed = 0;        // stages armed at least once (bit mask)
            uint32_t armed_parity = 0; // parity of the last arming, per stage
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < args.num_tiles; tile += gridDim.x) {
                int tm, tn;
                tile_coords(tile, args.tiles_m, args.tiles_n, args.group_m, tm, tn);
                const int m0 = tm * BM, n0 = tn * BN;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], Cfg::STAGE_BYTES);
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    unsigned char *sA = smem + stage * Cfg::STAGE_BYTES;
                    unsigned char *sB = sA + Cfg::A_BYTES;
                    const int k0 = kb * BK;
                    if (!args.a_mn_major) {
                        tma_load_2d(sA, &tmA, &full[stage], k0, m0);
                    } else {
#pragma unroll
                        for (int j = 0; j < BM / SWZ; ++j)
                            tma_load_2d(sA + j * 128 * BK, &tmA, &full[stage], m0 + j * SWZ, k0);
                    }
                    if (!args.b_mn_major) {
                        tma_load_2d(sB, &tmB, &full[stage], k0, n0);
                    } else {
#pragma unroll
                        for (int j = 0; j < BN / SWZ; ++j)
                            tma_load_2d(sB + j * 128 * BK, &tmB, &full[stage], n0 + j * SWZ, k0);
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (*abort_flag) {
                // Unwinding: let every load already issued land before the
                // CTA's shared memory goes away.
                for (int s = 0; s < STAGES; ++s)
                    if (armed & (1u << s)) mbar_drain_wait(&full[s], (armed_parity >> s) & 1u, 100000000ull);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // --------------------------------------------------- MMA issuer --
            constexpr uint32_t kIdesc = mma_idesc(TcTraits<AB>::kFmt, TcTraits<AB>::kFmt, BM, BN);
            const uint32_t idesc = kIdesc | (args.a_mn_major << 15) | (args.b_mn_major << 16);
            // K-major: LBO unused (one swizzle row spans the k-block), SBO =
            // 8 rows x 128 B; k advances 32 B inside the swizzle row.
            // MN-major: LBO = bytes between 128-byte-wide MN blocks (one TMA
            // box), SBO = 8 k-rows x 128 B; k advances whole 8-row groups.
            const uint32_t a_lbo = args.a_mn_major ? 128u * BK : 16u;
            const uint32_t b_lbo = args.b_mn_major ? 128u * BK : 16u;
            const uint32_t a_kstep = args.a_mn_major ? 128u * Cfg::UMMA_K : 32u;
            const uint32_t b_kstep = args.b_mn_major ? 128u * Cfg::UMMA_K : 32u;
            uint32_t stage = 0, phase = 0;
            bool ok = true, issued = false;
            int local = 0;
            for (int tile = blockIdx.x; ok && tile < args.num_tiles; tile += gridDim.x, ++local) {
                const uint32_t acc = local & 1, acc_phase = (local >> 1) & 1;
                if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, args.status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait_bounded(&full[stage], phase, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + stage * Cfg::STAGE_BYTES);
                    const uint32_t b_addr = a_addr + Cfg::A_BYTES;
#pragma unroll
                    for (int ks = 0; ks < Cfg::KSTEPS; ++ks) {
                        const uint64_t ad = sw128_desc(a_addr + ks * a_kstep, a_lbo, 1024u);
                        const uint64_t bd = sw128_desc(b_addr + ks * b_kstep, b_lbo, 1024u);
                        tc_mma<TcTraits<AB>::kKind>(d_tmem, ad, bd, idesc, (kb | ks) != 0 ? 1u : 0u);
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
    } else {
        // ------------------------------------------------------- epilogue --
        const int quad = warp & 3;  // TMEM lanes this warp may read: 32*quad .. 32*quad+31
        const int row_in_tile = quad * 32 + lane;
        const EpiParams &e = args.e;
        int local = 0;
        for (int tile = blockIdx.x; tile < args.num_tiles; tile += gridDim.x, ++local) {
            const uint32_t acc = local & 1, acc_phase = (local >> 1) & 1;
            int tm, tn;
            tile_coords(tile, args.tiles_m, args.tiles_n, args.group_m, tm, tn);
            const int m0 = tm * BM, n0 = tn * BN;
            const bool got = mbar_wait_bounded(&tfull[acc], acc_phase, abort_flag, args.status);
            if (__any_sync(0xffffffffu, !got)) break;  // warp-uniform exit
            tc_fence_after();
            const int row = m0 + row_in_tile;
            const bool row_ok = row < M;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN;
            int nvalid = BN / 32;
            const int left = (N - n0 + 31) >> 5;  // chunks that start inside the matrix
            if (left < nvalid) nvalid = left;
            epilogue_row_chunks<OUT, BN / 32>(t_row, n0, nvalid, row, row_ok, e.bias + n0, e);
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

template <int AB, int OUT, int BN, int STAGES>
cudaError_t launch_tcgen05_cfg(const CUtensorMap &ta, const CUtensorMap &tb, const TcArgs &args, int grid,
                               cudaStream_t stream) {
    using Cfg = TcConfig<AB, BN, STAGES>;
    auto kern = gemm_tcgen05_kernel<AB, OUT, BN, STAGES>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    kern<<<grid, Cfg::THREADS, Cfg::SMEM_BYTES, stream>>>(ta, tb, args);
    return cudaGetLastError();
}

}  // namespace gb300
