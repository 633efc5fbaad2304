// gemm_mx.cu -- block-scaled ("MX") matrix product on the sm_103a tensor cores.
//
// Rigel section 1 lists fp4 and block-scaled MXFP4 next to fp8 among the
// low-precision rows of the matrix units without defining them; the formats
// are those of the OCP Microscaling (MX) specification v1.0: 32 consecutive
// elements along k share one E8M0 scale 2^(code - 127), elements are E4M3
// (MXFP8) or E2M1 (MXFP4).  The product is the dense one with every element
// multiplied by its block's scale:
//
//     C = cast(epilogue(alpha * sum_k (X^A[i][k/32] P^A[i][k]) (X^B[j][k/32] P^B[j][k])
//                       + beta*C + bias))
//
// and the tensor cores apply the scales themselves: tcgen05.mma
// kind::mxf8f6f4 (one scale per 32 k, K = 32 a instruction) or kind::mxf4
// (two scales, K = 64 of packed E2M1), each scale read from tensor memory.
//
// Roles (one SM per 128 x 256 output tile, persistent over tiles):
//   warp 0 (one lane)  TMA loads of 128 bytes of K of 128 rows of A and 256
//                      rows of B into a STAGES-deep ring (128-byte swizzle,
//                      zero fill past M, N and K), plus bulk copies of the
//                      stage's scale chunks (A's row block, B's two);
//   warp 1 (one lane)  tcgen05.cp of the chunks into the stage's tensor-memory
//                      scale slot (32x128b, replicated to the four lane
//                      groups: row r's scales in column r / 32 of the slot's
//                      part, so B's 256 rows take eight columns), then the
//                      block-scaled MMAs (N = 256) into the fp32 accumulator
//                      (columns 0-255; the scale slots follow);
//   warps 2-9          the shared epilogue (alpha, beta*C, bias, activation,
//                      cast), one row and half the columns per thread.
// The scales arrive row-major (M x K/32, N x K/32) and a pre-pass rewrites them
// into 512-byte chunks of 128 rows x 4 blocks in the order the tensor-memory
// copy expects (see MxArgs).
//
// Why 256 columns: every byte of a stage crosses shared memory twice (TMA
// write, MMA read), and a 128 x 128 tile moved 256 bytes a clock through it at
// the full MMA rate, twice what it delivers, so that kernel ran at a third of
// the tensor rate.  B 256 rows wide cuts that to 192.  A 256-column
// accumulator leaves tensor memory room for one accumulator beside the scale
// slots, so a tile's epilogue (eight warps) runs before the next tile's MMAs
// start, while the producer keeps loading the next tile's stages.  (Moving
// the accumulator into registers first, 128 values a thread, and releasing it
// at once spilled more than a kilobyte a thread at the 168-register cap of a
// 10-warp CTA.)
#include "epilogue.cuh"
#include "gemm_tcgen05.cuh"
#include "kernel_args.h"
#include "mx_traits.cuh"
#include "sm103_ptx.cuh"

namespace gb300 {

template <int ELEM, int STAGES_>
struct MxConfig {
    static constexpr int BM = 128, BN = 256;
    static constexpr int STAGES = STAGES_;
    static constexpr int ROW_BYTES = 128;                         // bytes of K per stage
    static constexpr int MMAS = 4;                                // 32 bytes of K each
    static constexpr int CHUNKS = MxTraits<ELEM>::kChunks;
    static constexpr int A_BYTES = BM * ROW_BYTES;
    static constexpr int B_BYTES = BN * ROW_BYTES;
    static constexpr int SFA_OFF = A_BYTES + B_BYTES;
    static constexpr int SFB_OFF = SFA_OFF + CHUNKS * 512;         // B's row blocks 0 and 1, CHUNKS each
    static constexpr int STAGE_TX = SFB_OFF + 2 * CHUNKS * 512;    // bytes a stage receives
    static constexpr int STAGE_BYTES = (STAGE_TX + 1023) / 1024 * 1024;
    static constexpr int ACC_COLS = BN;                           // one accumulator
    static constexpr int SF_SLOT_COLS = 12 * CHUNKS;              // A: 4 per chunk; B: 8 per chunk
    static constexpr int TMEM_COLS = 512;
    static constexpr int EPI_WARPS = 8;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
    static_assert(ACC_COLS + STAGES * SF_SLOT_COLS <= TMEM_COLS, "scale slots fit beside the accumulator");
    static_assert((2 * STAGES + 3) * 8 + 8 <= BAR_BYTES, "barriers fit their slot");
    static_assert(SMEM_BYTES <= 232448, "fits the 227 KB opt-in shared memory");
    static_assert(SMEM_BYTES > 232448 / 2, "one CTA per SM: it allocates all 512 TMEM columns");
};

template <int ELEM, int OUT, int STAGES>
__global__ void __launch_bounds__(MxConfig<ELEM, STAGES>::THREADS, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ MxArgs args) {
    using Cfg = MxConfig<ELEM, STAGES>;
    constexpr int BM = Cfg::BM, BN = Cfg::BN;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * Cfg::STAGE_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 1;
    uint64_t *mma_done = tempty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tfull, 1);
        mbar_init(tempty, Cfg::EPI_WARPS);
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
            // ----------------------------------------------------- producer --
            uint32_t stage = 0, phase = 0;
            uint32_t armed = 0, armed_parity = 0;
            bool ok = true;
            const long long rb_b = (N + 127) / 128;  // B's row blocks in the scale pack
            for (int tile = blockIdx.x; ok && tile < args.num_tiles; tile += gridDim.x) {
                int tm, tn;
                tile_coords(tile, args.tiles_m, args.tiles_n, args.group_m, tm, tn);
                const unsigned char *sfa_row = args.sfa + static_cast<long long>(tm) * args.kc_count * 512;
                // B's second row block of the tile; past N it does not exist in the
                // pack, and the first one stands in (those rows of B are zero-filled).
                const long long rb0 = 2LL * tn, rb1 = rb0 + 1 < rb_b ? rb0 + 1 : rb0;
                const unsigned char *sfb_row0 = args.sfb + rb0 * args.kc_count * 512;
                const unsigned char *sfb_row1 = args.sfb + rb1 * args.kc_count * 512;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], Cfg::STAGE_TX);
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    unsigned char *sA = smem + stage * Cfg::STAGE_BYTES;
                    tma_load_2d(sA, &tmA, &full[stage], kb * Cfg::ROW_BYTES, tm * BM);
                    tma_load_2d(sA + Cfg::A_BYTES, &tmB, &full[stage], kb * Cfg::ROW_BYTES, tn * BN);
                    const long long chunk = static_cast<long long>(kb) * Cfg::CHUNKS * 512;
                    bulk_load_1d(sA + Cfg::SFA_OFF, sfa_row + chunk, Cfg::CHUNKS * 512, &full[stage]);
                    bulk_load_1d(sA + Cfg::SFB_OFF, sfb_row0 + chunk, Cfg::CHUNKS * 512, &full[stage]);
                    bulk_load_1d(sA + Cfg::SFB_OFF + Cfg::CHUNKS * 512, sfb_row1 + chunk, Cfg::CHUNKS * 512,
                                 &full[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (*abort_flag) {
                // Unwinding: let every copy already issued land before the CTA's
                // shared memory goes away.
                for (int s = 0; s < STAGES; ++s)
                    if (armed & (1u << s)) mbar_drain_wait(&full[s], (armed_parity >> s) & 1u, 100000000ull);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // --------------------------------------------------- MMA issuer --
            uint32_t stage = 0, phase = 0;
            bool ok = true, issued = false;
            int local = 0;
            for (int tile = blockIdx.x; ok && tile < args.num_tiles; tile += gridDim.x, ++local) {
                if (!mbar_wait_bounded(tempty, (local & 1) ^ 1u, abort_flag, args.status)) break;
                tc_fence_after();
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait_bounded(&full[stage], phase, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + stage * Cfg::STAGE_BYTES);
                    const uint32_t b_addr = a_addr + Cfg::A_BYTES;
                    // this stage's scale slot: A's chunks (4 columns each), then B's
                    // (8 columns each: rows 0-127, then rows 128-255)
                    const uint32_t sfa_t = tmem_base + Cfg::ACC_COLS + stage * Cfg::SF_SLOT_COLS;
                    const uint32_t sfb_t = sfa_t + 4 * Cfg::CHUNKS;
#pragma unroll
                    for (int c = 0; c < Cfg::CHUNKS; ++c) {
                        tc_cp_32x128b_x4(sfa_t + 4 * c, plain16_desc(a_addr + Cfg::SFA_OFF + 512 * c));
                        tc_cp_32x128b_x4(sfb_t + 8 * c, plain16_desc(a_addr + Cfg::SFB_OFF + 512 * c));
                        tc_cp_32x128b_x4(sfb_t + 8 * c + 4,
                                         plain16_desc(a_addr + Cfg::SFB_OFF + Cfg::CHUNKS * 512 + 512 * c));
                    }
#pragma unroll
                    for (int ks = 0; ks < Cfg::MMAS; ++ks) {
                        // MXFP8: MMA ks uses block ks of the one chunk.  MXFP4: blocks
                        // 2 ks, 2 ks + 1 -- chunk ks / 2, bytes 2 (ks % 2) and the next.
                        const uint32_t chunk = Cfg::CHUNKS == 1 ? 0u : static_cast<uint32_t>(ks >> 1);
                        const uint32_t sf_id = Cfg::CHUNKS == 1 ? static_cast<uint32_t>(ks)
                                                                : static_cast<uint32_t>((ks & 1) * 2);
                        const uint32_t idesc = mma_idesc_bs(MxTraits<ELEM>::kFmt, BM, BN, sf_id, sf_id);
                        const uint64_t ad = sw128_desc(a_addr + ks * 32, 16u, 1024u);
                        const uint64_t bd = sw128_desc(b_addr + ks * 32, 16u, 1024u);
                        tc_mma_bs<MxTraits<ELEM>::kKind>(tmem_base, ad, bd, idesc, sfa_t + 4 * chunk,
                                                         sfb_t + 8 * chunk, (kb | ks) != 0 ? 1u : 0u);
                    }
                    issued = true;
                    tc_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) tc_commit(tfull);
            }
            if (*abort_flag && issued) {
                tc_commit(mma_done);
                mbar_drain_wait(mma_done, 0, 100000000ull);
            }
        }
    } else {
        // ------------------------------------------------------- epilogue --
        const int quad = warp & 3;           // TMEM lanes this warp may read: 32*quad .. 32*quad+31
        const int half = (warp - 2) >> 2;    // which 128 of the tile's 256 columns
        const EpiParams &e = args.e;
        int local = 0;
        for (int tile = blockIdx.x; tile < args.num_tiles; tile += gridDim.x, ++local) {
            int tm, tn;
            tile_coords(tile, args.tiles_m, args.tiles_n, args.group_m, tm, tn);
            const int m0 = tm * BM, col_base = tn * BN + half * 128;
            const bool got = mbar_wait_bounded(tfull, local & 1, abort_flag, args.status);
            if (__any_sync(0xffffffffu, !got)) break;  // warp-uniform exit
            tc_fence_after();
            const int row = m0 + quad * 32 + lane;
            const bool row_ok = row < M;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + half * 128;
            int nvalid = (N - col_base + 31) >> 5;  // chunks that start inside the matrix
            nvalid = nvalid < 0 ? 0 : (nvalid > 4 ? 4 : nvalid);
            epilogue_row_chunks<OUT, 4, false>(t_row, col_base, nvalid, row, row_ok, e.bias + col_base, e);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty);
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

// Row-major scale codes (rows x blocks, row pitch `blocks`) into the chunk
// layout of MxArgs: one thread per destination byte; scales of rows or blocks
// past the operand read as 127 (2^0).
__global__ void mx_sf_pack_kernel(const unsigned char *__restrict__ src, long long rows, long long blocks,
                                  unsigned char *__restrict__ dst, long long total, long long kc_count) {
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long chunk = i >> 9;
        const int within = static_cast<int>(i & 511);
        const long long rb = chunk / kc_count, kc = chunk - rb * kc_count;
        const int l = within >> 4, g = (within >> 2) & 3, j = within & 3;
        const long long row = rb * 128 + g * 32 + l, blk = kc * 4 + j;
        dst[i] = (row < rows && blk < blocks) ? src[row * blocks + blk] : static_cast<unsigned char>(127);
    }
}

template <int ELEM, int OUT>
cudaError_t launch_mx_cfg(const CUtensorMap &ta, const CUtensorMap &tb, const MxArgs &args, int grid,
                          cudaStream_t stream) {
    constexpr int STAGES = 4;
    using Cfg = MxConfig<ELEM, STAGES>;
    auto kern = gemm_mx_kernel<ELEM, OUT, STAGES>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    kern<<<grid, Cfg::THREADS, Cfg::SMEM_BYTES, stream>>>(ta, tb, args);
    return cudaGetLastError();
}

cudaError_t launch_mx(int elem, int out, const CUtensorMap &ta, const CUtensorMap &tb, const MxArgs &args, int grid,
                      cudaStream_t stream) {
    if (elem == kMxE4M3) {
        if (out == kDtF32) return launch_mx_cfg<kMxE4M3, kDtF32>(ta, tb, args, grid, stream);
        if (out == kDtF16) return launch_mx_cfg<kMxE4M3, kDtF16>(ta, tb, args, grid, stream);
        if (out == kDtBF16) return launch_mx_cfg<kMxE4M3, kDtBF16>(ta, tb, args, grid, stream);
    } else if (elem == kMxE2M1) {
        if (out == kDtF32) return launch_mx_cfg<kMxE2M1, kDtF32>(ta, tb, args, grid, stream);
        if (out == kDtF16) return launch_mx_cfg<kMxE2M1, kDtF16>(ta, tb, args, grid, stream);
        if (out == kDtBF16) return launch_mx_cfg<kMxE2M1, kDtBF16>(ta, tb, args, grid, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_mx_sf_pack(const unsigned char *src, long long rows, long long blocks, unsigned char *dst,
                              long long row_blocks, long long kc_count, cudaStream_t stream) {
    const long long total = row_blocks * kc_count * 512;
    if (total <= 0) return cudaSuccess;
    const long long want = (total + 255) / 256;
    const int grid = static_cast<int>(want < 4096 ? want : 4096);
    mx_sf_pack_kernel<<<grid, 256, 0, stream>>>(src, rows, blocks, dst, total, kc_count);
    return cudaGetLastError();
}

}  // namespace gb300
