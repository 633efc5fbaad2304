// gemm_mx_pair.cu -- the block-scaled ("MX") product on SM pairs.
//
// Same operation as gemm_mx.cu (OCP MX v1.0 elements and E8M0 block scales,
// applied by the tensor cores from tensor memory), on 256 x 256 output tiles
// per pair of SMs (tcgen05 cta_group::2): each CTA stages 128 rows of A and
// 128 rows of B per k-block, and the pair's MMA (M = 256, N = 256) reads A
// from each CTA's own shared memory and B from both.  Every byte a CTA stages
// feeds twice the multiply-adds of the one-SM kernel's 128 x 256 tile, so
// shared memory moves 128 bytes a clock at the full MMA rate instead of 192.
//
// Scale factors: the leader's tcgen05.cp (cta_group::2) copies each CTA's
// staged chunks into that CTA's own tensor memory, at the same columns in
// both.  Each CTA's tensor memory holds the scales of ITS 128 rows of A (4
// columns per chunk, row r's in column r / 32) and of ALL 256 rows of the
// tile's B (8 columns per chunk: rows 0-127, then 128-255) -- each SM's
// tensor core multiplies its own rows of A by every column of B.  Integer
// tests with a scale per row and block pin this: of the four placements
// (A's own rows or both blocks, B's likewise) only this one is exact, and
// the others are wrong exactly in the peer's half of the tile.
//
// Roles per CTA (10 warps): warp 0 lane 0 loads (TMA, completion counted on
// the leader's barrier); warp 1 lane 0 of the leader copies the scales and
// issues the MMAs; warps 2-9 run the epilogue of the CTA's 128 rows.  One
// 256-column accumulator: a tile's epilogue runs before the next tile's MMAs,
// while the loads of the next tile proceed.
#include "epilogue.cuh"
#include "gemm_tcgen05.cuh"
#include "kernel_args.h"
#include "mx_traits.cuh"
#include "sm103_ptx.cuh"

namespace gb300 {

namespace {

template <int ELEM, int STAGES_>
struct MxpConfig {
    static constexpr int BM = 128, BN = 256, BNH = 128;     // per CTA: 128 rows of A, 128 of B
    static constexpr int STAGES = STAGES_;
    static constexpr int ROW_BYTES = 128;
    static constexpr int MMAS = 4;
    static constexpr int CHUNKS = MxTraits<ELEM>::kChunks;
    static constexpr int A_BYTES = BM * ROW_BYTES;
    static constexpr int B_BYTES = BNH * ROW_BYTES;
    static constexpr int SF_BLOCK = CHUNKS * 512;             // one 128-row block's chunks of a stage
    static constexpr int SFA_OFF = A_BYTES + B_BYTES;         // the CTA's own row block of A
    static constexpr int SFB_OFF = SFA_OFF + SF_BLOCK;        // B's two row blocks of the tile
    static constexpr int STAGE_TX = SFB_OFF + 2 * SF_BLOCK;   // bytes one CTA receives per stage
    static constexpr int STAGE_BYTES = (STAGE_TX + 1023) / 1024 * 1024;
    static constexpr int ACC_COLS = BN;
    static constexpr int SF_SLOT_COLS = 12 * CHUNKS;          // A: 4 per chunk, B: 8 per chunk
    static constexpr int TMEM_COLS = 512;
    static constexpr int EPI_WARPS = 8;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
    static_assert(ACC_COLS + STAGES * SF_SLOT_COLS <= TMEM_COLS, "scale slots fit beside the accumulator");
    static_assert((2 * STAGES + 3) * 8 + 16 <= BAR_BYTES, "barriers fit their slot");
    static_assert(SMEM_BYTES <= 232448, "fits the 227 KB opt-in shared memory");
};

}  // namespace

template <int ELEM, int OUT, int STAGES>
__global__ void __launch_bounds__(MxpConfig<ELEM, STAGES>::THREADS, 1)
    gemm_mx_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                        const __grid_constant__ MxArgs args) {
    using Cfg = MxpConfig<ELEM, STAGES>;
    constexpr int BM = Cfg::BM, BNH = Cfg::BNH;

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
    const uint32_t rank = cluster_ctarank();  // 0 leader, 1 peer
    const int cluster = blockIdx.x / 2;
    const int nclusters = gridDim.x / 2;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);   // the leader's expect_tx arrive covers both CTAs' bytes
            mbar_init(&empty[s], 1);  // the leader's multicast commit
        }
        mbar_init(tfull, 1);
        mbar_init(tempty, 2 * Cfg::EPI_WARPS);  // both CTAs' epilogue warps (the leader's copy is used)
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmSFA);
        tma_prefetch_desc(&tmSFB);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish_pair();
    }
    __syncwarp();
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t full0_leader = mapa_shared(smem_u32(&full[0]), 0);
    const uint32_t tempty_leader = mapa_shared(smem_u32(tempty), 0);
    const uint32_t abort_local = smem_u32(const_cast<int *>(abort_flag));
    const int M = args.e.M, N = args.e.N;
    const int num_kb = args.num_kb;

    if (warp == 0) {
        if (lane == 0) {
            // ----------------------------------------------------- producer --
            uint32_t stage = 0, phase = 0;
            bool ok = true, issued = false;
            const long long rbs_a = (M + 127) / 128, rbs_b = (N + 127) / 128;
            for (int tile = cluster; ok && tile < args.num_tiles; tile += nclusters) {
                int tm, tn;
                tile_coords(tile, args.tiles_m, args.tiles_n, args.group_m, tm, tn);
                const int m0 = tm * 2 * BM, n0 = tn * 2 * BNH;
                // Row blocks of the scale chunks: A's of this CTA's rows, B's two; a
                // block past the operand's end is replaced by its last (those rows
                // of the operand are zero-filled).
                long long ra = 2LL * tm + rank, rb0 = 2LL * tn, rb1 = 2LL * tn + 1;
                ra = ra < rbs_a ? ra : rbs_a - 1;
                rb0 = rb0 < rbs_b ? rb0 : rbs_b - 1;
                rb1 = rb1 < rbs_b ? rb1 : rbs_b - 1;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!pair_wait<2>(&empty[stage], phase ^ 1u, abort_flag, args.status, abort_local, rank)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fbar = full0_leader + 8u * stage;
                    if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2u * Cfg::STAGE_TX);
                    issued = true;
                    unsigned char *sA = smem + stage * Cfg::STAGE_BYTES;
                    const uint64_t pol = l2_policy_evict_last();
                    tma_load_2d_pair(sA, &tmA, fbar, kb * Cfg::ROW_BYTES, m0 + static_cast<int>(rank) * BM, pol);
                    tma_load_2d_pair(sA + Cfg::A_BYTES, &tmB, fbar, kb * Cfg::ROW_BYTES,
                                     n0 + static_cast<int>(rank) * BNH, pol);
                    // scale chunks: rows of 256 bytes, 2 per chunk; a block's chunks of
                    // stage kb start at row 2 * (rb * kc_count + kb * CHUNKS)
                    const int kcs = args.kc_count;
                    const int c0 = kb * Cfg::CHUNKS;
                    tma_load_2d_pair(sA + Cfg::SFA_OFF, &tmSFA, fbar, 0, static_cast<int>(2 * (ra * kcs + c0)), pol);
                    tma_load_2d_pair(sA + Cfg::SFB_OFF, &tmSFB, fbar, 0, static_cast<int>(2 * (rb0 * kcs + c0)), pol);
                    tma_load_2d_pair(sA + Cfg::SFB_OFF + Cfg::SF_BLOCK, &tmSFB, fbar, 0,
                                     static_cast<int>(2 * (rb1 * kcs + c0)), pol);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (*abort_flag && issued) {
                // Unwinding: loads in flight complete within microseconds.
                const unsigned long long t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 200000ull) sleep_ns(10000);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // -------------------------------------------- MMA issuer (leader) --
            uint32_t stage = 0, phase = 0;
            bool ok = true, issued = false;
            int local = 0;
            for (int tile = cluster; ok && tile < args.num_tiles; tile += nclusters, ++local) {
                if (!pair_wait<2>(tempty, (local & 1) ^ 1u, abort_flag, args.status, abort_local, rank)) break;
                tc_fence_after();
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!pair_wait<2>(&full[stage], phase, abort_flag, args.status, abort_local, rank)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + stage * Cfg::STAGE_BYTES);
                    const uint32_t b_addr = a_addr + Cfg::A_BYTES;
                    const uint32_t sfa_t = tmem_base + Cfg::ACC_COLS + stage * Cfg::SF_SLOT_COLS;
                    const uint32_t sfb_t = sfa_t + 4 * Cfg::CHUNKS;
#pragma unroll
                    for (int c = 0; c < Cfg::CHUNKS; ++c) {
                        // A: chunk c at columns +4c; B: chunk c of rows 0-127 at +8c, of rows 128-255 at +8c+4
                        tc_cp_32x128b_x4_pair(sfa_t + 4 * c, plain16_desc(a_addr + Cfg::SFA_OFF + 512 * c));
                        tc_cp_32x128b_x4_pair(sfb_t + 8 * c, plain16_desc(a_addr + Cfg::SFB_OFF + 512 * c));
                        tc_cp_32x128b_x4_pair(sfb_t + 8 * c + 4,
                                              plain16_desc(a_addr + Cfg::SFB_OFF + Cfg::SF_BLOCK + 512 * c));
                    }
#pragma unroll
                    for (int ks = 0; ks < Cfg::MMAS; ++ks) {
                        const uint32_t chunk = Cfg::CHUNKS == 1 ? 0u : static_cast<uint32_t>(ks >> 1);
                        const uint32_t sf_id = Cfg::CHUNKS == 1 ? static_cast<uint32_t>(ks)
                                                                : static_cast<uint32_t>((ks & 1) * 2);
                        const uint32_t idesc = mma_idesc_bs(MxTraits<ELEM>::kFmt, 2 * BM, 2 * BNH, sf_id, sf_id);
                        const uint64_t ad = sw128_desc(a_addr + ks * 32, 16u, 1024u);
                        const uint64_t bd = sw128_desc(b_addr + ks * 32, 16u, 1024u);
                        tc_mma_bs_pair<MxTraits<ELEM>::kKind>(tmem_base, ad, bd, idesc, sfa_t + 4 * chunk,
                                                               sfb_t + 8 * chunk, (kb | ks) != 0 ? 1u : 0u);
                    }
                    issued = true;
                    tc_commit_pair(&empty[stage], 0x3);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) tc_commit_pair(tfull, 0x3);
            }
            if (*abort_flag && issued) {
                tc_commit_pair(mma_done, 0x1);
                mbar_drain_wait(mma_done, 0, 100000000ull);
            }
        }
    } else {
        // ------------------------------------------------------- epilogue --
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;
        const EpiParams &e = args.e;
        int local = 0;
        for (int tile = cluster; tile < args.num_tiles; tile += nclusters, ++local) {
            int tm, tn;
            tile_coords(tile, args.tiles_m, args.tiles_n, args.group_m, tm, tn);
            const int row = tm * 2 * BM + static_cast<int>(rank) * BM + quad * 32 + lane;
            const int col_base = tn * 2 * BNH + half * 128;
            const bool got = pair_wait<2>(tfull, local & 1, abort_flag, args.status, abort_local, rank);
            if (__any_sync(0xffffffffu, !got)) break;
            tc_fence_after();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + half * 128;
            int nvalid = (N - col_base + 31) >> 5;
            nvalid = nvalid < 0 ? 0 : (nvalid > 4 ? 4 : nvalid);
            epilogue_row_chunks<OUT, 4, false>(t_row, col_base, nvalid, row, row < M, e.bias + col_base, e);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(tempty_leader);
        }
    }

    __syncwarp();
    tc_fence_before();
    cluster_sync_all();  // no CTA leaves while its peer may still signal into it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    }
}

template <int ELEM, int OUT>
cudaError_t launch_mx_pair_cfg(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tsa,
                               const CUtensorMap &tsb, const MxArgs &args, int clusters, cudaStream_t stream) {
    constexpr int STAGES = 6;
    using Cfg = MxpConfig<ELEM, STAGES>;
    auto kern = gemm_mx_pair_kernel<ELEM, OUT, STAGES>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, ta, tb, tsa, tsb, args);
}

cudaError_t launch_mx_pair(int elem, int out, const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tsa,
                           const CUtensorMap &tsb, const MxArgs &args, int clusters, cudaStream_t stream) {
    if (elem == kMxE4M3) {
        if (out == kDtF32) return launch_mx_pair_cfg<kMxE4M3, kDtF32>(ta, tb, tsa, tsb, args, clusters, stream);
        if (out == kDtF16) return launch_mx_pair_cfg<kMxE4M3, kDtF16>(ta, tb, tsa, tsb, args, clusters, stream);
        if (out == kDtBF16) return launch_mx_pair_cfg<kMxE4M3, kDtBF16>(ta, tb, tsa, tsb, args, clusters, stream);
    } else if (elem == kMxE2M1) {
        if (out == kDtF32) return launch_mx_pair_cfg<kMxE2M1, kDtF32>(ta, tb, tsa, tsb, args, clusters, stream);
        if (out == kDtF16) return launch_mx_pair_cfg<kMxE2M1, kDtF16>(ta, tb, tsa, tsb, args, clusters, stream);
        if (out == kDtBF16) return launch_mx_pair_cfg<kMxE2M1, kDtBF16>(ta, tb, tsa, tsb, args, clusters, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gb300
