// gemm_tcgen05_pair.cuh -- the GEMM on pairs of SMs (tcgen05 cta_group::2).
//
// Same roles as the one-SM kernel (gemm_tcgen05.cuh), but a cluster of two
// CTAs on two SMs computes one 256 x BN output tile with one MMA stream:
//
//   * each CTA's producer loads its own 128 rows of A and its own BN/2
//     columns of B into its own shared memory, and counts the bytes on the
//     LEADER CTA's full[s] barrier (TMA with cta_group::2);
//   * the leader's MMA thread issues tcgen05.mma.cta_group::2 256 x BN x K;
//     the hardware reads A rows 0-127 / B columns 0..BN/2-1 from the leader's
//     shared memory and the rest from the peer's, and writes accumulator rows
//     0-127 to the leader's tensor memory and 128-255 to the peer's;
//   * tcgen05.commit multicasts to both CTAs: empty[s] frees both halves of a
//     stage, tfull[acc] starts both CTAs' epilogues;
//   * each CTA's eight epilogue warps drain their own tensor memory (two warps
//     per 32-lane quadrant, each taking half of the columns) and arrive on the
//     leader's tempty[acc].
//
// Per SM and per 16-deep k slice, the MMA reads 4 KB of A and 16*BN bytes of
// B from shared memory and TMA writes as much: 128 B/clk at BN = 256, which
// fits the shared-memory bandwidth, where the one-SM 128 x 256 tile needs
// 192 B/clk.  BN is a runtime multiple of 32 up to 256, chosen by the host to
// balance waves of tiles over the clusters.
//
// With CL = 4 a cluster holds two such pairs that compute two tiles side by
// side along N (the same 256 rows of A).  Each CTA then fetches only half of
// its 128 rows of A and TMA multicasts them to the CTA in the same position of
// the other pair, so the two pairs read each A panel from L2 once: a quarter
// fewer operand bytes per SM (24 KB instead of 32 KB per stage).  A stage is
// free again only when both pairs' MMAs have read it, so every CTA's empty[s]
// takes one commit from each pair's leader and the two pairs run in lockstep.
#pragma once

#include "epilogue.cuh"
#include "gemm_tcgen05.cuh"
#include "kernel_args.h"
#include "sm103_ptx.cuh"

namespace gb300 {

// BNH: B columns one CTA stages per k-block (half the widest tile it runs).
// All instantiations use 128 (6 stages of 32 KB); a 64-column, 8-stage ring
// for 128-wide tiles measured no faster on GB300 (M=512, N=K=4096: 28.7 us
// either way), so it is not built.
template <int AB, int STAGES_, int BNH = 128>
struct PairConfig {
    static constexpr int BM = 128;  // rows per CTA (256 per pair)
    static constexpr int BN_MAX = 256;
    static constexpr int STAGES = STAGES_;
    static constexpr int ES = TcTraits<AB>::kBytes;
    static constexpr int SWZ = 128 / ES;
    static constexpr int BK = SWZ;
    static constexpr int UMMA_K = TcTraits<AB>::kUmmaK;
    static constexpr int KSTEPS = BK / UMMA_K;
    static constexpr int A_BYTES = BM * BK * ES;          // this CTA's rows of A
    // This CTA's columns of B (at most).  An N-contiguous B is loaded in whole
    // 128-byte swizzle rows (SWZ columns), so the slot is never narrower.
    static constexpr int B_COLS = BNH > SWZ ? BNH : SWZ;
    static constexpr int B_BYTES = B_COLS * BK * ES;
    // 3xTF32 keeps a hi and a lo copy of both tiles: [A hi][A lo][B hi][B lo].
    static constexpr bool X3 = (AB == kDtTF32x3);
    static constexpr int COPIES = X3 ? 2 : 1;
    static constexpr int A_LO = A_BYTES;                  // offset of A lo (3xTF32)
    static constexpr int B_OFF = COPIES * A_BYTES;        // offset of B (hi)
    static constexpr int B_LO = B_OFF + B_BYTES;          // offset of B lo (3xTF32)
    static constexpr int STAGE_BYTES = COPIES * (A_BYTES + B_BYTES);
    static constexpr int ACC_STRIDE = 256;                // TMEM columns between the two accumulators
    static constexpr int TMEM_COLS = 512;
    static constexpr int EPI_WARPS = 8;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    // Per epilogue warp: one staged 32-row x 64-byte box of C (TMA in and out).
    static constexpr int CSTAGE_BYTES = EPI_WARPS * kStageBoxBytes;
    static constexpr int BAR_BYTES = 256;
    // Bias staged per epilogue warp (up to 4 chunks of 32 columns), per accumulator.
    static constexpr int BIAS_BYTES = 2 * EPI_WARPS * 128 * 4;
    // Layout: [stages][C boxes][barriers][bias]; stages and boxes stay 1024-byte aligned.
    static constexpr int CSTAGE_OFF = STAGES * STAGE_BYTES;
    static constexpr int BAR_OFF = CSTAGE_OFF + CSTAGE_BYTES;
    static constexpr int BIAS_OFF = BAR_OFF + BAR_BYTES;
    static constexpr int SMEM_BYTES = 1024 + BIAS_OFF + BIAS_BYTES;
    static_assert((2 * STAGES + 5 + EPI_WARPS) * 8 + 8 <= BAR_BYTES, "barriers fit their slot");
    // A CTA's last tile stages its C boxes in the idle ring: per warp up to 4
    // chunks x 2 boxes (fp32 output) of 2 KB.
    static constexpr int BURST_BYTES_PER_WARP = 4 * 2 * kStageBoxBytes;
    static_assert(EPI_WARPS * BURST_BYTES_PER_WARP <= STAGES * STAGE_BYTES, "last-tile boxes fit the ring");
    static_assert(SMEM_BYTES <= 232448, "fits the 227 KB opt-in shared memory");
    static_assert(SMEM_BYTES > 232448 / 2, "one CTA per SM: the pair allocates all 512 TMEM columns");
};

// ----------------------------------------------------------- schedule --
// A cluster's work is a sequence of segments: (tile, k-blocks [kb_begin,
// kb_end)).  First its piece [u0, u1) of the stream-K unit range (the k-blocks
// of tiles dp_tiles .. num_tiles-1 in one line), cut at tile boundaries; then
// whole tiles c, c + clusters, ... below dp_tiles.  Kinds: FULL (all k-blocks
// of a tile), OWNER (starts at k-block 0 but stops early: later clusters hold
// the rest), PART (starts inside a tile).  Since pieces are contiguous, only a
// cluster's first segment can be a PART, so each cluster fills at most one
// partial slot; the OWNER of a tile is the cluster whose piece holds its first
// k-block (its last stream-K segment).  PARTs never wait on anything, OWNERs
// wait only on PARTs of later clusters: no cycle.  Doing the stream-K piece
// first lets the fix-up epilogues overlap the whole tiles' main loops, and
// every cluster ends on an ordinary epilogue.
enum SegKind { kSegFull = 0, kSegOwner = 1, kSegPart = 2 };

struct Segment {
    int tile, kb_begin, kb_end, kind;
    long long sk_tile;  // index among the stream-K tiles (-1 for whole tiles)
};

struct SegmentIter {
    int next_dp, nclusters, dp_tiles, num_kb;
    long long u, u_end;
    __device__ __forceinline__ SegmentIter(const TcArgs &a, int cluster, int nclusters_)
        : next_dp(cluster), nclusters(nclusters_), dp_tiles(a.dp_tiles), num_kb(a.num_kb),
          u(a.sk_units > 0 ? a.sk_cut[cluster] : 0), u_end(a.sk_units > 0 ? a.sk_cut[cluster + 1] : 0) {}
    __device__ __forceinline__ bool next(Segment &s) {
        if (u >= u_end) {
            if (next_dp >= dp_tiles) return false;
            s.tile = next_dp;
            s.kb_begin = 0;
            s.kb_end = num_kb;
            s.kind = kSegFull;
            s.sk_tile = -1;
            next_dp += nclusters;
            return true;
        }
        const long long t = u / num_kb;
        const long long tile_end = (t + 1) * num_kb;
        s.kb_begin = static_cast<int>(u - t * num_kb);
        s.kb_end = static_cast<int>((u_end < tile_end ? u_end : tile_end) - t * num_kb);
        s.tile = dp_tiles + static_cast<int>(t);
        s.sk_tile = t;
        s.kind = s.kb_begin != 0 ? kSegPart : (s.kb_end == num_kb ? kSegFull : kSegOwner);
        u = t * num_kb + s.kb_end;
        return true;
    }
};

// Last cluster whose piece overlaps stream-K tile t, whose first k-block is
// in `owner`'s piece: the last cluster whose piece starts before the tile's end.
__device__ __forceinline__ int last_contributor(const TcArgs &a, long long t, int owner, int nclusters) {
    const long long end = (t + 1) * a.num_kb;
    int c = owner;
    while (c + 1 < nclusters && static_cast<long long>(a.sk_cut[c + 1]) < end) ++c;
    return c;
}

// Index (in floats) of column group q (4 columns) of chunk ci, row r, inside
// one CTA's partial slot: a warp's 32 rows of one group are 512 contiguous bytes.
__device__ __forceinline__ long long partial_index(int ci, int q, int r) {
    return ((static_cast<long long>(ci) * 8 + q) * 128 + r) * 4;
}

// PART epilogue: this thread's raw fp32 accumulators of chunks c0 .. c0+n-1 to
// its cluster's partial slot (coalesced 16-byte stores, L2 only).  The slot is
// read once, by the tile's owner a few tiles' time later, and then dropped
// from L2 (owner_row_chunks), so its lines are the last L2 evicts: written
// with the ordinary priority, operand panels and C pushed many of them out to
// HBM before the owner came (with both measures, a 4096^3 launch moves 157
// instead of 172 MB through DRAM).
__device__ __forceinline__ void store_partial_chunks(uint32_t t_base, int c0, int n, int r, float *slot) {
    if (n <= 0) return;
    const uint64_t pol = l2_policy_evict_last();
    uint32_t ra[32], rb[32];
    __syncwarp();
    tmem_ld_issue(t_base, ra);
    tmem_ld_wait(ra);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (i >= n) break;
        uint32_t(&cur)[32] = (i & 1) ? rb : ra;
        uint32_t(&nxt)[32] = (i & 1) ? ra : rb;
        const bool more = i + 1 < n;
        if (more) tmem_ld_issue(t_base + (i + 1) * 32, nxt);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 v = make_float4(__uint_as_float(cur[4 * q]), __uint_as_float(cur[4 * q + 1]),
                                         __uint_as_float(cur[4 * q + 2]), __uint_as_float(cur[4 * q + 3]));
            st_global_cg_v4_hint(slot + partial_index(c0 + i, q, r), v, pol);
        }
        __syncwarp();
        if (more) tmem_ld_wait(nxt);
    }
}

// OWNER epilogue: like epilogue_row_chunks, with the partial sums of
// `ncontrib` later clusters (slots slot0, slot0 + slot_stride, ...) added to
// the accumulators before alpha / beta / bias / GELU / cast.  Each partial
// line is discarded from L2 once the warp has added it: the slot is scratch
// that the next writer fills again, so it never needs to reach HBM.  Slots
// are 128-byte aligned (the workspace is 256-byte aligned, a slot 128 KB).
// With e.c_tma the chunks go through the warp's staged C box (rows row0 ..
// row0+31, row0 < M) instead.  Returns false if a wait for C gave up.
template <int OUT, bool SC>
__device__ __forceinline__ bool owner_row_chunks(uint32_t t_base, int col_base, int c0, int nvalid, int row,
                                                 bool row_ok, int r, const float *slot0, long long slot_stride,
                                                 int ncontrib, const float *bias_base, const EpiParams &e,
                                                 int row0, const CUtensorMap *tmC, unsigned char *cbuf,
                                                 uint64_t *cbar, uint32_t &cphase, volatile int *abort_flag,
                                                 unsigned int *status, float bias_lane) {
    using OutT = typename Elem<OUT>::T;
    OutT *crow = reinterpret_cast<OutT *>(e.C) + (long long)(row_ok ? row : 0) * e.ldc;
    const OutT *rrow = (SC && row_ok) ? residual_row<OUT>(e, row) : nullptr;
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
#pragma unroll 1
        for (int k = 0; k < ncontrib; ++k) {
            const float *src = slot0 + k * slot_stride;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 p = __ldcg(reinterpret_cast<const float4 *>(src + partial_index(c0 + i, q, r)));
                v[4 * q] += p.x; v[4 * q + 1] += p.y; v[4 * q + 2] += p.z; v[4 * q + 3] += p.w;
            }
        }
        // A value that needs every partial load of this chunk, consumed before
        // the warp converges: past the __syncwarp no lane has a load of the
        // lines below outstanding.
        float dep = 0.0f;
#pragma unroll
        for (int q = 0; q < 8; ++q) dep += v[4 * q];
        asm volatile("" ::"f"(dep));
        __syncwarp();
        if ((r & 7) == 0) {  // lanes 0, 8, 16, 24: one 128-byte line each of the warp's 512 bytes
#pragma unroll 1
            for (int k = 0; k < ncontrib; ++k)
#pragma unroll
                for (int q = 0; q < 8; ++q) discard_l2_line(slot0 + k * slot_stride + partial_index(c0 + i, q, r));
        }
        const int col0 = col_base + i * 32;
        // E4M3 outputs never move through shared memory (the host gives them no C map).
        const bool staged = OUT != kDtE4M3 && e.c_tma;
        if (!staged) product_scale_chunk<SC>(v, e, row, col0, false);  // the TMA path scales in epilogue_chunk32_tma
        if (staged) {
            if constexpr (OUT != kDtE4M3) {
                if (ok && row0 < (e.swap ? e.N : e.M))
                    ok = epilogue_chunk32_tma<OUT, SC>(v, col0, row0, bias_base + i * 32, bias_lane, e, tmC, cbuf,
                                                       cbar, cphase, abort_flag, status);
            }
        } else if (row_ok) {
            const OutT *rchunk = rrow != nullptr ? rrow + col0 : nullptr;
            if (e.c_vec && col0 + 32 <= e.N)
                epilogue_chunk32_fast<OUT, SC>(v, crow + col0, bias_base + i * 32, e, rchunk);
            else
                epilogue_chunk32_safe<OUT, SC>(v, crow + col0, col0, e, rchunk);
        }
    }
    __syncwarp();
    return ok;
}

// CL: CTAs per cluster, 2 (one pair) or 4 (two pairs sharing A by multicast).
// SC: built for calls with product scales, fp8 output, amax or a residual
// (gemm_ex); without, that code is left out.
// Registers: an SM's 65,536 registers sit in four sub-partitions of 16,384,
// and a 10-warp CTA places three warps on two of them, so a thread gets at
// most 170 (168 in steps of 8).  Built with 200 (__maxnreg__), GB300 reports
// no resident cluster for the kernel.
template <int AB, int OUT, int STAGES, int BNH, int CL, bool SC>
__global__ void __launch_bounds__(PairConfig<AB, STAGES, BNH>::THREADS, 1)
    gemm_tcgen05_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmC, const __grid_constant__ TcArgs args) {
    using Cfg = PairConfig<AB, STAGES, BNH>;
    constexpr int BM = Cfg::BM, BK = Cfg::BK, SWZ = Cfg::SWZ;
    static_assert(CL == 2 || (CL == 4 && !Cfg::X3), "two pairs per cluster only for single-copy operands");
    constexpr int PAIRS = CL / 2;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::BAR_OFF);
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *mma_done = tempty + 2;
    uint64_t *cbar = mma_done + 1;  // one per epilogue warp: its C box has landed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(cbar + Cfg::EPI_WARPS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *bias_stage = reinterpret_cast<float *>(smem + Cfg::BIAS_OFF);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t prank = rank & 1u;   // position in the pair: 0 leader, 1 peer
    const uint32_t pidx = rank >> 1;    // which pair of the cluster
    const uint32_t lead = rank & ~1u;   // cluster rank of this pair's leader
    const int cluster = blockIdx.x / CL;
    const int nclusters = gridDim.x / CL;
    const int bn = args.bn;
    const int bnh = bn >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);   // the leader's expect_tx arrive covers both CTAs' bytes
            mbar_init(&empty[s], PAIRS);  // one multicast commit per pair reading the stage
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 2 * Cfg::EPI_WARPS);  // both CTAs' epilogue warps (leader's copy is used)
        }
        mbar_init(mma_done, 1);
        for (int w = 0; w < Cfg::EPI_WARPS; ++w) mbar_init(&cbar[w], 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (args.e.c_tma) tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish_pair();
    }
    __syncwarp();
    tc_fence_before();
    cluster_sync_all();  // both CTAs' barriers initialised and TMEM allocated
    tc_fence_after();
    // Everything above touches only this CTA's own resources, so it may overlap
    // the previous grid in the stream; every global-memory access below waits.
    grid_dep_wait();
    grid_dep_launch();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t full0_leader = mapa_shared(smem_u32(&full[0]), lead);
    const uint32_t tempty0_leader = mapa_shared(smem_u32(&tempty[0]), lead);
    const uint32_t abort_local = smem_u32(const_cast<int *>(abort_flag));

    const int M = args.e.M, N = args.e.N;
    const int num_kb = args.num_kb;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer --
            uint32_t stage = 0, phase = 0;
            bool ok = true, issued = false;
            const uint64_t pol_ab = l2_policy_evict_last();
            SegmentIter it(args, cluster, nclusters);
            Segment seg;
            while (ok && it.next(seg)) {
                int tm, tn;
                tile_coords(seg.tile, args.tiles_m, args.tiles_n, args.group_m, tm, tn);
                tn = tn * PAIRS + static_cast<int>(pidx);
                const int m0 = tm * 2 * BM + static_cast<int>(prank) * BM;
                const int n0 = tn * bn + static_cast<int>(prank) * bnh;
                for (int kb = seg.kb_begin; kb < seg.kb_end; ++kb) {
                    if (!pair_wait<CL>(&empty[stage], phase ^ 1u, abort_flag, args.status, abort_local, rank)) {
                        ok = false;
                        break;
                    }
                    // Only the leader arms the phase, with both CTAs' bytes; the
                    // peer's loads complete on the leader's barrier (a
                    // completion may precede the arming within a phase: the
                    // phase cannot end before the leader's arrive).  This keeps
                    // cluster-scope fences off the per-k-block path.
                    const uint32_t fbar = full0_leader + 8u * stage;
                    if (prank == 0) mbar_arrive_expect_tx(&full[stage], 2u * args.stage_tx);
                    issued = true;
                    unsigned char *sA = smem + stage * Cfg::STAGE_BYTES;
                    unsigned char *sB = sA + Cfg::B_OFF;
                    const int k0 = kb * BK;
                    if constexpr (Cfg::X3) {
                        // hi and lo halves of the stacked K-major arrays
                        tma_load_2d_pair(sA, &tmA, fbar, k0, m0, pol_ab);
                        tma_load_2d_pair(sA + Cfg::A_LO, &tmA, fbar, k0, m0 + args.lo_row_a, pol_ab);
                        tma_load_2d_pair(sB, &tmB, fbar, k0, n0, pol_ab);
                        tma_load_2d_pair(sA + Cfg::B_LO, &tmB, fbar, k0, n0 + args.lo_row_b, pol_ab);
                    } else if constexpr (CL == 4) {
                        // This CTA's share of the A rows, delivered to both pairs.
                        const uint16_t amask = static_cast<uint16_t>((1u << prank) | (4u << prank));
                        if (!args.a_mn_major) {
                            tma_load_2d_pair_mc(sA + pidx * (BM / 2) * 128, &tmA, fbar, k0,
                                                m0 + static_cast<int>(pidx) * (BM / 2), amask, pol_ab);
                        } else {
                            // BM / SWZ boxes of SWZ rows; the host runs this only when that is even.
                            for (int j = static_cast<int>(pidx); j < BM / SWZ; j += PAIRS)
                                tma_load_2d_pair_mc(sA + j * 128 * BK, &tmA, fbar, m0 + j * SWZ, k0, amask,
                                                    pol_ab);
                        }
                    } else if (!args.a_mn_major) {
                        tma_load_2d_pair(sA, &tmA, fbar, k0, m0, pol_ab);
                    } else {
#pragma unroll
                        for (int j = 0; j < BM / SWZ; ++j)
                            tma_load_2d_pair(sA + j * 128 * BK, &tmA, fbar, m0 + j * SWZ, k0, pol_ab);
                    }
                    if constexpr (!Cfg::X3) {
                        if (!args.b_mn_major) {
                            tma_load_2d_pair(sB, &tmB, fbar, k0, n0, pol_ab);
                        } else {
                            for (int j = 0; j * SWZ < bnh; ++j)
                                tma_load_2d_pair(sB + j * 128 * BK, &tmB, fbar, n0 + j * SWZ, k0, pol_ab);
                        }
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (*abort_flag && issued) {
                // Unwinding: loads in flight complete within microseconds; give
                // them time to land before this CTA's shared memory is released.
                const unsigned long long t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 200000ull) sleep_ns(10000);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && prank == 0) {
            // --------------------------------------------- MMA issuer (leader) --
            // Stages are released in every CTA that multicast into this pair's;
            // the accumulator is published to this pair only.
            constexpr uint16_t kEmptyMask = CL == 4 ? 0xF : 0x3;
            const uint16_t pair_mask = static_cast<uint16_t>(0x3u << lead);
            const uint32_t idesc = mma_idesc(TcTraits<AB>::kFmt, TcTraits<AB>::kFmt, 2 * BM, bn) |
                                   (args.a_mn_major << 15) | (args.b_mn_major << 16);
            const uint32_t a_lbo = args.a_mn_major ? 128u * BK : 16u;
            const uint32_t b_lbo = args.b_mn_major ? 128u * BK : 16u;
            const uint32_t a_kstep = args.a_mn_major ? 128u * Cfg::UMMA_K : 32u;
            const uint32_t b_kstep = args.b_mn_major ? 128u * Cfg::UMMA_K : 32u;
            uint32_t stage = 0, phase = 0;
            bool ok = true, issued = false;
            int local = 0;
            SegmentIter it(args, cluster, nclusters);
            Segment seg;
            for (; ok && it.next(seg); ++local) {
                const uint32_t acc = local & 1, acc_phase = (local >> 1) & 1;
                if (!pair_wait<CL>(&tempty[acc], acc_phase ^ 1u, abort_flag, args.status, abort_local, rank)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * Cfg::ACC_STRIDE;
                for (int kb = seg.kb_begin; kb < seg.kb_end; ++kb) {
                    if (!pair_wait<CL>(&full[stage], phase, abort_flag, args.status, abort_local, rank)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + stage * Cfg::STAGE_BYTES);
                    const uint32_t b_addr = a_addr + Cfg::B_OFF;
#pragma unroll
                    for (int ks = 0; ks < Cfg::KSTEPS; ++ks) {
                        const uint32_t acc_in = (kb != seg.kb_begin || ks != 0) ? 1u : 0u;
                        const uint64_t ad = sw128_desc(a_addr + ks * a_kstep, a_lbo, 1024u);
                        const uint64_t bd = sw128_desc(b_addr + ks * b_kstep, b_lbo, 1024u);
                        if constexpr (Cfg::X3) {
                            // 3xTF32: A*B ~ A_lo*B_hi + A_hi*B_lo + A_hi*B_hi, small terms first
                            const uint64_t ad_lo = sw128_desc(a_addr + Cfg::A_LO + ks * a_kstep, a_lbo, 1024u);
                            const uint64_t bd_lo = sw128_desc(a_addr + Cfg::B_LO + ks * b_kstep, b_lbo, 1024u);
                            tc_mma_pair<TcTraits<AB>::kKind>(d_tmem, ad_lo, bd, idesc, acc_in);
                            tc_mma_pair<TcTraits<AB>::kKind>(d_tmem, ad, bd_lo, idesc, 1u);
                            tc_mma_pair<TcTraits<AB>::kKind>(d_tmem, ad, bd, idesc, 1u);
                        } else {
                            tc_mma_pair<TcTraits<AB>::kKind>(d_tmem, ad, bd, idesc, acc_in);
                        }
                    }
                    issued = true;
                    tc_commit_pair(&empty[stage], kEmptyMask);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) tc_commit_pair(&tfull[acc], pair_mask);
            }
            if (*abort_flag && issued) {
                tc_commit_pair(mma_done, static_cast<uint16_t>(1u << rank));
                mbar_drain_wait(mma_done, 0, 100000000ull);
            }
        }
    } else {
        // ------------------------------------------------------- epilogue --
        const int ew = warp - 2;           // 0..7
        const int quad = warp & 3;         // TMEM lanes 32*quad .. 32*quad+31
        const int half = ew >> 2;          // which half of the tile's columns
        const int nchunks = bn >> 5;
        const int c_begin = half ? (nchunks + 1) >> 1 : 0;
        const int c_end = half ? nchunks : (nchunks + 1) >> 1;
        const EpiParams &e = args.e;
        const int r = quad * 32 + lane;  // this thread's row inside the CTA's 128
        unsigned char *cbuf = smem + Cfg::CSTAGE_OFF + ew * kStageBoxBytes;
        uint32_t cphase = 0;
        int local = 0;
        SegmentIter it(args, cluster, nclusters);
        Segment seg;
        for (; it.next(seg); ++local) {
            const uint32_t acc = local & 1, acc_phase = (local >> 1) & 1;
            SegmentIter peek = it;
            Segment after;
            // After the last segment's accumulator is ready, every MMA has
            // completed and no load is pending: the operand ring is idle.
            const bool last = !peek.next(after);
            int tm, tn;
            tile_coords(seg.tile, args.tiles_m, args.tiles_n, args.group_m, tm, tn);
            tn = tn * PAIRS + static_cast<int>(pidx);
            // Accumulator rows (TMEM lanes) and columns: output rows and columns,
            // or output columns and rows when the kernel computes C^T (e.swap).
            const int row0 = tm * 2 * BM + static_cast<int>(prank) * BM + quad * 32;  // the warp's first lane row
            const int row = row0 + lane;
            const int n_tile = tn * bn;
            float *bias_s = bias_stage + (acc * Cfg::EPI_WARPS + ew) * 128;
            float bias_lane = 0.0f;
            if (seg.kind != kSegPart) {
                if (e.swap)
                    bias_lane = epilogue_prefetch_t<OUT>(n_tile + c_begin * 32, c_end - c_begin, row0, e, last);
                else
                    epilogue_prefetch<OUT>(bias_s, n_tile + c_begin * 32, c_end - c_begin, row, row < M, e, last);
            }
            const bool got = pair_wait<CL>(&tfull[acc], acc_phase, abort_flag, args.status, abort_local, rank);
            if (__any_sync(0xffffffffu, !got)) break;
            tc_fence_after();
            const int lane_extent = e.swap ? N : M, col_extent = e.swap ? M : N;
            const bool row_ok = row < lane_extent;
            const uint32_t t_row =
                tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * Cfg::ACC_STRIDE;
            const int col_base = n_tile + c_begin * 32;
            int nvalid = c_end - c_begin;
            const int left = (col_extent - col_base + 31) >> 5;  // chunks that start inside the matrix
            if (left < nvalid) nvalid = left;
            bool fail = false;
            if (seg.kind == kSegFull) {
                if (OUT == kDtE4M3 || !e.c_tma) {
                    epilogue_row_chunks<OUT, 4, SC>(t_row + c_begin * 32, col_base, nvalid, row, row_ok, bias_s, e);
                } else {
                    if constexpr (OUT != kDtE4M3) {
                        if (row0 < lane_extent && last)
                            fail = !epilogue_rows_tma_burst<OUT, SC>(
                                t_row + c_begin * 32, col_base, nvalid, row0, bias_s, bias_lane, e, &tmC,
                                smem + ew * Cfg::BURST_BYTES_PER_WARP, &cbar[ew], cphase, abort_flag, args.status);
                        else if (row0 < lane_extent)
                            fail = !epilogue_rows_tma<OUT, SC>(t_row + c_begin * 32, col_base, nvalid, row0, bias_s,
                                                               bias_lane, e, &tmC, cbuf, &cbar[ew], cphase, abort_flag,
                                                               args.status);
                    }
                }
            } else if (seg.kind == kSegPart) {
                float *slot = args.partial + (static_cast<long long>(cluster) * CL + rank) * kPartialFloatsPerCta;
                store_partial_chunks(t_row + c_begin * 32, c_begin, nvalid, r, slot);
                __threadfence();
                __syncwarp();
                if (lane == 0) st_release_gpu(&args.flags[(cluster * CL + rank) * 8 + ew], args.epoch);
            } else {
                const int c_last = last_contributor(args, seg.sk_tile, cluster, nclusters);
                const int ncontrib = c_last - cluster;
                for (int k = 1; k <= ncontrib && !fail; ++k) {
                    const unsigned int *f = &args.flags[((cluster + k) * CL + rank) * 8 + ew];
                    fail = !flag_wait_bounded(f, args.epoch, abort_flag, args.status);
                }
                if (__any_sync(0xffffffffu, fail)) {
                    raise_abort_others<CL>(abort_local, rank);
                    break;
                }
                const float *slot0 =
                    args.partial + (static_cast<long long>(cluster + 1) * CL + rank) * kPartialFloatsPerCta;
                fail = !owner_row_chunks<OUT, SC>(t_row + c_begin * 32, col_base, c_begin, nvalid, row, row_ok, r, slot0,
                                              CL * kPartialFloatsPerCta, ncontrib, bias_s, e, row0, &tmC, cbuf,
                                              &cbar[ew], cphase, abort_flag, args.status, bias_lane);
                __syncwarp();
                if (lane == 0)
                    for (int k = 1; k <= ncontrib; ++k) args.flags[((cluster + k) * CL + rank) * 8 + ew] = 0u;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(tempty0_leader + 8u * acc);
            if (__any_sync(0xffffffffu, fail)) {
                raise_abort_others<CL>(abort_local, rank);
                break;
            }
        }
        // Staged stores still in flight must finish before the CTA's shared memory goes.
        if (lane == 0) bulk_wait<0>();
        __syncwarp();
    }

    __syncwarp();
    tc_fence_before();
    cluster_sync_all();  // no CTA leaves while its peer may still signal into it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    }
}

// `clusters` clusters of CL CTAs.  With CL = 4, args.tiles_n / num_tiles /
// dp_tiles / sk_units count pairs of side-by-side tiles, and the A map's box
// is half a pair tile's rows (K-major A) or one swizzle row (MN-major A, an
// even number of them per 128 rows).
template <int AB, int OUT, int STAGES, int BNH = 128, int CL = 2>
cudaError_t launch_pair_cfg(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc, const TcArgs &args,
                            int clusters,
                            cudaStream_t stream) {
    using Cfg = PairConfig<AB, STAGES, BNH>;
    // What one CTA's loads of a stage occupy must fit its slots.
    if (args.bn > 2 * BNH) return cudaErrorInvalidValue;
    if (args.stage_tx > static_cast<uint32_t>(Cfg::STAGE_BYTES)) return cudaErrorInvalidValue;
    // Two pairs split each CTA's A rows between them: whole boxes only.
    if (CL == 4 && args.a_mn_major && (Cfg::BM / Cfg::SWZ) % 2 != 0) return cudaErrorInvalidValue;
    // E4M3 outputs always run the build with scales (the host marks them scaled).
    auto kern = gemm_tcgen05_pair_kernel<AB, OUT, STAGES, BNH, CL, true>;
    if constexpr (OUT != kDtE4M3) {
        if (!args.e.scaled) kern = gemm_tcgen05_pair_kernel<AB, OUT, STAGES, BNH, CL, false>;
    }
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL * clusters, 1, 1);
    cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // The prologue may start while the previous grid drains (the kernel waits
    // for it before its first global-memory access).
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, args);
}

// Largest number of CL-CTA clusters of this kernel that can be resident at once.
template <int AB, int OUT, int STAGES, int BNH = 128, int CL = 2>
int pair_max_clusters() {
    using Cfg = PairConfig<AB, STAGES, BNH>;
    // Both builds have the same footprint; E4M3 outputs exist only with scales.
    auto kern = gemm_tcgen05_pair_kernel<AB, OUT, STAGES, BNH, CL, OUT == kDtE4M3>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL, 1, 1);
    cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace gb300
