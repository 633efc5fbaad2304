// gemm_mma_sync.cu -- the warp-level matrix-instruction baseline of the
// cheap-baseline gate (Rigel, section 3: a kernel counts as a win only when it
// beats the legacy warp-matrix path by 1.10x; section 4, signal 2: the
// four-way showdown).  On Apple GPUs that path is simdgroup_matrix 8x8; its
// counterpart here is mma.sync.m16n8k16 (fp16 / bf16 in, fp32 accumulate),
// issued by every warp from fragments it loads itself, as "X3: Metal GEMM"
// sections 3-4 do with simdgroup_multiply_accumulate.
//
// A conventional multistage kernel: 128 x 128 output tile per CTA, 8 warps of
// 64 x 32, k-slices of 32 staged by cp.async (16-byte chunks, zero fill
// outside the matrix) in a 3-deep ring, fragments by ldmatrix (transposing
// for M-contiguous A and N-contiguous B), the same epilogue as the SIMT
// kernel.  Measurement only: gemm_baseline() runs it, gemm() never does.
#include "epilogue.cuh"
#include "kernel_args.h"

namespace gb300 {

namespace {

constexpr int kMsBM = 128, kMsBN = 128, kMsBK = 32, kMsStages = 3, kMsThreads = 256;
// Shared-memory rows are padded by 16 bytes so that the 8 row addresses of an
// ldmatrix fall in distinct bank groups.
constexpr int kMsKRow = kMsBK + 8;     // halves per row of a K-contiguous slice (rows = M or N)
constexpr int kMsMNRow = kMsBM + 8;    // halves per row of an M/N-contiguous slice (rows = K)
constexpr int kMsSlot = 128 * kMsKRow; // halves per operand per stage (>= kMsBK * kMsMNRow)
static_assert(kMsSlot >= kMsBK * kMsMNRow, "either layout fits the slot");
constexpr int kMsSmemBytes = kMsStages * 2 * kMsSlot * 2;

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <bool TRANS>
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *row_addr) {
    if constexpr (TRANS)
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "r"(smem_u32(row_addr)));
    else
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "r"(smem_u32(row_addr)));
}

template <int AB>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if constexpr (AB == kDtF16)
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

// A_K: A is K-contiguous (else M-contiguous).  B_K: B is K-contiguous (else
// N-contiguous).  The contiguous extent of each operand is a multiple of 8
// elements and its rows start 16-byte aligned (checked by the host).
template <int AB, int OUT, bool A_K, bool B_K>
__global__ void __launch_bounds__(kMsThreads) gemm_mma_sync_kernel(const SimtArgs a) {
    using InT = typename Elem<AB>::T;
    using OutT = typename Elem<OUT>::T;
    extern __shared__ __align__(16) unsigned char ms_smem[];
    InT *sm = reinterpret_cast<InT *>(ms_smem);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wm = (warp >> 2) * 64, wn = (warp & 3) * 32;  // warp's sub-tile in the CTA tile
    const int m0 = blockIdx.y * kMsBM, n0 = blockIdx.x * kMsBN;
    const int M = a.e.M, N = a.e.N, K = a.K;
    const InT *A = static_cast<const InT *>(a.A);
    const InT *B = static_cast<const InT *>(a.B);

    auto slot_a = [&](int s) { return sm + (s * 2) * kMsSlot; };
    auto slot_b = [&](int s) { return sm + (s * 2 + 1) * kMsSlot; };

    // One k-slice: 128 x 32 elements of each operand = 512 chunks of 8, two per thread.
    auto load_slice = [&](int s, int k0) {
        InT *sa = slot_a(s), *sb = slot_b(s);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int c = tid + r * kMsThreads;
            if constexpr (A_K) {
                const int row = c >> 2, kc = (c & 3) * 8;
                const bool ok = m0 + row < M && k0 + kc < K;
                const InT *src = ok ? A + (long long)(m0 + row) * a.sam + (k0 + kc) : A;
                cp_async16(sa + row * kMsKRow + kc, src, ok);
            } else {
                const int k = c >> 4, mc = (c & 15) * 8;
                const bool ok = k0 + k < K && m0 + mc < M;
                const InT *src = ok ? A + (long long)(k0 + k) * a.sak + (m0 + mc) : A;
                cp_async16(sa + k * kMsMNRow + mc, src, ok);
            }
            if constexpr (B_K) {
                const int row = c >> 2, kc = (c & 3) * 8;
                const bool ok = n0 + row < N && k0 + kc < K;
                const InT *src = ok ? B + (long long)(n0 + row) * a.sbn + (k0 + kc) : B;
                cp_async16(sb + row * kMsKRow + kc, src, ok);
            } else {
                const int k = c >> 4, nc = (c & 15) * 8;
                const bool ok = k0 + k < K && n0 + nc < N;
                const InT *src = ok ? B + (long long)(k0 + k) * a.sbk + (n0 + nc) : B;
                cp_async16(sb + k * kMsMNRow + nc, src, ok);
            }
        }
    };

    float acc[4][4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int v = 0; v < 4; ++v) acc[i][j][v] = 0.0f;

    const int ktiles = (K + kMsBK - 1) / kMsBK;
#pragma unroll
    for (int s = 0; s < kMsStages - 1; ++s) {
        if (s < ktiles) load_slice(s, s * kMsBK);
        cp_async_commit();
    }
    for (int kt = 0; kt < ktiles; ++kt) {
        cp_async_wait<kMsStages - 2>();
        __syncthreads();  // slice kt landed for every thread; slice kt-1's slot is free
        const int nxt = kt + kMsStages - 1;
        if (nxt < ktiles) load_slice(nxt % kMsStages, nxt * kMsBK);
        cp_async_commit();
        const InT *sa = slot_a(kt % kMsStages), *sb = slot_b(kt % kMsStages);
#pragma unroll
        for (int kk = 0; kk < kMsBK; kk += 16) {
            uint32_t af[4][4], bf[2][4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int mb = wm + i * 16;
                if constexpr (A_K) {
                    // matrices: rows 0-7 / 8-15 (lanes 0-15) at k 0-7, then at k 8-15 (lanes 16-31)
                    ldsm_x4<false>(af[i], sa + (mb + (lane & 15)) * kMsKRow + kk + (lane >> 4) * 8);
                } else {
                    // stored rows are k: lanes give k = kk + (lane&7) + 8*(lane>>4), m offset 8*((lane>>3)&1)
                    ldsm_x4<true>(af[i], sa + (kk + (lane & 7) + (lane >> 4) * 8) * kMsMNRow + mb +
                                             ((lane >> 3) & 1) * 8);
                }
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int nb = wn + j * 16;  // two n8 blocks per ldmatrix.x4
                if constexpr (B_K) {
                    // stored rows are n: n = (lane&7) + 8*(lane>>4), k offset 8*((lane>>3)&1)
                    ldsm_x4<false>(bf[j], sb + (nb + (lane & 7) + (lane >> 4) * 8) * kMsKRow + kk +
                                              ((lane >> 3) & 1) * 8);
                } else {
                    // stored rows are k: k = (lane&7) + 8*((lane>>3)&1), n offset 8*(lane>>4)
                    ldsm_x4<true>(bf[j], sb + (kk + (lane & 7) + ((lane >> 3) & 1) * 8) * kMsMNRow + nb +
                                             (lane >> 4) * 8);
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) mma16816<AB>(acc[i][j], af[i], bf[j >> 1][(j & 1) * 2], bf[j >> 1][(j & 1) * 2 + 1]);
        }
    }
    cp_async_wait<0>();

    // Thread (g, t) = (lane / 4, lane % 4) holds rows g and g + 8, columns 2t and 2t + 1 of each 16 x 8 block.
    OutT *C = static_cast<OutT *>(a.e.C);
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int row = m0 + wm + i * 16 + g + (v >> 1) * 8;
                const int col = n0 + wn + j * 8 + 2 * t + (v & 1);
                if (row < M && col < N) {
                    const float b = (a.e.epilogue != kEpiNone) ? a.e.bias[col] : 0.0f;
                    epilogue_store_one<OUT>(acc[i][j][v], C + (long long)row * a.e.ldc + col, b, a.e);
                }
            }
}

template <int AB, int OUT, bool A_K, bool B_K>
cudaError_t launch_ms(const SimtArgs &a, cudaStream_t s) {
    auto kern = gemm_mma_sync_kernel<AB, OUT, A_K, B_K>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMsSmemBytes);
    if (err != cudaSuccess) return err;
    dim3 grid((a.e.N + kMsBN - 1) / kMsBN, (a.e.M + kMsBM - 1) / kMsBM);
    kern<<<grid, kMsThreads, kMsSmemBytes, s>>>(a);
    return cudaGetLastError();
}

template <int AB, int OUT>
cudaError_t launch_ms_layout(const SimtArgs &a, bool a_k, bool b_k, cudaStream_t s) {
    if (a_k && b_k) return launch_ms<AB, OUT, true, true>(a, s);
    if (a_k) return launch_ms<AB, OUT, true, false>(a, s);
    if (b_k) return launch_ms<AB, OUT, false, true>(a, s);
    return launch_ms<AB, OUT, false, false>(a, s);
}

}  // namespace

cudaError_t launch_mma_sync(int ab, int out, const SimtArgs &a, bool a_k_contig, bool b_k_contig, cudaStream_t s) {
    if ((a.e.M + kMsBM - 1) / kMsBM > 65535) return cudaErrorInvalidConfiguration;
    switch (ab * 4 + out) {
    case kDtF16 * 4 + kDtF16: return launch_ms_layout<kDtF16, kDtF16>(a, a_k_contig, b_k_contig, s);
    case kDtF16 * 4 + kDtF32: return launch_ms_layout<kDtF16, kDtF32>(a, a_k_contig, b_k_contig, s);
    case kDtF16 * 4 + kDtBF16: return launch_ms_layout<kDtF16, kDtBF16>(a, a_k_contig, b_k_contig, s);
    case kDtBF16 * 4 + kDtBF16: return launch_ms_layout<kDtBF16, kDtBF16>(a, a_k_contig, b_k_contig, s);
    case kDtBF16 * 4 + kDtF32: return launch_ms_layout<kDtBF16, kDtF32>(a, a_k_contig, b_k_contig, s);
    case kDtBF16 * 4 + kDtF16: return launch_ms_layout<kDtBF16, kDtF16>(a, a_k_contig, b_k_contig, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gb300
