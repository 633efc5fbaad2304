// kernel_args.h -- argument blocks passed by value from the host library to
// the kernels, and the launcher entry points each kernel file exports to the
// host library (internal; not part of the C ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime_api.h>

namespace gb300 {

// Element type and epilogue codes, numbered like gemm_dtype_t / gemm_epilogue_t.
enum : int { kDtF32 = 0, kDtF16 = 1, kDtBF16 = 2, kDtE4M3 = 3 };
// Internal operand format of the tensor-core fp32 path: each operand split into
// a tf32 "hi" and an fp32 "lo" part, stacked in one K-major array (3xTF32).
enum : int { kDtTF32x3 = 4 };
enum : int { kEpiNone = 0, kEpiBias = 1, kEpiBiasGelu = 2, kEpiBiasGeluTanh = 3, kEpiBiasSilu = 4,
             kEpiBiasRelu = 5 };

// Everything the epilogue needs: output geometry and the scalars.
struct EpiParams {
    int M, N;
    void *C;          // M x ldc row-major output (input too when beta != 0)
    long long ldc;    // elements
    const float *bias;
    float alpha, beta;
    int epilogue;
    int c_vec;        // C base and row pitch allow 16-byte vector access
    int c_tma;        // pair kernel: C moves through shared memory by TMA (the kernel's C map is valid)
    int swap;         // pair kernel: the MMA computes C^T = B^T A^T (TMEM lanes are output columns)
    // Product scales (gemm_ex), device pointers, each NULL when absent: the product
    // term is alpha * alpha_scale[0] * row_scale[i] * col_scale[j] * acc.
    int scaled;       // any product scale, out_scale or amax is present, or the output is E4M3
    const float *alpha_scale, *row_scale, *col_scale;
    const float *out_scale;  // E4M3 output: stores y / out_scale[0] (NULL = 1)
    float *amax;             // atomically raised to max |y| over the outputs (NULL = not kept)
    // Post-activation residual (gemm_ex): y = act(z) + R[i][j], R an M x ldr
    // row-major array of the output type; NULL when absent (then `scaled` may be 0).
    const void *residual;
    long long ldr;           // elements
    int r_vec;               // R's base and row pitch allow 16-byte vector loads
};

// Most clusters a stream-K schedule spreads over (the cut table's size).
constexpr int kMaxSkClusters = 128;

// tcgen05 path: operands come through the two tensor maps.
struct TcArgs {
    EpiParams e;
    int K;
    int tiles_m, tiles_n, num_tiles, num_kb, group_m;
    uint32_t a_mn_major, b_mn_major;  // 1: the M (resp. N) index is the contiguous one
    unsigned int *status;             // device status word (timeouts)
    int bn;                           // pair kernel: tile width (multiple of 32, <= 256)
    uint32_t stage_tx;                // pair kernel: bytes one CTA's loads deliver per stage
    // Pair kernel schedule.  Tiles [0, dp_tiles) are computed whole, cluster c
    // taking c, c + clusters, ...; the k-blocks of tiles [dp_tiles, num_tiles)
    // form one range of sk_units = (num_tiles - dp_tiles) * num_kb units that
    // is cut into `clusters` contiguous pieces (stream-K): cluster c's piece is
    // units [sk_cut[c], sk_cut[c + 1]).  The cuts start at 0, end at sk_units
    // and never decrease; only trailing pieces may be empty.
    int dp_tiles;
    long long sk_units;
    unsigned int sk_cut[kMaxSkClusters + 1];
    float *partial;                   // stream-K: per CTA, 128 x 256 fp32 partial sums
    unsigned int *flags;              // stream-K: per CTA, 8 epilogue warps
    unsigned int epoch;               // stream-K: value a flag takes when its partial is ready (never 0)
    int lo_row_a, lo_row_b;           // 3xTF32: first row of the "lo" half in the stacked A / B arrays
};

// Floats of stream-K partial sums one CTA of a cluster writes, and flags per cluster.
constexpr long long kPartialFloatsPerCta = 128LL * 256LL;
constexpr int kFlagsPerCluster = 2 * 8;

// SIMT path: operands as (pointer, stride) views, any strides.
struct SimtArgs {
    EpiParams e;
    int K;
    const void *A;
    long long sam, sak;
    const void *B;
    long long sbk, sbn;
};

// Quantized matrix product (4-bit codes, 64 per group along K; see gemm_q4.cu).
struct Q4Args {
    EpiParams e;              // M rows of x / C, N outputs per row, C, ldc, alpha, beta, bias, epilogue
    int K;
    const void *X;            // M x ldx row-major, fp16 or bf16
    long long ldx;
    const uint32_t *Wq;       // N * K/8 words: code of (n, k) in bits 4*(k%8) of word n*K/8 + k/8
    const uint32_t *SB;       // N * K/64 words: binary16 scale (low half) and bias (high half) of group (n, g)
    unsigned int *status;     // device status word (timeouts of the tensor-core kernel's waits)
    int w_pitch;              // tensor-core kernel: width in bytes of its weight box, min(160, K / 2)
};

// Block-scaled (MX) product: elements of A (M x K) and of B given as its
// transpose (N x K), both K-contiguous, with one E8M0 scale per 32 consecutive
// k of a row.  Element types: E4M3 one per byte (MXFP8), E2M1 two per byte,
// even k in the low nibble (MXFP4).
enum : int { kMxE4M3 = 0, kMxE2M1 = 1 };

// Scale factors as the kernel reads them (written by the pack pre-pass): for
// each operand, 512-byte chunks of 128 rows x 4 blocks of 32 k; chunk (rb, kc)
// at byte (rb * kc_count + kc) * 512, and inside it the scale of row
// 128 rb + 32 g + l and block 4 kc + j at byte 16 l + 4 g + j -- the layout
// tcgen05.cp ... 32x128b.warpx4 turns into the tensor-memory scale layout of
// the block-scaled MMA (row r's scales at lane r, column r / 32, byte j).
struct MxArgs {
    EpiParams e;
    int K;                          // elements
    int tiles_m, tiles_n, num_tiles, num_kb, group_m;  // num_kb: stages of 128 bytes of K
    const unsigned char *sfa, *sfb; // chunked scales of A and B
    int kc_count;                   // chunk columns per 128-row block (a multiple of the chunks per stage)
    unsigned int *status;
};

// Launchers (each returns the launch's cudaError_t), defined by the kernel files.
//   one-SM tcgen05 kernel, `bn` = 256 or 128, `grid` CTAs:
cudaError_t launch_tcgen05_f16(int out, int bn, const CUtensorMap &, const CUtensorMap &, const TcArgs &, int grid,
                               cudaStream_t);
cudaError_t launch_tcgen05_bf16(int out, int bn, const CUtensorMap &, const CUtensorMap &, const TcArgs &, int grid,
                                cudaStream_t);
cudaError_t launch_tcgen05_e4m3(int out, int bn, const CUtensorMap &, const CUtensorMap &, const TcArgs &, int grid,
                                cudaStream_t);
//   pair kernel (tile width in args.bn), `clusters` clusters of `cl` CTAs (2: one
//   pair; 4: two pairs sharing A by multicast, the schedule counting pairs of
//   side-by-side tiles); the third map describes C (read only when args.e.c_tma != 0):
cudaError_t launch_pair_f16(int out, int cl, const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                            const TcArgs &, int clusters, cudaStream_t);
cudaError_t launch_pair_bf16(int out, int cl, const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                             const TcArgs &, int clusters, cudaStream_t);
cudaError_t launch_pair_e4m3(int out, int cl, const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                             const TcArgs &, int clusters, cudaStream_t);
int pair_max_clusters_f16(int out, int cl);
int pair_max_clusters_bf16(int out, int cl);
int pair_max_clusters_e4m3(int out, int cl);
//   3xTF32 pair kernel (fp32 output) and the hi/lo split pre-pass:
cudaError_t launch_pair_tf32x3(int out, const CUtensorMap &, const CUtensorMap &, const CUtensorMap &, const TcArgs &, int clusters,
                               cudaStream_t);
int pair_max_clusters_tf32x3(int out);
cudaError_t launch_tf32_split(const float *src, long long rows, long long cols, long long s_row, long long s_col,
                              float *dst, long long pitch, cudaStream_t stream);
//   CUDA-core kernels:
cudaError_t launch_simt(int ab, int out, const SimtArgs &args, cudaStream_t stream);
//   warp-level mma.sync baseline (fp16 / bf16; operand layouts by contiguity):
cudaError_t launch_mma_sync(int ab, int out, const SimtArgs &args, bool a_k_contig, bool b_k_contig,
                            cudaStream_t stream);
cudaError_t launch_epilogue_only(int out, const EpiParams &e, cudaStream_t stream);
cudaError_t launch_bias_gelu(int out, const EpiParams &e, cudaStream_t stream);
//   4-bit quantized product for up to kQ4MaxRows rows of x, and the dequantisation pass:
constexpr int kQ4MaxRows = 8;
//   4-bit decode: with a map of the codes (K/2 bytes x N rows, box w_pitch x 32 rows) the tensor-core
//   kernel (TMA staging, mma.sync), without one (nullptr) the CUDA-core kernel
cudaError_t launch_q4_gemv(int x_dtype, int out, const CUtensorMap *tmW, const Q4Args &args, cudaStream_t stream);
cudaError_t launch_q4_dequantize(int out, long long N, long long K, const uint32_t *Wq, const uint32_t *SB, void *W,
                                 cudaStream_t stream);
//   4-bit prefill (more than kQ4MaxRows rows of x): x by a map over (K, M) with 64 x 128 boxes
//   (128-byte swizzle), the codes by a map over (K/2 bytes, N) with 32 x 128 boxes; `grid` CTAs
cudaError_t launch_q4_prefill(int x_dtype, int out, const CUtensorMap &tmX, const CUtensorMap &tmW, const Q4Args &args,
                              int grid, cudaStream_t stream);
//   block-scaled product (one SM per 128 x 128 tile) and its scale-factor pack pre-pass:
cudaError_t launch_mx(int elem, int out, const CUtensorMap &ta, const CUtensorMap &tb, const MxArgs &args, int grid,
                      cudaStream_t stream);
// The same product on SM pairs, 256 x 256 tiles: tsa / tsb map the chunked
// scales as rows of 256 bytes (two per chunk), boxes of 2 x chunks-per-stage
// rows; `clusters` CTA pairs.
cudaError_t launch_mx_pair(int elem, int out, const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tsa,
                           const CUtensorMap &tsb, const MxArgs &args, int clusters, cudaStream_t stream);
cudaError_t launch_mx_sf_pack(const unsigned char *src, long long rows, long long blocks, unsigned char *dst,
                              long long row_blocks, long long kc_count, cudaStream_t stream);
cudaError_t launch_wait_selftest(const unsigned int *never_set, unsigned long long limit_ns, unsigned int *status,
                                 cudaStream_t stream);

}  // namespace gb300
