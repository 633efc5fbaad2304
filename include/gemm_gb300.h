/*
 * gemm_gb300.h -- C ABI of the GB300 (sm_103a) dense GEMM with fused epilogue.
 *
 * Operation (one call):
 *
 *     z[i][j] = alpha * sum_k A[i][k] * B[k][j]  +  beta * C[i][j]  +  bias[j]
 *     C[i][j] = cast_out( epilogue(z[i][j]) )        for 0 <= i < M, 0 <= j < N
 *
 * with fp32 accumulation whatever the input type, the epilogue applied to the
 * accumulators in registers and the result stored once.  Defined on the pages
 * by: "Case Study: Steel's BlockMMA" (the paragraph on the ending where fusion
 * plugs in -- store_result applies the Epilogue to every accumulator, and
 * apply_epilogue reads an input C for alpha*AB + beta*C; AccumType = float;
 * transposition by the A_str_m / A_str_k stride constants), "Case Study: The
 * Tiled GEMM" (the fused alpha*AB + beta*C store), "X3: Metal GEMM" sections
 * 2, 4 and 5 (out-of-range operand elements read as zero; the masked,
 * casting write-back that never touches elements outside M x N) and Rigel
 * (abstract and section 1: GEMM + bias + GELU fused into one kernel).
 *
 * Conventions shared by every entry point
 *   - All pointers except those documented as host pointers are DEVICE
 *     pointers on the current CUDA device.  The caller owns every buffer;
 *     the library allocates nothing per call and keeps no pointer after a
 *     call returns.
 *   - Strides and leading dimensions are in ELEMENTS, not bytes.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *     A returned GEMM_OK means the work was enqueued; device-side failures
 *     are reported later by gemm_device_status().
 *   - No entry point prints, aborts or traps.  Argument errors return a
 *     status code before anything is enqueued.
 */
#ifndef GEMM_GB300_H
#define GEMM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *gemm_stream_t;

/* Element types.  E4M3 is OCP FP8 E4M3 ("fn": finite, saturating, NaN = S.1111.111). */
typedef enum {
    GEMM_F32 = 0,
    GEMM_F16 = 1,
    GEMM_BF16 = 2,
    GEMM_E4M3 = 3
} gemm_dtype_t;

/* Epilogues, applied to z before the cast: none, or bias[j] added and then
 * an activation.  GELU is the exact erf form 0.5*z*(1 + erf(z/sqrt(2))) (the
 * pages' bias+GELU fusion, Rigel section 1); the others use the same
 * pluggable place ("Case Study: Steel's BlockMMA", the Epilogue functor):
 * GELU's tanh form 0.5*z*(1 + tanh(sqrt(2/pi)*(z + 0.044715*z^3))), SiLU
 * z/(1 + exp(-z)) and ReLU max(z, 0).  Every one needs a bias. */
typedef enum {
    GEMM_EPI_NONE = 0,
    GEMM_EPI_BIAS = 1,
    GEMM_EPI_BIAS_GELU = 2,
    GEMM_EPI_BIAS_GELU_TANH = 3,
    GEMM_EPI_BIAS_SILU = 4,
    GEMM_EPI_BIAS_RELU = 5
} gemm_epilogue_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,   /* negative size, ldc < N, bad enum, NULL where a buffer is needed */
    GEMM_ERR_UNSUPPORTED = 2,   /* dtype combination the library does not implement */
    GEMM_ERR_MISALIGNED = 3,    /* reserved: every stride/alignment has a path, so not returned today */
    GEMM_ERR_WORKSPACE = 4,     /* workspace missing or smaller than gemm_workspace_size() */
    GEMM_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed (launch, attribute, tensor map) */
    GEMM_ERR_TIMEOUT = 6        /* a device-side wait gave up (reported by gemm_device_status) */
} gemm_status_t;

/* Which kernel family a call runs on (see gemm_query_path).  fp32 inputs report
 * GEMM_PATH_SIMT, the path without a workspace; given a workspace of
 * gemm_workspace_size() bytes they run as 3xTF32 on the tensor cores. */
typedef enum {
    GEMM_PATH_NOOP = 0,           /* M == 0 or N == 0: nothing to do */
    GEMM_PATH_EPILOGUE_ONLY = 1,  /* K == 0 or alpha == 0: C = cast(epilogue(beta*C + bias)) */
    GEMM_PATH_TCGEN05 = 2,        /* TMA -> shared memory -> tcgen05.mma (TMEM accumulators) */
    GEMM_PATH_SIMT = 3            /* CUDA-core FFMA kernel (fp32 inputs, or strides TMA cannot take) */
} gemm_path_t;

/*
 * gemm -- C = cast(epilogue(alpha*A*B + beta*C + bias)), C updated in place.
 *
 *   M, N, K        problem sizes, each >= 0.  M == 0 or N == 0 is a no-op.
 *                  K == 0 (or alpha == 0) gives C = cast(epilogue(beta*C + bias))
 *                  and reads neither A nor B (BLAS convention).
 *   ab_dtype       element type of A and B: F32, F16, BF16 or E4M3.
 *   A              element (i, k) is A[i*a_stride_m + k*a_stride_k].
 *   B              element (k, j) is B[k*b_stride_k + j*b_stride_n].
 *                  Transposition is expressed only through these strides; any
 *                  non-negative strides are accepted.  When one stride of an
 *                  operand is 1, the base is 16-byte aligned and the other
 *                  stride is a multiple of 16 bytes, the operand is streamed
 *                  by TMA; otherwise the call runs on the SIMT kernel.
 *   C, ldc         row-major M x N output (and input when beta != 0) inside an
 *                  M x ldc buffer, ldc >= N.  Columns N..ldc-1 and anything
 *                  outside the M x N block are never written.
 *   c_dtype        F32, F16 or BF16.  F32 inputs require F32 output; E4M3
 *                  inputs require BF16 or F32 output.
 *   alpha, beta    fp32 scalars.  beta == 0: C is not read (NaNs in C do not
 *                  propagate).  For fp8 with per-tensor dequantisation scales
 *                  s_a, s_b, pass alpha * s_a * s_b.
 *   bias           fp32[N] device array, required (non-NULL) for every
 *                  epilogue other than GEMM_EPI_NONE, ignored for NONE.
 *   epilogue       a gemm_epilogue_t; the order is z = alpha*AB + beta*C +
 *                  bias, then the activation, then the cast (round to nearest
 *                  even).
 *   workspace      optional device scratch, 256-byte aligned, owned by the
 *   workspace_bytes  caller: with at least gemm_workspace_size(...) bytes the
 *                  last waves of output tiles are split along K over all SM
 *                  pairs (stream-K: partial sums go through the workspace);
 *                  with less, or NULL / 0, whole tiles only.  Calls that share
 *                  a workspace must not run concurrently.  Its contents need no
 *                  initialisation (each call tags its flags with a fresh value).
 *   stream         CUDA stream the work is enqueued on.
 *
 * Aliasing: C must not overlap A, B or bias.  Returns GEMM_OK once enqueued.
 */
gemm_status_t gemm(int64_t M, int64_t N, int64_t K,
                   gemm_dtype_t ab_dtype,
                   const void *A, int64_t a_stride_m, int64_t a_stride_k,
                   const void *B, int64_t b_stride_k, int64_t b_stride_n,
                   void *C, int64_t ldc, gemm_dtype_t c_dtype,
                   float alpha, float beta,
                   const float *bias, gemm_epilogue_t epilogue,
                   void *workspace, size_t workspace_bytes,
                   gemm_stream_t stream);

/*
 * Scales of gemm_ex, each a DEVICE pointer read when the kernel runs (so a
 * scale computed by an earlier kernel needs no host round trip), each
 * optional (NULL = absent):
 *   alpha_scale  fp32[1]  per-tensor product scale, e.g. s_a * s_b of fp8 operands;
 *   row_scale    fp32[M]  per row of A / C (per token);
 *   col_scale    fp32[N]  per column of B / C (per output channel);
 *   out_scale    fp32[1]  E4M3 output only: C stores y / out_scale[0] (NULL = 1),
 *                         rounded to nearest even and saturated to +-448;
 *   amax         fp32[1]  raised atomically to max |y| over the M x N outputs,
 *                         y being the activated value (plus the residual)
 *                         before out_scale and the cast; the caller sets it
 *                         (e.g. to 0) beforehand.
 *   residual     M x ldr row-major array of the OUTPUT type (F32, F16 or BF16;
 *                         not with an E4M3 output), added after the activation:
 *                         y = act(z) + residual[i][j] -- the post-activation
 *                         residual of a transformer block.  ldr >= N (elements);
 *                         columns N..ldr-1 are never read.  It must not overlap
 *                         C.  NULL = none (ldr ignored).
 * The product term becomes alpha * alpha_scale[0] * row_scale[i] *
 * col_scale[j] * sum_k A[i][k] B[k][j]; beta*C, the bias and the residual are
 * not scaled.  ("Case Study: Steel's BlockMMA", the paragraph on the ending
 * where fusion plugs in: the epilogue is a functor applied to every
 * accumulator before the store; these are its per-row / per-column forms, the
 * fp8 output with its amax the quantising store of a low-precision path, and
 * the residual one more input of that functor.)
 */
typedef struct {
    const float *alpha_scale;
    const float *row_scale;
    const float *col_scale;
    const float *out_scale;
    float *amax;
    const void *residual;
    int64_t ldr;
} gemm_scales_t;

/*
 * gemm_ex -- gemm() with the scales and the residual above (scales may be
 * NULL: then exactly gemm()).  Same arguments, conventions and errors, plus
 * c_dtype E4M3 (fp8 output, from F16, BF16 or E4M3 inputs, beta == 0;
 * otherwise GEMM_ERR_UNSUPPORTED).  The scale and residual arrays are checked
 * against their device allocations like every other buffer; a residual with
 * an E4M3 output is GEMM_ERR_UNSUPPORTED, ldr < N GEMM_ERR_INVALID_ARG.  With
 * K == 0 or alpha == 0 the product scales are not read (out_scale, amax and
 * the residual still apply).
 */
gemm_status_t gemm_ex(int64_t M, int64_t N, int64_t K,
                      gemm_dtype_t ab_dtype,
                      const void *A, int64_t a_stride_m, int64_t a_stride_k,
                      const void *B, int64_t b_stride_k, int64_t b_stride_n,
                      void *C, int64_t ldc, gemm_dtype_t c_dtype,
                      float alpha, float beta,
                      const float *bias, gemm_epilogue_t epilogue,
                      const gemm_scales_t *scales,
                      void *workspace, size_t workspace_bytes,
                      gemm_stream_t stream);

/*
 * gemm_workspace_size -- bytes of device scratch that let gemm() use its
 * fastest path.  fp16 / bf16 / fp8 inputs: the stream-K schedule on the
 * current device, 256 KB of partial sums and 64 bytes of flags per pair of SMs
 * (about 19 MB on a 152-SM GB300), independent of M, N, K; 0 when the device
 * cannot be queried.  fp32 inputs: the 3xTF32 split of both operands, hi and
 * lo copies in K-major rows padded to 16 bytes, 2*(M+N)*ceil4(K)*4 bytes
 * (each half rounded up to 256); with it gemm() runs fp32 on the tensor
 * cores, without it on the FFMA kernel.  Never fails.
 */
size_t gemm_workspace_size(int64_t M, int64_t N, int64_t K, gemm_dtype_t ab_dtype);

/* How the tcgen05 pair kernel distributes tiles (a per-thread setting). */
typedef enum {
    GEMM_SCHED_AUTO = 0,     /* stream-K for the last waves when the tiles do not divide evenly */
    GEMM_SCHED_TILES = 1,    /* whole tiles only */
    GEMM_SCHED_STREAM_K = 2  /* every tile's k-blocks in one range split over all SM pairs */
} gemm_schedule_t;

/*
 * gemm_set_schedule -- schedule of the calling thread's later gemm() calls on
 * the pair kernel (stream-K still needs a large enough workspace); other
 * threads keep their own setting.  Meant for tuning and tests.
 * GEMM_ERR_INVALID_ARG for an unknown value; never touches the device.
 */
gemm_status_t gemm_set_schedule(gemm_schedule_t schedule);

/*
 * Operand order of the pair kernel.  The kernel can compute C = A*B as
 * C^T = B^T * A^T, with B's transpose as the MMA's first operand and C^T's
 * rows written as C's columns.  On GB300 a second MMA operand that is
 * N-contiguous (B stored K x N row-major) keeps the tensor pipe measurably
 * less busy than a K-contiguous one (79.5 % vs 86.5 % of cycles, bf16
 * 8192^3), so AUTO transposes exactly that case for fp16 / bf16 inputs: A
 * K-contiguous, B N-contiguous, 16-bit output, C base and pitch usable by
 * TMA (fp8 inputs measured no faster transposed and keep the given order).
 * The result is the same product; only the summation order inside fp32
 * accumulation may differ.
 */
typedef enum {
    GEMM_ORDER_AUTO = 0,        /* transpose when it is the faster orientation (above) */
    GEMM_ORDER_AS_GIVEN = 1,    /* never transpose */
    GEMM_ORDER_TRANSPOSED = 2   /* transpose whenever the output allows (16-bit, TMA-able C) */
} gemm_operand_order_t;

/*
 * gemm_set_operand_order -- operand order of the calling thread's later
 * gemm() calls on the pair kernel; other threads keep their own setting.
 * Meant for tuning and tests.  GEMM_ERR_INVALID_ARG for an unknown value;
 * never touches the device.
 */
gemm_status_t gemm_set_operand_order(gemm_operand_order_t order);

/*
 * Cluster shape of the pair kernel.  A cluster can hold two SM pairs that
 * compute two output tiles side by side along N, over the same rows of A:
 * each CTA then fetches half of its A rows and the TMA multicasts them to the
 * CTA in the same place of the other pair, so every A panel crosses from L2
 * to shared memory once per two tiles (a quarter fewer operand bytes per SM).
 * Tiles, results and the summation order are the same either way.  Four-CTA
 * clusters may fit on fewer SMs (GB300: 144 of 152), so AUTO uses them where
 * that costs less than the traffic saves: when the tile columns pair up
 * evenly and either no SM is lost or the problem has at most four waves of
 * tiles.  Both shapes need A's tile rows to split into whole TMA boxes (any
 * K-contiguous A; an M-contiguous A with 16-bit elements).  ON forces
 * two-pair clusters wherever A splits, even with an odd number of tile
 * columns (the last pair then computes a tile outside the matrix and stores
 * nothing).
 *
 * A multicast load's tensor map may cover only the calling GPU's own memory:
 * the pair kernel's first operand (A, or B when it computes C^T = B^T A^T)
 * must be a device allocation of the current device, else the call runs
 * one-pair clusters whatever the setting (pinned host memory or another
 * GPU's memory is read by plain per-CTA TMA loads).
 */
typedef enum {
    GEMM_MCAST_AUTO = 0,   /* two-pair clusters where they measured faster (above) */
    GEMM_MCAST_OFF = 1,    /* one pair per cluster */
    GEMM_MCAST_ON = 2      /* two pairs per cluster wherever A's rows split between them */
} gemm_multicast_t;

/*
 * gemm_set_multicast -- cluster shape of the calling thread's later gemm()
 * calls on the pair kernel; other threads keep their own setting.  Meant for
 * tuning and tests.  GEMM_ERR_INVALID_ARG for an unknown value; never touches
 * the device.
 */
gemm_status_t gemm_set_multicast(gemm_multicast_t mode);

/*
 * gemm_query_path -- validate the same arguments gemm() takes and report, in
 * *path (host pointer), which kernel family gemm() would launch.  Launches
 * nothing and touches no device memory.  Returns the status gemm() would
 * return before enqueueing.
 */
gemm_status_t gemm_query_path(int64_t M, int64_t N, int64_t K,
                              gemm_dtype_t ab_dtype,
                              const void *A, int64_t a_stride_m, int64_t a_stride_k,
                              const void *B, int64_t b_stride_k, int64_t b_stride_n,
                              const void *C, int64_t ldc, gemm_dtype_t c_dtype,
                              float alpha, float beta,
                              const float *bias, gemm_epilogue_t epilogue,
                              gemm_path_t *path);

/* Tile policy of the tcgen05 path (a per-thread setting; see gemm_set_tile_policy). */
typedef enum {
    GEMM_TILE_AUTO = 0,     /* cost model: wave balance over the SMs and shared-memory bandwidth */
    GEMM_TILE_1SM_256 = 1,  /* one SM per 128 x 256 output tile */
    GEMM_TILE_1SM_128 = 2,  /* one SM per 128 x 128 output tile */
    GEMM_TILE_PAIR = 3      /* a cluster of two SMs per 256 x bn output tile (cta_group::2 MMA) */
} gemm_tile_policy_t;

/*
 * gemm_set_tile_policy -- choose how the calling thread's later gemm() calls
 * tile the output on the tcgen05 path; other threads keep their own setting.
 * `bn` is used with
 * GEMM_TILE_PAIR only: a multiple of 32 in 128..256, or 0 to let the cost
 * model pick the width.  Meant for tuning and tests; GEMM_TILE_AUTO (the
 * default) is the right choice otherwise.  Returns GEMM_ERR_INVALID_ARG for an
 * unknown policy or width; never touches the device.
 */
gemm_status_t gemm_set_tile_policy(gemm_tile_policy_t policy, int bn);

/*
 * gemm_query_tile -- the tile the tcgen05 path would use on the current device
 * for an M x N x K problem: *kind = 1 for one SM per tile, 2 for a pair of SMs;
 * *bn = tile width; *units = tiles in flight at once (CTAs, or two-CTA
 * clusters).  All three are host pointers.  Reads device attributes; launches
 * nothing.  GEMM_ERR_CUDA if the device cannot be queried.
 */
gemm_status_t gemm_query_tile(int64_t M, int64_t N, int64_t K, gemm_dtype_t ab_dtype, gemm_dtype_t c_dtype,
                              int *kind, int *bn, int *units);

/*
 * What the calling thread's last gemm() (or gemm_builtin_scratch()) call
 * enqueued, for tuning, tests and reports.  No counterpart on the pages.
 */
typedef struct {
    int path;          /* gemm_path_t of the kernel family launched (NOOP when nothing was) */
    int kind;          /* tcgen05 path: 1 one SM per tile, 2 a pair of SMs per tile; else 0 */
    int bn;            /* tcgen05 path: tile width in columns of the MMA's output */
    int transposed;    /* 1 when the pair kernel ran C^T = B^T A^T */
    int cluster_ctas;  /* CTAs per cluster: 1 (one-SM kernel), 2 (one pair) or 4 (two pairs sharing A) */
    int grid_ctas;     /* CTAs of the tcgen05 GEMM kernel (0 on the other paths) */
    int tiles;         /* its scheduling units: output tiles, or pairs of tiles side by side for
                          4-CTA clusters (0 on the other paths) */
    int stream_k_tiles;/* of those, units whose k-blocks are split over all clusters */
    int tf32x3;        /* 1 when fp32 inputs ran as 3xTF32 (split pre-pass + tensor cores) */
} gemm_launch_info_t;

/*
 * gemm_last_launch -- copy the calling thread's record of its last gemm()
 * call that returned GEMM_OK into *info (host pointer).  A call that failed
 * leaves the record as it was.  GEMM_ERR_INVALID_ARG for info == NULL.
 * Touches no device.
 */
gemm_status_t gemm_last_launch(gemm_launch_info_t *info);

/*
 * gemm_builtin_scratch -- gemm() for callers that cannot allocate device
 * memory.  (The pages have no counterpart: this is a deployment convenience
 * of this library, not part of the method.)
 *
 * gemm() takes the stream-K scratch (partial sums and ready flags) from a
 * workspace the caller allocates.  Code that cannot call cudaMalloc or any
 * allocating routine where it multiplies -- inside CUDA stream capture, on
 * real-time paths, or in processes whose device memory belongs to another
 * allocator -- calls this instead: same arguments and result as gemm()
 * without the workspace pair, with the scratch taken from a fixed array of
 * 20,976,640 bytes (enough for 80 pairs of SMs) that the library reserves in
 * device memory on every device that loads it, for as long as it is loaded.
 * It allocates nothing.
 *
 *   - The first call on a device looks the array's device address up
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call shares the one array and leaves its contents behind; nothing
 *     in it needs clearing between calls.  Calls that overlap on the GPU (on
 *     different streams, or from different threads) race on it: serialise
 *     them.
 *   - A device with more than 80 pairs of SMs needs a larger stream-K
 *     workspace than the array holds: such calls return GEMM_ERR_WORKSPACE
 *     (use gemm() with a workspace there).
 *   - fp32 inputs run on the CUDA-core FFMA kernel here, as gemm() without a
 *     workspace does: the 3xTF32 split needs a workspace that grows with M,
 *     N and K, which no fixed array can hold (about 8x slower at 4096^3).
 *   - Other errors as gemm().
 */
gemm_status_t gemm_builtin_scratch(int64_t M, int64_t N, int64_t K,
                                   gemm_dtype_t ab_dtype,
                                   const void *A, int64_t a_stride_m, int64_t a_stride_k,
                                   const void *B, int64_t b_stride_k, int64_t b_stride_n,
                                   void *C, int64_t ldc, gemm_dtype_t c_dtype,
                                   float alpha, float beta,
                                   const float *bias, gemm_epilogue_t epilogue,
                                   gemm_stream_t stream);

/*
 * gemm_bias_gelu -- the UNFUSED second pass, for measuring what fusion saves
 * (Rigel abstract: fused GEMM + bias + GELU against the decomposed path):
 * C[i][j] = cast(GELU(C[i][j] + bias[j])) in place, for an M x N block of an
 * M x ldc row-major buffer of type c_dtype (F32, F16 or BF16).  bias is fp32[N]
 * on the device.  Asynchronous on `stream`; same error behaviour as gemm().
 */
gemm_status_t gemm_bias_gelu(int64_t M, int64_t N, void *C, int64_t ldc, gemm_dtype_t c_dtype,
                             const float *bias, gemm_stream_t stream);

/*
 * Products with 4-bit group-quantized weights.  "X3: Metal GEMM" section 7
 * names quantized matmul -- a memory-bound GEMV when decoding, a GEMM when
 * filling the prompt -- as the main LLM workload; the pages give no storage
 * format, so this library takes the affine one with groups of 64 along K:
 *
 *     W[n][k] = s[n][k/64] * q[n][k] + b[n][k/64],   q[n][k] in 0..15,
 *
 * W being N x K (output features x input features).
 *   Wq          N*K/8 32-bit words, 16-byte aligned: q[n][k] is bits
 *               4*(k%8) .. 4*(k%8)+3 of word n*K/8 + k/8.
 *   scale_bias  N*K/64 pairs of binary16 values (s, b), in that order, one
 *               pair per group (n, g) at pair index n*K/64 + g; 4-byte aligned.
 */

/*
 * gemm_q4 -- C = cast(epilogue(alpha * x W^T + beta*C + bias)) for M rows of
 * x (M == 0 or N == 0 is a no-op).
 *   x_dtype     F16 or BF16.  X is M x ldx row-major, 16-byte aligned base,
 *               ldx >= K with ldx*2 a multiple of 16.
 *   K           a multiple of 64.
 *   C, c_dtype, ldc, alpha, beta, bias, epilogue: as in gemm(), with the
 *               output M x N and bias fp32[N]; the same fused epilogues.
 * Decode (1 <= M <= 8) runs an HBM-streaming kernel (gemm_q4_kernel_t below).
 * Prefill (M > 8) runs on the tensor cores with the dequantisation fused in:
 * each 64-k group of W is expanded to x's 16-bit type, round(s*q + b), straight
 * into tensor memory as the MMA's operand (never written to memory), and
 * multiplied with x in fp32 accumulation -- the rounding of W that
 * gemm_q4_dequantize followed by gemm() also has (at most 2^-11 of each |W|
 * for F16 x, 2^-8 for BF16).  Asynchronous on `stream`; errors as gemm().
 */
gemm_status_t gemm_q4(int64_t M, int64_t N, int64_t K, gemm_dtype_t x_dtype,
                      const void *X, int64_t ldx,
                      const uint32_t *Wq, const void *scale_bias,
                      void *C, int64_t ldc, gemm_dtype_t c_dtype,
                      float alpha, float beta,
                      const float *bias, gemm_epilogue_t epilogue,
                      gemm_stream_t stream);

/*
 * gemm_q4_ws -- gemm_q4 with a caller-owned workspace, for long prompts.  The
 * fused prefill converts each 64-k group of W once per 128 rows of x, so from
 * a few hundred rows of x up it is faster to expand W once into 16 bits and
 * run the dense tensor-core kernel (GB300, N = K = 4096: fused 31 / 33 / 60 /
 * 187 us at M = 64 / 256 / 1024 / 4096 against 35 / 35 / 37 / 93 us for
 * gemm_q4_dequantize + gemm()).  When gemm_q4_workspace_size(M, N, K,
 * x_dtype) is non-zero and the workspace (256-byte aligned device memory, not
 * overlapping any operand) holds that many bytes, the call does exactly
 * that: W into the workspace as x_dtype (the same rounding of W as the fused
 * kernel), then gemm() with the rest of the workspace for its partial sums.
 * Otherwise it runs gemm_q4.  Same arguments, results within the same
 * tolerances, and errors as gemm_q4; asynchronous on `stream`.
 */
gemm_status_t gemm_q4_ws(int64_t M, int64_t N, int64_t K, gemm_dtype_t x_dtype,
                         const void *X, int64_t ldx,
                         const uint32_t *Wq, const void *scale_bias,
                         void *C, int64_t ldc, gemm_dtype_t c_dtype,
                         float alpha, float beta,
                         const float *bias, gemm_epilogue_t epilogue,
                         void *workspace, size_t workspace_bytes,
                         gemm_stream_t stream);

/*
 * gemm_q4_workspace_size -- bytes of workspace gemm_q4_ws uses for this shape:
 * 0 below GEMM_Q4_DEQUANT_ROWS rows of x (the fused kernel is faster there) or
 * for an x_dtype other than F16 / BF16, else the 16-bit W (256-byte rounded)
 * plus gemm_workspace_size(M, N, K, x_dtype).  Pure function of its
 * arguments; touches no device.
 */
#define GEMM_Q4_DEQUANT_ROWS 384
size_t gemm_q4_workspace_size(int64_t M, int64_t N, int64_t K, gemm_dtype_t x_dtype);

/*
 * The kernel behind gemm_q4.  Both compute the same sums (per 64-k group,
 * s * sum_k x q + b * sum_k x, in fp32) and meet the same tolerances; they
 * differ in how the weights move and where the products are formed.
 */
typedef enum {
    GEMM_Q4_AUTO = 0,   /* the one measured faster for the number of rows of x */
    GEMM_Q4_FFMA = 1,   /* CUDA-core kernel: 16-byte loads into registers, codes to fp32, f32x2 multiply-add */
    GEMM_Q4_MMA = 2     /* tensor-core kernel: codes and x staged in shared memory by bulk copies, exact
                           16-bit codes times x by mma.sync.m16n8k16 (rows of x as the 8 columns) */
} gemm_q4_kernel_t;

/*
 * gemm_set_q4_kernel -- kernel of the calling thread's later gemm_q4() calls;
 * other threads keep their own setting.  Meant for tuning and tests.
 * GEMM_ERR_INVALID_ARG for an unknown value; never touches the device.
 */
gemm_status_t gemm_set_q4_kernel(gemm_q4_kernel_t kind);

/*
 * The calling thread's tuning settings, as the gemm_set_* calls left them
 * (every thread starts with all of them AUTO and bn 0).  No counterpart on
 * the pages.
 */
typedef struct {
    int tile_policy;    /* gemm_tile_policy_t */
    int tile_bn;        /* pair tile width forced with GEMM_TILE_PAIR, 0 = cost model */
    int schedule;       /* gemm_schedule_t */
    int operand_order;  /* gemm_operand_order_t */
    int multicast;      /* gemm_multicast_t */
    int q4_kernel;      /* gemm_q4_kernel_t */
} gemm_tuning_t;

/*
 * gemm_get_tuning -- copy the calling thread's settings into *out (host
 * pointer).  GEMM_ERR_INVALID_ARG for out == NULL; touches no device.
 */
gemm_status_t gemm_get_tuning(gemm_tuning_t *out);

/*
 * gemm_q4_dequantize -- W[n][k] = round(s*q + b) into the N x K row-major
 * device array W of type w_dtype (F16 or BF16; 16-byte aligned), for
 * gemm(M, N, K, w_dtype, X, ldx, 1, W, 1, K, ...) to multiply (W^T as B,
 * K-contiguous) -- the unfused alternative to gemm_q4's prefill, for a W
 * used by many calls.  The rounding to 16 bits is the only difference from the
 * exact product: at most 2^-11 (F16) or 2^-8 (BF16) of each |W| value.
 * K a multiple of 64.  Asynchronous on `stream`; errors as gemm().
 */
gemm_status_t gemm_q4_dequantize(int64_t N, int64_t K, const uint32_t *Wq, const void *scale_bias,
                                 void *W, gemm_dtype_t w_dtype, gemm_stream_t stream);

/*
 * Block-scaled ("microscaling", MX) products.  Rigel section 1 lists fp4 and
 * block-scaled MXFP4 next to fp8 among the low-precision rows of the matrix
 * units without defining them; the formats here are those of the OCP
 * Microscaling Formats (MX) specification v1.0.  Each block of 32 consecutive
 * k of a row shares one scale, an E8M0 code c standing for 2^(c - 127) (0xFF:
 * NaN), and each element is an E4M3 (MXFP8) or E2M1 (MXFP4) number:
 *
 *     a[i][k] = 2^(a_scale[i][k/32] - 127) * PA[i][k],  b[k][j] likewise with
 *     b_scale[j][k/32] and PB[j][k]
 *     C = cast(epilogue(alpha * sum_k a[i][k] b[k][j] + beta*C + bias))
 *
 * with gemm()'s epilogues, output types (F32, F16, BF16) and conventions.
 */
typedef enum {
    GEMM_MX_E4M3 = 0,   /* MXFP8: one E4M3 element per byte */
    GEMM_MX_E2M1 = 1    /* MXFP4: two E2M1 elements per byte, even k in the low nibble */
} gemm_mx_elem_t;

/*
 * gemm_mx -- the block-scaled product above on the tensor cores
 * (tcgen05.mma kind::mxf8f6f4 / kind::mxf4, scales applied by the MMA): up
 * to 128 rows of A one SM per 128 x 256 output tile, beyond that SM pairs
 * (cta_group::2) per 256 x 256 tile.
 *   K              a multiple of 32 (whole scale blocks); M, N, K >= 0.
 *   A, lda         M x K elements, row-major (K-contiguous), row pitch lda
 *                  ELEMENTS (lda >= K; even for E2M1).  16-byte aligned base,
 *                  row pitch a multiple of 16 bytes, else GEMM_ERR_MISALIGNED.
 *   a_scale        M x K/32 E8M0 codes, row-major (pitch K/32 bytes), device.
 *   B, ldb         B given as its transpose: N x K elements, K-contiguous, row
 *                  pitch ldb elements, same alignment rules.
 *   b_scale        N x K/32 E8M0 codes, row-major.
 *   C, ldc, c_dtype, alpha, beta, bias, epilogue: as in gemm() (c_dtype F32,
 *                  F16 or BF16; alpha == 0 or K == 0 reads neither operands
 *                  nor scales).
 *   workspace      device scratch, 256-byte aligned, of at least
 *                  gemm_mx_workspace_size() bytes (GEMM_ERR_WORKSPACE
 *                  otherwise): the scales rearranged for the tensor cores.
 *                  Calls sharing it must not overlap; no initialisation needed.
 * Asynchronous on `stream`; errors as gemm().
 */
gemm_status_t gemm_mx(int64_t M, int64_t N, int64_t K, gemm_mx_elem_t elem,
                      const void *A, int64_t lda, const uint8_t *a_scale,
                      const void *B, int64_t ldb, const uint8_t *b_scale,
                      void *C, int64_t ldc, gemm_dtype_t c_dtype,
                      float alpha, float beta,
                      const float *bias, gemm_epilogue_t epilogue,
                      void *workspace, size_t workspace_bytes,
                      gemm_stream_t stream);

/*
 * gemm_mx_workspace_size -- bytes of workspace gemm_mx needs: 512 bytes per
 * 128 rows of A and of B per 128 (E4M3) or 256 (E2M1) k, each half rounded up
 * to 256 bytes.  0 for invalid sizes (K not a multiple of 32).  Never fails,
 * touches no device.
 */
size_t gemm_mx_workspace_size(int64_t M, int64_t N, int64_t K, gemm_mx_elem_t elem);

/*
 * Baselines of the cheap-baseline gate (Rigel section 3; section 4, signal
 * 2): a claim that the tensor path is fast stands only once the trivial
 * explanations have run and lost -- a GEMM on the ordinary ALUs, and the
 * legacy warp-matrix instruction (simdgroup_matrix on the pages).  For
 * measurement and tests only; gemm() never runs them.
 */
typedef enum {
    GEMM_BASELINE_SIMT = 0,     /* threadgroup-tiled CUDA-core FFMA kernel (no matrix instructions) */
    GEMM_BASELINE_MMA_SYNC = 1  /* warp-level mma.sync.m16n8k16 kernel, fp16 / bf16 inputs */
} gemm_baseline_t;

/*
 * gemm_baseline -- the same operation and arguments as gemm() (no workspace),
 * computed by the baseline kernel `kind`.  GEMM_BASELINE_SIMT takes every
 * combination gemm() takes.  GEMM_BASELINE_MMA_SYNC takes F16 or BF16 inputs
 * whose operands are TMA-streamable in gemm()'s sense (one unit stride,
 * 16-byte aligned base and other stride) and whose contiguous extents (K for
 * a K-contiguous operand, M or N otherwise) are multiples of 8; anything else
 * returns GEMM_ERR_UNSUPPORTED.  K == 0, alpha == 0, M == 0 and N == 0
 * behave as in gemm().  Asynchronous on `stream`; errors as gemm().
 */
gemm_status_t gemm_baseline(gemm_baseline_t kind, int64_t M, int64_t N, int64_t K,
                            gemm_dtype_t ab_dtype,
                            const void *A, int64_t a_stride_m, int64_t a_stride_k,
                            const void *B, int64_t b_stride_k, int64_t b_stride_n,
                            void *C, int64_t ldc, gemm_dtype_t c_dtype,
                            float alpha, float beta,
                            const float *bias, gemm_epilogue_t epilogue,
                            gemm_stream_t stream);

/*
 * gemm_device_status -- synchronise `stream`, then return and clear the
 * device-side status word of the current device: GEMM_ERR_TIMEOUT if any
 * kernel gave up on a bounded wait since the last call, GEMM_ERR_CUDA if the
 * synchronisation itself failed, GEMM_OK otherwise.
 */
gemm_status_t gemm_device_status(gemm_stream_t stream);

/*
 * gemm_wait_selftest -- exercise the bounded waits the GEMM kernels rely on
 * instead of hanging.  Enqueues on `stream` a one-warp kernel that waits on an
 * mbarrier nobody arrives at and then on *never_set (a device word the caller
 * guarantees nobody sets to 0xFFFFFFFF during the call), each for at most
 * limit_ns nanoseconds (1 .. 1e9).  Each wait that gives up records a timeout,
 * so the next gemm_device_status() returns GEMM_ERR_TIMEOUT; the CUDA context
 * stays usable.  (Failure-detection aid; the pages have no counterpart.)
 */
gemm_status_t gemm_wait_selftest(const unsigned int *never_set, uint64_t limit_ns, gemm_stream_t stream);

/* gemm_status_string -- static, NUL-terminated description of a status code. */
const char *gemm_status_string(gemm_status_t status);

/* gemm_version -- static version string of the library build. */
const char *gemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_GB300_H */
