// gemm_simt.cu -- CUDA-core kernels:
//   * gemm_simt_kernel: register-blocked FFMA GEMM for fp32 inputs (IEEE fp32
//     fused multiply-add, k ascending per output) and the general fallback for
//     operand strides the TMA unit cannot take.  It is the threadgroup-tiled
//     kernel of "X3: Metal GEMM" section 2 grown to a 128x128 tile with an 8x8
//     register block per thread (the TM/TN register blocking of "Case Study:
//     Steel's BlockMMA"): stage a k-slice of A and B in shared memory with zero
//     fill outside the matrix, barrier, multiply from registers, barrier.
//   * epilogue_only_kernel: K == 0 or alpha == 0 (C = epilogue(beta*C + bias)).
//   * bias_gelu_kernel: the unfused bias+GELU pass over a finished GEMM output,
//     used only to measure what fusing saves (Rigel, abstract and section 1).
//   * wait_selftest_kernel: runs the bounded waits of the GEMM kernels against
//     events that never happen, so tests can see them give up and report.
#include "epilogue.cuh"
#include "kernel_args.h"
#include "sm103_ptx.cuh"

namespace gb300 {

namespace {

constexpr int kSimtBM = 128, kSimtBN = 128, kSimtBK = 8, kSimtThreads = 256;

template <int AB, int OUT>
__global__ void __launch_bounds__(kSimtThreads) gemm_simt_kernel(const SimtArgs a) {
    using InT = typename Elem<AB>::T;
    using OutT = typename Elem<OUT>::T;
    __shared__ float As[kSimtBK][kSimtBM + 4];
    __shared__ float Bs[kSimtBK][kSimtBN + 4];

    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const int m0 = blockIdx.y * kSimtBM, n0 = blockIdx.x * kSimtBN;
    const int M = a.e.M, N = a.e.N, K = a.K;
    const InT *A = static_cast<const InT *>(a.A);
    const InT *B = static_cast<const InT *>(a.B);
    // Walk the contiguous dimension with consecutive threads where there is one.
    const bool a_k_contig = (a.sak == 1);
    const bool b_n_contig = (a.sbn == 1);

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

    for (int k0 = 0; k0 < K; k0 += kSimtBK) {
#pragma unroll
        for (int r = 0; r < (kSimtBM * kSimtBK) / kSimtThreads; ++r) {
            const int e = tid + r * kSimtThreads;
            const int m = a_k_contig ? e / kSimtBK : e % kSimtBM;
            const int k = a_k_contig ? e % kSimtBK : e / kSimtBM;
            const int gm = m0 + m, gk = k0 + k;
            As[k][m] = (gm < M && gk < K) ? Elem<AB>::load(A + (long long)gm * a.sam + (long long)gk * a.sak) : 0.0f;
        }
#pragma unroll
        for (int r = 0; r < (kSimtBN * kSimtBK) / kSimtThreads; ++r) {
            const int e = tid + r * kSimtThreads;
            const int n = b_n_contig ? e % kSimtBN : e / kSimtBK;
            const int k = b_n_contig ? e / kSimtBN : e % kSimtBK;
            const int gn = n0 + n, gk = k0 + k;
            Bs[k][n] = (gn < N && gk < K) ? Elem<AB>::load(B + (long long)gk * a.sbk + (long long)gn * a.sbn) : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kSimtBK; ++k) {
            float av[8], bv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) av[i] = As[k][ty + 16 * i];
#pragma unroll
            for (int j = 0; j < 8; ++j) bv[j] = Bs[k][tx + 16 * j];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }

    OutT *C = static_cast<OutT *>(a.e.C);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = m0 + ty + 16 * i;
        if (row >= M) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int col = n0 + tx + 16 * j;
            if (col < N) {
                const float b = (a.e.epilogue != kEpiNone) ? a.e.bias[col] : 0.0f;
                const OutT *r = a.e.residual ? residual_row<OUT>(a.e, row) + col : nullptr;
                const float y = epilogue_store_one<OUT>(acc[i][j] * product_scale(a.e, row, col),
                                                        C + (long long)row * a.e.ldc + col, b, a.e, r);
                amax = fmaxf(amax, fabsf(y));
            }
        }
    }
    if (a.e.amax) amax_push(amax, a.e.amax);
}

template <int OUT>
__global__ void epilogue_only_kernel(const EpiParams e) {
    using OutT = typename Elem<OUT>::T;
    OutT *C = static_cast<OutT *>(e.C);
    const long long total = (long long)e.M * e.N;
    float amax = 0.0f;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long i = idx / e.N, j = idx - i * e.N;
        const float b = (e.epilogue != kEpiNone) ? e.bias[j] : 0.0f;
        const OutT *r = e.residual ? residual_row<OUT>(e, static_cast<int>(i)) + j : nullptr;
        amax = fmaxf(amax, fabsf(epilogue_store_one<OUT>(0.0f, C + i * e.ldc + j, b, e, r)));
    }
    if (e.amax) amax_push(amax, e.amax);
}

template <int OUT>
__global__ void bias_gelu_kernel(const EpiParams e) {
    using OutT = typename Elem<OUT>::T;
    OutT *C = static_cast<OutT *>(e.C);
    const long long total = (long long)e.M * e.N;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long i = idx / e.N, j = idx - i * e.N;
        OutT *p = C + i * e.ldc + j;
        *p = Elem<OUT>::cvt(activate_one<OUT>(Elem<OUT>::load(p) + e.bias[j], kEpiBiasGelu, false));
    }
}

// One warp: lane 0 waits on an mbarrier that nobody arrives at, then on a
// global flag that nobody sets, each for at most limit_ns; each wait that gives
// up records a timeout in the status word.  Returns in about 2 * limit_ns.
__global__ void wait_selftest_kernel(const unsigned int *never_set, unsigned long long limit_ns,
                                     unsigned int *status) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        volatile int *ab = &abort_flag;
        mbar_wait_bounded(&bar, 0, ab, status, limit_ns);
        *ab = 0;
        flag_wait_bounded(never_set, 0xFFFFFFFFu, ab, status, limit_ns);
    }
}

int elementwise_grid(long long total, int threads) {
    long long blocks = (total + threads - 1) / threads;
    const long long cap = 152LL * 16;  // a few waves over the SMs; the loops are grid-stride
    if (blocks > cap) blocks = cap;
    return static_cast<int>(blocks < 1 ? 1 : blocks);
}

template <int AB, int OUT>
cudaError_t launch_simt_t(const SimtArgs &a, cudaStream_t s) {
    dim3 grid((a.e.N + kSimtBN - 1) / kSimtBN, (a.e.M + kSimtBM - 1) / kSimtBM);
    gemm_simt_kernel<AB, OUT><<<grid, kSimtThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt(int ab, int out, const SimtArgs &a, cudaStream_t s) {
    if ((a.e.N + kSimtBN - 1) / kSimtBN > 2147483647 || (a.e.M + kSimtBM - 1) / kSimtBM > 65535)
        return cudaErrorInvalidConfiguration;
    switch (ab * 4 + out) {
    case kDtF32 * 4 + kDtF32: return launch_simt_t<kDtF32, kDtF32>(a, s);
    case kDtF16 * 4 + kDtF16: return launch_simt_t<kDtF16, kDtF16>(a, s);
    case kDtF16 * 4 + kDtF32: return launch_simt_t<kDtF16, kDtF32>(a, s);
    case kDtF16 * 4 + kDtBF16: return launch_simt_t<kDtF16, kDtBF16>(a, s);
    case kDtBF16 * 4 + kDtBF16: return launch_simt_t<kDtBF16, kDtBF16>(a, s);
    case kDtBF16 * 4 + kDtF32: return launch_simt_t<kDtBF16, kDtF32>(a, s);
    case kDtBF16 * 4 + kDtF16: return launch_simt_t<kDtBF16, kDtF16>(a, s);
    case kDtE4M3 * 4 + kDtBF16: return launch_simt_t<kDtE4M3, kDtBF16>(a, s);
    case kDtE4M3 * 4 + kDtF32: return launch_simt_t<kDtE4M3, kDtF32>(a, s);
    case kDtF16 * 4 + kDtE4M3: return launch_simt_t<kDtF16, kDtE4M3>(a, s);
    case kDtBF16 * 4 + kDtE4M3: return launch_simt_t<kDtBF16, kDtE4M3>(a, s);
    case kDtE4M3 * 4 + kDtE4M3: return launch_simt_t<kDtE4M3, kDtE4M3>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_epilogue_only(int out, const EpiParams &e, cudaStream_t s) {
    const int threads = 256;
    const int grid = elementwise_grid((long long)e.M * e.N, threads);
    switch (out) {
    case kDtF32: epilogue_only_kernel<kDtF32><<<grid, threads, 0, s>>>(e); break;
    case kDtF16: epilogue_only_kernel<kDtF16><<<grid, threads, 0, s>>>(e); break;
    case kDtBF16: epilogue_only_kernel<kDtBF16><<<grid, threads, 0, s>>>(e); break;
    case kDtE4M3: epilogue_only_kernel<kDtE4M3><<<grid, threads, 0, s>>>(e); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(const unsigned int *never_set, unsigned long long limit_ns, unsigned int *status,
                                 cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(never_set, limit_ns, status);
    return cudaGetLastError();
}

cudaError_t launch_bias_gelu(int out, const EpiParams &e, cudaStream_t s) {
    const int threads = 256;
    const int grid = elementwise_grid((long long)e.M * e.N, threads);
    switch (out) {
    case kDtF32: bias_gelu_kernel<kDtF32><<<grid, threads, 0, s>>>(e); break;
    case kDtF16: bias_gelu_kernel<kDtF16><<<grid, threads, 0, s>>>(e); break;
    case kDtBF16: bias_gelu_kernel<kDtBF16><<<grid, threads, 0, s>>>(e); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace gb300
