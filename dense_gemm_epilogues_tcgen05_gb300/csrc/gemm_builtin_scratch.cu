// gemm_builtin_scratch.cu -- gemm() for callers that cannot allocate device
// memory.
//
// The stream-K schedule of the pair kernel needs scratch memory for partial
// sums and ready flags, which gemm() takes from a caller-allocated workspace.
// Some callers cannot call cudaMalloc (or any allocating library routine) at
// the point where they multiply: code running inside CUDA stream capture,
// real-time paths where allocation latency is not allowed, or processes whose
// device memory is owned by another allocator.  gemm_builtin_scratch gives
// them the same computation with the scratch taken from a fixed array that
// this file reserves in device memory (static storage of the library module).
// It allocates nothing.
//
// The array lives as long as the library is loaded, on every device that
// loads this module; it is sized for up to kBuiltinMaxPairs pairs of SMs.
#include <cuda_runtime_api.h>

#include <cstdint>
#include <mutex>

#include "../../include/gemm_gb300.h"
#include "kernel_args.h"

namespace {

constexpr int kBuiltinMaxPairs = 80;
// Partial sums (2 CTAs x 128 x 256 fp32 per pair) and ready flags (16 words
// per pair, rounded up to 256 bytes): the stream-K workspace of 80 pairs.
constexpr size_t kBuiltinScratchBytes =
    static_cast<size_t>(kBuiltinMaxPairs) * 2 * gb300::kPartialFloatsPerCta * 4 +
    ((static_cast<size_t>(kBuiltinMaxPairs) * gb300::kFlagsPerCluster * 4 + 255) / 256) * 256;

}  // namespace

// Zero at module load; afterwards every call leaves its last contents.  The
// kernels never need it cleared: a flag counts as set only when it holds the
// current call's epoch, and each call resets the flags it consumed.
static __device__ __align__(256) unsigned char g_builtin_scratch[kBuiltinScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices];  // device address of g_builtin_scratch, per device

// Device address of the array on the current device; looked up once per device.
gemm_status_t builtin_scratch(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_builtin_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return GEMM_OK;
}

}  // namespace

extern "C" {

gemm_status_t gemm_builtin_scratch(int64_t M, int64_t N, int64_t K, gemm_dtype_t ab_dtype, const void *A,
                                   int64_t a_stride_m, int64_t a_stride_k, const void *B, int64_t b_stride_k,
                                   int64_t b_stride_n, void *C, int64_t ldc, gemm_dtype_t c_dtype, float alpha,
                                   float beta, const float *bias, gemm_epilogue_t epilogue, gemm_stream_t stream) {
    gemm_path_t path;
    gemm_status_t st = gemm_query_path(M, N, K, ab_dtype, A, a_stride_m, a_stride_k, B, b_stride_k, b_stride_n, C,
                                       ldc, c_dtype, alpha, beta, bias, epilogue, &path);
    if (st != GEMM_OK) return st;
    if (path != GEMM_PATH_TCGEN05)  // the other kernels use no scratch
        return gemm(M, N, K, ab_dtype, A, a_stride_m, a_stride_k, B, b_stride_k, b_stride_n, C, ldc, c_dtype,
                    alpha, beta, bias, epilogue, nullptr, 0, stream);
    void *scratch = nullptr;
    if ((st = builtin_scratch(&scratch)) != GEMM_OK) return st;
    // The stream-K workspace grows with the number of SM pairs of the device.
    if (gemm_workspace_size(M, N, K, ab_dtype) > kBuiltinScratchBytes) return GEMM_ERR_WORKSPACE;
    return gemm(M, N, K, ab_dtype, A, a_stride_m, a_stride_k, B, b_stride_k, b_stride_n, C, ldc, c_dtype, alpha,
                beta, bias, epilogue, scratch, kBuiltinScratchBytes, stream);
}

}  // extern "C"
