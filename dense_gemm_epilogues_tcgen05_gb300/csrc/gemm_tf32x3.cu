// gemm_tf32x3.cu -- fp32 inputs on the tensor cores (3xTF32).
//
// An fp32 value splits into x = hi + lo with hi = tf32(x) (10 explicit
// fraction bits, round to nearest) and lo = x - hi, exact in fp32 because hi
// and x share their leading bits.  Then
//     A*B = A_hi*B_hi + A_hi*B_lo + A_lo*B_hi + A_lo*B_lo,
// and the last product (relative size 2^-22) is dropped; the tensor core rounds
// lo to tf32 once more (relative 2^-11 of lo), so each product keeps ~2^-21
// relative accuracy, well inside the 1e-5 bound of fp32 outputs where plain
// TF32 (~2^-11 per product) is not.  The pair kernel runs the three products
// as three tcgen05.mma kind::tf32 per k-step into one fp32 accumulator, small
// terms first.
//
// tf32_split_kernel is the pre-pass: it reads an operand through any strides
// (32 x 32 tiles staged in shared memory, coalesced along whichever dimension
// is contiguous) and writes hi then lo as one stacked K-major array
// [rows x pitch | rows x pitch] into the caller's workspace.
#include "gemm_tcgen05.cuh"
#include "gemm_tcgen05_pair.cuh"

namespace gb300 {

namespace {

__device__ __forceinline__ float tf32_round(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

__global__ void tf32_split_kernel(const float *__restrict__ src, long long rows, long long cols, long long s_row,
                                  long long s_col, float *__restrict__ dst, long long pitch) {
    __shared__ float tile[32][33];
    const bool col_contig = (s_col == 1) || (s_row != 1);  // read along the contiguous dimension
    const long long lo_off = rows * pitch;
    for (long long r0 = static_cast<long long>(blockIdx.y) * 32; r0 < rows; r0 += 32LL * gridDim.y) {
        for (long long c0 = static_cast<long long>(blockIdx.x) * 32; c0 < cols; c0 += 32LL * gridDim.x) {
            for (int i = threadIdx.y; i < 32; i += blockDim.y) {
                const int tr = col_contig ? i : threadIdx.x;
                const int tc = col_contig ? threadIdx.x : i;
                const long long r = r0 + tr, c = c0 + tc;
                tile[tr][tc] = (r < rows && c < cols) ? src[r * s_row + c * s_col] : 0.0f;
            }
            __syncthreads();
            for (int i = threadIdx.y; i < 32; i += blockDim.y) {
                const long long r = r0 + i, c = c0 + threadIdx.x;
                if (r < rows && c < cols) {
                    const float x = tile[i][threadIdx.x];
                    const float hi = tf32_round(x);
                    dst[r * pitch + c] = hi;
                    dst[lo_off + r * pitch + c] = x - hi;
                }
            }
            __syncthreads();
        }
    }
}

}  // namespace

cudaError_t launch_tf32_split(const float *src, long long rows, long long cols, long long s_row, long long s_col,
                              float *dst, long long pitch, cudaStream_t stream) {
    long long gx = (cols + 31) / 32, gy = (rows + 31) / 32;
    if (gx > 4096) gx = 4096;
    if (gy > 4096) gy = 4096;
    tf32_split_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), dim3(32, 8), 0, stream>>>(
        src, rows, cols, s_row, s_col, dst, pitch);
    return cudaGetLastError();
}

cudaError_t launch_pair_tf32x3(int out, const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc, const TcArgs &args,
                               int clusters, cudaStream_t stream) {
    if (out == kDtF32) return launch_pair_cfg<kDtTF32x3, kDtF32, 3>(ta, tb, tc, args, clusters, stream);
    return cudaErrorInvalidValue;
}

int pair_max_clusters_tf32x3(int out) {
    if (out == kDtF32) return pair_max_clusters<kDtTF32x3, kDtF32, 3>();
    return 0;
}

}  // namespace gb300
