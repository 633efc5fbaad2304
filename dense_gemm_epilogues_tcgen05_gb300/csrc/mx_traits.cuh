// mx_traits.cuh -- what the two block-scaled kernels (gemm_mx.cu, one SM per
// tile; gemm_mx_pair.cu, SM pairs) share about the element types: scale
// chunks per 128-byte k-block, MMA kind, and the instruction descriptor's
// element format.
#pragma once
#include "kernel_args.h"
#include "sm103_ptx.cuh"

namespace gb300 {

template <int ELEM> struct MxTraits;
template <> struct MxTraits<kMxE4M3> {
    static constexpr int kChunks = 1;          // 128 bytes of K = 128 elements = 4 blocks = one chunk
    static constexpr int kKind = kKindMxf8f6f4;
    static constexpr uint32_t kFmt = 0;        // E4M3
};
template <> struct MxTraits<kMxE2M1> {
    static constexpr int kChunks = 2;          // 128 bytes of K = 256 elements = 8 blocks = two chunks
    static constexpr int kKind = kKindMxf4;
    static constexpr uint32_t kFmt = 1;        // E2M1 (kind::mxf4)
};

}  // namespace gb300
