// gemm_tcgen05_bf16.cu -- tcgen05 GEMM instantiations for bf16 A/B operands.
// One-SM kernel: tile widths 256 (4-stage ring) and 128 (6-stage ring).
// Pair kernel: 256 x BN tiles on two SMs, 6-stage ring of 32 KB per CTA; clusters
// of one pair or of two pairs sharing A by multicast (cl = 2 or 4 CTAs).
#include "gemm_tcgen05.cuh"
#include "gemm_tcgen05_pair.cuh"

namespace gb300 {

cudaError_t launch_tcgen05_bf16(int out, int bn, const CUtensorMap &ta, const CUtensorMap &tb, const TcArgs &args,
                                 int grid, cudaStream_t stream) {
    if (out == kDtBF16 && bn == 256) return launch_tcgen05_cfg<kDtBF16, kDtBF16, 256, 4>(ta, tb, args, grid, stream);
    if (out == kDtBF16 && bn == 128) return launch_tcgen05_cfg<kDtBF16, kDtBF16, 128, 6>(ta, tb, args, grid, stream);
    if (out == kDtF32 && bn == 256) return launch_tcgen05_cfg<kDtBF16, kDtF32, 256, 4>(ta, tb, args, grid, stream);
    if (out == kDtF32 && bn == 128) return launch_tcgen05_cfg<kDtBF16, kDtF32, 128, 6>(ta, tb, args, grid, stream);
    if (out == kDtF16 && bn == 256) return launch_tcgen05_cfg<kDtBF16, kDtF16, 256, 4>(ta, tb, args, grid, stream);
    if (out == kDtF16 && bn == 128) return launch_tcgen05_cfg<kDtBF16, kDtF16, 128, 6>(ta, tb, args, grid, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_pair_bf16(int out, int cl, const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc, const TcArgs &args,
                              int clusters, cudaStream_t stream) {
    if (cl == 4) {
        if (out == kDtBF16) return launch_pair_cfg<kDtBF16, kDtBF16, 6, 128, 4>(ta, tb, tc, args, clusters, stream);
        if (out == kDtF32) return launch_pair_cfg<kDtBF16, kDtF32, 6, 128, 4>(ta, tb, tc, args, clusters, stream);
        if (out == kDtF16) return launch_pair_cfg<kDtBF16, kDtF16, 6, 128, 4>(ta, tb, tc, args, clusters, stream);
        if (out == kDtE4M3) return launch_pair_cfg<kDtBF16, kDtE4M3, 6, 128, 4>(ta, tb, tc, args, clusters, stream);
        return cudaErrorInvalidValue;
    }
    if (out == kDtBF16) return launch_pair_cfg<kDtBF16, kDtBF16, 6>(ta, tb, tc, args, clusters, stream);
    if (out == kDtF32) return launch_pair_cfg<kDtBF16, kDtF32, 6>(ta, tb, tc, args, clusters, stream);
    if (out == kDtF16) return launch_pair_cfg<kDtBF16, kDtF16, 6>(ta, tb, tc, args, clusters, stream);
    if (out == kDtE4M3) return launch_pair_cfg<kDtBF16, kDtE4M3, 6>(ta, tb, tc, args, clusters, stream);
    return cudaErrorInvalidValue;
}

int pair_max_clusters_bf16(int out, int cl) {
    if (cl == 4) {
        if (out == kDtBF16) return pair_max_clusters<kDtBF16, kDtBF16, 6, 128, 4>();
        if (out == kDtF32) return pair_max_clusters<kDtBF16, kDtF32, 6, 128, 4>();
        if (out == kDtF16) return pair_max_clusters<kDtBF16, kDtF16, 6, 128, 4>();
        if (out == kDtE4M3) return pair_max_clusters<kDtBF16, kDtE4M3, 6, 128, 4>();
        return 0;
    }
    if (out == kDtBF16) return pair_max_clusters<kDtBF16, kDtBF16, 6>();
    if (out == kDtF32) return pair_max_clusters<kDtBF16, kDtF32, 6>();
    if (out == kDtF16) return pair_max_clusters<kDtBF16, kDtF16, 6>();
    if (out == kDtE4M3) return pair_max_clusters<kDtBF16, kDtE4M3, 6>();
    return 0;
}

}  // namespace gb300
