// gemm_tcgen05_f16.cu -- tcgen05 GEMM instantiations for f16 A/B operands.
// Tile widths: 256 (4-stage ring) and 128 (6-stage ring), both 192 KB of stages.
#include "gemm_tcgen05.cuh"

namespace gb300 {

cudaError_t launch_tcgen05_f16(int out, int bn, const CUtensorMap &ta, const CUtensorMap &tb, const TcArgs &args,
                                 int grid, cudaStream_t stream) {
    if (out == kDtF16 && bn == 256) return launch_tcgen05_cfg<kDtF16, kDtF16, 256, 4>(ta, tb, args, grid, stream);
    if (out == kDtF16 && bn == 128) return launch_tcgen05_cfg<kDtF16, kDtF16, 128, 6>(ta, tb, args, grid, stream);
    if (out == kDtF32 && bn == 256) return launch_tcgen05_cfg<kDtF16, kDtF32, 256, 4>(ta, tb, args, grid, stream);
    if (out == kDtF32 && bn == 128) return launch_tcgen05_cfg<kDtF16, kDtF32, 128, 6>(ta, tb, args, grid, stream);
    if (out == kDtBF16 && bn == 256) return launch_tcgen05_cfg<kDtF16, kDtBF16, 256, 4>(ta, tb, args, grid, stream);
    if (out == kDtBF16 && bn == 128) return launch_tcgen05_cfg<kDtF16, kDtBF16, 128, 6>(ta, tb, args, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gb300
