// gemm_tcgen05_e4m3.cu -- tcgen05 GEMM instantiations for e4m3 A/B operands.
// Tile widths: 256 (4-stage ring) and 128 (6-stage ring), both 192 KB of stages.
#include "gemm_tcgen05.cuh"

namespace gb300 {

cudaError_t launch_tcgen05_e4m3(int out, int bn, const CUtensorMap &ta, const CUtensorMap &tb, const TcArgs &args,
                                 int grid, cudaStream_t stream) {
    if (out == kDtBF16 && bn == 256) return launch_tcgen05_cfg<kDtE4M3, kDtBF16, 256, 4>(ta, tb, args, grid, stream);
    if (out == kDtBF16 && bn == 128) return launch_tcgen05_cfg<kDtE4M3, kDtBF16, 128, 6>(ta, tb, args, grid, stream);
    if (out == kDtF32 && bn == 256) return launch_tcgen05_cfg<kDtE4M3, kDtF32, 256, 4>(ta, tb, args, grid, stream);
    if (out == kDtF32 && bn == 128) return launch_tcgen05_cfg<kDtE4M3, kDtF32, 128, 6>(ta, tb, args, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gb300
