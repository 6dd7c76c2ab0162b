// kernel_rs.cu -- instantiations of the fused chunk-scheduled kernel for
// the GEMM-RS operator (128x256 and 128x128 tiles).
#include "fused.cuh"

namespace syn {

cudaError_t launch_fused_rs(const KernelParams &p, const TensorMaps &tm, int tile_n, int grid,
                            cudaStream_t st) {
    if (tile_n == 256) return launch_fused_t<OP_RS, 256>(p, tm, grid, st);
    if (tile_n == 128) return launch_fused_t<OP_RS, 128>(p, tm, grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace syn
