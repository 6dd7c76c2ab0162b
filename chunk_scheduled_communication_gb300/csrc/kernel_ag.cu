// kernel_ag.cu -- instantiations of the fused chunk-scheduled kernel for
// the AG-GEMM operator (128x256 and 128x128 tiles).
#include "fused.cuh"

namespace syn {

cudaError_t launch_fused_ag(const KernelParams &p, const TensorMaps &tm, int tile_n, int grid,
                            cudaStream_t st) {
    if (tile_n == 256) return launch_fused_t<OP_AG, 256>(p, tm, grid, st);
    if (tile_n == 128) return launch_fused_t<OP_AG, 128>(p, tm, grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace syn

namespace syn {

int fused_smem_bytes(int op, int tile_n) {
    if (op == OP_AG) return tile_n == 256 ? KCfg<OP_AG, 256>::SMEM_ALLOC : KCfg<OP_AG, 128>::SMEM_ALLOC;
    if (op == OP_RS) return tile_n == 256 ? KCfg<OP_RS, 256>::SMEM_ALLOC : KCfg<OP_RS, 128>::SMEM_ALLOC;
    return tile_n == 256 ? KCfg<OP_AR, 256>::SMEM_ALLOC : KCfg<OP_AR, 128>::SMEM_ALLOC;
}

}  // namespace syn
