// kernel_rs.cu -- compiled instances of the fused chunk-scheduled kernel
// for the GEMM-RS operator (every tile shape / pipeline depth / staging-buffer
// combination that dispatch_cfg lists, single CTA and CTA pair).
#include "fused.cuh"

namespace syn {

cudaError_t launch_fused_rs(const KernelParams &p, const TensorMaps &tm, const LaunchCfg &lc,
                            cudaStream_t st) {
    return launch_op<OP_RS>(p, tm, lc, st);
}

int smem_bytes_rs(const LaunchCfg &lc) { return smem_bytes_op<OP_RS>(lc); }

int max_clusters_rs(const LaunchCfg &lc) { return max_clusters_op<OP_RS>(lc); }

int epi_tma_rs(const LaunchCfg &lc) { return epi_tma_op<OP_RS>(lc); }

}  // namespace syn
