// kernel_ag.cu -- compiled instances of the fused chunk-scheduled kernel
// for the AG-GEMM operator (every tile shape / pipeline depth / staging-buffer
// combination that dispatch_cfg lists, single CTA and CTA pair).
#include "fused.cuh"

namespace syn {

cudaError_t launch_fused_ag(const KernelParams &p, const TensorMaps &tm, const LaunchCfg &lc,
                            cudaStream_t st) {
    return launch_op<OP_AG>(p, tm, lc, st);
}

int smem_bytes_ag(const LaunchCfg &lc) { return smem_bytes_op<OP_AG>(lc); }

int max_clusters_ag(const LaunchCfg &lc) { return max_clusters_op<OP_AG>(lc); }

}  // namespace syn

namespace syn {

int smem_bytes_rs(const LaunchCfg &lc);
int smem_bytes_ar(const LaunchCfg &lc);
int max_clusters_rs(const LaunchCfg &lc);
int max_clusters_ar(const LaunchCfg &lc);

int fused_smem_bytes(int op, const LaunchCfg &lc) {
    if (op == OP_AG) return smem_bytes_ag(lc);
    if (op == OP_RS) return smem_bytes_rs(lc);
    return smem_bytes_ar(lc);
}

int fused_max_clusters(int op, const LaunchCfg &lc) {
    if (op == OP_AG) return max_clusters_ag(lc);
    if (op == OP_RS) return max_clusters_rs(lc);
    return max_clusters_ar(lc);
}

}  // namespace syn
