// gemm_dgrad.cu -- backward data-gradient GEMM variants (chain rule of the
// column-then-row MLP of "Megatron-LM：NVIDIA 的大规模并行训练方案", 张量并行原理).
//   dgrad_h: dY_i = (dZ.B_i^T) * GeLU'(Y_i), the GeLU derivative fused in the epilogue.
//   dgrad_x: dX = sum_i dY_i.A_i^T, shards summed as split-K in TMEM (the
//            backward counterpart of the row-parallel AllReduce).
#include "gemm.cuh"

namespace tpmlp {
TPMLP_GEMM_LAUNCHER(launch_dgrad_h, false, false, EPI_DGELU)
// Selective recompute: the same GEMM also rebuilds H_i = GeLU(Y_i) from the
// saved pre-activation it already reads, so the forward pass need not keep H.
TPMLP_GEMM_LAUNCHER(launch_dgrad_h_recompute, false, false, EPI_DGELU_H)
TPMLP_GEMM_LAUNCHER(launch_dgrad_x, false, false, EPI_BF16)
}  // namespace tpmlp
