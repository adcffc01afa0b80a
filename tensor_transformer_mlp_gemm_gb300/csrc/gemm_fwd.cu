// gemm_fwd.cu -- forward-pass GEMM variants.
//   column_fwd: Y_i = X.A_i + b1_i and H_i = GeLU(Y_i) in one epilogue
//               ("Megatron-LM：NVIDIA 的大规模并行训练方案", 张量并行原理 column
//               split; 融合优化技术 Bias + GeLU fusion).
//   row_fwd:    Z = sum_i H_i.B_i + b2, shards summed as split-K in TMEM
//               (same page, 张量并行原理 row split).
#include "gemm.cuh"

namespace tpmlp {
TPMLP_GEMM_LAUNCHER(launch_column_fwd, false, true, EPI_BIAS_GELU)
TPMLP_GEMM_LAUNCHER(launch_row_fwd, false, true, EPI_BIAS)
}  // namespace tpmlp
