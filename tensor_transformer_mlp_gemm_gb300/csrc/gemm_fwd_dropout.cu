// gemm_fwd_dropout.cu -- the row-parallel GEMM of the sequence-parallel
// sublayer: Out = X + Dropout(sum_i H_i.B_i + b2), the dropout mask drawn in
// the epilogue from Philox4x32-10 and the residual X read per token chunk
// ("Megatron-LM：NVIDIA 的大规模并行训练方案", 并行训练范式 / 序列并行: Dropout
// along the sequence dimension).
#include "gemm.cuh"

namespace tpmlp {
TPMLP_GEMM_LAUNCHER(launch_row_fwd_dropout, false, true, EPI_BIAS_DROP_RES)
}  // namespace tpmlp
