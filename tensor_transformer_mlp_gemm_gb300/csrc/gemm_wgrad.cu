// gemm_wgrad.cu -- weight-gradient GEMMs dA_i = X^T.dY_i and dB_i = H_i^T.dZ.
// Both contract over tokens, so both operands are read MN-major directly from
// the token-major activations (no transposed copies); fp32 results.
#include "gemm.cuh"

namespace tpmlp {
TPMLP_GEMM_LAUNCHER(launch_wgrad, true, true, EPI_F32)
}  // namespace tpmlp
