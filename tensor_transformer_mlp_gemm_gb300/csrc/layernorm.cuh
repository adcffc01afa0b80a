// layernorm.cuh -- the elementwise and row-reduction kernels of the
// sequence-parallel sublayer Out = X + Dropout(MLP(LN(X))), each run per token
// chunk ("Megatron-LM：NVIDIA 的大规模并行训练方案", 并行训练范式 / 序列并行).
//   ln_forward:       Xn = (X - mean) * rstd * gamma + beta per token row, with
//                     mean and rstd = 1 / sqrt(var + eps) (biased variance)
//                     kept for the backward pass
//   dropout_backward: dZ = keep ? dOut / (1 - p) : 0 (the keep bits the
//                     forward pass stored) and the column sums of dZ (db2)
//   ln_backward:      dX = rstd * (g - mean(g) - xhat * mean(g * xhat)) + dOut,
//                     g = dXn * gamma, dgamma = sum dXn * xhat and dbeta =
//                     sum dXn.  Rows of at most 4096 elements: one pass over
//                     blocks of token rows gives dX and per-block partial
//                     sums; wider rows: one CTA per token row for dX, then
//                     the column sums over row splits.  Either way the
//                     partials are added in a fixed order (no atomics anywhere).
// All three are bound by HBM traffic.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

#include "philox.cuh"

namespace tpmlp {

constexpr int LN_THREADS = 256;
constexpr int LN_MAX_VEC = 8;                          // 8-element vectors per thread
constexpr int LN_MAX_H = LN_THREADS * LN_MAX_VEC * 8;  // 16384
constexpr int LN_WARP_MAX_H = 32 * 16 * 8;             // rows the one-warp forward kernel takes
constexpr int LN_MAX_CHUNKS = 8;

struct LnChunks {
    const void* in[LN_MAX_CHUNKS];
    int n;           // chunks (the kernels find a row's chunk as row / rows)
    long long rows;  // rows per chunk
};

struct LnForwardParams {
    LnChunks x;                  // bf16 [rows, h] per chunk
    void* y[LN_MAX_CHUNKS];      // bf16 Xn, same chunking
    const void* gamma;           // bf16 [h]
    const void* beta;            // bf16 [h]
    float* mean;                 // fp32 [T]
    float* rstd;                 // fp32 [T]
    int h;
    float eps;
};

struct DropoutBackwardParams {
    LnChunks dout;               // bf16 [rows, h] per chunk
    void* dz[LN_MAX_CHUNKS];     // bf16, same chunking
    int h;
    DropoutParams drop;          // drop.mask: the keep bits the forward pass stored
    float* part;                 // fp32 [splits][h] partial column sums of dZ
    int splits;                  // row splits
    long long rows_per_split;
};

// Row splits of the dropout backward pass (which also sums dZ's columns):
// enough 64-column CTAs to cover the GPU about sixteen times, at least 128
// rows per split, at most LN_MAX_SPLITS.
int dropout_splits(long long T, long long h, int sm_count);

struct LnBackwardParams {
    LnChunks x;                  // bf16 X (the sublayer input)
    const void* dxn[LN_MAX_CHUNKS];   // bf16 gradient of Xn, same chunking
    const void* dres[LN_MAX_CHUNKS];  // bf16 gradient through the residual path (dOut)
    void* dx[LN_MAX_CHUNKS];          // bf16 output
    const void* gamma;           // bf16 [h]
    const float* mean;
    const float* rstd;
    float* part;                 // fp32 [splits][2][h] partial dgamma, dbeta
    int h;
    long long rows_per_block;    // rows per split of the dgamma / dbeta pass
};

constexpr int LN_MAX_SPLITS = 64;
constexpr int LN_FUSED_MAX_BLOCKS = 512;

// Rows of at most LN_WARP_MAX_H elements take the fused LayerNorm backward:
// dX and the dgamma / dbeta partial sums in one pass over row blocks.
inline bool ln_backward_fused(long long h) { return h <= LN_WARP_MAX_H; }

// Bytes of partial sums the dgamma / dbeta sums need.
inline size_t ln_partial_bytes(long long h) {
    const size_t splits = ln_backward_fused(h) ? LN_FUSED_MAX_BLOCKS : LN_MAX_SPLITS;
    return splits * 2 * static_cast<size_t>(h) * sizeof(float);
}
// Row splits of the dgamma / dbeta sums.  Fused pass: one block of rows per
// CTA, two CTAs per SM.  Separate pass: enough 64-column CTAs to cover the
// GPU about sixteen times (many short CTAs, so the last to start ends soon
// after the rest), at least 128 rows per split.
inline int ln_param_splits(long long T, long long h, int sm_count) {
    if (ln_backward_fused(h)) {
        long long b = 2LL * sm_count;
        if (b > LN_FUSED_MAX_BLOCKS) b = LN_FUSED_MAX_BLOCKS;
        if (b > T) b = T;
        return static_cast<int>(b < 1 ? 1 : b);
    }
    const long long strips = (h + 63) / 64;
    long long s = (16LL * sm_count + strips - 1) / strips;
    const long long by_rows = T / 128 > 0 ? T / 128 : 1;
    if (s > by_rows) s = by_rows;
    if (s > LN_MAX_SPLITS) s = LN_MAX_SPLITS;
    return static_cast<int>(s < 1 ? 1 : s);
}
// Kernel launches of the LayerNorm backward.
inline int ln_backward_launches(long long h) { return ln_backward_fused(h) ? 2 : 3; }

cudaError_t launch_ln_forward(const LnForwardParams& p, long long T, cudaStream_t st);
// Two launches: dZ with its per-split column sums, then db2 = their
// fixed-order sum.
cudaError_t launch_dropout_backward(const DropoutBackwardParams& p, long long T, float* db2,
                                    cudaStream_t st);
// ln_backward_launches(h) launches: dX with the dgamma / dbeta partial sums
// over `splits` row blocks (one pass for rows of at most LN_WARP_MAX_H
// elements, a dX pass and a partial-sum pass for wider rows), then one
// fixed-order finish for both outputs.
cudaError_t launch_ln_backward(const LnBackwardParams& p, long long T, int splits, float* dgamma,
                               float* dbeta, cudaStream_t st);

}  // namespace tpmlp
