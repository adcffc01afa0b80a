// colsum.cuh -- bias gradients: column sums of bf16 matrices into fp32.
//   db1 = sum over tokens of dY (per shard block), db2 = sum over tokens of dZ
//   (over all sequence chunks).
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

namespace tpmlp {

constexpr int CS_THREADS = 256;   // 8 column vectors x 32 row slots
constexpr int CS_COLS = 64;       // columns per CTA (one 128-byte line per row)
constexpr int CS_MAX_SPLITS = 64; // row splits; partial sums [splits][n_out] fp32
constexpr int CS_MAX_PARTS = 8;

enum ColsumMode : int {
    CS_ROWS_CONCAT = 0,  // parts stacked along rows, one output of ncols
    CS_COLS_CONCAT = 1   // part p sums into out[p*ncols .. (p+1)*ncols)
};

struct ColsumParams {
    const void* src[CS_MAX_PARTS];  // bf16 [rows_per_part, ncols] each
    int nparts;
    long long rows_per_part;
    int ncols;
    int mode;
    int splits;                  // row splits (1 = write `out` directly)
    long long rows_per_split;
    float* out;                  // fp32 [n_out]
    float* partial;              // fp32 [splits][n_out] when splits > 1
};

// Chooses splits so that enough CTAs stream the input; returns the grid.
dim3 colsum_plan(ColsumParams& p, int sm_count);
// Bytes of partial-sum scratch colsum needs for n_out outputs.
inline size_t colsum_scratch_bytes(long long n_out) {
    return static_cast<size_t>(CS_MAX_SPLITS) * static_cast<size_t>(n_out) * sizeof(float);
}
// Launches the column sum (one kernel, plus a fixed-order finishing kernel
// when the rows are split).  Deterministic: no atomics.
cudaError_t launch_colsum(const ColsumParams& p, dim3 grid, cudaStream_t stream, int* launches);

// fp32 column sums of a [rows, ld] partial-sum matrix (its first ncols
// columns): out[c] = sum over r of part[r * ld + c], r in increasing order
// within each of 16 row lanes, the 16 lanes then added in lane order.  ncols
// and ld multiples of 4, part and out 16-byte aligned.
cudaError_t launch_colsum_f32(const float* part, long long rows, long long ld, long long ncols,
                              float* out, cudaStream_t stream);
// The same over the first 2 * ncols columns in one launch: out0[c] for c < ncols,
// out1[c] for column ncols + c (two row-interleaved sums, e.g. [rows][2][ncols]).
cudaError_t launch_colsum_f32_pair(const float* part, long long rows, long long ld,
                                   long long ncols, float* out0, float* out1,
                                   cudaStream_t stream);

}  // namespace tpmlp
