// gemm_params.h -- host-visible description of one launch of the tcgen05
// GEMM (tile sizes, operand partitioning, epilogue kind) and the launchers
// of its variants.  Shared by the C-ABI translation unit and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "philox.cuh"

namespace tpmlp {

// A CTA pair (cluster of 2) computes a CLUSTER_M x TN tile with
// tcgen05.mma.cta_group::2: each CTA stages its own BM rows of A and its own
// TN/2 rows of B per K step and holds BM rows x TN columns of the accumulator.
// TN is BN (narrow tiles, two accumulators) or BN_WIDE (one accumulator).
constexpr int BM = 128;            // tile rows per CTA (TMEM lanes)
constexpr int CLUSTER_M = 2 * BM;  // tile rows per CTA pair
constexpr int BN = 256;       // narrow tile columns (TMEM columns per accumulator)
constexpr int BN_WIDE = 512;  // wide tile columns (the whole of TMEM)
// tile-width policy of the bf16-output GEMMs (tpmlp_set_wide_tiles): the
// default takes wide tiles for GEMMs of at least WIDE_MIN_KSTEPS K steps
constexpr int WIDE_TILES_DEEP_K = 3;
constexpr int WIDE_MIN_KSTEPS = 256;
constexpr int BK = 64;        // K per stage: one 128-byte swizzle row of bf16
constexpr int STAGES = 6;
constexpr int A_STAGE_BYTES = BM * BK * 2;
constexpr int B_ROWS = BN / 2;     // B rows (output columns) staged per CTA
constexpr int B_STAGE_BYTES = B_ROWS * BK * 2;
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr int GEMM_THREADS = 192;
constexpr int TMEM_COLS = 2 * BN;
constexpr int BAR_BYTES = 256;
constexpr int EPI_WARPS = 4;
constexpr int EPI_CHUNK = 32;                 // accumulator columns per epilogue step
constexpr int EPI_BUF_BYTES = 4096;           // one staged 32 x 32 chunk (fp32, or 2 x bf16)
constexpr int EPI_STAGE_BYTES = EPI_WARPS * 2 * EPI_BUF_BYTES;  // double-buffered per warp
// fp32 output pacing: one BK step of a pair's 256 x 256 MMAs takes 4 x 128 SM
// clocks; chunk c of a tile is stored no earlier than c x PACE_CLK_PER_KBLOCK x
// (the tile's K steps) clocks after its accumulator arrived, which spreads the
// eight chunk stores over about two thirds of the next tile's MMA time (7 x 48
// of 512 clocks per K step; measured best among 20..96 on the weight gradients
// of the 175B-class layer).
constexpr int PACE_CLK_PER_KBLOCK = 48;
constexpr int GEMM_SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_STAGE_BYTES + BAR_BYTES;
constexpr int MAX_MAPS = 8;
// Tail split: when the tiles do not fill the last wave of pairs, the leftover
// tiles' K ranges are split across the idle pairs.  Each split unit writes an
// fp32 partial tile; the last unit of a tile to finish sums them in a fixed
// order and runs the epilogue.
constexpr int MAX_SPLIT_UNITS = 128;       // partial tiles the workspace holds
constexpr int MAX_SPLITS = 8;              // K splits per leftover tile
constexpr int DEFAULT_SPLIT_MIN_KBLOCKS = 128;  // split only tiles this deep in K
constexpr int MN_CHUNK = 64;                      // elements per 128-byte row
constexpr int MN_CHUNK_BYTES = MN_CHUNK * BK * 2;  // one MN-major box [BK][64]

// How the tensor maps of an operand (or the output pointers) are indexed.
enum Part : int {
    PART_SINGLE = 0,  // one map; K coordinate runs over all segments
    PART_GROUP = 1,   // map g; K coordinate runs over all segments
    PART_KSEG = 2,    // map s; K coordinate within the segment
    PART_ROW = 3      // map row0 / rows_per_map (token chunks); K over all segments
};

// Output i of a tile goes through out_map[i] (first output) and
// out_map[MAX_MAPS + i] (second output), i = group or token chunk.
enum Epi : int {
    EPI_BIAS_GELU = 1,  // out 1 = bf16(acc + bias), out 2 = bf16(GeLU(acc + bias))
    EPI_BIAS = 2,       // out 1 = bf16(acc + bias)
    EPI_DGELU = 3,      // out 1 = bf16(acc * GeLU'(in0))
    EPI_BF16 = 4,       // out 1 = bf16(acc)
    EPI_F32 = 5,        // out 1 = acc (fp32)
    EPI_DGELU_H = 6,    // out 1 = bf16(acc * GeLU'(in0)), out 2 = bf16(GeLU(in0)) (recompute)
    EPI_BIAS_DROP_RES = 7  // out 1 = bf16(in0 + dropout(acc + bias)) (sequence-parallel sublayer)
};

// Error-word bits (which role gave up).
constexpr unsigned ERR_PRODUCER = 1u, ERR_MMA = 2u, ERR_EPILOGUE = 4u, ERR_DRAIN = 8u;

struct GemmParams {
    CUtensorMap a_map[MAX_MAPS];
    CUtensorMap b_map[MAX_MAPS];
    int M, N, K;            // per-group output rows/cols; K per segment
    int groups, ksegs;
    int a_part, b_part;
    int a_rows_per_map, b_rows_per_map;
    int a_nmaps, b_nmaps;   // encoded maps; PART_ROW indices are clamped to them
    // MN-major operands whose row count is a multiple of 64 are encoded as 3-D
    // maps {64, K, rows / 64} so one copy fetches every 64-row chunk of a box
    int a_mn3d, b_mn3d;
    // tail split (set by the launcher; units = 0 means every tile is whole)
    int dp_tiles;           // tiles computed whole, in schedule order 0..dp_tiles-1
    int splits;             // K splits per leftover tile
    int units;              // leftover tiles x splits
    int split_min_kblocks;  // split only when a tile has at least this many K steps
    int head_prefetch;      // at a tile's start, prefetch this many K steps of the next
                            // tile's operands into L2 (0 = off)
    CUtensorMap part_map;   // fp32 [MAX_SPLIT_UNITS * CLUSTER_M, BN] partial tiles
    const float* partial;   // same buffer, for the summing loads
    int* counters;          // [MAX_SPLIT_UNITS][2] arrivals per leftover tile and CTA
    int tn;                 // tile columns: BN or BN_WIDE (set with mtiles, ntiles)
    int mtiles, ntiles, total_tiles, band;  // pair tiles of CLUSTER_M x tn
    // epilogue: TMA store maps (box 32 x 32, 128-byte swizzle for fp32,
    // 64-byte swizzle for bf16) and the saved pre-activation for EPI_DGELU
    CUtensorMap out_map[2 * MAX_MAPS];
    const void* in0[MAX_MAPS];
    const void* bias;
    long long ld_in;         // leading dimension of in0 (elements)
    int out_part;            // PART_GROUP or PART_ROW
    int out_rows_per_part;   // rows per output chunk for PART_ROW
    int bias_group_stride;   // bias offset per group (EPI_BIAS_GELU, EPI_BIAS)
    DropoutParams drop;      // EPI_BIAS_DROP_RES: mask of element (m, n) = Philox word of m * N + n
    // EPI_DGELU / EPI_DGELU_H: column sums of the fp32 output (the bias gradient
    // db1), one row per 32-row group of the output: colsum_part[r / 32][g * N + n]
    // (null: none)
    float* colsum_part;
    long long colsum_ld;     // floats per partial row (groups x N)
    // control
    unsigned int* err;
    unsigned long long timeout_ns;
    int stall_producer;      // failure-detection self-test: issue no loads
};

// Launchers, one per (operand majorness, epilogue) variant.  Each launches a
// persistent grid of CTA pairs (at most one pair per tile, at most as many
// pairs as fit on the GPU at once).
//   column_fwd : A K-major,  B MN-major, EPI_BIAS_GELU  (Y_i, H_i)
//   row_fwd    : A K-major,  B MN-major, EPI_BIAS       (Z; column-linear Y_i)
//   dgrad_h    : A K-major,  B K-major,  EPI_DGELU      (dY_i)
//   dgrad_x    : A K-major,  B K-major,  EPI_BF16       (dX; row-linear dX_i)
//   wgrad      : A MN-major, B MN-major, EPI_F32        (dA_i, dB_i; linear dW_i)
cudaError_t launch_column_fwd(const GemmParams& p, cudaStream_t stream);
cudaError_t launch_row_fwd(const GemmParams& p, cudaStream_t stream);
cudaError_t launch_dgrad_h(const GemmParams& p, cudaStream_t stream);
//   row_fwd_dropout: A K-major, B MN-major, EPI_BIAS_DROP_RES (Out = X + Dropout(Z))
cudaError_t launch_row_fwd_dropout(const GemmParams& p, cudaStream_t stream);
//   dgrad_h_recompute: A K-major, B K-major, EPI_DGELU_H (dY_i and H_i = GeLU(Y_i))
cudaError_t launch_dgrad_h_recompute(const GemmParams& p, cudaStream_t stream);
cudaError_t launch_dgrad_x(const GemmParams& p, cudaStream_t stream);
cudaError_t launch_wgrad(const GemmParams& p, cudaStream_t stream);

}  // namespace tpmlp
