// block_internal.h -- the MLP block's passes on explicit device buffers, shared
// by the C-ABI units that run the block: tpmlp.cu (the block's own calls) and
// sp_layer.cu (the sequence-parallel sublayer around it).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "abi_internal.h"
#include "philox.cuh"
#include "tpmlp.h"

namespace tpmlp {
namespace block {

// Workspace byte offsets of the standard calls.
struct Layout {
    size_t y, h, dy, part1, part2, split_part, split_cnt, total;
};

// Device buffers one forward/backward pair works in.  The standard calls
// carve them all out of one workspace; the recompute calls take the saved
// pre-activation Y apart from a scratch area that holds the rest.
struct Regions {
    uint8_t* y;           // Y shards [t][T][fi] bf16 (kept from forward to backward)
    uint8_t* h;           // H shards (kept in the standard calls; scratch with recompute)
    uint8_t* dy;          // dY shards (scratch)
    uint8_t* part1;       // db1 partial sums (scratch)
    uint8_t* part2;       // db2 partial sums (scratch)
    uint8_t* split_part;  // tail-split partial tiles (scratch)
    uint8_t* split_cnt;   // tail-split counters (scratch)
};

struct Shapes {
    int T, h, f, t, fi, chunks, Tc;
};

// The row GEMM's epilogue for the sequence-parallel sublayer:
// Out = residual + Dropout(Z), the residual given per token chunk.
struct RowEpilogue {
    const void* const* residual;
    DropoutParams drop;
};

Layout layout_of(const tpmlp_dims& d);
tpmlp_status check_dims(const tpmlp_dims* d);
Regions regions_of(uint8_t* ws, const Layout& L);
Shapes shapes_of(const tpmlp_dims& d);
// With no tokens the weight and bias gradients are zero.
tpmlp_status zero_weight_grads(const Shapes& s, void* const* dA_shards, void* db1,
                               void* const* dB_shards, void* db2, cudaStream_t st);
// The forward pass (column GEMM + bias + GeLU, row GEMM + b2 or `ep`).
tpmlp_status run_forward(const Shapes& s, const abi::DeviceInfo* dev, const void* const* X,
                         const void* const* A_shards, const void* b1,
                         const void* const* B_shards, const void* b2, void* const* Z,
                         const Regions& R, cudaStream_t st, const RowEpilogue* ep);
// The backward pass; recompute = true rebuilds H from the saved Y; with
// db2_given the caller has already written db2 (its column sums of dZ).
tpmlp_status run_backward(const Shapes& s, const abi::DeviceInfo* dev, const void* const* dZ,
                          const void* const* X, const void* const* A_shards,
                          const void* const* B_shards, void* const* dX, void* const* dA_shards,
                          void* db1, void* const* dB_shards, void* db2, const Regions& R,
                          bool recompute, cudaStream_t st, bool db2_given = false);

}  // namespace block
}  // namespace tpmlp
