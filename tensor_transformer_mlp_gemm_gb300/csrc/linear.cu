// linear.cu -- the C ABI of the tensor-parallel linear layers (declared in
// include/tpmlp.h): the column- and row-parallel halves of the MLP block
// without the GeLU, as the attention projections use them.
//
//   column parallel  forward   Y_i = X.W_i + b_i          row_fwd kernel, t groups
//                    backward  dX = sum_i dY_i.W_i^T      dgrad_x kernel, t k-segments
//                              dW_i = X^T.dY_i            wgrad kernel, t groups
//                              db = column sums of dY     colsum
//   row parallel     forward   Z = sum_i X_i.W_i + b      row_fwd kernel, t k-segments
//                    backward  dX_i = dZ.W_i^T            dgrad_x kernel, t groups
//                              dW_i = X_i^T.dZ            wgrad kernel, t groups
//                              db = column sums of dZ     colsum
//
// Sources (page title, section): "2、分布式训练基础：数据并行、模型并行、流水线并行的基本概念与区别",
// "2.2 模型并行 —— 张量并行 / 核心原理" (Y = XW; column split [W1, W2];
// row split [W1; W2] with X = [X1, X2] and a summing AllReduce; the QKV
// projection column parallel and the output projection row parallel);
// "Megatron-LM：NVIDIA 的大规模并行训练方案", "Megatron-LM 核心架构 / 张量并行原理"
// and "并行训练范式 / 序列并行" (token chunks in, token chunks out).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "abi_internal.h"
#include "colsum.cuh"
#include "gemm_params.h"
#include "tpmlp.h"

#define TPMLP_API extern "C" __attribute__((visibility("default")))

namespace tpmlp {
namespace {

using namespace abi;

enum class Split { Column, Row };

// Shapes of one linear layer; `shard` is out / t (column) or in / t (row).
struct Lin {
    int T, in, out, t, chunks, Tc, shard;
};

tpmlp_status check_linear(const tpmlp_linear_dims* d, Split k) {
    if (!d) return TPMLP_ERR_INVALID_ARG;
    if (d->tokens < 0 || d->in_features <= 0 || d->out_features <= 0 || d->t <= 0 ||
        d->seq_chunks <= 0)
        return TPMLP_ERR_INVALID_ARG;
    const int64_t split = k == Split::Column ? d->out_features : d->in_features;
    const int64_t other = k == Split::Column ? d->in_features : d->out_features;
    if (split % d->t != 0) return TPMLP_ERR_INVALID_ARG;
    if (d->tokens % d->seq_chunks != 0) return TPMLP_ERR_INVALID_ARG;
    if (d->t > kMaxShards || d->seq_chunks > kMaxShards) return TPMLP_ERR_UNSUPPORTED;
    if ((split / d->t) % 8 != 0 || other % 8 != 0) return TPMLP_ERR_UNSUPPORTED;
    const int64_t lim = (int64_t(1) << 31) - 1;
    if (d->tokens > lim || d->in_features > lim || d->out_features > lim)
        return TPMLP_ERR_UNSUPPORTED;
    if (d->seq_chunks > 1 && (d->tokens / d->seq_chunks) % BM != 0) return TPMLP_ERR_UNSUPPORTED;
    return TPMLP_OK;
}

Lin lin_of(const tpmlp_linear_dims& d, Split k) {
    Lin s;
    s.T = static_cast<int>(d.tokens);
    s.in = static_cast<int>(d.in_features);
    s.out = static_cast<int>(d.out_features);
    s.t = d.t;
    s.chunks = d.seq_chunks;
    s.Tc = s.T / s.chunks;
    s.shard = (k == Split::Column ? s.out : s.in) / s.t;
    return s;
}

// Scratch workspace: bias-gradient partial sums | tail-split tiles | counters.
struct Scratch {
    void* colsum;
    void* split_part;
    void* split_cnt;
};

size_t colsum_bytes(const tpmlp_linear_dims& d) {
    return align256(colsum_scratch_bytes(d.out_features));
}

size_t scratch_bytes(const tpmlp_linear_dims& d) {
    return colsum_bytes(d) + split_part_bytes() + split_cnt_bytes();
}

Scratch scratch_of(const tpmlp_linear_dims& d, void* ws) {
    uint8_t* b = static_cast<uint8_t*>(ws);
    const size_t c = colsum_bytes(d);
    return Scratch{b, b + c, b + c + split_part_bytes()};
}

// dW shards are [in, oi] (column) or [ii, out] (row): shard * other fp32 each.
tpmlp_status zero_linear_grads(const Lin& s, Split k, void* const* dW, void* db, cudaStream_t st) {
    const size_t other = static_cast<size_t>(k == Split::Column ? s.in : s.out);
    const size_t wbytes = other * static_cast<size_t>(s.shard) * sizeof(float);
    for (int i = 0; i < s.t; ++i) TPMLP_CUDA(cudaMemsetAsync(dW[i], 0, wbytes, st));
    TPMLP_CUDA(cudaMemsetAsync(db, 0, static_cast<size_t>(s.out) * sizeof(float), st));
    return TPMLP_OK;
}

tpmlp_status bias_grad(const DeviceInfo* dev, const void* const* src, int nparts,
                       long long rows_per_part, int ncols, int mode, void* db, void* partial,
                       cudaStream_t st) {
    ColsumParams c;
    std::memset(&c, 0, sizeof(c));
    for (int i = 0; i < nparts; ++i) c.src[i] = src[i];
    c.nparts = nparts;
    c.rows_per_part = rows_per_part;
    c.ncols = ncols;
    c.mode = mode;
    c.out = static_cast<float*>(db);
    c.partial = static_cast<float*>(partial);
    const dim3 g = colsum_plan(c, dev->sm_count);
    TPMLP_CUDA(timed(TPMLP_KERNEL_BIAS_GRAD, c.splits > 1 ? 2 : 1, st,
                     [&] { return launch_colsum(c, g, st, nullptr); }));
    return TPMLP_OK;
}

// ---- column parallel ---------------------------------------------------------------------

tpmlp_status column_forward(const Lin& s, const DeviceInfo* dev, const void* const* X,
                            const void* const* W, const void* b, void* const* Y,
                            const Scratch& R, cudaStream_t st) {
    // Y_i = X.W_i + b_i: t groups, M = T, N = oi, K = in
    GemmParams p;
    base_params(p, *dev, s.T, s.shard, s.in, s.t, 1);
    choose_tile_width(p, *dev);
    for (int j = 0; j < s.chunks; ++j)
        if (!encode_kmajor(&p.a_map[j], X[j], s.in, s.Tc, BM)) return TPMLP_ERR_UNSUPPORTED;
    p.a_part = PART_ROW;
    p.a_nmaps = s.chunks;
    p.a_rows_per_map = s.Tc;
    for (int i = 0; i < s.t; ++i)
        if (!encode_mnmajor(&p.b_map[i], W[i], s.shard, s.in, &p.b_mn3d))
            return TPMLP_ERR_UNSUPPORTED;
    p.b_part = PART_GROUP;
    p.b_nmaps = s.t;
    for (int i = 0; i < s.t; ++i)
        if (!encode_out(&p.out_map[i], Y[i], s.shard, s.T, false)) return TPMLP_ERR_UNSUPPORTED;
    p.out_part = PART_GROUP;
    p.bias = b;
    p.bias_group_stride = s.shard;
    if (!attach_split(p, R.split_part, R.split_cnt)) return TPMLP_ERR_UNSUPPORTED;
    TPMLP_CUDA(timed(TPMLP_KERNEL_LINEAR_FWD, 1, st, [&] { return launch_row_fwd(p, st); }));
    return TPMLP_OK;
}

tpmlp_status column_backward(const Lin& s, const DeviceInfo* dev, const void* const* dY,
                             const void* const* X, const void* const* W, void* const* dX,
                             void* const* dW, void* db, const Scratch& R, cudaStream_t st) {
    // dX = sum_i dY_i.W_i^T: M = T, N = in, K = oi per segment; rows back into chunks
    {
        GemmParams p;
        base_params(p, *dev, s.T, s.in, s.shard, 1, s.t);
        choose_tile_width(p, *dev);
        for (int i = 0; i < s.t; ++i) {
            if (!encode_kmajor(&p.a_map[i], dY[i], s.shard, s.T, BM)) return TPMLP_ERR_UNSUPPORTED;
            if (!encode_kmajor(&p.b_map[i], W[i], s.shard, s.in, B_ROWS))
                return TPMLP_ERR_UNSUPPORTED;
        }
        p.a_part = p.b_part = PART_KSEG;
        p.a_nmaps = p.b_nmaps = s.t;
        for (int j = 0; j < s.chunks; ++j)
            if (!encode_out(&p.out_map[j], dX[j], s.in, s.Tc, false)) return TPMLP_ERR_UNSUPPORTED;
        p.out_part = PART_ROW;
        p.out_rows_per_part = s.Tc;
        if (!attach_split(p, R.split_part, R.split_cnt)) return TPMLP_ERR_UNSUPPORTED;
        TPMLP_CUDA(timed(TPMLP_KERNEL_LINEAR_DGRAD, 1, st, [&] { return launch_dgrad_x(p, st); }));
    }
    // dW_i = X^T.dY_i: t groups, M = in, N = oi, K = Tc per chunk segment
    {
        GemmParams p;
        base_params(p, *dev, s.in, s.shard, s.Tc, s.t, s.chunks);
        for (int j = 0; j < s.chunks; ++j)
            if (!encode_mnmajor(&p.a_map[j], X[j], s.in, s.Tc, &p.a_mn3d)) return TPMLP_ERR_UNSUPPORTED;
        p.a_part = PART_KSEG;
        p.a_nmaps = s.chunks;
        for (int i = 0; i < s.t; ++i)
            if (!encode_mnmajor(&p.b_map[i], dY[i], s.shard, s.T, &p.b_mn3d)) return TPMLP_ERR_UNSUPPORTED;
        p.b_part = PART_GROUP;
        p.b_nmaps = s.t;
        for (int i = 0; i < s.t; ++i)
            if (!encode_out(&p.out_map[i], dW[i], s.shard, s.in, true)) return TPMLP_ERR_UNSUPPORTED;
        p.out_part = PART_GROUP;
        if (!attach_split(p, R.split_part, R.split_cnt)) return TPMLP_ERR_UNSUPPORTED;
        TPMLP_CUDA(timed(TPMLP_KERNEL_LINEAR_WGRAD, 1, st, [&] { return launch_wgrad(p, st); }));
    }
    // db = column sums of dY, shard i into db[i*oi, (i+1)*oi)
    return bias_grad(dev, dY, s.t, s.T, s.shard, CS_COLS_CONCAT, db, R.colsum, st);
}

// ---- row parallel ---------------------------------------------------------------------------

tpmlp_status row_forward(const Lin& s, const DeviceInfo* dev, const void* const* X,
                         const void* const* W, const void* b, void* const* Z, const Scratch& R,
                         cudaStream_t st) {
    // Z = sum_i X_i.W_i + b: M = T, N = out, K = ii per segment; rows into chunks
    GemmParams p;
    base_params(p, *dev, s.T, s.out, s.shard, 1, s.t);
    choose_tile_width(p, *dev);
    for (int i = 0; i < s.t; ++i) {
        if (!encode_kmajor(&p.a_map[i], X[i], s.shard, s.T, BM)) return TPMLP_ERR_UNSUPPORTED;
        if (!encode_mnmajor(&p.b_map[i], W[i], s.out, s.shard, &p.b_mn3d))
            return TPMLP_ERR_UNSUPPORTED;
    }
    p.a_part = p.b_part = PART_KSEG;
    p.a_nmaps = p.b_nmaps = s.t;
    for (int j = 0; j < s.chunks; ++j)
        if (!encode_out(&p.out_map[j], Z[j], s.out, s.Tc, false)) return TPMLP_ERR_UNSUPPORTED;
    p.out_part = PART_ROW;
    p.out_rows_per_part = s.Tc;
    p.bias = b;
    if (!attach_split(p, R.split_part, R.split_cnt)) return TPMLP_ERR_UNSUPPORTED;
    TPMLP_CUDA(timed(TPMLP_KERNEL_LINEAR_FWD, 1, st, [&] { return launch_row_fwd(p, st); }));
    return TPMLP_OK;
}

tpmlp_status row_backward(const Lin& s, const DeviceInfo* dev, const void* const* dZ,
                          const void* const* X, const void* const* W, void* const* dX,
                          void* const* dW, void* db, const Scratch& R, cudaStream_t st) {
    // dX_i = dZ.W_i^T: t groups, M = T, N = ii, K = out; dZ gathered from its chunks
    {
        GemmParams p;
        base_params(p, *dev, s.T, s.shard, s.out, s.t, 1);
        choose_tile_width(p, *dev);
        for (int j = 0; j < s.chunks; ++j)
            if (!encode_kmajor(&p.a_map[j], dZ[j], s.out, s.Tc, BM)) return TPMLP_ERR_UNSUPPORTED;
        p.a_part = PART_ROW;
        p.a_nmaps = s.chunks;
        p.a_rows_per_map = s.Tc;
        for (int i = 0; i < s.t; ++i)
            if (!encode_kmajor(&p.b_map[i], W[i], s.out, s.shard, B_ROWS))
                return TPMLP_ERR_UNSUPPORTED;
        p.b_part = PART_GROUP;
        p.b_nmaps = s.t;
        for (int i = 0; i < s.t; ++i)
            if (!encode_out(&p.out_map[i], dX[i], s.shard, s.T, false)) return TPMLP_ERR_UNSUPPORTED;
        p.out_part = PART_GROUP;
        if (!attach_split(p, R.split_part, R.split_cnt)) return TPMLP_ERR_UNSUPPORTED;
        TPMLP_CUDA(timed(TPMLP_KERNEL_LINEAR_DGRAD, 1, st, [&] { return launch_dgrad_x(p, st); }));
    }
    // dW_i = X_i^T.dZ: t groups, M = ii, N = out, K = Tc per chunk segment
    {
        GemmParams p;
        base_params(p, *dev, s.shard, s.out, s.Tc, s.t, s.chunks);
        for (int i = 0; i < s.t; ++i)
            if (!encode_mnmajor(&p.a_map[i], X[i], s.shard, s.T, &p.a_mn3d)) return TPMLP_ERR_UNSUPPORTED;
        p.a_part = PART_GROUP;
        p.a_nmaps = s.t;
        for (int j = 0; j < s.chunks; ++j)
            if (!encode_mnmajor(&p.b_map[j], dZ[j], s.out, s.Tc, &p.b_mn3d)) return TPMLP_ERR_UNSUPPORTED;
        p.b_part = PART_KSEG;
        p.b_nmaps = s.chunks;
        for (int i = 0; i < s.t; ++i)
            if (!encode_out(&p.out_map[i], dW[i], s.out, s.shard, true)) return TPMLP_ERR_UNSUPPORTED;
        p.out_part = PART_GROUP;
        if (!attach_split(p, R.split_part, R.split_cnt)) return TPMLP_ERR_UNSUPPORTED;
        TPMLP_CUDA(timed(TPMLP_KERNEL_LINEAR_WGRAD, 1, st, [&] { return launch_wgrad(p, st); }));
    }
    // db = column sums of dZ over all chunks
    return bias_grad(dev, dZ, s.chunks, s.Tc, s.out, CS_ROWS_CONCAT, db, R.colsum, st);
}

// The argument checks shared by the four calls: the t weight shards, and,
// when T > 0, `nin` input pointers, `nout` output pointers (per shard or per
// chunk) and the workspace.
tpmlp_status check_common(const Lin& s, const void* const* W, const void* const* in, int nin,
                          void* const* outs, int nout, void* workspace) {
    TPMLP_TRY(check_ptrs(W, s.t));
    if (s.T > 0) {
        TPMLP_TRY(check_ptrs(in, nin));
        TPMLP_TRY(check_ptrs(reinterpret_cast<const void* const*>(outs), nout));
        TPMLP_TRY(check_ptr(workspace));
    }
    return TPMLP_OK;
}

}  // namespace
}  // namespace tpmlp

using namespace tpmlp;
using namespace tpmlp::abi;

TPMLP_API size_t tpmlp_linear_workspace_bytes(const tpmlp_linear_dims* dims) {
    if (!dims) return 0;
    // both kinds need the same scratch; accept dims valid for either split
    if (check_linear(dims, Split::Column) != TPMLP_OK && check_linear(dims, Split::Row) != TPMLP_OK)
        return 0;
    return scratch_bytes(*dims);
}

TPMLP_API tpmlp_status tpmlp_column_linear_forward(const tpmlp_linear_dims* dims,
                                                   const void* const* X,
                                                   const void* const* W_shards, const void* b,
                                                   void* const* Y_shards, void* workspace,
                                                   void* stream) {
    TPMLP_TRY(check_linear(dims, Split::Column));
    const Lin s = lin_of(*dims, Split::Column);
    TPMLP_TRY(check_ptr(b));
    TPMLP_TRY(check_common(s, W_shards, X, s.chunks, Y_shards, s.t, workspace));
    DeviceInfo* dev = nullptr;
    TPMLP_TRY(device_info(&dev));
    if (s.T == 0) return TPMLP_OK;
    return column_forward(s, dev, X, W_shards, b, Y_shards, scratch_of(*dims, workspace),
                          static_cast<cudaStream_t>(stream));
}

TPMLP_API tpmlp_status tpmlp_column_linear_backward(const tpmlp_linear_dims* dims,
                                                    const void* const* dY_shards,
                                                    const void* const* X,
                                                    const void* const* W_shards,
                                                    void* const* dX, void* const* dW_shards,
                                                    void* db, void* workspace, void* stream) {
    TPMLP_TRY(check_linear(dims, Split::Column));
    const Lin s = lin_of(*dims, Split::Column);
    TPMLP_TRY(check_ptrs(reinterpret_cast<const void* const*>(dW_shards), s.t));
    TPMLP_TRY(check_ptr(db));
    TPMLP_TRY(check_common(s, W_shards, dY_shards, s.t, dX, s.chunks, workspace));
    if (s.T > 0) TPMLP_TRY(check_ptrs(X, s.chunks));
    DeviceInfo* dev = nullptr;
    TPMLP_TRY(device_info(&dev));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (s.T == 0) return zero_linear_grads(s, Split::Column, dW_shards, db, st);
    return column_backward(s, dev, dY_shards, X, W_shards, dX, dW_shards, db,
                           scratch_of(*dims, workspace), st);
}

TPMLP_API tpmlp_status tpmlp_row_linear_forward(const tpmlp_linear_dims* dims,
                                                const void* const* X_shards,
                                                const void* const* W_shards, const void* b,
                                                void* const* Z, void* workspace, void* stream) {
    TPMLP_TRY(check_linear(dims, Split::Row));
    const Lin s = lin_of(*dims, Split::Row);
    TPMLP_TRY(check_ptr(b));
    TPMLP_TRY(check_common(s, W_shards, X_shards, s.t, Z, s.chunks, workspace));
    DeviceInfo* dev = nullptr;
    TPMLP_TRY(device_info(&dev));
    if (s.T == 0) return TPMLP_OK;
    return row_forward(s, dev, X_shards, W_shards, b, Z, scratch_of(*dims, workspace),
                       static_cast<cudaStream_t>(stream));
}

TPMLP_API tpmlp_status tpmlp_row_linear_backward(const tpmlp_linear_dims* dims,
                                                 const void* const* dZ,
                                                 const void* const* X_shards,
                                                 const void* const* W_shards,
                                                 void* const* dX_shards, void* const* dW_shards,
                                                 void* db, void* workspace, void* stream) {
    TPMLP_TRY(check_linear(dims, Split::Row));
    const Lin s = lin_of(*dims, Split::Row);
    TPMLP_TRY(check_ptrs(reinterpret_cast<const void* const*>(dW_shards), s.t));
    TPMLP_TRY(check_ptr(db));
    TPMLP_TRY(check_common(s, W_shards, dZ, s.chunks, dX_shards, s.t, workspace));
    if (s.T > 0) TPMLP_TRY(check_ptrs(X_shards, s.t));
    DeviceInfo* dev = nullptr;
    TPMLP_TRY(device_info(&dev));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (s.T == 0) return zero_linear_grads(s, Split::Row, dW_shards, db, st);
    return row_backward(s, dev, dZ, X_shards, W_shards, dX_shards, dW_shards, db,
                        scratch_of(*dims, workspace), st);
}
