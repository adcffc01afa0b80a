// sp_layer.cu -- C ABI of the sequence-parallel sublayer around the MLP block
// (declared in include/tpmlp.h):
//
//   forward   ln_forward     Xn = LN(X) per token chunk (mean, rstd kept)
//             column_fwd     Y_i = Xn.A_i + b1_i, H_i = GeLU(Y_i)
//             row_fwd_dropout Out = X + Dropout(sum_i H_i.B_i + b2)
//   backward  dropout_backward dZ = keep ? dOut / (1 - p) : 0
//             the block's backward on dZ and Xn    (dXn, dA, db1, dB, db2)
//             ln_backward    dX = LN'(dXn) + dOut, dgamma, dbeta
//
// Sources: "Megatron-LM：NVIDIA 的大规模并行训练方案", "并行训练范式 / 序列并行"
// (LayerNorm and Dropout along the sequence dimension on top of tensor
// parallelism) and "Megatron-LM 核心架构 / 张量并行原理" (the block).  The
// dropout mask is Philox4x32-10 (Salmon et al., SC'11) on the element index.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "abi_internal.h"
#include "block_internal.h"
#include "layernorm.cuh"
#include "tpmlp.h"

#define TPMLP_API extern "C" __attribute__((visibility("default")))

namespace tpmlp {
namespace {

using namespace abi;
using namespace block;

// After the block's workspace: Xn | mean | rstd | dZ | dXn | LayerNorm partials |
// dropout keep bits | partial column sums of dZ.
struct SpLayout {
    Layout blk;
    size_t xn, mean, rstd, dz, dxn, part, mask, dpart, total;
};

long long mask_words_of(long long h) { return (h + 31) / 32; }

SpLayout sp_layout_of(const tpmlp_dims& d) {
    SpLayout L;
    L.blk = layout_of(d);
    const size_t act = align256(static_cast<size_t>(d.tokens) * static_cast<size_t>(d.hidden) * 2);
    const size_t row = align256(static_cast<size_t>(d.tokens) * sizeof(float));
    L.xn = L.blk.total;
    L.mean = L.xn + act;
    L.rstd = L.mean + row;
    L.dz = L.rstd + row;
    L.dxn = L.dz + act;
    L.part = L.dxn + act;
    L.mask = L.part + align256(ln_partial_bytes(d.hidden));
    L.dpart = L.mask + align256(static_cast<size_t>(d.tokens) *
                                static_cast<size_t>(mask_words_of(d.hidden)) * sizeof(uint32_t));
    L.total = L.dpart + align256(static_cast<size_t>(LN_MAX_SPLITS) *
                                 static_cast<size_t>(d.hidden) * sizeof(float));
    return L;
}

tpmlp_status check_sp(const tpmlp_dims* d, const tpmlp_sp_params* sp) {
    TPMLP_TRY(check_dims(d));
    if (!sp) return TPMLP_ERR_INVALID_ARG;
    if (!(sp->eps >= 0.0f) || !std::isfinite(sp->eps)) return TPMLP_ERR_INVALID_ARG;
    if (!(sp->dropout_p >= 0.0 && sp->dropout_p < 1.0)) return TPMLP_ERR_INVALID_ARG;
    if (d->hidden > LN_MAX_H) return TPMLP_ERR_UNSUPPORTED;
    return TPMLP_OK;
}

DropoutParams dropout_of(const tpmlp_sp_params& sp) {
    DropoutParams dp;
    dp.seed = sp.seed;
    dp.offset = sp.offset;
    dp.thresh = static_cast<uint64_t>(std::floor((1.0 - sp.dropout_p) * 4294967296.0));
    dp.scale = static_cast<float>(1.0 / (1.0 - sp.dropout_p));
    return dp;
}

// chunk pointers into a [T, h] bf16 buffer stored chunk after chunk
void chunk_ptrs(uint8_t* base, const Shapes& s, void** out) {
    for (int j = 0; j < s.chunks; ++j)
        out[j] = base + static_cast<size_t>(j) * s.Tc * s.h * 2;
}

}  // namespace
}  // namespace tpmlp

using namespace tpmlp;
using namespace tpmlp::abi;
using namespace tpmlp::block;

TPMLP_API size_t tpmlp_sp_workspace_bytes(const tpmlp_dims* dims) {
    if (check_dims(dims) != TPMLP_OK || dims->hidden > LN_MAX_H) return 0;
    return sp_layout_of(*dims).total;
}

TPMLP_API tpmlp_status tpmlp_sp_workspace_layout(const tpmlp_dims* dims, size_t* xn_offset,
                                                 size_t* dz_offset) {
    TPMLP_TRY(check_dims(dims));
    if (dims->hidden > LN_MAX_H) return TPMLP_ERR_UNSUPPORTED;
    const SpLayout L = sp_layout_of(*dims);
    if (xn_offset) *xn_offset = L.xn;
    if (dz_offset) *dz_offset = L.dz;
    return TPMLP_OK;
}

TPMLP_API tpmlp_status tpmlp_sp_forward(const tpmlp_dims* dims, const tpmlp_sp_params* sp,
                                        const void* const* X, const void* gamma,
                                        const void* beta, const void* const* A_shards,
                                        const void* b1, const void* const* B_shards,
                                        const void* b2, int t, void* const* Out, void* workspace,
                                        void* stream) {
    TPMLP_TRY(check_sp(dims, sp));
    if (t != dims->t) return TPMLP_ERR_INVALID_ARG;
    const Shapes s = shapes_of(*dims);
    TPMLP_TRY(check_ptrs(A_shards, s.t));
    TPMLP_TRY(check_ptrs(B_shards, s.t));
    TPMLP_TRY(check_ptr(gamma));
    TPMLP_TRY(check_ptr(beta));
    TPMLP_TRY(check_ptr(b1));
    TPMLP_TRY(check_ptr(b2));
    if (s.T > 0) {
        TPMLP_TRY(check_ptrs(X, s.chunks));
        TPMLP_TRY(check_ptrs(reinterpret_cast<const void* const*>(Out), s.chunks));
        TPMLP_TRY(check_ptr(workspace));
    }
    DeviceInfo* dev = nullptr;
    TPMLP_TRY(device_info(&dev));
    if (s.T == 0) return TPMLP_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const SpLayout L = sp_layout_of(*dims);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    void* xn[LN_MAX_CHUNKS];
    chunk_ptrs(ws + L.xn, s, xn);

    LnForwardParams ln;
    std::memset(&ln, 0, sizeof(ln));
    for (int j = 0; j < s.chunks; ++j) {
        ln.x.in[j] = X[j];
        ln.y[j] = xn[j];
    }
    ln.x.n = s.chunks;
    ln.x.rows = s.Tc;
    ln.gamma = gamma;
    ln.beta = beta;
    ln.mean = reinterpret_cast<float*>(ws + L.mean);
    ln.rstd = reinterpret_cast<float*>(ws + L.rstd);
    ln.h = s.h;
    ln.eps = sp->eps;
    TPMLP_CUDA(timed(TPMLP_KERNEL_LAYERNORM_FWD, 1, st,
                     [&] { return launch_ln_forward(ln, s.T, st); }));

    RowEpilogue ep;
    ep.residual = X;
    ep.drop = dropout_of(*sp);
    // the row GEMM's epilogue also stores the mask's bits for the backward pass
    ep.drop.mask = reinterpret_cast<uint32_t*>(ws + L.mask);
    ep.drop.mask_words = mask_words_of(s.h);
    return run_forward(s, dev, xn, A_shards, b1, B_shards, b2, Out, regions_of(ws, L.blk), st, &ep);
}

TPMLP_API tpmlp_status tpmlp_sp_backward(const tpmlp_dims* dims, const tpmlp_sp_params* sp,
                                         const void* const* dOut, const void* const* X,
                                         const void* gamma, const void* const* A_shards,
                                         const void* const* B_shards, void* workspace,
                                         void* const* dX, void* dgamma, void* dbeta,
                                         void* const* dA_shards, void* db1,
                                         void* const* dB_shards, void* db2, void* stream) {
    TPMLP_TRY(check_sp(dims, sp));
    const Shapes s = shapes_of(*dims);
    TPMLP_TRY(check_ptrs(A_shards, s.t));
    TPMLP_TRY(check_ptrs(B_shards, s.t));
    TPMLP_TRY(check_ptrs(reinterpret_cast<const void* const*>(dA_shards), s.t));
    TPMLP_TRY(check_ptrs(reinterpret_cast<const void* const*>(dB_shards), s.t));
    TPMLP_TRY(check_ptr(gamma));
    TPMLP_TRY(check_ptr(dgamma));
    TPMLP_TRY(check_ptr(dbeta));
    TPMLP_TRY(check_ptr(db1));
    TPMLP_TRY(check_ptr(db2));
    if (s.T > 0) {
        TPMLP_TRY(check_ptrs(dOut, s.chunks));
        TPMLP_TRY(check_ptrs(X, s.chunks));
        TPMLP_TRY(check_ptrs(reinterpret_cast<const void* const*>(dX), s.chunks));
        TPMLP_TRY(check_ptr(workspace));
    }
    DeviceInfo* dev = nullptr;
    TPMLP_TRY(device_info(&dev));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (s.T == 0) {
        TPMLP_CUDA(cudaMemsetAsync(dgamma, 0, static_cast<size_t>(s.h) * sizeof(float), st));
        TPMLP_CUDA(cudaMemsetAsync(dbeta, 0, static_cast<size_t>(s.h) * sizeof(float), st));
        return zero_weight_grads(s, dA_shards, db1, dB_shards, db2, st);
    }
    const SpLayout L = sp_layout_of(*dims);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    void *xn[LN_MAX_CHUNKS], *dz[LN_MAX_CHUNKS], *dxn[LN_MAX_CHUNKS];
    chunk_ptrs(ws + L.xn, s, xn);
    chunk_ptrs(ws + L.dz, s, dz);
    chunk_ptrs(ws + L.dxn, s, dxn);

    DropoutBackwardParams db;
    std::memset(&db, 0, sizeof(db));
    for (int j = 0; j < s.chunks; ++j) {
        db.dout.in[j] = dOut[j];
        db.dz[j] = dz[j];
    }
    db.dout.n = s.chunks;
    db.dout.rows = s.Tc;
    db.h = s.h;
    db.drop = dropout_of(*sp);
    db.drop.mask = reinterpret_cast<uint32_t*>(ws + L.mask);  // written by the forward pass
    db.drop.mask_words = mask_words_of(s.h);
    db.part = reinterpret_cast<float*>(ws + L.dpart);
    db.splits = dropout_splits(s.T, s.h, dev->sm_count);
    db.rows_per_split = (s.T + db.splits - 1) / db.splits;
    // dZ and, from the same pass, db2 = its column sums
    TPMLP_CUDA(timed(TPMLP_KERNEL_DROPOUT_BWD, 2, st, [&] {
        return launch_dropout_backward(db, s.T, static_cast<float*>(db2), st);
    }));

    TPMLP_TRY(run_backward(s, dev, dz, xn, A_shards, B_shards, dxn, dA_shards, db1, dB_shards,
                           db2, regions_of(ws, L.blk), false, st, /*db2_given=*/true));

    LnBackwardParams lb;
    std::memset(&lb, 0, sizeof(lb));
    for (int j = 0; j < s.chunks; ++j) {
        lb.x.in[j] = X[j];
        lb.dxn[j] = dxn[j];
        lb.dres[j] = dOut[j];
        lb.dx[j] = dX[j];
    }
    lb.x.n = s.chunks;
    lb.x.rows = s.Tc;
    lb.gamma = gamma;
    lb.mean = reinterpret_cast<const float*>(ws + L.mean);
    lb.rstd = reinterpret_cast<const float*>(ws + L.rstd);
    lb.part = reinterpret_cast<float*>(ws + L.part);
    lb.h = s.h;
    const int splits = ln_param_splits(s.T, s.h, dev->sm_count);
    lb.rows_per_block = (s.T + splits - 1) / splits;
    TPMLP_CUDA(timed(TPMLP_KERNEL_LAYERNORM_BWD, ln_backward_launches(s.h), st, [&] {
        return launch_ln_backward(lb, s.T, splits, static_cast<float*>(dgamma),
                                  static_cast<float*>(dbeta), st);
    }));
    return TPMLP_OK;
}
