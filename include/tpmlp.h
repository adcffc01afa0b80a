/*
 * tpmlp.h -- C ABI of libtpmlp: the tensor-parallel Transformer MLP block,
 * forward and backward, on one sm_103 GPU, and the column- and row-parallel
 * linear layers it is made of (the attention projections).
 *
 *     Z = GeLU(X.A + b1).B + b2
 *
 * Sources (page title, section):
 *   [FGO]    "Megatron-LM：NVIDIA 的大规模并行训练方案", section
 *            "Megatron-LM 核心架构 / 张量并行原理": Y = XA; A split by
 *            columns [A_1, A_2] gives Y_i = X.A_i (column parallel); A split
 *            by rows with X split by columns gives Y = sum_i X_i.A_i summed by
 *            an AllReduce (row parallel); the MLP's first linear is column
 *            parallel and its second row parallel.
 *   [FGO-F]  same page, "融合优化技术": Bias + GeLU fused into one kernel.
 *   [FGO-SP] same page, "并行训练范式 / 序列并行": sequence parallelism on
 *            top of tensor parallelism, along the sequence dimension.
 *   [CH2]    "2、分布式训练基础：数据并行、模型并行、流水线并行的基本概念与区别",
 *            "2.2 模型并行 —— 张量并行 / 核心原理": column-parallel split
 *            [W1, W2], row-parallel split [W1; W2] with X = [X1, X2] and an
 *            AllReduce sum.
 *
 * All t shards live on the one GPU; the row-parallel AllReduce of the
 * forward pass (and its conjugate in the backward pass) becomes an on-chip
 * split-K accumulation over the shards.  In the sequence-parallel variant X
 * and dZ arrive as seq_chunks token chunks and Z and dX leave in the same
 * chunking: the gather before the column-parallel GEMM is done by addressing
 * the chunks directly, the reduce-scatter after the row-parallel GEMM by the
 * split-K accumulation plus a row-to-chunk mapping in the GEMM's epilogue.
 *
 * Conventions for every call:
 *   - All matrices are dense, row-major, with the shapes given below.
 *     Notation: T = tokens, h = hidden, f = ffn, fi = f / t, Tc = T / seq_chunks.
 *   - All buffer pointers are DEVICE pointers on the current CUDA device,
 *     owned by the caller, 16-byte aligned.  The library never allocates
 *     or frees device memory during a forward/backward call.
 *   - Pointer-array arguments ("const void* const*") are HOST arrays of
 *     device pointers (one per shard or per chunk); the library copies the
 *     pointers during the call and does not keep the host array.
 *   - Calls are asynchronous on the given stream (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream).  A returned TPMLP_OK means the
 *     work was validated and enqueued; device-side failures (a bounded wait
 *     that expired) are reported by tpmlp_sync_check().
 *   - Validation failures return an error before anything is launched and
 *     leave every output untouched.  Nothing crosses the ABI as an exception.
 *   - Results are bitwise reproducible run to run (no atomics in any sum).
 *   - Thread-compatible: concurrent calls from several host threads are
 *     allowed on different streams with different workspaces.
 *
 * Requirements (else TPMLP_ERR_UNSUPPORTED): an sm_103 device; h and fi
 * multiples of 8; 1 <= t <= 8; 1 <= seq_chunks <= 8 dividing T, and, when
 * seq_chunks > 1, Tc a multiple of 128; T, h, f below 2^31.
 */
#ifndef TPMLP_H
#define TPMLP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TPMLP_OK = 0,
    TPMLP_ERR_INVALID_ARG = 1,  /* null pointer, bad dims, t mismatch */
    TPMLP_ERR_UNSUPPORTED = 2,  /* shape/alignment/device outside the requirements */
    TPMLP_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed */
    TPMLP_ERR_TIMEOUT = 4       /* a bounded device wait expired (see tpmlp_sync_check) */
} tpmlp_status;

typedef struct {
    int64_t tokens;      /* T: micro-batch x sequence rows, sequence-major */
    int64_t hidden;      /* h */
    int64_t ffn;         /* f */
    int32_t t;           /* tensor-parallel shards (1..8) */
    int32_t seq_chunks;  /* 1, or the sequence-parallel degree (normally t) */
} tpmlp_dims;

/* Bytes of device workspace a forward/backward pair needs: the saved
 * pre-activation Y and activation H (written by tpmlp_forward, read by
 * tpmlp_backward), the gradient dY (written and read by tpmlp_backward) and
 * the bias-gradient partial sums.  The caller allocates it (256-byte aligned
 * is best) and keeps it alive from the forward to the matching backward. */
size_t tpmlp_workspace_bytes(const tpmlp_dims* dims);

/* Byte offsets inside the workspace of Y, H and dY, each stored shard-major
 * as t blocks [T, fi] bf16 (shard i at offset + i*T*fi*2).  Any output may be
 * NULL.  Lets a caller inspect the saved activations. */
tpmlp_status tpmlp_workspace_layout(const tpmlp_dims* dims, size_t* y_offset,
                                    size_t* h_offset, size_t* dy_offset);

/* Forward pass ([FGO] 张量并行原理, [CH2] 2.2, [FGO-F] 融合优化技术):
 *   for each shard i:  Y_i = X.A_i + b1[i*fi:(i+1)*fi],  H_i = GeLU(Y_i)
 *   Z = (sum_i H_i.B_i) + b2          (b2 added once, after the shard sum)
 * GeLU is the tanh form 0.5 y (1 + tanh(sqrt(2/pi) (y + 0.044715 y^3))).
 *   X        [seq_chunks] chunks of [Tc, h] bf16 (chunk j = token rows j*Tc..)
 *   A_shards [t] shards of [h, fi] bf16   (column block i of A)
 *   b1       [f] bf16
 *   B_shards [t] shards of [fi, h] bf16   (row block i of B)
 *   b2       [h] bf16
 *   t        must equal dims->t
 *   Z        [seq_chunks] chunks of [Tc, h] bf16 (output)
 *   workspace  >= tpmlp_workspace_bytes(dims) bytes; Y and H are saved there
 * Products accumulate in fp32 on the tensor cores; bias and GeLU are applied
 * in fp32 in the GEMM epilogue; Y, H and Z are rounded to bf16 once. */
tpmlp_status tpmlp_forward(const tpmlp_dims* dims,
                           const void* const* X,
                           const void* const* A_shards, const void* b1,
                           const void* const* B_shards, const void* b2,
                           int t,
                           void* const* Z,
                           void* workspace, void* stream);

/* Backward pass: the chain rule of tpmlp_forward for upstream gradient dZ.
 *   dY_i = (dZ.B_i^T) * GeLU'(Y_i)   (kept in the workspace, bf16)
 *   dX   = sum_i dY_i.A_i^T          (the backward AllReduce, on chip)
 *   dA_i = X^T.dY_i,  dB_i = H_i^T.dZ,
 *   db1  = column sums of dY, db2 = column sums of dZ.
 *   dZ        [seq_chunks] chunks of [Tc, h] bf16
 *   X, A_shards, B_shards   as passed to tpmlp_forward
 *   workspace the workspace of the matching tpmlp_forward (Y, H read; dY written)
 *   dX        [seq_chunks] chunks of [Tc, h] bf16 (output)
 *   dA_shards [t] of [h, fi] fp32 (output, overwritten)
 *   db1       [f] fp32 (output, overwritten)
 *   dB_shards [t] of [fi, h] fp32 (output, overwritten)
 *   db2       [h] fp32 (output, overwritten)
 * With T = 0 the weight and bias gradients are set to zero. */
tpmlp_status tpmlp_backward(const tpmlp_dims* dims,
                            const void* const* dZ,
                            const void* const* X,
                            const void* const* A_shards,
                            const void* const* B_shards,
                            void* workspace,
                            void* const* dX,
                            void* const* dA_shards, void* db1,
                            void* const* dB_shards, void* db2,
                            void* stream);

/* Selective recompute ("融合优化技术" and "高级特性 / 选择性激活重计算" on
 * "Megatron-LM：NVIDIA 的大规模并行训练方案": keep part of the activations,
 * recompute the rest in the backward pass).  Same block, same results for
 * Z, dX, dA, db1 and db2 (bitwise); dB is computed from H = GeLU(Y) rebuilt
 * from the saved bf16 Y, so it may differ from tpmlp_backward's in the last
 * bits.  Only Y (T x f bf16) is kept between the forward and the backward
 * pass ("saved", per layer); H, dY and the partial sums live in "scratch",
 * which holds nothing between calls and can be shared by all layers that run
 * on one stream.  The dH GEMM's epilogue rebuilds H from Y as it computes dY.
 *   saved   >= *saved_bytes device bytes: written by the forward, read by the backward
 *   scratch >= *scratch_bytes device bytes: used during either call only
 * Other arguments, layouts and errors as tpmlp_forward / tpmlp_backward. */
tpmlp_status tpmlp_recompute_workspace_bytes(const tpmlp_dims* dims, size_t* saved_bytes,
                                             size_t* scratch_bytes);
tpmlp_status tpmlp_forward_recompute(const tpmlp_dims* dims,
                                     const void* const* X,
                                     const void* const* A_shards, const void* b1,
                                     const void* const* B_shards, const void* b2,
                                     int t,
                                     void* const* Z,
                                     void* saved, void* scratch, void* stream);
tpmlp_status tpmlp_backward_recompute(const tpmlp_dims* dims,
                                      const void* const* dZ,
                                      const void* const* X,
                                      const void* const* A_shards,
                                      const void* const* B_shards,
                                      void* saved, void* scratch,
                                      void* const* dX,
                                      void* const* dA_shards, void* db1,
                                      void* const* dB_shards, void* db2,
                                      void* stream);

/* ---- Tensor-parallel linear layers ------------------------------------------
 * The two halves of the block without the GeLU, as the attention projections
 * use them ([CH2] 2.2: the QKV projection is column parallel, the output
 * projection row parallel; [FGO] 张量并行原理).  Same kernels, conventions,
 * sequence-parallel chunking and error behaviour as tpmlp_forward /
 * tpmlp_backward.  Notation: T = tokens, in = in_features, out =
 * out_features, Tc = T / seq_chunks.
 *
 * Requirements (else TPMLP_ERR_UNSUPPORTED) as for the block, with:
 *   column parallel: t divides out (else TPMLP_ERR_INVALID_ARG); in and
 *                    oi = out / t multiples of 8;
 *   row parallel:    t divides in (else TPMLP_ERR_INVALID_ARG); ii = in / t
 *                    and out multiples of 8.
 * The workspace holds only scratch (tail-split partial tiles, bias-gradient
 * partial sums); nothing in it lives from one call to the next, so one
 * workspace may serve every linear layer that runs on one stream. */
typedef struct {
    int64_t tokens;        /* T */
    int64_t in_features;   /* in: K of the forward product */
    int64_t out_features;  /* out: N of the forward product */
    int32_t t;             /* shards (1..8): of out (column) or of in (row) */
    int32_t seq_chunks;    /* 1, or the sequence-parallel degree */
} tpmlp_linear_dims;

/* Bytes of scratch workspace any linear-layer call with these dims needs. */
size_t tpmlp_linear_workspace_bytes(const tpmlp_linear_dims* dims);

/* Column-parallel forward:  Y_i = X.W_i + b[i*oi:(i+1)*oi]
 *   X        [seq_chunks] chunks of [Tc, in] bf16 (gathered on the fly)
 *   W_shards [t] of [in, oi] bf16 (column block i of W)
 *   b        [out] bf16
 *   Y_shards [t] of [T, oi] bf16 (output)
 * Backward for upstream dY_i:
 *   dX = sum_i dY_i.W_i^T  (on-chip shard sum; written back in chunks)
 *   dW_i = X^T.dY_i,  db = column sums of [dY_1 .. dY_t]
 *   dY_shards [t] of [T, oi] bf16;  X, W_shards as in the forward
 *   dX        [seq_chunks] chunks of [Tc, in] bf16 (output)
 *   dW_shards [t] of [in, oi] fp32 (output, overwritten)
 *   db        [out] fp32 (output, overwritten)
 * With T = 0 the forward does nothing and the backward zeroes dW and db. */
tpmlp_status tpmlp_column_linear_forward(const tpmlp_linear_dims* dims,
                                         const void* const* X,
                                         const void* const* W_shards, const void* b,
                                         void* const* Y_shards,
                                         void* workspace, void* stream);
tpmlp_status tpmlp_column_linear_backward(const tpmlp_linear_dims* dims,
                                          const void* const* dY_shards,
                                          const void* const* X,
                                          const void* const* W_shards,
                                          void* const* dX,
                                          void* const* dW_shards, void* db,
                                          void* workspace, void* stream);

/* Row-parallel forward:  Z = (sum_i X_i.W_i) + b   (b added once, after the
 * shard sum -- the AllReduce of [CH2] 2.2 done on chip)
 *   X_shards [t] of [T, ii] bf16 (column block i of the input)
 *   W_shards [t] of [ii, out] bf16 (row block i of W)
 *   b        [out] bf16
 *   Z        [seq_chunks] chunks of [Tc, out] bf16 (output, reduce-scattered)
 * Backward for upstream dZ:
 *   dX_i = dZ.W_i^T,  dW_i = X_i^T.dZ,  db = column sums of dZ
 *   dZ        [seq_chunks] chunks of [Tc, out] bf16;  X_shards, W_shards as in the forward
 *   dX_shards [t] of [T, ii] bf16 (output)
 *   dW_shards [t] of [ii, out] fp32 (output, overwritten)
 *   db        [out] fp32 (output, overwritten)
 * With T = 0 the forward does nothing and the backward zeroes dW and db. */
tpmlp_status tpmlp_row_linear_forward(const tpmlp_linear_dims* dims,
                                      const void* const* X_shards,
                                      const void* const* W_shards, const void* b,
                                      void* const* Z,
                                      void* workspace, void* stream);
tpmlp_status tpmlp_row_linear_backward(const tpmlp_linear_dims* dims,
                                       const void* const* dZ,
                                       const void* const* X_shards,
                                       const void* const* W_shards,
                                       void* const* dX_shards,
                                       void* const* dW_shards, void* db,
                                       void* workspace, void* stream);

/* ---- Sequence-parallel LayerNorm / Dropout sublayer ---------------------------
 * "Megatron-LM：NVIDIA 的大规模并行训练方案", "并行训练范式 / 序列并行": on top
 * of tensor parallelism, LayerNorm and Dropout are distributed along the
 * sequence dimension, each rank working on its token chunk.  The sublayer
 * around the block is the pre-LayerNorm residual block
 *
 *   Out = X + Dropout(MLP(LN(X)))
 *   LN(X) = (X - mean) * rstd * gamma + beta per token row over h,
 *           mean and var the row's mean and (biased) variance, rstd = 1/sqrt(var + eps)
 *   Dropout(z) = keep ? z / (1 - p) : 0
 *
 * keep for element (r, n) of the [T, h] output, e = r * h + n (r the token
 * row over all chunks): Philox4x32-10 (Salmon, Moraes, Dror and Shaw,
 * "Parallel random numbers: as easy as 1, 2, 3", SC'11) with key
 * (seed_lo, seed_hi) and counter (lo, hi, 0, 0) of offset + e / 4; word e % 4
 * of its output is compared with floor((1 - p) * 2^32) (keep iff below).
 * The same element keeps the same mask in the forward and the backward call.
 *
 * The forward pass runs LN per token chunk, then the block on LN(X) with the
 * dropout and the residual add fused into the row GEMM's epilogue, which also
 * stores the mask as bits in the workspace; the backward pass undoes the
 * dropout on dOut from those bits (summing dZ's columns into db2 on the way),
 * runs the block's backward pass, then LN's backward with the residual
 * gradient dOut added:
 *   dX = LN'(dXn) + dOut,  dgamma = sum_r dXn * xhat,  dbeta = sum_r dXn
 * Layouts, chunking, conventions and errors as tpmlp_forward / tpmlp_backward,
 * with h <= 16384 (else TPMLP_ERR_UNSUPPORTED), eps >= 0 and 0 <= p < 1
 * (else TPMLP_ERR_INVALID_ARG).  gamma, beta [h] bf16; dgamma, dbeta [h] fp32.
 * The workspace (tpmlp_sp_workspace_bytes) holds the block's workspace plus
 * LN(X), the row statistics, the dropout mask's bits (T x ceil(h / 32) 32-bit
 * words), dZ and the gradient of LN(X); it must be kept from the forward call
 * to the matching backward call. */
typedef struct {
    float eps;           /* LayerNorm epsilon (e.g. 1e-5) */
    double dropout_p;    /* probability of dropping an element, 0 <= p < 1 */
    uint64_t seed;       /* Philox key */
    uint64_t offset;     /* Philox counter offset, in blocks of 4 elements */
} tpmlp_sp_params;

size_t tpmlp_sp_workspace_bytes(const tpmlp_dims* dims);
/* Byte offsets in that workspace of LN(X) and of dZ (= dOut with the dropout
 * undone, written by tpmlp_sp_backward), each a [T, h] bf16 tensor stored
 * chunk after chunk.  Either output may be NULL. */
tpmlp_status tpmlp_sp_workspace_layout(const tpmlp_dims* dims, size_t* xn_offset,
                                       size_t* dz_offset);
tpmlp_status tpmlp_sp_forward(const tpmlp_dims* dims, const tpmlp_sp_params* sp,
                              const void* const* X, const void* gamma, const void* beta,
                              const void* const* A_shards, const void* b1,
                              const void* const* B_shards, const void* b2, int t,
                              void* const* Out, void* workspace, void* stream);
tpmlp_status tpmlp_sp_backward(const tpmlp_dims* dims, const tpmlp_sp_params* sp,
                               const void* const* dOut, const void* const* X,
                               const void* gamma, const void* const* A_shards,
                               const void* const* B_shards, void* workspace,
                               void* const* dX, void* dgamma, void* dbeta,
                               void* const* dA_shards, void* db1,
                               void* const* dB_shards, void* db2, void* stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char* tpmlp_status_string(tpmlp_status s);

/* Synchronises the stream, then reports: TPMLP_ERR_CUDA if a CUDA error is
 * pending, TPMLP_ERR_TIMEOUT if a kernel of this library gave up on a bounded
 * wait since the last check (the device error word is then cleared), else
 * TPMLP_OK.  Kernels that time out stop early, leave their outputs
 * incomplete, release their tensor memory and return; the context stays
 * usable. */
tpmlp_status tpmlp_sync_check(void* stream);

/* Tail split of the GEMMs.  When a GEMM's output tiles do not fill the last
 * wave of CTA pairs, the K ranges of the leftover tiles are split across the
 * pairs that would otherwise idle; each part writes an fp32 partial tile into
 * the workspace and the last part to finish sums them in a fixed order (the
 * result stays bitwise reproducible) before the fused epilogue.  This is done
 * only for tiles at least `kblocks` 64-deep K steps long (default 128); 0
 * turns it off.  Affects launches enqueued after the call. */
tpmlp_status tpmlp_set_split_min_kblocks(int kblocks);

/* Head prefetch of the GEMMs: when a CTA pair starts a tile, it asks L2 for
 * the first `kblocks` 64-deep K steps of its next tile's operands, a whole
 * tile ahead of the loads that use them.  Helps GEMMs with short K ranges per
 * tile (the weight gradients, K = tokens), whose tile starts otherwise wait for
 * data fetched from DRAM; costs one extra TMA instruction per prefetched box.
 * 0 turns it off; 0..64, else TPMLP_ERR_INVALID_ARG.  Results do not depend on
 * it.  Affects launches enqueued after the call. */
tpmlp_status tpmlp_set_head_prefetch(int kblocks);

/* Tile width of the GEMMs with bf16 outputs (every GEMM but the weight
 * gradients).  A CTA pair computes either 256 x 256 output tiles (two
 * accumulators in tensor memory: a tile's epilogue runs under the next
 * tile's MMAs) or 256 x 512 tiles (one accumulator in two halves, K steps in
 * three phases so each half drains under MMAs on the other), which move a
 * quarter fewer operand bytes from L2 per FLOP.  mode 0 always 256; 1 picks
 * 512 where its tiles fill the GPU's waves at least as well as 256-wide ones;
 * 2 always 512; 3 (default) picks 512 for GEMMs of at least 256 K steps of 64
 * (summed over the row-parallel shards), where the one-half phases are a
 * small share and the lower operand traffic lowers the power drawn.  0 to 3,
 * else TPMLP_ERR_INVALID_ARG.  Half 0 of a wide tile sums K in the narrow
 * tile's order (bitwise equal columns); half 1 starts its sum further along K
 * (equal within rounding).  Affects launches enqueued after the call. */
tpmlp_status tpmlp_set_wide_tiles(int mode);

/* TMA tensor-map cache.  Every call encodes one tensor map per operand shard,
 * token chunk and output of each GEMM it launches; the library keeps the
 * encoded maps in a cache keyed by every argument of the encoding (base
 * address, element type, extents, strides, box, swizzle), so a repeated call
 * on the same buffers encodes nothing.  A buffer at a new address is a new key
 * (a stale entry is never used for another address).  At most 4096 maps are
 * kept; when the cache is full it is emptied.  Thread-safe (one mutex).
 * tpmlp_map_cache_stats reports the hits, misses (encodings) and entries so
 * far; any pointer may be NULL.  Always TPMLP_OK. */
tpmlp_status tpmlp_map_cache_stats(uint64_t* hits, uint64_t* misses, uint64_t* entries);

/* Self-test of the cache logic on the host (no GPU, no driver): runs a fixed
 * sequence against a private cache of capacity 4 with a stand-in encoder and
 * writes out[0..7] = hits, misses, encoder calls, final entries, 1 if a hit
 * returned the bytes of the first encoding, 1 if a new address gave another
 * map, the capacity, and the key size in bytes.  n >= 8, else
 * TPMLP_ERR_INVALID_ARG. */
tpmlp_status tpmlp_selftest_map_cache(uint64_t* out, int n);

/* Upper bound, in nanoseconds, on any single wait inside a kernel of this
 * library (default 2e9).  Affects launches enqueued after the call. */
tpmlp_status tpmlp_set_wait_timeout_ns(uint64_t ns);

/* Failure-detection self-test.  Runs one 128 x 256 x 64 GEMM tile whose
 * loader deliberately issues no loads, so the tensor-core issuer's wait on
 * its first stage can only end by the bounded-wait limit; the kernel then
 * records the timeout, drains, frees its tensor memory and returns.
 *   a  [128, 64] bf16 device buffer, b [256, 64] bf16, c [128, 256] bf16
 *   (valid buffers of at least those sizes; c may be partially written).
 * Synchronises the stream and returns what tpmlp_sync_check returns:
 * TPMLP_ERR_TIMEOUT when the failure was detected as designed. */
tpmlp_status tpmlp_selftest_stalled_gemm(const void* a, const void* b, void* c,
                                         uint64_t timeout_ns, void* stream);

/* Explicit sequence-parallel gather and scatter ("Megatron-LM：NVIDIA 的大规模
 * 并行训练方案", 并行训练范式 / 序列并行: the tensor-parallel block gathers the
 * sequence chunks before its column-parallel GEMM and reduce-scatters its
 * output to them after the row-parallel GEMM).  tpmlp_forward / tpmlp_backward
 * do both without copies, through one tensor map per chunk and an epilogue that
 * writes each row into its chunk; these calls make the copies explicit.
 *   tpmlp_sp_gather:  out[T, cols] = concatenation along tokens of the
 *                     dims->seq_chunks chunks [T / seq_chunks, cols]
 *   tpmlp_sp_scatter: chunk j = rows [j T / seq_chunks, (j + 1) T / seq_chunks)
 *                     of in[T, cols]
 * bf16 (any 2-byte element), row-major, cols a multiple of 8 (else
 * TPMLP_ERR_UNSUPPORTED), 16-byte-aligned device pointers, at most 8 chunks;
 * dims->tokens and dims->seq_chunks are read, the rest of dims is not.  One
 * kernel on `stream`, asynchronous; nothing is allocated. */
tpmlp_status tpmlp_sp_gather(const tpmlp_dims* dims, const void* const* chunks, int64_t cols,
                             void* out, void* stream);
tpmlp_status tpmlp_sp_scatter(const tpmlp_dims* dims, const void* in, int64_t cols,
                              void* const* chunks, void* stream);

/* Column sums of one bf16 matrix [rows, cols] into fp32 out[cols] -- the
 * reduction tpmlp_backward uses for its bias gradients (db2 is the column
 * sums of dZ) -- for callers that cannot allocate device memory.  The pages
 * have no counterpart to this call; it exists for the library's users.
 *
 * Who needs it: tpmlp_backward takes its scratch from a caller-allocated
 * workspace.  A caller embedded in another runtime whose device memory is
 * owned by that runtime's pool cannot add a cudaMalloc of its own (it would
 * escape the pool's budget, and cudaFree synchronises the whole device); a
 * latency-critical loop may forbid allocation after start-up.  This call
 * allocates nothing: it keeps its partial sums in a static 4 MiB device
 * array (1,048,576 floats) inside the library, which every GPU that loads the
 * library holds until the process exits.
 *   src   device bf16 [rows, cols], row-major, 16-byte aligned
 *   rows  >= 0 (rows = 0 writes zeros), below 2^31
 *   cols  multiple of 8, at most 1,048,576; larger returns TPMLP_ERR_UNSUPPORTED
 *   out   device fp32 [cols], 16-byte aligned, overwritten
 * The first call on a device does a one-time set-up (looks up the array's
 * device address); make that first call before any stream capture.  All
 * calls on a device share the array and the last call's contents stay in it;
 * nothing in it needs clearing, but calls that overlap on the GPU (unordered
 * streams) race on it.  Asynchronous on `stream`, like every other call. */
tpmlp_status tpmlp_column_sums_noalloc(const void* src, int64_t rows, int64_t cols, void* out,
                                       void* stream);

/* Kernel-level timing.  Between tpmlp_profile_begin and tpmlp_profile_end
 * the library records a CUDA event pair on the launch stream around each of
 * its kernel launches (at most `capacity` launches).  tpmlp_profile_end
 * synchronises on those events and writes, for each kernel kind k <
 * nkinds, the summed milliseconds ms[k] and the launch count launches[k];
 * it returns the number of launches recorded, or -1 on error. */
enum {
    TPMLP_KERNEL_COLUMN_FWD = 0,  /* Y_i = X.A_i + b1, H_i = GeLU(Y_i) */
    TPMLP_KERNEL_ROW_FWD = 1,     /* Z = sum_i H_i.B_i + b2 */
    TPMLP_KERNEL_DGRAD_H = 2,     /* dY_i = (dZ.B_i^T) * GeLU'(Y_i) */
    TPMLP_KERNEL_DGRAD_X = 3,     /* dX = sum_i dY_i.A_i^T */
    TPMLP_KERNEL_WGRAD_B = 4,     /* dB_i = H_i^T.dZ */
    TPMLP_KERNEL_WGRAD_A = 5,     /* dA_i = X^T.dY_i */
    TPMLP_KERNEL_BIAS_GRAD = 6,   /* db1, db2, linear db column sums (all launches) */
    TPMLP_KERNEL_LINEAR_FWD = 7,  /* linear layers: Y_i = X.W_i + b, Z = sum_i X_i.W_i + b */
    TPMLP_KERNEL_LINEAR_DGRAD = 8,  /* linear layers: dX = sum_i dY_i.W_i^T, dX_i = dZ.W_i^T */
    TPMLP_KERNEL_LINEAR_WGRAD = 9,  /* linear layers: dW_i */
    TPMLP_KERNEL_LAYERNORM_FWD = 10,  /* sequence-parallel sublayer: LN(X) and row statistics */
    TPMLP_KERNEL_LAYERNORM_BWD = 11,  /* sequence-parallel sublayer: dX, dgamma, dbeta (2 launches; 3 for h > 4096) */
    TPMLP_KERNEL_DROPOUT_BWD = 12,    /* sequence-parallel sublayer: dZ from dOut and the mask, db2 (2 launches) */
    TPMLP_KERNEL_SP_COPY = 13,        /* tpmlp_sp_gather / tpmlp_sp_scatter */
    TPMLP_KERNEL_KINDS = 14
};
tpmlp_status tpmlp_profile_begin(int capacity);
/* The same, with event pairs only around the launches of the kernel kinds
 * whose bits are set in `kinds` (bit k = kind k): timing one kind costs the
 * others no event records.  TPMLP_ERR_INVALID_ARG for capacity <= 0, kinds
 * == 0 or a bit at or above TPMLP_KERNEL_KINDS. */
tpmlp_status tpmlp_profile_begin_kinds(int capacity, uint32_t kinds);
int tpmlp_profile_end(double* ms, int* launches, int nkinds);
const char* tpmlp_kernel_name(int kind);

#ifdef __cplusplus
}
#endif

#endif /* TPMLP_H */
