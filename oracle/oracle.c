/*
 * oracle.c -- fp64 CPU oracle for the tensor-parallel Transformer MLP block
 *
 *     Z = GeLU(X.A + b1).B + b2,  A split by columns into t shards, B by rows.
 *
 * TEST INFRASTRUCTURE.  This file is the slow, obviously correct definition
 * the CUDA path is checked against.  Only the test suite, the smoke check and
 * the benchmark's CPU-baseline leg may load it.  It shares no code, header,
 * table or helper with the CUDA library, and it never calls into it.
 *
 * Sources (page title, section):
 *   [FGO]  "Megatron-LM：NVIDIA 的大规模并行训练方案" (freeguideonline.com),
 *          section "Megatron-LM 核心架构 / 张量并行原理" (column split,
 *          row split, MLP = column then row) and "融合优化技术" (Bias+GeLU).
 *   [CH2]  "2、分布式训练基础：数据并行、模型并行、流水线并行的基本概念与区别",
 *          section "2.2 模型并行 —— 张量并行 / 核心原理" (Y = XW, column and
 *          row parallel linear layers).
 *   [FGO-SP] same page as [FGO], section "并行训练范式 / 序列并行".
 *
 * Everything is fp64.  Inputs are whatever values the caller passes (the
 * tests pass the exact bf16 values upcast to double).  Matrices are dense
 * row-major.  Shard i of A is the column block A[:, i*fi:(i+1)*fi] stored as
 * its own [h, fi] array; shard i of B is the row block B[i*fi:(i+1)*fi, :]
 * stored as its own [fi, h] array; fi = f / t.
 *
 * Readings where the pages are silent (each one is listed in the design
 * notes):
 *   - "GeLU" is the tanh form of Hendrycks & Gimpel (2016):
 *       GeLU(x) = x/2 * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3))).
 *   - b2 is added once, after the shard partial products are summed (after
 *     the row-parallel "AllReduce" of [FGO]/[CH2]); b1 is one [f] vector whose
 *     slice [i*fi, (i+1)*fi) belongs to shard i.
 *   - The backward pass is the chain rule of this forward pass (the pages do
 *     not write it down): with dZ = dL/dZ,
 *       dH_i = dZ.B_i^T, dY_i = dH_i * GeLU'(Y_i), dX = sum_i dY_i.A_i^T,
 *       dA_i = X^T.dY_i, dB_i = H_i^T.dZ, db1 = column sums of dY,
 *       db2 = column sums of dZ.
 *
 *   - The attention projections are the same two halves without the GeLU
 *     ([CH2] 2.2: the QKV projection column parallel, the output projection
 *     row parallel); their biases follow the same placement as b1 and b2.
 *     Pinned by tests/test_oracle_linear_pins.py.
 *   - Sequence parallelism places LayerNorm and Dropout on each rank's token
 *     chunk ([FGO-SP]); the sublayer around the block is read as the usual
 *     pre-LayerNorm residual block Out = X + Dropout(MLP(LN(X))), LayerNorm
 *     with the biased variance and eps, Dropout with a Philox4x32-10 mask
 *     (details at oracle_dropout_keep).  Pinned by tests/test_oracle_sp_pins.py.
 *
 * Parallelism: OpenMP over output rows only; every output element is a
 * plain sum taken in index order.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- threads ----------------------------------------------------------- */

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_get_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- GeLU, tanh form ----------------------------------------------------
 * u(x) = sqrt(2/pi) * (x + 0.044715 x^3)
 * GeLU(x)  = 0.5 x (1 + tanh u)
 * GeLU'(x) = 0.5 (1 + tanh u) + 0.5 x (1 - tanh^2 u) du/dx,
 *            du/dx = sqrt(2/pi) * (1 + 3 * 0.044715 x^2)
 */
static double gelu_k0(void) { return sqrt(2.0 / acos(-1.0)); }
static const double GELU_K1 = 0.044715;

double oracle_gelu(double x) {
    double u = gelu_k0() * (x + GELU_K1 * x * x * x);
    return 0.5 * x * (1.0 + tanh(u));
}

double oracle_gelu_grad(double x) {
    double k0 = gelu_k0();
    double u = k0 * (x + GELU_K1 * x * x * x);
    double th = tanh(u);
    double du = k0 * (1.0 + 3.0 * GELU_K1 * x * x);
    return 0.5 * (1.0 + th) + 0.5 * x * (1.0 - th * th) * du;
}

/* ---- forward ------------------------------------------------------------
 * Column-parallel first linear ([CH2] 2.2 column split, [FGO] 张量并行原理):
 *   for each shard i:  Y_i = X.A_i + b1[i*fi:(i+1)*fi],  H_i = GeLU(Y_i)
 *   (bias and GeLU applied together, [FGO] 融合优化技术)
 * Row-parallel second linear ([CH2] 2.2 row split):
 *   Z = (sum_i H_i.B_i) + b2
 * Outputs: Y[i], H[i] are [T, fi]; Z is [T, h].
 */
void oracle_forward(int64_t T, int64_t h, int64_t f, int t,
                    const double *X,
                    const double *const *A, const double *b1,
                    const double *const *B, const double *b2,
                    double *const *Y, double *const *H, double *Z) {
    const int64_t fi = f / t;
    for (int i = 0; i < t; ++i) {
        const double *Ai = A[i];
        double *Yi = Y[i], *Hi = H[i];
        #pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < T; ++r) {
            double *yrow = Yi + r * fi;
            for (int64_t j = 0; j < fi; ++j) yrow[j] = 0.0;
            for (int64_t k = 0; k < h; ++k) {
                const double x = X[r * h + k];
                const double *arow = Ai + k * fi;
                for (int64_t j = 0; j < fi; ++j) yrow[j] += x * arow[j];
            }
            for (int64_t j = 0; j < fi; ++j) {
                yrow[j] += b1[i * fi + j];
                Hi[r * fi + j] = oracle_gelu(yrow[j]);
            }
        }
    }
    /* row-parallel partial products, summed over shards (the on-chip stand-in
     * for the AllReduce), then the bias once */
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < T; ++r) {
        double *zrow = Z + r * h;
        for (int64_t n = 0; n < h; ++n) zrow[n] = 0.0;
        for (int i = 0; i < t; ++i) {
            const double *Hi = H[i], *Bi = B[i];
            for (int64_t j = 0; j < fi; ++j) {
                const double hv = Hi[r * fi + j];
                const double *brow = Bi + j * h;
                for (int64_t n = 0; n < h; ++n) zrow[n] += hv * brow[n];
            }
        }
        for (int64_t n = 0; n < h; ++n) zrow[n] += b2[n];
    }
}

/* ---- backward -----------------------------------------------------------
 * Chain rule of oracle_forward for upstream gradient dZ = dL/dZ [T, h]:
 *   dH_i = dZ.B_i^T                   [T, fi]
 *   dY_i = dH_i * GeLU'(Y_i)          [T, fi]   (written to dY[i])
 *   dX   = sum_i dY_i.A_i^T           [T, h]    (sum over shards, as the
 *                                                 backward AllReduce)
 *   dA_i = X^T.dY_i                   [h, fi]
 *   dB_i = H_i^T.dZ                   [fi, h]
 *   db1[i*fi + j] = sum_r dY_i[r, j]  [f]
 *   db2[n] = sum_r dZ[r, n]           [h]
 */
void oracle_backward(int64_t T, int64_t h, int64_t f, int t,
                     const double *X,
                     const double *const *A, const double *const *B,
                     const double *const *Y, const double *const *H,
                     const double *dZ,
                     double *const *dY, double *dX,
                     double *const *dA, double *db1,
                     double *const *dB, double *db2) {
    const int64_t fi = f / t;
    /* dY_i */
    for (int i = 0; i < t; ++i) {
        const double *Bi = B[i], *Yi = Y[i];
        double *dYi = dY[i];
        #pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < T; ++r) {
            for (int64_t j = 0; j < fi; ++j) {
                double dh = 0.0;
                const double *brow = Bi + j * h;
                for (int64_t n = 0; n < h; ++n) dh += dZ[r * h + n] * brow[n];
                dYi[r * fi + j] = dh * oracle_gelu_grad(Yi[r * fi + j]);
            }
        }
    }
    /* dX = sum_i dY_i.A_i^T */
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < T; ++r) {
        for (int64_t k = 0; k < h; ++k) {
            double acc = 0.0;
            for (int i = 0; i < t; ++i) {
                const double *arow = A[i] + k * fi;
                const double *dyrow = dY[i] + r * fi;
                for (int64_t j = 0; j < fi; ++j) acc += dyrow[j] * arow[j];
            }
            dX[r * h + k] = acc;
        }
    }
    /* dA_i = X^T.dY_i */
    for (int i = 0; i < t; ++i) {
        const double *dYi = dY[i];
        double *dAi = dA[i];
        #pragma omp parallel for schedule(static)
        for (int64_t k = 0; k < h; ++k) {
            double *out = dAi + k * fi;
            for (int64_t j = 0; j < fi; ++j) out[j] = 0.0;
            for (int64_t r = 0; r < T; ++r) {
                const double x = X[r * h + k];
                const double *dyrow = dYi + r * fi;
                for (int64_t j = 0; j < fi; ++j) out[j] += x * dyrow[j];
            }
        }
    }
    /* dB_i = H_i^T.dZ */
    for (int i = 0; i < t; ++i) {
        const double *Hi = H[i];
        double *dBi = dB[i];
        #pragma omp parallel for schedule(static)
        for (int64_t j = 0; j < fi; ++j) {
            double *out = dBi + j * h;
            for (int64_t n = 0; n < h; ++n) out[n] = 0.0;
            for (int64_t r = 0; r < T; ++r) {
                const double hv = Hi[r * fi + j];
                const double *dzrow = dZ + r * h;
                for (int64_t n = 0; n < h; ++n) out[n] += hv * dzrow[n];
            }
        }
    }
    /* db1: column sums of dY, shard by shard */
    for (int i = 0; i < t; ++i) {
        const double *dYi = dY[i];
        for (int64_t j = 0; j < fi; ++j) {
            double s = 0.0;
            for (int64_t r = 0; r < T; ++r) s += dYi[r * fi + j];
            db1[i * fi + j] = s;
        }
    }
    /* db2: column sums of dZ */
    for (int64_t n = 0; n < h; ++n) {
        double s = 0.0;
        for (int64_t r = 0; r < T; ++r) s += dZ[r * h + n];
        db2[n] = s;
    }
}

/* ---- sampled outputs ----------------------------------------------------
 * The same definitions as above, evaluated only for selected outputs, so a
 * full-size problem can be checked one output at a time.
 *
 * oracle_rows: for each selected token row r = rows[q]:
 *   Zr[q, :]  = Z[r, :]   and   dXr[q, :] = dX[r, :]
 * (needs row r of Y_i, H_i and dY_i for every shard, computed here).  When
 * Yr, Hr, dYr are not NULL they receive those rows too, shard after shard:
 *   Yr[q, i*fi + j] = Y_i[r, j], likewise H_i and dY_i   ([nrows, f] each).
 */
void oracle_rows(int64_t T, int64_t h, int64_t f, int t,
                 const double *X,
                 const double *const *A, const double *b1,
                 const double *const *B, const double *b2,
                 const double *dZ,
                 int64_t nrows, const int64_t *rows,
                 double *Zr, double *dXr,
                 double *Yr, double *Hr, double *dYr) {
    const int64_t fi = f / t;
    (void)T;
    #pragma omp parallel for schedule(dynamic)
    for (int64_t q = 0; q < nrows; ++q) {
        const int64_t r = rows[q];
        double *z = Zr + q * h;
        double *dx = dXr + q * h;
        for (int64_t n = 0; n < h; ++n) { z[n] = 0.0; dx[n] = 0.0; }
        for (int i = 0; i < t; ++i) {
            const double *Ai = A[i], *Bi = B[i];
            for (int64_t j = 0; j < fi; ++j) {
                double y = 0.0;
                for (int64_t k = 0; k < h; ++k) y += X[r * h + k] * Ai[k * fi + j];
                y += b1[i * fi + j];
                const double hv = oracle_gelu(y);
                double dh = 0.0;
                for (int64_t n = 0; n < h; ++n) dh += dZ[r * h + n] * Bi[j * h + n];
                const double dy = dh * oracle_gelu_grad(y);
                for (int64_t n = 0; n < h; ++n) z[n] += hv * Bi[j * h + n];
                for (int64_t k = 0; k < h; ++k) dx[k] += dy * Ai[k * fi + j];
                if (Yr) Yr[q * f + i * fi + j] = y;
                if (Hr) Hr[q * f + i * fi + j] = hv;
                if (dYr) dYr[q * f + i * fi + j] = dy;
            }
        }
        for (int64_t n = 0; n < h; ++n) z[n] += b2[n];
    }
}

/* oracle_cols: for each selected ffn column c = cols[q] (global index in
 * [0, f), shard i = c / fi, local column j = c % fi):
 *   dAc[q, :] = dA_i[:, j]   (length h)
 *   dBc[q, :] = dB_i[j, :]   (length h)
 *   db1c[q]   = db1[c]
 * (needs column j of Y_i, H_i and dY_i over all T rows, computed here).
 */
void oracle_cols(int64_t T, int64_t h, int64_t f, int t,
                 const double *X,
                 const double *const *A, const double *b1,
                 const double *const *B,
                 const double *dZ,
                 int64_t ncols, const int64_t *cols,
                 double *dAc, double *dBc, double *db1c) {
    const int64_t fi = f / t;
    #pragma omp parallel for schedule(dynamic)
    for (int64_t q = 0; q < ncols; ++q) {
        const int64_t c = cols[q];
        const int i = (int)(c / fi);
        const int64_t j = c % fi;
        const double *Ai = A[i], *Bi = B[i];
        double *da = dAc + q * h;
        double *db = dBc + q * h;
        double s1 = 0.0;
        for (int64_t n = 0; n < h; ++n) { da[n] = 0.0; db[n] = 0.0; }
        for (int64_t r = 0; r < T; ++r) {
            double y = 0.0;
            for (int64_t k = 0; k < h; ++k) y += X[r * h + k] * Ai[k * fi + j];
            y += b1[c];
            const double hv = oracle_gelu(y);
            double dh = 0.0;
            for (int64_t n = 0; n < h; ++n) dh += dZ[r * h + n] * Bi[j * h + n];
            const double dy = dh * oracle_gelu_grad(y);
            for (int64_t k = 0; k < h; ++k) da[k] += X[r * h + k] * dy;
            for (int64_t n = 0; n < h; ++n) db[n] += hv * dZ[r * h + n];
            s1 += dy;
        }
        db1c[q] = s1;
    }
}

/* db2 alone (column sums of dZ), for full-size problems. */
void oracle_db2(int64_t T, int64_t h, const double *dZ, double *db2) {
    #pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < h; ++n) {
        double s = 0.0;
        for (int64_t r = 0; r < T; ++r) s += dZ[r * h + n];
        db2[n] = s;
    }
}

/* ---- tensor-parallel linear layers ------------------------------------------
 * The two halves of the block without the GeLU, as used for the attention
 * projections ([CH2] 2.2: QKV projection column parallel, output projection
 * row parallel; [FGO] 张量并行原理).  in = input width, out = output width.
 *
 * Column parallel, W split by columns into t shards W_i [in, oi], oi = out/t:
 *   Y_i = X.W_i + b[i*oi:(i+1)*oi]                     Y_i [T, oi]
 * backward for upstream dY_i:
 *   dX = sum_i dY_i.W_i^T, dW_i = X^T.dY_i, db = column sums of [dY_1..dY_t]
 */
void oracle_column_linear_forward(int64_t T, int64_t in, int64_t out, int t,
                                  const double *X, const double *const *W,
                                  const double *b, double *const *Y) {
    const int64_t oi = out / t;
    for (int i = 0; i < t; ++i) {
        const double *Wi = W[i];
        double *Yi = Y[i];
        #pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < T; ++r) {
            double *yrow = Yi + r * oi;
            for (int64_t j = 0; j < oi; ++j) yrow[j] = 0.0;
            for (int64_t k = 0; k < in; ++k) {
                const double x = X[r * in + k];
                const double *wrow = Wi + k * oi;
                for (int64_t j = 0; j < oi; ++j) yrow[j] += x * wrow[j];
            }
            for (int64_t j = 0; j < oi; ++j) yrow[j] += b[i * oi + j];
        }
    }
}

void oracle_column_linear_backward(int64_t T, int64_t in, int64_t out, int t,
                                   const double *X, const double *const *W,
                                   const double *const *dY, double *dX,
                                   double *const *dW, double *db) {
    const int64_t oi = out / t;
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < T; ++r) {
        for (int64_t k = 0; k < in; ++k) {
            double acc = 0.0;
            for (int i = 0; i < t; ++i) {
                const double *wrow = W[i] + k * oi;
                const double *dyrow = dY[i] + r * oi;
                for (int64_t j = 0; j < oi; ++j) acc += dyrow[j] * wrow[j];
            }
            dX[r * in + k] = acc;
        }
    }
    for (int i = 0; i < t; ++i) {
        const double *dYi = dY[i];
        double *dWi = dW[i];
        #pragma omp parallel for schedule(static)
        for (int64_t k = 0; k < in; ++k) {
            double *o = dWi + k * oi;
            for (int64_t j = 0; j < oi; ++j) o[j] = 0.0;
            for (int64_t r = 0; r < T; ++r) {
                const double x = X[r * in + k];
                const double *dyrow = dYi + r * oi;
                for (int64_t j = 0; j < oi; ++j) o[j] += x * dyrow[j];
            }
        }
        for (int64_t j = 0; j < oi; ++j) {
            double s = 0.0;
            for (int64_t r = 0; r < T; ++r) s += dYi[r * oi + j];
            db[i * oi + j] = s;
        }
    }
}

/* Row parallel, W split by rows into t shards W_i [ii, out], ii = in/t, and
 * the input split by columns into X_i [T, ii]:
 *   Z = (sum_i X_i.W_i) + b                            Z [T, out]
 * backward for upstream dZ:
 *   dX_i = dZ.W_i^T, dW_i = X_i^T.dZ, db = column sums of dZ
 */
void oracle_row_linear_forward(int64_t T, int64_t in, int64_t out, int t,
                               const double *const *X, const double *const *W,
                               const double *b, double *Z) {
    const int64_t ii = in / t;
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < T; ++r) {
        double *zrow = Z + r * out;
        for (int64_t n = 0; n < out; ++n) zrow[n] = 0.0;
        for (int i = 0; i < t; ++i) {
            for (int64_t k = 0; k < ii; ++k) {
                const double x = X[i][r * ii + k];
                const double *wrow = W[i] + k * out;
                for (int64_t n = 0; n < out; ++n) zrow[n] += x * wrow[n];
            }
        }
        for (int64_t n = 0; n < out; ++n) zrow[n] += b[n];
    }
}

void oracle_row_linear_backward(int64_t T, int64_t in, int64_t out, int t,
                                const double *const *X, const double *const *W,
                                const double *dZ, double *const *dX,
                                double *const *dW, double *db) {
    const int64_t ii = in / t;
    for (int i = 0; i < t; ++i) {
        const double *Wi = W[i], *Xi = X[i];
        double *dXi = dX[i], *dWi = dW[i];
        #pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < T; ++r) {
            for (int64_t k = 0; k < ii; ++k) {
                double acc = 0.0;
                const double *wrow = Wi + k * out;
                for (int64_t n = 0; n < out; ++n) acc += dZ[r * out + n] * wrow[n];
                dXi[r * ii + k] = acc;
            }
        }
        #pragma omp parallel for schedule(static)
        for (int64_t k = 0; k < ii; ++k) {
            double *o = dWi + k * out;
            for (int64_t n = 0; n < out; ++n) o[n] = 0.0;
            for (int64_t r = 0; r < T; ++r) {
                const double x = Xi[r * ii + k];
                const double *dzrow = dZ + r * out;
                for (int64_t n = 0; n < out; ++n) o[n] += x * dzrow[n];
            }
        }
    }
    for (int64_t n = 0; n < out; ++n) {
        double s = 0.0;
        for (int64_t r = 0; r < T; ++r) s += dZ[r * out + n];
        db[n] = s;
    }
}

/* ---- sequence-parallel LayerNorm / Dropout sublayer --------------------------
 * "在张量并行的基础上，LayerNorm 和 Dropout 沿序列维度分布" ([FGO-SP] 序列并行):
 * with sequence parallelism the LayerNorm before the column-parallel GEMM and
 * the Dropout after the row-parallel GEMM run on each rank's token chunk.  The
 * pages give no formula for the sublayer; the reading taken (the usual
 * pre-LayerNorm residual block) is
 *
 *   Xn  = LN(X) = (X - mean) * rstd * gamma + beta,   per token row, over h
 *         mean = sum_n X[n] / h,  var = sum_n (X[n] - mean)^2 / h,
 *         rstd = 1 / sqrt(var + eps)
 *   Z   = MLP(Xn)                      (the block above, b2 included)
 *   Out = X + Dropout(Z),  Dropout(z) = keep ? z / (1 - p) : 0
 *
 * keep for element (r, n) of the [T, h] output: Philox4x32-10 (Salmon, Moraes,
 * Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11) with
 * key (seed_lo, seed_hi) and counter (lo, hi, 0, 0) of c = offset + e / 4,
 * e = r * h + n; word e % 4 of the output u, and keep iff u < thresh, thresh =
 * floor((1 - p) * 2^32) (an integer in [0, 2^32]).
 */

static void philox_round(uint32_t *c, const uint32_t *k) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c[0];
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c[2];
    const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    const uint32_t n0 = hi1 ^ c[1] ^ k[0];
    const uint32_t n2 = hi0 ^ c[3] ^ k[1];
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
}

void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    uint32_t k[2] = {key[0], key[1]};
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k[0] += 0x9E3779B9u;
            k[1] += 0xBB67AE85u;
        }
        philox_round(c, k);
    }
    for (int i = 0; i < 4; ++i) out[i] = c[i];
}

/* keep[e] (0/1) for e in [0, count) of a [T, h] tensor starting at element e0 */
void oracle_dropout_keep(uint64_t seed, uint64_t offset, uint64_t thresh, int64_t e0,
                         int64_t count, uint8_t *keep) {
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    for (int64_t i = 0; i < count; ++i) {
        const uint64_t e = (uint64_t)(e0 + i);
        const uint64_t c = offset + e / 4;
        const uint32_t ctr[4] = {(uint32_t)c, (uint32_t)(c >> 32), 0u, 0u};
        uint32_t u[4];
        oracle_philox4x32_10(ctr, key, u);
        keep[i] = (uint64_t)u[e % 4] < thresh ? 1 : 0;
    }
}

/* LayerNorm forward over rows of X [T, h]: Xn, and the per-row mean and rstd */
void oracle_layernorm_forward(int64_t T, int64_t h, const double *X, const double *gamma,
                              const double *beta, double eps, double *Xn, double *mean,
                              double *rstd) {
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < T; ++r) {
        const double *x = X + r * h;
        double s = 0.0;
        for (int64_t n = 0; n < h; ++n) s += x[n];
        const double mu = s / (double)h;
        double v = 0.0;
        for (int64_t n = 0; n < h; ++n) v += (x[n] - mu) * (x[n] - mu);
        const double rs = 1.0 / sqrt(v / (double)h + eps);
        for (int64_t n = 0; n < h; ++n) Xn[r * h + n] = (x[n] - mu) * rs * gamma[n] + beta[n];
        mean[r] = mu;
        rstd[r] = rs;
    }
}

/* LayerNorm backward: dX from dXn, and dgamma, dbeta (column sums over rows)
 *   xhat = (x - mean) * rstd,  g = dXn * gamma,
 *   dX = rstd * (g - mean_n(g) - xhat * mean_n(g * xhat))
 *   dgamma = sum_r dXn * xhat,  dbeta = sum_r dXn */
void oracle_layernorm_backward(int64_t T, int64_t h, const double *X, const double *gamma,
                               const double *mean, const double *rstd, const double *dXn,
                               double *dX, double *dgamma, double *dbeta) {
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < T; ++r) {
        const double *x = X + r * h;
        const double *dy = dXn + r * h;
        double sg = 0.0, sgx = 0.0;
        for (int64_t n = 0; n < h; ++n) {
            const double xh = (x[n] - mean[r]) * rstd[r];
            const double g = dy[n] * gamma[n];
            sg += g;
            sgx += g * xh;
        }
        const double mg = sg / (double)h, mgx = sgx / (double)h;
        for (int64_t n = 0; n < h; ++n) {
            const double xh = (x[n] - mean[r]) * rstd[r];
            dX[r * h + n] = rstd[r] * (dy[n] * gamma[n] - mg - xh * mgx);
        }
    }
    for (int64_t n = 0; n < h; ++n) {
        double sgm = 0.0, sbt = 0.0;
        for (int64_t r = 0; r < T; ++r) {
            const double xh = (X[r * h + n] - mean[r]) * rstd[r];
            sgm += dXn[r * h + n] * xh;
            sbt += dXn[r * h + n];
        }
        dgamma[n] = sgm;
        dbeta[n] = sbt;
    }
}

/* ---- sampled rows of the sequence-parallel sublayer ---------------------
 * Out[r, :] and dX[r, :] of Out = X + Dropout(MLP(LN(X))) for the selected
 * token rows r = rows[q] of a [T, h] problem, with upstream gradient dOut.
 * Every quantity of a token row depends only on that row (LayerNorm is over
 * h, the mask of element (r, n) is fixed by its index r * h + n), so each row
 * is the composition, in order, of the definitions above applied to one row:
 *   LN forward of X[r]                     -> xn, mean, rstd
 *   keep[n] of element r * h + n
 *   dz = dOut[r] * keep * scale             (dropout backward)
 *   the block on the one-row input xn      -> z, dxn  (oracle_rows)
 *   Out[r] = X[r] + keep * scale * z
 *   LN backward of X[r] for dxn, plus dOut[r] (the residual path)
 * scale = 1 / (1 - p) and thresh = floor((1 - p) * 2^32) come from the caller.
 */
void oracle_sp_rows(int64_t T, int64_t h, int64_t f, int t,
                    const double *X, const double *gamma, const double *beta, double eps,
                    const double *const *A, const double *b1,
                    const double *const *B, const double *b2,
                    uint64_t seed, uint64_t offset, uint64_t thresh, double scale,
                    const double *dOut, int64_t nrows, const int64_t *rows,
                    double *Outr, double *dXr) {
    (void)T;
    #pragma omp parallel for schedule(dynamic)
    for (int64_t q = 0; q < nrows; ++q) {
        const int64_t r = rows[q];
        const double *xr = X + r * h;
        const double *dor = dOut + r * h;
        double *buf = (double *)malloc(sizeof(double) * (size_t)(7 * h + 2));
        uint8_t *keep = (uint8_t *)malloc((size_t)h);
        if (!buf || !keep) { free(buf); free(keep); continue; }
        double *xn = buf, *dz = buf + h, *zr = buf + 2 * h, *dxn = buf + 3 * h;
        double *dxl = buf + 4 * h, *dgb = buf + 5 * h;  /* this row's dgamma, dbeta (unused) */
        double *stats = buf + 7 * h;                     /* mean, rstd */
        const int64_t zero = 0;
        oracle_layernorm_forward(1, h, xr, gamma, beta, eps, xn, &stats[0], &stats[1]);
        oracle_dropout_keep(seed, offset, thresh, r * h, h, keep);
        for (int64_t n = 0; n < h; ++n) dz[n] = dor[n] * (double)keep[n] * scale;
        oracle_rows(1, h, f, t, xn, A, b1, B, b2, dz, 1, &zero, zr, dxn, NULL, NULL, NULL);
        for (int64_t n = 0; n < h; ++n) Outr[q * h + n] = xr[n] + (double)keep[n] * scale * zr[n];
        oracle_layernorm_backward(1, h, xr, gamma, &stats[0], &stats[1], dxn, dxl, dgb, dgb + h);
        for (int64_t n = 0; n < h; ++n) dXr[q * h + n] = dxl[n] + dor[n];
        free(buf);
        free(keep);
    }
}
