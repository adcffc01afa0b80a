"""Pins for the oracle's tensor-parallel linear layers, each against something
other than the oracle.

Sources (page title, section):
  [FGO] "Megatron-LM：NVIDIA 的大规模并行训练方案", "Megatron-LM 核心架构 / 张量并行原理"
  [CH2] "2、分布式训练基础：数据并行、模型并行、流水线并行的基本概念与区别",
        "2.2 模型并行 —— 张量并行 / 核心原理"

The attention projections of a tensor-parallel layer are the two halves of
the MLP block without the GeLU: the QKV projection is column parallel
(Y_i = X.W_i + b_i), the output projection row parallel
(Z = sum_i X_i.W_i + b).

What pins what:
  * small integer inputs, every output and gradient brute-forced with Python
    integer loops (exact, no numpy);
  * numpy float64 matmuls on random shapes;
  * the adjoint identities of a linear map: <dY, Y - b> = <dX, X> = <dW, W>;
  * sharding invariance: t shards give the same bits as one shard;
  * the MLP block is column linear -> GeLU -> row linear.
"""
import numpy as np
import pytest

import oracle

from test_oracle_pins import _gelu_np, _split_cols, _split_rows


def _int_mat(rng, r, c, lo=-4, hi=5):
    return rng.integers(lo, hi, size=(r, c)).astype(np.float64)


def _py_matmul(P, Q):
    """Exact integer product by plain loops."""
    P, Q = P.astype(np.int64).tolist(), Q.astype(np.int64).tolist()
    n, k, m = len(P), len(Q), len(Q[0]) if Q else 0
    return np.array([[sum(P[r][q] * Q[q][c] for q in range(k)) for c in range(m)]
                     for r in range(n)], dtype=np.float64).reshape(n, m)


def _py_colsum(P):
    P = P.astype(np.int64).tolist()
    return np.array([sum(row[c] for row in P) for c in range(len(P[0]))], dtype=np.float64)


@pytest.mark.parametrize("T,din,dout,t", [(3, 4, 6, 2), (5, 3, 9, 3), (4, 8, 8, 4)])
def test_column_linear_exact_integers(T, din, dout, t):
    rng = np.random.default_rng(T * 100 + t)
    X, W, dY = _int_mat(rng, T, din), _int_mat(rng, din, dout), _int_mat(rng, T, dout)
    b = rng.integers(-6, 7, size=dout).astype(np.float64)
    r = oracle.column_linear(X, _split_cols(W, t), b, _split_cols(dY, t))
    Y = _py_matmul(X, W) + b
    assert np.array_equal(np.concatenate(r["Y"], 1), Y)
    assert np.array_equal(r["dX"], _py_matmul(dY, W.T))
    assert np.array_equal(np.concatenate(r["dW"], 1), _py_matmul(X.T, dY))
    assert np.array_equal(r["db"], _py_colsum(dY))


@pytest.mark.parametrize("T,din,dout,t", [(3, 6, 4, 2), (5, 9, 3, 3), (4, 8, 8, 4)])
def test_row_linear_exact_integers(T, din, dout, t):
    rng = np.random.default_rng(T * 100 + t + 7)
    X, W, dZ = _int_mat(rng, T, din), _int_mat(rng, din, dout), _int_mat(rng, T, dout)
    b = rng.integers(-6, 7, size=dout).astype(np.float64)
    r = oracle.row_linear(_split_cols(X, t), _split_rows(W, t), b, dZ)
    assert np.array_equal(r["Z"], _py_matmul(X, W) + b)
    assert np.array_equal(np.concatenate(r["dX"], 1), _py_matmul(dZ, W.T))
    assert np.array_equal(np.concatenate(r["dW"], 0), _py_matmul(X.T, dZ))
    assert np.array_equal(r["db"], _py_colsum(dZ))


def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


@pytest.mark.parametrize("T,din,dout,t", [(17, 24, 36, 3), (9, 40, 16, 2)])
def test_linear_layers_against_numpy(T, din, dout, t):
    rng = np.random.default_rng(T + din)
    X, W = rng.standard_normal((T, din)), rng.standard_normal((din, dout))
    b, dY = rng.standard_normal(dout), rng.standard_normal((T, dout))
    c = oracle.column_linear(X, _split_cols(W, t), b, _split_cols(dY, t))
    assert _rel(np.concatenate(c["Y"], 1), X @ W + b) < 1e-13
    assert _rel(c["dX"], dY @ W.T) < 1e-13
    assert _rel(np.concatenate(c["dW"], 1), X.T @ dY) < 1e-13
    assert _rel(c["db"], dY.sum(0)) < 1e-13
    r = oracle.row_linear(_split_cols(X, t), _split_rows(W, t), b, dY)
    assert _rel(r["Z"], X @ W + b) < 1e-13
    assert _rel(np.concatenate(r["dX"], 1), dY @ W.T) < 1e-13
    assert _rel(np.concatenate(r["dW"], 0), X.T @ dY) < 1e-13
    assert _rel(r["db"], dY.sum(0)) < 1e-13


def test_adjoint_identities():
    rng = np.random.default_rng(21)
    T, din, dout, t = 11, 12, 18, 3
    X, W = rng.standard_normal((T, din)), rng.standard_normal((din, dout))
    b, dY = rng.standard_normal(dout), rng.standard_normal((T, dout))
    c = oracle.column_linear(X, _split_cols(W, t), b, _split_cols(dY, t))
    lhs = np.sum(dY * (np.concatenate(c["Y"], 1) - b))
    assert np.isclose(lhs, np.sum(c["dX"] * X), rtol=1e-12)
    assert np.isclose(lhs, np.sum(np.concatenate(c["dW"], 1) * W), rtol=1e-12)
    r = oracle.row_linear(_split_cols(X, t), _split_rows(W, t), b, dY)
    lhs = np.sum(dY * (r["Z"] - b))
    assert np.isclose(lhs, np.sum(np.concatenate(r["dX"], 1) * X), rtol=1e-12)
    assert np.isclose(lhs, np.sum(np.concatenate(r["dW"], 0) * W), rtol=1e-12)


def test_sharding_invariance_bitwise():
    rng = np.random.default_rng(5)
    T, din, dout = 7, 24, 24
    X, W = rng.standard_normal((T, din)), rng.standard_normal((din, dout))
    b, dY = rng.standard_normal(dout), rng.standard_normal((T, dout))
    c1 = oracle.column_linear(X, [W], b, [dY])
    r1 = oracle.row_linear([X], [W], b, dY)
    for t in (2, 3, 4):
        c = oracle.column_linear(X, _split_cols(W, t), b, _split_cols(dY, t))
        assert np.array_equal(np.concatenate(c["Y"], 1), c1["Y"][0])
        assert np.array_equal(c["dX"], c1["dX"])
        assert np.array_equal(np.concatenate(c["dW"], 1), c1["dW"][0])
        r = oracle.row_linear(_split_cols(X, t), _split_rows(W, t), b, dY)
        assert np.array_equal(r["Z"], r1["Z"])
        assert np.array_equal(np.concatenate(r["dX"], 1), r1["dX"][0])


def test_mlp_block_is_column_gelu_row():
    rng = np.random.default_rng(8)
    T, h, f, t = 6, 8, 16, 2
    X, A, B = rng.standard_normal((T, h)), rng.standard_normal((h, f)), rng.standard_normal((f, h))
    b1, b2 = rng.standard_normal(f), rng.standard_normal(h)
    c = oracle.column_linear(X, _split_cols(A, t), b1)
    H = [_gelu_np(y) for y in c["Y"]]
    r = oracle.row_linear(H, _split_rows(B, t), b2)
    blk = oracle.forward(X, _split_cols(A, t), b1, _split_rows(B, t), b2)
    assert _rel(r["Z"], blk["Z"]) < 1e-13


def test_empty_token_batch():
    W = np.ones((4, 6))
    c = oracle.column_linear(np.zeros((0, 4)), _split_cols(W, 2), np.ones(6),
                             [np.zeros((0, 3))] * 2)
    assert c["Y"][0].shape == (0, 3) and not c["db"].any() and not c["dW"][1].any()
    r = oracle.row_linear([np.zeros((0, 2))] * 2, _split_rows(W, 2), np.ones(6), np.zeros((0, 6)))
    assert r["Z"].shape == (0, 6) and not r["db"].any() and not r["dW"][0].any()
