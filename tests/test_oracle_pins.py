"""Pins for the fp64 oracle, each against something other than the oracle.

Sources (page title, section):
  [FGO] "Megatron-LM：NVIDIA 的大规模并行训练方案", "Megatron-LM 核心架构 / 张量并行原理"
  [CH2] "2、分布式训练基础：数据并行、模型并行、流水线并行的基本概念与区别",
        "2.2 模型并行 —— 张量并行 / 核心原理"

What pins what:
  * exact special case  -- with pre-activations in {0} or |y| >= 10 the tanh in
    GeLU rounds to exactly +-1, so GeLU is exactly max(y, 0) except GeLU(0)=0,
    GeLU' is exactly 1 / 0 / 0.5, and the whole block (every output and
    gradient) reduces to integer matrix products that numpy evaluates exactly;
  * numpy float64 matmuls on the unsharded block, random tiny shapes;
  * the column-split identity Y = [X.A_1, ..., X.A_t]  ([FGO], [CH2]);
  * the row-split identity  Z = sum_i H_i.B_i + b2 equal to the unsharded H.B + b2;
  * GeLU closed-form facts, GeLU' against a central difference, the tanh form
    against the erf form;
  * db = column sums, against numpy;
  * central finite differences of L = sum(Z * dZ) for every input entry;
  * sampled row/column outputs equal to the full computation.
"""
import math

import numpy as np
import pytest

import oracle


def _gelu_np(x):
    # tanh-form GeLU (Hendrycks & Gimpel 2016), used only where GeLU itself is
    # pinned independently below
    c = math.sqrt(2.0 / math.pi)
    return 0.5 * x * (1.0 + np.tanh(c * (x + 0.044715 * x ** 3)))


def _split_cols(A, t):
    fi = A.shape[1] // t
    return [np.ascontiguousarray(A[:, i * fi:(i + 1) * fi]) for i in range(t)]


def _split_rows(B, t):
    fi = B.shape[0] // t
    return [np.ascontiguousarray(B[i * fi:(i + 1) * fi, :]) for i in range(t)]


def _rand_block(rng, T, h, f, scale_w=0.5):
    X = rng.standard_normal((T, h))
    A = rng.standard_normal((h, f)) * scale_w
    b1 = rng.standard_normal(f) * 0.3
    B = rng.standard_normal((f, h)) * scale_w
    b2 = rng.standard_normal(h) * 0.3
    dZ = rng.standard_normal((T, h))
    return X, A, b1, B, b2, dZ


def _run(X, A, b1, B, b2, dZ, t):
    return oracle.forward_backward(X, _split_cols(A, t), b1, _split_rows(B, t), b2, dZ)


# ---------------------------------------------------------------------------
# exact special case: saturated GeLU, integer arithmetic


def _saturated_case(rng, T, h, f):
    """Inputs whose pre-activations Y are multiples of 10: |Y| >= 10 or Y == 0."""
    X = rng.integers(-3, 4, size=(T, h)).astype(np.float64)
    A = 10.0 * rng.integers(-2, 3, size=(h, f)).astype(np.float64)
    b1 = 10.0 * rng.integers(-2, 3, size=f).astype(np.float64)
    B = rng.integers(-4, 5, size=(f, h)).astype(np.float64)
    b2 = rng.integers(-8, 9, size=h).astype(np.float64) / 4.0
    dZ = rng.integers(-3, 4, size=(T, h)).astype(np.float64)
    return X, A, b1, B, b2, dZ


def _saturated_expected(X, A, b1, B, b2, dZ):
    Xi, Ai, Bi, dZi = (a.astype(np.int64) for a in (X, A, B, dZ))
    Y = Xi @ Ai + b1.astype(np.int64)                    # exact integers
    H = np.where(Y > 0, Y, 0)                            # GeLU at |y| >= 10 or 0
    gp = np.where(Y > 0, 1.0, np.where(Y == 0, 0.5, 0.0))  # GeLU' there
    Z = (H @ Bi).astype(np.float64) + b2
    dY = (dZi @ Bi.T).astype(np.float64) * gp            # halves are exact
    dX = dY @ A.T
    dA = X.T @ dY
    dB = (H.T @ dZi).astype(np.float64)
    return {"Y": Y.astype(np.float64), "H": H.astype(np.float64), "Z": Z, "dY": dY,
            "dX": dX, "dA": dA, "dB": dB, "db1": dY.sum(0), "db2": dZ.sum(0)}


def _cat(lst, axis):
    return np.concatenate(lst, axis=axis)


def test_exact_saturated_hand_case():
    # T=2, h=2, f=4, t=2: the small case worked by hand in the design notes.
    X = np.array([[1., 2.], [2., -1.]])
    A = np.array([[10., 0., -10., 10.], [0., 10., 10., -10.]])
    b1 = np.array([0., -20., 10., 0.])
    B = np.array([[1., 0.], [2., 1.], [0., -1.], [1., 1.]])
    b2 = np.array([0.5, -0.25])
    dZ = np.array([[1., -1.], [2., 0.]])
    out = _run(X, A, b1, B, b2, dZ, t=2)
    # pre-activations: row 0 -> [10, 0, 20, -10], row 1 -> [20, -30, -20, 30]
    assert np.array_equal(_cat(out["Y"], 1), [[10., 0., 20., -10.], [20., -30., -20., 30.]])
    assert np.array_equal(_cat(out["H"], 1), [[10., 0., 20., 0.], [20., 0., 0., 30.]])
    # Z row 0 = 10*B[0] + 20*B[2] + b2 ; row 1 = 20*B[0] + 30*B[3] + b2
    assert np.array_equal(out["Z"], [[10.5, -20.25], [50.5, 29.75]])
    exp = _saturated_expected(X, A, b1, B, b2, dZ)
    for k in ("dX", "dA", "dB", "db1", "db2"):
        got = out[k] if not isinstance(out[k], list) else _cat(out[k], 1 if k == "dA" else 0)
        assert np.array_equal(got, exp[k]), k
    assert np.array_equal(_cat(out["dY"], 1), [[1., 0.5, 1., 0.], [2., 0., 0., 2.]])


@pytest.mark.parametrize("T,h,f,t", [(3, 4, 8, 2), (5, 3, 12, 3), (4, 8, 16, 4), (1, 5, 6, 1)])
def test_exact_saturated_random(T, h, f, t):
    rng = np.random.default_rng(100 + T * h + f + t)
    X, A, b1, B, b2, dZ = _saturated_case(rng, T, h, f)
    out = _run(X, A, b1, B, b2, dZ, t)
    exp = _saturated_expected(X, A, b1, B, b2, dZ)
    assert np.array_equal(_cat(out["Y"], 1), exp["Y"])
    assert np.array_equal(_cat(out["H"], 1), exp["H"])
    assert np.array_equal(out["Z"], exp["Z"])
    assert np.array_equal(_cat(out["dY"], 1), exp["dY"])
    assert np.array_equal(out["dX"], exp["dX"])
    assert np.array_equal(_cat(out["dA"], 1), exp["dA"])
    assert np.array_equal(_cat(out["dB"], 0), exp["dB"])
    assert np.array_equal(out["db1"], exp["db1"])
    assert np.array_equal(out["db2"], exp["db2"])


# ---------------------------------------------------------------------------
# library routine: numpy float64 on the unsharded block


def _rel(a, b):
    return np.linalg.norm(np.asarray(a) - np.asarray(b)) / max(np.linalg.norm(b), 1e-300)


@pytest.mark.parametrize("T,h,f,t", [(7, 5, 12, 3), (16, 8, 32, 4), (3, 16, 8, 1), (9, 12, 24, 2)])
def test_random_block_against_numpy(T, h, f, t):
    rng = np.random.default_rng(T * 1000 + h * 10 + f + t)
    X, A, b1, B, b2, dZ = _rand_block(rng, T, h, f)
    out = _run(X, A, b1, B, b2, dZ, t)
    Y = X @ A + b1
    H = _gelu_np(Y)
    Z = H @ B + b2
    assert _rel(_cat(out["Y"], 1), Y) < 1e-13
    assert _rel(_cat(out["H"], 1), H) < 1e-13
    assert _rel(out["Z"], Z) < 1e-12
    # gradients: numpy matmuls, with the oracle's dY (whose GeLU' is pinned by
    # the finite-difference test below)
    dY = _cat(out["dY"], 1)
    assert _rel(out["dX"], dY @ A.T) < 1e-12
    assert _rel(_cat(out["dA"], 1), X.T @ dY) < 1e-12
    assert _rel(_cat(out["dB"], 0), H.T @ dZ) < 1e-12
    assert _rel(out["db1"], dY.sum(0)) < 1e-13
    assert _rel(out["db2"], dZ.sum(0)) < 1e-13


# ---------------------------------------------------------------------------
# sharding identities


def test_column_split_identity_bitwise():
    rng = np.random.default_rng(7)
    X, A, b1, B, b2, dZ = _rand_block(rng, 11, 16, 32)
    one = oracle.forward(X, [A], b1, [B], b2)
    two = oracle.forward(X, _split_cols(A, 2), b1, _split_rows(B, 2), b2)
    four = oracle.forward(X, _split_cols(A, 4), b1, _split_rows(B, 4), b2)
    # Y = [X.A_1, ..., X.A_t]: every element is the same ordered sum
    assert np.array_equal(_cat(two["Y"], 1), one["Y"][0])
    assert np.array_equal(_cat(four["Y"], 1), one["Y"][0])
    assert np.array_equal(_cat(four["H"], 1), one["H"][0])


def test_row_split_and_sharding_invariance():
    rng = np.random.default_rng(8)
    X, A, b1, B, b2, dZ = _rand_block(rng, 12, 16, 64)
    ref = _run(X, A, b1, B, b2, dZ, 1)
    for t in (2, 4, 8):
        got = _run(X, A, b1, B, b2, dZ, t)
        # Z = sum_i H_i.B_i + b2 equals the unsharded H.B + b2
        assert _rel(got["Z"], ref["Z"]) < 1e-13
        assert _rel(got["dX"], ref["dX"]) < 1e-13
        assert np.array_equal(_cat(got["dA"], 1), ref["dA"][0])
        assert np.array_equal(_cat(got["dB"], 0), ref["dB"][0])
        assert np.array_equal(got["db1"], ref["db1"])
        assert np.array_equal(got["db2"], ref["db2"])
        # the partial products really are summed: each shard alone is not Z
        part = oracle.forward(X, _split_cols(A, t)[:1], b1[: 64 // t], _split_rows(B, t)[:1], b2)
        assert _rel(part["Z"], ref["Z"]) > 1e-3


def test_b2_added_once():
    rng = np.random.default_rng(9)
    X, A, b1, B, _, dZ = _rand_block(rng, 4, 8, 16)
    zero = np.zeros(8)
    bump = np.full(8, 3.0)
    for t in (1, 2, 4):
        z0 = oracle.forward(X, _split_cols(A, t), b1, _split_rows(B, t), zero)["Z"]
        z1 = oracle.forward(X, _split_cols(A, t), b1, _split_rows(B, t), bump)["Z"]
        assert np.allclose(z1 - z0, 3.0, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# GeLU closed form


def test_gelu_closed_form():
    assert oracle.gelu(0.0) == 0.0
    assert oracle.gelu_grad(0.0) == 0.5
    assert oracle.gelu(30.0) == 30.0 and oracle.gelu(-30.0) == 0.0
    assert oracle.gelu_grad(30.0) == 1.0 and oracle.gelu_grad(-30.0) == 0.0
    for x in np.linspace(-7, 7, 281):
        g, gm = oracle.gelu(x), oracle.gelu(-x)
        # tanh is odd, so GeLU(x) - GeLU(-x) = x and GeLU'(x) + GeLU'(-x) = 1
        assert abs((g - gm) - x) <= 1e-14 * max(1.0, abs(x))
        assert abs(oracle.gelu_grad(x) + oracle.gelu_grad(-x) - 1.0) <= 1e-14
        # GeLU' against a central difference of GeLU
        e = 1e-5
        fd = (oracle.gelu(x + e) - oracle.gelu(x - e)) / (2 * e)
        assert abs(fd - oracle.gelu_grad(x)) <= 1e-8
    # the tanh form stays within 5e-4 of the exact erf form x*Phi(x) on [-6, 6]
    worst = max(abs(oracle.gelu(x) - 0.5 * x * (1 + math.erf(x / math.sqrt(2))))
                for x in np.linspace(-6, 6, 2401))
    assert 1e-4 < worst <= 5e-4


# ---------------------------------------------------------------------------
# finite differences of L = sum(Z * dZ), so dL/dZ = dZ


def test_finite_difference_gradients():
    T, h, f, t = 8, 8, 16, 2
    rng = np.random.default_rng(11)
    X, A, b1, B, b2, dZ = _rand_block(rng, T, h, f, scale_w=0.6)
    out = _run(X, A, b1, B, b2, dZ, t)
    grads = {"X": out["dX"], "A": _cat(out["dA"], 1), "b1": out["db1"],
             "B": _cat(out["dB"], 0), "b2": out["db2"]}
    params = {"X": X, "A": A, "b1": b1, "B": B, "b2": b2}

    def loss(p):
        z = oracle.forward(p["X"], _split_cols(p["A"], t), p["b1"],
                           _split_rows(p["B"], t), p["b2"])["Z"]
        return float(np.sum(z * dZ))

    eps = 1e-6
    for name, val in params.items():
        g = grads[name]
        fd = np.empty_like(val)
        flat = val.reshape(-1)
        for idx in range(flat.size):
            keep = flat[idx]
            flat[idx] = keep + eps
            lp = loss(params)
            flat[idx] = keep - eps
            lm = loss(params)
            flat[idx] = keep
            fd.reshape(-1)[idx] = (lp - lm) / (2 * eps)
        err = np.abs(fd - g).max() / np.abs(g).max()
        assert err <= 1e-6, (name, err)


# ---------------------------------------------------------------------------
# sampled outputs equal the full computation


def test_sampled_rows_and_cols_equal_full():
    rng = np.random.default_rng(12)
    T, h, f, t = 20, 16, 48, 3
    X, A, b1, B, b2, dZ = _rand_block(rng, T, h, f)
    As, Bs = _split_cols(A, t), _split_rows(B, t)
    full = oracle.forward_backward(X, As, b1, Bs, b2, dZ)
    rows = [0, 7, 19, 3]
    r = oracle.rows(X, As, b1, Bs, b2, dZ, rows, activations=True)
    assert np.array_equal(r["Z"], full["Z"][rows])
    assert np.array_equal(r["dX"], full["dX"][rows])
    assert np.array_equal(r["Y"], _cat(full["Y"], 1)[rows])
    assert np.array_equal(r["H"], _cat(full["H"], 1)[rows])
    assert np.array_equal(r["dY"], _cat(full["dY"], 1)[rows])
    plain = oracle.rows(X, As, b1, Bs, b2, dZ, rows)
    assert set(plain) == {"Z", "dX"} and np.array_equal(plain["Z"], r["Z"])
    cols = [0, 15, 16, 47, 30]
    c = oracle.cols(X, As, b1, Bs, dZ, cols)
    dA, dB = _cat(full["dA"], 1), _cat(full["dB"], 0)
    assert np.array_equal(c["dA_cols"], dA[:, cols].T)
    assert np.array_equal(c["dB_rows"], dB[cols, :])
    assert np.array_equal(c["db1"], full["db1"][cols])
    assert np.array_equal(oracle.db2(dZ), full["db2"])


def test_sequence_parallel_chunks():
    rng = np.random.default_rng(13)
    T, h, f, t = 16, 8, 32, 4
    X, A, b1, B, b2, dZ = _rand_block(rng, T, h, f)
    As, Bs = _split_cols(A, t), _split_rows(B, t)
    full = oracle.forward_backward(X, As, b1, Bs, b2, dZ)
    sp = oracle.forward_backward_sp(np.split(X, 4), As, b1, Bs, b2, np.split(dZ, 4))
    for j in range(4):
        assert np.array_equal(sp["Z_chunks"][j], full["Z"][4 * j:4 * j + 4])
        assert np.array_equal(sp["dX_chunks"][j], full["dX"][4 * j:4 * j + 4])
    assert np.array_equal(sp["db2"], full["db2"])


def test_empty_token_batch():
    rng = np.random.default_rng(14)
    _, A, b1, B, b2, _ = _rand_block(rng, 1, 8, 16)
    X = np.zeros((0, 8)); dZ = np.zeros((0, 8))
    out = _run(X, A, b1, B, b2, dZ, 2)
    assert out["Z"].shape == (0, 8) and out["dX"].shape == (0, 8)
    assert np.array_equal(_cat(out["dA"], 1), np.zeros((8, 16)))
    assert np.array_equal(_cat(out["dB"], 0), np.zeros((16, 8)))
    assert np.array_equal(out["db1"], np.zeros(16))
    assert np.array_equal(out["db2"], np.zeros(8))
