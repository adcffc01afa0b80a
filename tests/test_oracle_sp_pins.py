"""Pins for the oracle's sequence-parallel LayerNorm / Dropout sublayer,
each against something other than the oracle.

Sources: "Megatron-LM：NVIDIA 的大规模并行训练方案", "并行训练范式 / 序列并行"
(LayerNorm and Dropout distributed along the sequence dimension on top of
tensor parallelism).  The sublayer Out = X + Dropout(MLP(LN(X))) is the
usual pre-LayerNorm residual block (a reading); the dropout mask comes from
Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as
easy as 1, 2, 3", SC'11).

What pins what:
  * Philox4x32-10: the algorithm's published known-answer vectors;
  * the mask: p = 0 keeps everything; its counter layout (element e reads
    word e % 4 of block offset + e / 4) against the pinned generator; any
    sub-range equals the same slice of the whole mask; the keep rate is
    within 5 sigma of 1 - p;
  * LayerNorm: h = 2 with eps = 0 gives exactly -+gamma + beta; rows come
    out with mean 0 and mean square 1; invariance under per-row affine maps
    of the input; central finite differences for dX, dgamma, dbeta;
  * the sublayer: Out - X = keep / (1 - p) * MLP(LN(X)); central finite
    differences of sum(dOut * Out) for X (both paths), gamma, beta, b2 and
    one weight entry, with the mask held fixed;
  * the sublayer's sampled rows (sp_rows, used at full size): bitwise equal
    to the same rows of the whole pinned sublayer, for several dropout rates,
    mask offsets, shard counts and row orders.
"""
import numpy as np
import pytest

import oracle

from test_oracle_pins import _split_cols, _split_rows

# Philox4x32-10 known-answer vectors published with the algorithm:
# (counter, key) -> output
KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,want", KAT)
def test_philox_known_answers(ctr, key, want):
    assert tuple(oracle.philox4x32_10(ctr, key)) == want


def test_dropout_threshold_and_p0():
    assert oracle.dropout_threshold(0.0) == 2**32
    assert oracle.dropout_threshold(0.5) == 2**31
    assert oracle.dropout_threshold(0.1) == int(0.9 * 2**32)
    assert oracle.dropout_keep(16, 24, 0.0, seed=5).all()
    with pytest.raises(ValueError):
        oracle.dropout_threshold(1.0)


def test_dropout_counter_layout():
    seed, offset, p = 0x0123456789ABCDEF, 7, 0.3
    thr = oracle.dropout_threshold(p)
    keep = oracle.dropout_keep(6, 10, p, seed, offset)
    key = (seed & 0xFFFFFFFF, seed >> 32)
    for e in range(60):
        c = offset + e // 4
        u = oracle.philox4x32_10((c & 0xFFFFFFFF, c >> 32, 0, 0), key)[e % 4]
        assert keep[e] == (1 if u < thr else 0), e


def test_dropout_slices_and_offsets():
    full = oracle.dropout_keep(40, 64, 0.25, seed=99, offset=3)
    assert np.array_equal(oracle.dropout_keep(40, 64, 0.25, 99, 3, e0=777, count=500),
                          full[777:1277])
    # an offset of k blocks is a shift of 4k elements
    shifted = oracle.dropout_keep(40, 64, 0.25, seed=99, offset=5)
    assert np.array_equal(shifted[:2000], full[8:2008])


def test_dropout_keep_rate():
    n, p = 1 << 20, 0.1
    k = oracle.dropout_keep(1024, 1024, p, seed=2024).mean()
    sigma = np.sqrt(p * (1 - p) / n)
    assert abs(k - (1 - p)) < 5 * sigma
    assert 0 < oracle.dropout_keep(64, 64, 0.9, seed=1).sum() < 64 * 64


def test_layernorm_two_features_exact():
    X = np.array([[1.0, 3.0], [5.0, -7.0], [0.25, 0.5]])
    gamma, beta = np.array([2.0, -0.5]), np.array([0.125, 1.0])
    r = oracle.layernorm(X, gamma, beta, eps=0.0)
    sign = np.sign(X[:, 1:2] - X[:, 0:1]) * np.array([-1.0, 1.0])
    assert np.array_equal(r["Xn"], sign * gamma + beta)


def test_layernorm_moments_and_affine_invariance():
    rng = np.random.default_rng(3)
    X = rng.standard_normal((9, 40)) * 3 + 1
    one, zero = np.ones(40), np.zeros(40)
    r = oracle.layernorm(X, one, zero, eps=0.0)
    assert np.allclose(r["Xn"].mean(1), 0, atol=1e-13)
    assert np.allclose((r["Xn"] ** 2).mean(1), 1, atol=1e-12)
    a = rng.uniform(0.5, 4.0, (9, 1)); c = rng.standard_normal((9, 1))
    g, b = rng.standard_normal(40), rng.standard_normal(40)
    assert np.allclose(oracle.layernorm(a * X + c, g, b, 0.0)["Xn"],
                       oracle.layernorm(X, g, b, 0.0)["Xn"], atol=1e-12)


def test_layernorm_backward_finite_differences():
    rng = np.random.default_rng(4)
    T, h, eps = 3, 7, 1e-5
    X, g, b = rng.standard_normal((T, h)), rng.standard_normal(h), rng.standard_normal(h)
    dY = rng.standard_normal((T, h))
    r = oracle.layernorm(X, g, b, eps, dXn=dY)
    L = lambda X_, g_, b_: float(np.sum(dY * oracle.layernorm(X_, g_, b_, eps)["Xn"]))
    step = 1e-6
    for (i, j) in [(0, 0), (1, 3), (2, 6)]:
        Xp, Xm = X.copy(), X.copy(); Xp[i, j] += step; Xm[i, j] -= step
        assert abs((L(Xp, g, b) - L(Xm, g, b)) / (2 * step) - r["dX"][i, j]) < 1e-6
    for j in range(h):
        gp, gm = g.copy(), g.copy(); gp[j] += step; gm[j] -= step
        assert abs((L(X, gp, b) - L(X, gm, b)) / (2 * step) - r["dgamma"][j]) < 1e-6
        bp, bm = b.copy(), b.copy(); bp[j] += step; bm[j] -= step
        assert abs((L(X, g, bp) - L(X, g, bm)) / (2 * step) - r["dbeta"][j]) < 1e-6


def _sp_case(rng, T=5, h=8, f=16, t=2):
    X = rng.standard_normal((T, h))
    gamma, beta = 1 + 0.2 * rng.standard_normal(h), 0.1 * rng.standard_normal(h)
    A = rng.standard_normal((h, f)) * 0.4
    B = rng.standard_normal((f, h)) * 0.4
    b1, b2 = 0.1 * rng.standard_normal(f), 0.1 * rng.standard_normal(h)
    dOut = rng.standard_normal((T, h))
    return X, gamma, beta, _split_cols(A, t), b1, _split_rows(B, t), b2, dOut


def test_sp_layer_dropout_scaling():
    rng = np.random.default_rng(5)
    X, g, b, A, b1, B, b2, _ = _sp_case(rng)
    r = oracle.sp_layer(X, g, b, 1e-5, A, b1, B, b2, p=0.5, seed=11)
    mlp = oracle.forward(oracle.layernorm(X, g, b, 1e-5)["Xn"], A, b1, B, b2)["Z"]
    assert np.allclose(r["Out"] - X, r["keep"] * 2.0 * mlp, rtol=1e-14, atol=1e-14)
    assert 0 < r["keep"].sum() < r["keep"].size


def test_sp_layer_backward_finite_differences():
    rng = np.random.default_rng(6)
    X, g, b, A, b1, B, b2, dOut = _sp_case(rng)
    eps, p, seed = 1e-5, 0.25, 77
    r = oracle.sp_layer(X, g, b, eps, A, b1, B, b2, p, seed, dOut=dOut)
    assert 0 < r["keep"].sum() < r["keep"].size

    def L(X_=X, g_=g, b_=b, A_=A, b2_=b2):
        return float(np.sum(dOut * oracle.sp_layer(X_, g_, b_, eps, A_, b1, B, b2_, p,
                                                   seed)["Out"]))
    step = 1e-6

    def fd(make):
        return (L(**make(+step)) - L(**make(-step))) / (2 * step)

    for (i, j) in [(0, 0), (2, 5), (4, 7)]:
        def mk(d, i=i, j=j):
            Xd = X.copy(); Xd[i, j] += d; return {"X_": Xd}
        assert abs(fd(mk) - r["dX"][i, j]) < 1e-6
    for j in (0, 3, 7):
        def mg(d, j=j):
            gd = g.copy(); gd[j] += d; return {"g_": gd}

        def mb(d, j=j):
            bd = b.copy(); bd[j] += d; return {"b_": bd}

        def m2(d, j=j):
            bd = b2.copy(); bd[j] += d; return {"b2_": bd}
        assert abs(fd(mg) - r["dgamma"][j]) < 1e-6
        assert abs(fd(mb) - r["dbeta"][j]) < 1e-6
        assert abs(fd(m2) - r["db2"][j]) < 1e-6

    def ma(d):
        A2 = [a.copy() for a in A]; A2[1][2, 3] += d; return {"A_": A2}
    assert abs(fd(ma) - r["dA"][1][2, 3]) < 1e-6


@pytest.mark.parametrize("T,h,f,t,p,offset", [
    (24, 16, 32, 2, 0.3, 5),
    (9, 8, 24, 3, 0.0, 0),
    (40, 12, 16, 1, 0.5, 123),
])
def test_sp_rows_equal_sp_layer_bitwise(T, h, f, t, p, offset):
    rng = np.random.default_rng(T * 31 + h)
    X = rng.standard_normal((T, h))
    A = rng.standard_normal((h, f)) * 0.3
    B = rng.standard_normal((f, h)) * 0.3
    b1 = rng.standard_normal(f) * 0.1
    b2 = rng.standard_normal(h) * 0.1
    dOut = rng.standard_normal((T, h))
    gamma = 1.0 + 0.1 * rng.standard_normal(h)
    beta = 0.1 * rng.standard_normal(h)
    As, Bs = _split_cols(A, t), _split_rows(B, t)
    full = oracle.sp_layer(X, gamma, beta, 1e-5, As, b1, Bs, b2, p, 77, offset, dOut=dOut)
    rows = [0, T - 1, T // 2, 1, T // 3]
    got = oracle.sp_rows(X, gamma, beta, 1e-5, As, b1, Bs, b2, p, 77, offset, dOut, rows)
    assert np.array_equal(got["Out"], full["Out"][rows])
    assert np.array_equal(got["dX"], full["dX"][rows])
