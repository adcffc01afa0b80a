"""Planted mistakes: each mutation of oracle.c (a dropped term, a wrong sign,
a wrong index, a transposed operand) must make at least one independent pin
in test_oracle_pins.py fail.  The mutants are compiled and run on the CPU."""
import os
import subprocess

import pytest

import oracle
import test_oracle_linear_pins as lin
import test_oracle_pins as pins
import test_oracle_sp_pins as sp

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, original text, mutated text); each original occurs exactly once
MUTATIONS = [
    ("b2 added twice", "zrow[n] += b2[n];", "zrow[n] += 2.0 * b2[n];"),
    ("b1 slice of shard 0 for every shard", "yrow[j] += b1[i * fi + j];", "yrow[j] += b1[j];"),
    ("GeLU' sign", "0.5 * x * (1.0 - th * th) * du", "0.5 * x * (1.0 + th * th) * du"),
    ("GeLU' dropped factor 3", "(1.0 + 3.0 * GELU_K1 * x * x)", "(1.0 + GELU_K1 * x * x)"),
    ("GeLU sign of tanh", "return 0.5 * x * (1.0 + tanh(u));", "return 0.5 * x * (1.0 - tanh(u));"),
    ("dX drops last shard", "            for (int i = 0; i < t; ++i) {\n                const double *arow",
     "            for (int i = 0; i + 1 < t; ++i) {\n                const double *arow"),
    ("dX transposed weight index", "const double *arow = A[i] + k * fi;",
     "const double *arow = A[i] + (k % fi) * fi;"),
    ("dB from Y instead of H", "const double *Hi = H[i];\n        double *dBi", "const double *Hi = Y[i];\n        double *dBi"),
    ("dA drops first token", "for (int64_t r = 0; r < T; ++r) {\n                const double x = X[r * h + k];",
     "for (int64_t r = 1; r < T; ++r) {\n                const double x = X[r * h + k];"),
    ("db1 sign", "db1[i * fi + j] = s;", "db1[i * fi + j] = -s;"),
    ("dH uses dZ transposed", "for (int64_t n = 0; n < h; ++n) dh += dZ[r * h + n] * brow[n];\n                dYi",
     "for (int64_t n = 0; n < h; ++n) dh += dZ[(n % T) * h + (r % h)] * brow[n];\n                dYi"),
    # tensor-parallel linear layers
    ("column linear: bias of shard 0", "yrow[j] += b[i * oi + j];", "yrow[j] += b[j];"),
    ("column linear: dX drops last shard", "for (int i = 0; i < t; ++i) {\n                const double *wrow = W[i]",
     "for (int i = 0; i + 1 < t; ++i) {\n                const double *wrow = W[i]"),
    ("column linear: dW pairs tokens in reverse", "const double *dyrow = dYi + r * oi;\n                for (int64_t j = 0; j < oi; ++j) o[j]",
     "const double *dyrow = dYi + (T - 1 - r) * oi;\n                for (int64_t j = 0; j < oi; ++j) o[j]"),
    ("column linear: db sign", "db[i * oi + j] = s;", "db[i * oi + j] = -s;"),
    ("row linear: bias twice", "zrow[n] += b[n];", "zrow[n] += 2.0 * b[n];"),
    ("row linear: dX skips last output column", "for (int64_t n = 0; n < out; ++n) acc += dZ[r * out + n] * wrow[n];",
     "for (int64_t n = 0; n + 1 < out; ++n) acc += dZ[r * out + n] * wrow[n];"),
    ("row linear: dW drops first token", "for (int64_t r = 0; r < T; ++r) {\n                const double x = Xi[r * ii + k];",
     "for (int64_t r = 1; r < T; ++r) {\n                const double x = Xi[r * ii + k];"),
    ("row linear: db from the first row only", "for (int64_t r = 0; r < T; ++r) s += dZ[r * out + n];",
     "for (int64_t r = 0; r < 1; ++r) s += dZ[r * out + n];"),
    # sequence-parallel LayerNorm / Dropout sublayer
    ("philox: Weyl key constant", "k[0] += 0x9E3779B9u;", "k[0] += 0x9E3779B8u;"),
    ("philox: second multiplier on the wrong word", "(uint64_t)0xCD9E8D57u * c[2];",
     "(uint64_t)0xCD9E8D57u * c[0];"),
    ("dropout: next output word", "keep[i] = (uint64_t)u[e % 4] < thresh", "keep[i] = (uint64_t)u[(e + 1) % 4] < thresh"),
    ("dropout: counter off by one element", "const uint64_t c = offset + e / 4;",
     "const uint64_t c = offset + (e + 1) / 4;"),
    ("layernorm: unbiased variance", "const double rs = 1.0 / sqrt(v / (double)h + eps);",
     "const double rs = 1.0 / sqrt(v / (double)(h - 1) + eps);"),
    ("layernorm: beta dropped", "Xn[r * h + n] = (x[n] - mu) * rs * gamma[n] + beta[n];",
     "Xn[r * h + n] = (x[n] - mu) * rs * gamma[n];"),
    ("layernorm backward: mean term dropped", "dX[r * h + n] = rstd[r] * (dy[n] * gamma[n] - mg - xh * mgx);",
     "dX[r * h + n] = rstd[r] * (dy[n] * gamma[n] - xh * mgx);"),
    ("layernorm backward: dgamma without xhat", "sgm += dXn[r * h + n] * xh;", "sgm += dXn[r * h + n];"),
    # sampled rows (full-size parity)
    ("sampled rows: H holds the pre-activation", "if (Hr) Hr[q * f + i * fi + j] = hv;",
     "if (Hr) Hr[q * f + i * fi + j] = y;"),
    ("sampled sublayer rows: mask of the sample index, not the token row",
     "oracle_dropout_keep(seed, offset, thresh, r * h, h, keep);",
     "oracle_dropout_keep(seed, offset, thresh, q * h, h, keep);"),
]

PIN_CALLS = [
    lambda: pins.test_exact_saturated_random(3, 4, 8, 2),
    lambda: pins.test_exact_saturated_random(4, 8, 16, 4),
    lambda: pins.test_random_block_against_numpy(7, 5, 12, 3),
    lambda: pins.test_gelu_closed_form(),
    lambda: pins.test_b2_added_once(),
    lambda: lin.test_column_linear_exact_integers(3, 4, 6, 2),
    lambda: lin.test_row_linear_exact_integers(3, 6, 4, 2),
    lambda: sp.test_philox_known_answers(*sp.KAT[2]),
    lambda: sp.test_dropout_counter_layout(),
    lambda: sp.test_layernorm_two_features_exact(),
    lambda: sp.test_layernorm_moments_and_affine_invariance(),
    lambda: sp.test_layernorm_backward_finite_differences(),
    lambda: sp.test_sp_layer_backward_finite_differences(),
    lambda: pins.test_sampled_rows_and_cols_equal_full(),
    lambda: sp.test_sp_rows_equal_sp_layer_bitwise(24, 16, 32, 2, 0.3, 5),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique: {name}"
    mut = tmp_path / "oracle_mut.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                    "-o", str(lib), str(mut), "-lm"], check=True)
    caught = []
    with oracle._library(str(lib)):
        for call in PIN_CALLS:
            try:
                call()
            except AssertionError:
                caught.append(call)
    assert caught, f"no pin caught the planted mistake: {name}"
