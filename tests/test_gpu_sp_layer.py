"""Parity of the sequence-parallel sublayer Out = X + Dropout(MLP(LN(X)))
(LayerNorm and Dropout per token chunk) through the C ABI, against the fp64
oracle.

Small and ragged layers are compared element by element against the full
oracle, and the dropout mask exactly (every element the oracle drops is an
exact zero of the GPU's dZ, and only those).  The 16384 x 4096 sequence-
parallel workload is compared on sampled rows (Out, dX from the oracle's
sampled sublayer rows, sp_rows: one row in each 128-row half of every 256-row
pair tile) and sampled columns of the weight gradients (one in each 128-wide
half of every 256-wide tile of every shard, from the block's inputs LN(X) and
dZ inside the oracle's sublayer, sp_block_inputs); LayerNorm's dgamma and
dbeta are checked element by element at the small sizes only.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from guard import GuardBands
from parity import gate, shard_tile_samples, tile_samples
from tensor_transformer_mlp_gemm_gb300.inputs import (WORKLOADS, column_shards, custom,
                                                      make_sp_inputs, row_shards)

pytestmark = pytest.mark.gpu

EPS = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _setup(gpu):
    oracle.set_threads(len(os.sched_getaffinity(0)))
    from tensor_transformer_mlp_gemm_gb300.build import build
    build()
    yield


def _layer(w, inputs, p, seed=1234):
    from tensor_transformer_mlp_gemm_gb300.sp import DeviceSPLayer
    return DeviceSPLayer(w, inputs, eps=EPS, dropout_p=p, seed=seed)


def _cat(xs, axis):
    return torch.cat([x.cpu() for x in xs], dim=axis)


def _report(rep):
    # max |error| over the bound, then (beyond the bf16 rounding allowance) what the gate compares
    print(" ".join(f"{k}:{v['max_abs'] / v['bound']:.2f}({v['max_excess'] / v['bound']:.2f})"
                   for k, v in rep.items()))


def _run_full(w, p, seed=0):
    rep = {}
    inputs = make_sp_inputs(w, seed)
    lay = _layer(w, inputs, p)
    g = GuardBands()
    g.guard(lay, ["Out", "dX", "dA", "dB", "db1", "db2", "dgamma", "dbeta", "ws"])
    g.watch_inputs(lay, ["X", "dOut", "A", "B", "b1", "b2", "gamma", "beta"])
    lay.step()
    from tensor_transformer_mlp_gemm_gb300 import binding
    assert binding.tpmlp_sync_check() == binding.TPMLP_OK
    g.check()
    ref = oracle.sp_layer(inputs["X"], inputs["gamma"], inputs["beta"], EPS,
                          column_shards(inputs["A"], w.t), inputs["b1"],
                          row_shards(inputs["B"], w.t), inputs["b2"], p, 1234, dOut=inputs["dZ"])
    torch.cuda.synchronize()
    gate("Xn", lay.workspace_tensor("xn").cpu(), ref["Xn"], rep)
    dz = lay.workspace_tensor("dz").cpu()
    dropped = ref["keep"] == 0
    assert torch.all(dz[torch.from_numpy(dropped)] == 0), "kept where the oracle drops"
    # a kept element is zero only where dOut is (the inputs hold a few exact zeros)
    nonzero = inputs["dZ"].float().numpy() != 0
    assert torch.all(dz[torch.from_numpy(~dropped & nonzero)] != 0), "dropped where the oracle keeps"
    gate("dZ", dz, ref["dZ"], rep)
    gate("Out", _cat(lay.Out, 0), ref["Out"], rep)
    gate("dX", _cat(lay.dX, 0), ref["dX"], rep)
    gate("dgamma", lay.dgamma, ref["dgamma"], rep)
    gate("dbeta", lay.dbeta, ref["dbeta"], rep)
    gate("dA", _cat(lay.dA, 1), np.concatenate(ref["dA"], 1), rep)
    gate("dB", _cat(lay.dB, 0), np.concatenate(ref["dB"], 0), rep)
    gate("db1", lay.db1, ref["db1"], rep)
    gate("db2", lay.db2, ref["db2"], rep)
    _report(rep)
    return lay, ref


@pytest.mark.parametrize("T,h,f,t,chunks,p", [
    (512, 256, 1024, 4, 4, 0.1),    # four token chunks
    (333, 264, 1032, 3, 1, 0.2),    # ragged M, N and K tails
    (256, 2048, 2048, 8, 2, 0.5),   # eight shards, wide rows
    (128, 256, 1024, 2, 1, 0.0),    # no dropout: Out = X + MLP(LN(X))
    (256, 6144, 1024, 2, 2, 0.1),   # LayerNorm rows of 3 vectors per thread (4-vector kernels)
    (128, 16384, 512, 1, 1, 0.1),   # the widest rows the LayerNorm kernels take (h = 16384)
    (2048, 4096, 256, 2, 4, 0.1),   # fused LayerNorm backward: row blocks across chunk edges
    (256, 3000, 512, 2, 2, 0.1),    # fused LayerNorm backward, second vector per thread partly used
    (1536, 4104, 256, 1, 3, 0.1),   # rows just above the fused backward's widest (4096)
])
def test_sp_layer_full(T, h, f, t, chunks, p):
    # weights with the workloads' standard deviation (0.02)
    _run_full(custom(T, h, f, t, seq_chunks=chunks), p, seed=2)


@pytest.mark.parametrize("T,h,f,t,chunks,p", [
    (512, 256, 1024, 4, 4, 0.1),
    (333, 264, 1032, 3, 1, 0.2),
])
def test_sp_layer_wide_tiles_full(T, h, f, t, chunks, p):
    """The dropout + residual epilogue and the rest on 256 x 512 pair tiles."""
    from tensor_transformer_mlp_gemm_gb300 import binding
    binding.tpmlp_set_wide_tiles(2)
    try:
        _run_full(custom(T, h, f, t, seq_chunks=chunks), p, seed=6)
    finally:
        binding.tpmlp_set_wide_tiles(binding.WIDE_TILES_DEFAULT)


def test_sp_layer_deterministic_and_seeded():
    w = custom(512, 256, 1024, 4, seq_chunks=4)
    inputs = make_sp_inputs(w, 3)
    a, b, c = _layer(w, inputs, 0.1), _layer(w, inputs, 0.1), _layer(w, inputs, 0.1, seed=99)
    for lay in (a, b, c):
        lay.step()
    torch.cuda.synchronize()
    for x, y in zip(a.Out + a.dX + a.dA + a.dB, b.Out + b.dX + b.dA + b.dB):
        assert torch.equal(x, y)
    assert torch.equal(a.dgamma, b.dgamma) and torch.equal(a.dbeta, b.dbeta)
    assert not torch.equal(a.workspace_tensor("dz"), c.workspace_tensor("dz"))


def test_sp_layer_empty_batch_zeroes_gradients():
    w = custom(0, 64, 256, 2)
    lay = _layer(w, make_sp_inputs(w, 0), 0.1)
    for x in lay.dA + lay.dB + [lay.db1, lay.db2, lay.dgamma, lay.dbeta]:
        x.fill_(7.0)
    lay.step()
    torch.cuda.synchronize()
    for x in lay.dA + lay.dB + [lay.db1, lay.db2, lay.dgamma, lay.dbeta]:
        assert torch.count_nonzero(x) == 0


FULL_ORACLE = os.environ.get("TPMLP_FULL_ORACLE") == "1"


@pytest.mark.skipif(not FULL_ORACLE, reason="every element of the 16384 x 4096 sublayer against "
                    "the fp64 oracle takes about four minutes of host time; "
                    "TPMLP_FULL_ORACLE=1 runs it")
def test_sp_h4096_full_every_element():
    """The 16384 x 4096 sequence-parallel sublayer, every element of LN(X), dZ
    (and the mask exactly), Out, dX, dgamma, dbeta, dA, dB, db1 and db2 against
    the full fp64 oracle: the one-pass LayerNorm backward over its 304 row
    blocks and the finish of their partial sums at full size."""
    _run_full(WORKLOADS["sp_h4096"], 0.1, seed=0)


def test_sp_h4096_sampled():
    w = WORKLOADS["sp_h4096"]
    p, seed = 0.1, 1234
    inputs = make_sp_inputs(w, 0)
    lay = _layer(w, inputs, p, seed)
    lay.step()
    torch.cuda.synchronize()
    rep = {}
    A, B = column_shards(inputs["A"], w.t), row_shards(inputs["B"], w.t)
    # a token row in each 128-row half of every 256-row pair tile
    rows = tile_samples(w.tokens, 31)
    r = oracle.sp_rows(inputs["X"], inputs["gamma"], inputs["beta"], EPS, A, inputs["b1"], B,
                       inputs["b2"], p, seed, 0, inputs["dZ"], rows)
    Out = torch.cat(lay.Out, 0)
    dX = torch.cat(lay.dX, 0)
    idx = torch.from_numpy(rows).to(Out.device)
    gate("Out[rows]", Out[idx].cpu(), r["Out"], rep)
    gate("dX[rows]", dX[idx].cpu(), r["dX"], rep)
    # weight-gradient columns (both halves of every 256-wide tile of every
    # shard) from the block's inputs inside the sublayer
    bi = oracle.sp_block_inputs(inputs["X"], inputs["gamma"], inputs["beta"], EPS, p, seed, 0,
                                dOut=inputs["dZ"])
    cols = shard_tile_samples(w.ffn, w.t, 32)
    c = oracle.cols(bi["Xn"], A, inputs["b1"], B, bi["dZ"], cols)
    fi = w.ffn // w.t
    gate("dA[:,cols]", torch.stack([lay.dA[int(q) // fi][:, int(q) % fi].cpu() for q in cols]),
         c["dA_cols"], rep)
    gate("dB[cols,:]", torch.stack([lay.dB[int(q) // fi][int(q) % fi, :].cpu() for q in cols]),
         c["dB_rows"], rep)
    gate("db1[cols]", lay.db1.cpu()[cols], c["db1"], rep)
    gate("db2", lay.db2, oracle.db2(bi["dZ"]), rep)
    _report(rep)
