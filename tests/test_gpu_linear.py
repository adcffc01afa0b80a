"""Parity of the tensor-parallel linear layers (the attention projections:
QKV column parallel, output projection row parallel) through the C ABI,
against the fp64 oracle.

Small and ragged layers are compared element by element against the full
oracle; the 175B-class projections (QKV 12288 x 36864 and the 12288 x 12288
output projection, 8 shards) on sampled rows and columns that the oracle
computes from just those rows or columns of the inputs, which is exact: row r
of Y and dX depends only on row r of X and dY, column j of dW and db only on
column j of dY.  Plus GPU-side invariants: the MLP block equals its two
linear halves bitwise, sequence-parallel equals plain bitwise, reruns are
bitwise equal.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from guard import GuardBands
from parity import gate, shard_tile_samples, tile_samples
from tensor_transformer_mlp_gemm_gb300.inputs import (LINEAR_WORKLOADS, column_shards, custom,
                                                      custom_linear, make_inputs,
                                                      make_linear_inputs, row_shards)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup(gpu):
    oracle.set_threads(len(os.sched_getaffinity(0)))
    from tensor_transformer_mlp_gemm_gb300.build import build
    build()
    yield


def _layer(w, inputs, **kw):
    from tensor_transformer_mlp_gemm_gb300.linear import DeviceLinear
    return DeviceLinear(w, inputs, **kw)


def _cat(xs, axis):
    return torch.cat([x.cpu() for x in xs], dim=axis)


def _full(lin, device=False):
    """Y (or Z), dX, dW, db of a layer in the unsharded layout (on the host
    unless device=True)."""
    mv = (lambda x: x) if device else (lambda x: x.cpu())
    cat = lambda xs, a: mv(torch.cat(list(xs), a))
    if lin.w.split == "column":
        return {"Y": cat(lin.Y, 1), "dX": cat(lin.dX, 0), "dW": cat(lin.dW, 1), "db": mv(lin.db)}
    return {"Y": cat(lin.Y, 0), "dX": cat(lin.dX, 1), "dW": cat(lin.dW, 0), "db": mv(lin.db)}


def _oracle(w, X, W, b, dY):
    """Full oracle outputs in the unsharded layout."""
    if w.split == "column":
        r = oracle.column_linear(X, column_shards(W, w.t), b, column_shards(dY, w.t))
        return {"Y": np.concatenate(r["Y"], 1), "dX": r["dX"], "dW": np.concatenate(r["dW"], 1),
                "db": r["db"]}
    r = oracle.row_linear(column_shards(X, w.t), row_shards(W, w.t), b, dY)
    return {"Y": r["Z"], "dX": np.concatenate(r["dX"], 1), "dW": np.concatenate(r["dW"], 0),
            "db": r["db"]}


def _run_full(w, seed=0):
    inputs = make_linear_inputs(w, seed)
    lin = _layer(w, inputs)
    g = GuardBands()
    g.guard(lin, ["Y", "dX", "dW", "db", "ws"])
    g.watch_inputs(lin, ["X", "W", "b", "dY"])
    lin.step()
    from tensor_transformer_mlp_gemm_gb300 import binding
    assert binding.tpmlp_sync_check() == binding.TPMLP_OK
    g.check()
    got = _full(lin)
    ref = _oracle(w, inputs["X"], inputs["W"], inputs["b"], inputs["dY"])
    for k in ("Y", "dX", "dW", "db"):
        gate(f"{w.split} {k}", got[k], ref[k])
    return lin


@pytest.mark.parametrize("name", ["qkv_tiny", "attn_out_tiny"])
def test_tiny_full(name):
    _run_full(LINEAR_WORKLOADS[name])


@pytest.mark.parametrize("split,T,din,dout,t,chunks", [
    ("column", 333, 264, 1032, 3, 1),   # ragged M, N, K tails, several tiles each way
    ("row", 333, 1032, 264, 3, 1),
    ("column", 77, 72, 272, 2, 1),      # smaller than one tile
    ("row", 77, 272, 72, 2, 1),
    ("column", 130, 520, 520, 1, 1),    # t = 1
    ("row", 256, 2048, 128, 8, 1),      # eight shards
    ("column", 512, 256, 1024, 4, 4),   # sequence-parallel token chunks
    ("row", 512, 1024, 256, 4, 4),
    ("column", 1024, 512, 2048, 8, 8),  # eight shards and eight token chunks
    ("row", 1024, 2048, 512, 8, 8),
])
def test_ragged_full(split, T, din, dout, t, chunks):
    _run_full(custom_linear(T, din, dout, t, split, sigma_w=0.05, seq_chunks=chunks), seed=3)


@pytest.fixture
def forced_tail_split():
    from tensor_transformer_mlp_gemm_gb300 import binding
    binding.tpmlp_set_split_min_kblocks(1)
    yield
    binding.tpmlp_set_split_min_kblocks(128)


@pytest.mark.parametrize("split", ["column", "row"])
def test_tail_split_full(forced_tail_split, split):
    _run_full(custom_linear(333, 264, 1032, 3, split, sigma_w=0.05) if split == "column"
              else custom_linear(333, 1032, 264, 3, split, sigma_w=0.05), seed=12)


def _assert_bitwise(a, b, what):
    if isinstance(a, list):
        for i, (x, y) in enumerate(zip(a, b)):
            _assert_bitwise(x, y, f"{what}[{i}]")
        return
    assert torch.equal(a, b), what


def test_mlp_block_equals_its_linear_halves():
    """Column linear = the block's pre-activation Y; row linear on the block's
    H = the block's Z; the linear backward calls reproduce the block's dX, dA
    (from its dY), dB (from its H and dZ) and db2 -- all bitwise, since both
    run the same kernels in the same accumulation order.  db1 agrees within
    the parity gate: the block sums dY in fp32 inside its dH GEMM, before
    rounding it to bf16, while the linear layer sums the bf16 dY it is given."""
    from tensor_transformer_mlp_gemm_gb300.block import DeviceBlock
    from tensor_transformer_mlp_gemm_gb300.linear import DeviceLinear
    w = custom(512, 256, 1024, 4, seq_chunks=4)
    inputs = make_inputs(w, 7)
    blk = DeviceBlock(w, inputs)
    blk.step()
    torch.cuda.synchronize()
    sv = blk.saved()
    cat = lambda xs, a: torch.cat([x.cpu() for x in xs], a)
    col_in = {"X": inputs["X"], "W": inputs["A"], "b": inputs["b1"],
              "dY": cat(sv["dY"], 1).to(torch.bfloat16)}
    col = DeviceLinear(custom_linear(512, 256, 1024, 4, "column", seq_chunks=4), col_in)
    col.step()
    row_in = {"X": cat(sv["H"], 1).to(torch.bfloat16), "W": inputs["B"], "b": inputs["b2"],
              "dY": inputs["dZ"]}
    row = DeviceLinear(custom_linear(512, 1024, 256, 4, "row", seq_chunks=4), row_in)
    row.step()
    torch.cuda.synchronize()
    _assert_bitwise(col.Y, [y for y in sv["Y"]], "Y")
    _assert_bitwise(row.Y, blk.Z, "Z")
    _assert_bitwise(col.dX, blk.dX, "dX")
    _assert_bitwise(col.dW, blk.dA, "dA")
    _assert_bitwise(row.dW, blk.dB, "dB")
    assert torch.equal(row.db, blk.db2)
    gate("db1 block vs column linear", blk.db1.cpu(), col.db.cpu())


def _rows_of(lin, which, rows):
    """Rows `rows` of the unsharded Y (or Z) or dX, gathered on the device."""
    xs = lin.Y if which == "Y" else lin.dX
    sharded = (lin.w.split == "column") == (which == "Y")  # t shards side by side
    if sharded:
        return torch.cat([x[rows.to(x.device)] for x in xs], 1).cpu()
    full = xs[0] if len(xs) == 1 else torch.cat(list(xs), 0)
    return full[rows.to(full.device)].cpu()


def _dw_cols(lin, cols):
    """Columns `cols` of the unsharded dW, gathered on the device."""
    if lin.w.split == "column":
        s = lin.w.shard
        return torch.stack([lin.dW[int(q) // s][:, int(q) % s] for q in cols], 1).cpu()
    full_cols = [torch.cat([d[:, int(q)] for d in lin.dW], 0) for q in cols]
    return torch.stack(full_cols, 1).cpu()


def _sampled(w, inputs, lin, rows, cols):
    """Y/dX rows and dW/db columns against the oracle on those rows/columns."""
    X, W, b, dY = inputs["X"], inputs["W"], inputs["b"], inputs["dY"]
    if w.split == "column":
        # rows of Y, dX: the oracle on the sampled rows of X and dY
        r = oracle.column_linear(X[rows], [W], b, [dY[rows]])
        gate("Y[rows]", _rows_of(lin, "Y", rows), r["Y"][0])
        gate("dX[rows]", _rows_of(lin, "dX", rows), r["dX"])
        # columns of dW, db: the oracle on the sampled columns of W, b, dY
        c = oracle.column_linear(X, [W[:, cols]], b[cols], [dY[:, cols]])
        dW = c["dW"][0]
    else:
        r = oracle.row_linear([X[rows]], [W], b, dY[rows])
        gate("Z[rows]", _rows_of(lin, "Y", rows), r["Z"])
        gate("dX[rows]", _rows_of(lin, "dX", rows), r["dX"][0])
        c = oracle.row_linear([X], [W[:, cols]], b[cols], dY[:, cols])
        dW = c["dW"][0]
    gate("dW[:,cols]", _dw_cols(lin, cols), dW)
    gate("db[cols]", lin.db.cpu()[cols], c["db"])


def _tile_covering(w, seed):
    """Token rows in both 128-row halves of every 256-row pair tile, and output
    columns in both 128-wide halves of every 256-wide tile (of every shard, for
    the column-parallel layer's sharded output)."""
    rows = tile_samples(w.tokens, seed)
    if w.split == "column":
        cols = shard_tile_samples(w.out_features, w.t, seed + 1)
    else:
        cols = tile_samples(w.out_features, seed + 1)
    return torch.from_numpy(rows), torch.from_numpy(cols)


@pytest.mark.parametrize("name", ["qkv_175b", "attn_out_175b"])
def test_175b_projections_sampled(name):
    w = LINEAR_WORKLOADS[name]
    inputs = make_linear_inputs(w, 0)
    lin = _layer(w, inputs)
    lin.step()
    torch.cuda.synchronize()
    rows, cols = _tile_covering(w, 21)
    _sampled(w, inputs, lin, rows, cols)
    Y0, dW0 = [y.clone() for y in lin.Y], lin.dW[5].clone()
    lin.step()
    torch.cuda.synchronize()
    _assert_bitwise(lin.Y, Y0, "Y rerun")
    assert torch.equal(lin.dW[5], dW0)


@pytest.mark.parametrize("name", ["qkv_sp_h4096", "attn_out_sp_h4096"])
def test_sequence_parallel_sampled_and_equal_to_plain(name):
    from dataclasses import replace
    w = LINEAR_WORKLOADS[name]
    inputs = make_linear_inputs(w, 0)
    sp = _layer(w, inputs)
    sp.step()
    torch.cuda.synchronize()
    rows, cols = _tile_covering(w, 23)
    _sampled(w, inputs, sp, rows, cols)
    plain = _layer(replace(w, seq_chunks=1), inputs)
    plain.step()
    torch.cuda.synchronize()
    a, b = _full(sp, device=True), _full(plain, device=True)
    for k in ("Y", "dX", "dW", "db"):
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("split", ["column", "row"])
def test_empty_token_batch_zeroes_gradients(split):
    w = custom_linear(0, 64, 256, 2, split)
    lin = _layer(w, make_linear_inputs(w, 0))
    for x in lin.dW + [lin.db]:
        x.fill_(7.0)
    lin.step()
    torch.cuda.synchronize()
    for x in lin.dW + [lin.db]:
        assert torch.count_nonzero(x) == 0


def test_rejects_bad_arguments_on_device():
    from tensor_transformer_mlp_gemm_gb300 import binding
    w = custom_linear(256, 256, 512, 2, "column")
    lin = _layer(w, make_linear_inputs(w, 0))
    off = lin.ws[2:].data_ptr()  # not 16-byte aligned
    with pytest.raises(binding.TpmlpError) as e:
        binding.tpmlp_column_linear_forward(lin.dims, lin.X, lin.W, lin.b, lin.Y, off)
    assert e.value.status == binding.TPMLP_ERR_UNSUPPORTED


@pytest.mark.parametrize("split", ["column", "row"])
@pytest.mark.parametrize("T,din,dout,t,chunks", [
    (333, 264, 1032, 3, 1),
    (512, 1024, 2048, 4, 4),
])
def test_wide_tiles_full(split, T, din, dout, t, chunks):
    """The linear layers' bf16-output GEMMs on 256 x 512 pair tiles."""
    from tensor_transformer_mlp_gemm_gb300 import binding
    binding.tpmlp_set_wide_tiles(2)
    try:
        if split == "column":
            _run_full(custom_linear(T, din, dout, t, split, sigma_w=0.05, seq_chunks=chunks), seed=5)
        else:
            _run_full(custom_linear(T, dout, din, t, split, sigma_w=0.05, seq_chunks=chunks), seed=5)
    finally:
        binding.tpmlp_set_wide_tiles(binding.WIDE_TILES_DEFAULT)
