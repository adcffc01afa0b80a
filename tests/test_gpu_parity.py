"""Parity of the CUDA path (through the C ABI) against the fp64 oracle.

Small and ragged problems are compared element by element against the full
oracle; the full-size workloads (the 1.3B-, 175B-class and sequence-parallel
layers) are compared on sampled rows/columns that the oracle computes one by
one, chosen so that every tile of every GEMM is reached: a token row in each
128-row half of every 256-row pair tile (rows of Z, dX and the saved Y, H,
dY), and an ffn column in each 128-wide half of every 256-wide output tile of
every shard (columns of dA, rows of dB, entries of db1); db2 in full.  Exact
GPU-side invariants ride along: sharded == unsharded and sequence-parallel ==
plain, bitwise.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from guard import GuardBands
from parity import compare_full, compare_sampled, shard_tile_samples, tile_samples
from tensor_transformer_mlp_gemm_gb300.inputs import (WORKLOADS, column_shards, custom,
                                                      make_inputs, row_shards)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup(gpu):
    oracle.set_threads(len(os.sched_getaffinity(0)))
    from tensor_transformer_mlp_gemm_gb300.build import build
    build()
    yield


def _block(w, inputs):
    from tensor_transformer_mlp_gemm_gb300.block import DeviceBlock
    return DeviceBlock(w, inputs)


def _oracle_full(w, inputs):
    return oracle.forward_backward(inputs["X"], column_shards(inputs["A"], w.t), inputs["b1"],
                                   row_shards(inputs["B"], w.t), inputs["b2"], inputs["dZ"])


def _run_full(w, seed=0):
    inputs = make_inputs(w, seed)
    blk = _block(w, inputs)
    # every output and the workspace inside sentinel-filled guard bands; the
    # inputs must come back unchanged
    g = GuardBands()
    g.guard(blk, ["Z", "dX", "dA", "dB", "db1", "db2", "ws"])
    g.watch_inputs(blk, ["X", "dZ", "A", "B", "b1", "b2"])
    blk.step()
    from tensor_transformer_mlp_gemm_gb300 import binding
    assert binding.tpmlp_sync_check() == binding.TPMLP_OK
    g.check()
    ref = _oracle_full(w, inputs)
    compare_full(blk, ref)
    return blk


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_full(seed):
    _run_full(WORKLOADS["tiny"], seed)


@pytest.mark.parametrize("T,h,f,t", [
    (333, 264, 1032, 3),   # ragged M, N and K tails, several tiles each way
    (77, 72, 272, 2),      # smaller than one tile in every dimension
    (130, 520, 520, 1),    # t = 1 (no sharding), one row past a tile
    (256, 128, 2048, 8),   # eight shards
])
def test_ragged_full(T, h, f, t):
    _run_full(custom(T, h, f, t, sigma_w=0.05), seed=3)


def test_small_gpt_full():
    _run_full(WORKLOADS["small_gpt"])


def test_sequence_parallel_small_full():
    # 4 chunks of 128 tokens: gather and reduce-scatter through chunk addressing
    _run_full(custom(512, 256, 1024, 4, seq_chunks=4), seed=4)


def _assert_bitwise(a, b, what):
    if isinstance(a, list):
        for i, (x, y) in enumerate(zip(a, b)):
            _assert_bitwise(x, y, f"{what}[{i}]")
        return
    assert torch.equal(a, b), what


def test_gpt_1p3b_sharded_equals_unsharded():
    w1, w4 = WORKLOADS["gpt_1p3b_t1"], WORKLOADS["gpt_1p3b_t4"]
    inputs = make_inputs(w4, 0)
    b1, b4 = _block(w1, inputs), _block(w4, inputs)
    b1.step()
    b4.step()
    torch.cuda.synchronize()
    # the shard sum walks K in the same order as the unsharded GEMM
    _assert_bitwise(b4.Z, b1.Z, "Z")
    _assert_bitwise(b4.dX, b1.dX, "dX")
    assert torch.equal(torch.cat(b4.dA, 1), b1.dA[0])
    assert torch.equal(torch.cat(b4.dB, 0), b1.dB[0])
    assert torch.equal(b4.db1, b1.db1) and torch.equal(b4.db2, b1.db2)
    compare_sampled(b4, inputs, w4, oracle, tile_samples(w4.tokens, 5),
                    shard_tile_samples(w4.ffn, w4.t, 6))


def test_gpt_175b_sampled():
    w = WORKLOADS["gpt_175b"]
    inputs = make_inputs(w, 0)
    blk = _block(w, inputs)
    blk.step()
    torch.cuda.synchronize()
    rows = tile_samples(w.tokens, 7)
    cols = shard_tile_samples(w.ffn, w.t, 8)
    assert len(rows) >= 2 * (w.tokens // 256) and len(cols) >= 2 * (w.ffn // 256)
    compare_sampled(blk, inputs, w, oracle, rows, cols)
    # the same step again gives the same bits
    Z0 = [z.clone() for z in blk.Z]
    dA0 = blk.dA[3].clone()
    blk.step()
    torch.cuda.synchronize()
    _assert_bitwise(blk.Z, Z0, "Z rerun")
    assert torch.equal(blk.dA[3], dA0)


FULL_ORACLE = os.environ.get("TPMLP_FULL_ORACLE") == "1"


@pytest.mark.skipif(not FULL_ORACLE, reason="every element of the full-size layers against the "
                    "fp64 oracle takes about four minutes of host time per layer; "
                    "TPMLP_FULL_ORACLE=1 runs it")
@pytest.mark.parametrize("name", ["gpt_175b", "sp_h4096"])
def test_full_size_every_element(name):
    """The 175B-class and sequence-parallel layers, every output and gradient
    element (Y, H, dY, Z, dX, dA, dB, db1, db2) against the full fp64 oracle."""
    w = WORKLOADS[name]
    inputs = make_inputs(w, 0)
    blk = _block(w, inputs)
    blk.step()
    torch.cuda.synchronize()
    ref = _oracle_full(w, inputs)
    rep = {}
    compare_full(blk, ref, rep)
    for k, m in rep.items():
        print(f"{name} {k}: rel_fro {m['rel_fro']:.3e} max_abs {m['max_abs']:.3e} "
              f"bound {m['bound']:.3e}")


def test_sequence_parallel_sampled_and_equal_to_plain():
    w = WORKLOADS["sp_h4096"]
    inputs = make_inputs(w, 0)
    sp = _block(w, inputs)
    sp.step()
    torch.cuda.synchronize()
    compare_sampled(sp, inputs, w, oracle, tile_samples(w.tokens, 9),
                    shard_tile_samples(w.ffn, w.t, 10))
    from dataclasses import replace
    plain = _block(replace(w, seq_chunks=1), inputs)
    plain.step()
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(sp.Z, 0), plain.Z[0])
    assert torch.equal(torch.cat(sp.dX, 0), plain.dX[0])
    _assert_bitwise(sp.dA, plain.dA, "dA")
    _assert_bitwise(sp.dB, plain.dB, "dB")
    assert torch.equal(sp.db1, plain.db1) and torch.equal(sp.db2, plain.db2)


def test_empty_token_batch_zeroes_gradients():
    w = custom(0, 64, 256, 2)
    inputs = make_inputs(w, 0)
    blk = _block(w, inputs)
    for x in blk.dA + blk.dB + [blk.db1, blk.db2]:
        x.fill_(7.0)
    blk.step()
    torch.cuda.synchronize()
    for x in blk.dA + blk.dB + [blk.db1, blk.db2]:
        assert torch.count_nonzero(x) == 0


def test_deterministic_rerun():
    w = custom(300, 256, 1024, 2)
    inputs = make_inputs(w, 11)
    a, b = _block(w, inputs), _block(w, inputs)
    a.step()
    b.step()
    torch.cuda.synchronize()
    _assert_bitwise(a.Z, b.Z, "Z")
    _assert_bitwise(a.dX, b.dX, "dX")
    _assert_bitwise(a.dA, b.dA, "dA")
    _assert_bitwise(a.dB, b.dB, "dB")
    assert torch.equal(a.db1, b.db1) and torch.equal(a.db2, b.db2)


@pytest.fixture
def forced_tail_split():
    """Split the leftover tiles of every GEMM, however short its K range, so
    the partial-tile path runs at sizes the full oracle covers."""
    from tensor_transformer_mlp_gemm_gb300 import binding
    binding.tpmlp_set_split_min_kblocks(1)
    yield
    binding.tpmlp_set_split_min_kblocks(128)


@pytest.mark.parametrize("T,h,f,t,chunks", [
    (128, 256, 1024, 2, 1),    # the tiny workload: every GEMM's tiles split
    (333, 264, 1032, 3, 1),    # ragged tails inside split tiles
    (512, 256, 1024, 4, 4),    # sequence-parallel chunks
    (512, 512, 2048, 2, 1),    # 16 leftover tiles of 4 units
    (333, 1024, 1536, 3, 1),   # 12 leftover tiles of 6 units
])
def test_tail_split_full(forced_tail_split, T, h, f, t, chunks):
    _run_full(custom(T, h, f, t, sigma_w=0.05, seq_chunks=chunks), seed=12)


def test_tail_split_deterministic(forced_tail_split):
    w = custom(333, 264, 1032, 3)
    inputs = make_inputs(w, 13)
    a, b = _block(w, inputs), _block(w, inputs)
    a.step()
    b.step()
    torch.cuda.synchronize()
    _assert_bitwise(a.Z, b.Z, "Z")
    _assert_bitwise(a.dX, b.dX, "dX")
    _assert_bitwise(a.dA, b.dA, "dA")
    _assert_bitwise(a.dB, b.dB, "dB")


def test_stalled_gemm_reports_timeout_and_context_survives():
    from tensor_transformer_mlp_gemm_gb300 import binding
    dev = torch.device("cuda:0")
    a = torch.zeros(128, 64, dtype=torch.bfloat16, device=dev)
    b = torch.zeros(256, 64, dtype=torch.bfloat16, device=dev)
    c = torch.zeros(128, 256, dtype=torch.bfloat16, device=dev)
    st = binding.tpmlp_selftest_stalled_gemm(a, b, c, 50_000_000)  # 50 ms
    assert st == binding.TPMLP_ERR_TIMEOUT
    assert binding.tpmlp_sync_check() == binding.TPMLP_OK  # the error word was cleared
    _run_full(WORKLOADS["tiny"], seed=5)                    # and the context still works


def test_rejects_bad_arguments_on_device():
    from tensor_transformer_mlp_gemm_gb300 import binding
    w = custom(256, 256, 512, 2)
    blk = _block(w, make_inputs(w, 0))
    with pytest.raises(binding.TpmlpError) as e:
        binding.tpmlp_forward(blk.dims, blk.X, blk.A, blk.b1, blk.B, blk.b2, 4, blk.Z, blk.ws)
    assert e.value.status == binding.TPMLP_ERR_INVALID_ARG
    off = blk.ws[2:].data_ptr()  # not 16-byte aligned
    with pytest.raises(binding.TpmlpError) as e:
        binding.tpmlp_forward(blk.dims, blk.X, blk.A, blk.b1, blk.B, blk.b2, 2, blk.Z, off)
    assert e.value.status == binding.TPMLP_ERR_UNSUPPORTED


@pytest.mark.parametrize("T,h,f,t,chunks", [
    (333, 264, 1032, 3, 1),    # ragged tails: prefetched boxes reach past the tensor edges
    (512, 256, 1024, 4, 4),    # token chunks
])
def test_head_prefetch_full_and_bitwise(T, h, f, t, chunks):
    """L2 prefetches of the next tile's first K steps never change a result."""
    from tensor_transformer_mlp_gemm_gb300 import binding
    w = custom(T, h, f, t, sigma_w=0.05, seq_chunks=chunks)
    inputs = make_inputs(w, 14)
    plain = _block(w, inputs)
    plain.step()
    binding.tpmlp_set_head_prefetch(4)
    try:
        pf = _run_full(w, seed=14)
    finally:
        binding.tpmlp_set_head_prefetch(0)
    torch.cuda.synchronize()
    _assert_bitwise(pf.Z, plain.Z, "Z")
    _assert_bitwise(pf.dX, plain.dX, "dX")
    _assert_bitwise(pf.dA, plain.dA, "dA")
    _assert_bitwise(pf.dB, plain.dB, "dB")


def test_tensor_map_cache_hits_on_repeat_and_misses_on_new_buffers():
    """A repeated step on the same buffers encodes no tensor map; a block on
    new buffers encodes its own; results do not depend on the cache."""
    from tensor_transformer_mlp_gemm_gb300 import binding
    w = custom(333, 264, 1032, 3)
    inputs = make_inputs(w, 15)
    a = _block(w, inputs)
    a.step()
    torch.cuda.synchronize()
    first = [z.clone() for z in a.Z] + [x.clone() for x in a.dA]
    s0 = binding.tpmlp_map_cache_stats()
    a.step()
    torch.cuda.synchronize()
    s1 = binding.tpmlp_map_cache_stats()
    assert s1["misses"] == s0["misses"], "a repeated step encoded tensor maps"
    assert s1["hits"] > s0["hits"]
    _assert_bitwise(a.Z + a.dA, first, "repeat")
    b = _block(w, inputs)
    b.step()
    torch.cuda.synchronize()
    s2 = binding.tpmlp_map_cache_stats()
    assert s2["misses"] > s1["misses"], "new buffers reused another buffer's maps"
    _assert_bitwise(b.Z + b.dA, first, "new buffers")


def test_profile_only_the_chosen_kinds():
    """tpmlp_profile_begin_kinds times the chosen kernel kinds only: one step of
    the block records launches of those kinds and none of the others."""
    from tensor_transformer_mlp_gemm_gb300 import binding
    w = custom(512, 256, 1024, 2)
    b = _block(w, make_inputs(w, 20))
    b.step()
    torch.cuda.synchronize()
    binding.tpmlp_profile_begin_kinds(64, ["column_fwd", "wgrad_a"])
    b.step()
    ms, count = binding.tpmlp_profile_end()
    assert count["column_fwd"] == 1 and count["wgrad_a"] == 1
    assert ms["column_fwd"] > 0 and ms["wgrad_a"] > 0
    assert all(count[k] == 0 for k in count if k not in ("column_fwd", "wgrad_a"))
    binding.tpmlp_profile_begin(64)
    b.step()
    _, every = binding.tpmlp_profile_end()
    assert every["row_fwd"] == 1 and every["dgrad_h"] == 1 and every["bias_grad"] >= 1


@pytest.fixture
def wide_tiles_forced():
    """Run every bf16-output GEMM with 256 x 512 pair tiles, whatever the size."""
    from tensor_transformer_mlp_gemm_gb300 import binding
    binding.tpmlp_set_wide_tiles(2)
    yield
    binding.tpmlp_set_wide_tiles(binding.WIDE_TILES_DEFAULT)


@pytest.mark.parametrize("T,h,f,t,chunks", [
    (128, 256, 1024, 2, 1),     # the tiny workload
    (333, 264, 1032, 3, 1),     # ragged M, N and K tails; wide tiles mostly past N
    (77, 72, 272, 2, 1),        # smaller than one tile in every dimension
    (512, 256, 1024, 4, 4),     # token chunks
    (300, 1040, 2064, 2, 1),    # several wide tiles per row, ragged last one
])
def test_wide_tiles_full(wide_tiles_forced, T, h, f, t, chunks):
    _run_full(custom(T, h, f, t, sigma_w=0.05, seq_chunks=chunks), seed=16)


@pytest.mark.parametrize("T,h,f,t,chunks", [
    (128, 256, 1024, 2, 1),
    (333, 264, 1032, 3, 1),
    (512, 256, 1024, 4, 4),
])
def test_wide_tiles_tail_split_full(wide_tiles_forced, forced_tail_split, T, h, f, t, chunks):
    _run_full(custom(T, h, f, t, sigma_w=0.05, seq_chunks=chunks), seed=17)


def test_wide_tiles_match_narrow():
    """Without the tail split, half 0 of a wide tile sums every output in the
    same order as a narrow tile (bitwise equal columns); half 1 starts its K
    sum further along (within the parity gate)."""
    from tensor_transformer_mlp_gemm_gb300 import binding
    from parity import gate
    w = custom(600, 1040, 2064, 2, seq_chunks=1)
    inputs = make_inputs(w, 18)
    binding.tpmlp_set_split_min_kblocks(0)
    try:
        binding.tpmlp_set_wide_tiles(0)
        narrow = _block(w, inputs)
        narrow.step()
        binding.tpmlp_set_wide_tiles(2)
        wide = _block(w, inputs)
        wide.step()
    finally:
        binding.tpmlp_set_wide_tiles(binding.WIDE_TILES_DEFAULT)
        binding.tpmlp_set_split_min_kblocks(128)
    torch.cuda.synchronize()
    sn, sw = narrow.saved(), wide.saved()
    fi = w.ffn // w.t
    half0 = (torch.arange(fi, device=sn["Y"][0].device) % 512) < 256
    for k in ("Y", "H", "dY"):
        for i in range(w.t):
            assert torch.equal(sw[k][i][:, half0], sn[k][i][:, half0]), f"{k}[{i}] half 0"
            gate(f"{k}[{i}] wide vs narrow", sw[k][i].cpu(), sn[k][i].cpu())
    gate("Z wide vs narrow", wide.Z[0].cpu(), narrow.Z[0].cpu())
    gate("dX wide vs narrow", wide.dX[0].cpu(), narrow.dX[0].cpu())
    for i in range(w.t):
        gate(f"dA[{i}] wide vs narrow", wide.dA[i].cpu(), narrow.dA[i].cpu())
        gate(f"dB[{i}] wide vs narrow", wide.dB[i].cpu(), narrow.dB[i].cpu())


def test_explicit_sp_gather_scatter():
    """tpmlp_sp_gather / tpmlp_sp_scatter: the gathered tensor is the chunks'
    concatenation, the scatter its inverse, and gather -> un-chunked block ->
    scatter gives the chunk-addressed block's outputs bitwise."""
    from dataclasses import replace
    from tensor_transformer_mlp_gemm_gb300 import binding
    w = custom(512, 264, 1056, 4, seq_chunks=4)
    inputs = make_inputs(w, 19)
    sp = _block(w, inputs)
    sp.step()
    plain = _block(replace(w, seq_chunks=1), inputs)
    g = GuardBands()
    g.guard(plain, ["X", "dZ"])
    binding.tpmlp_sp_gather(sp.dims, sp.X, w.hidden, plain.X[0])
    binding.tpmlp_sp_gather(sp.dims, sp.dZ, w.hidden, plain.dZ[0])
    torch.cuda.synchronize()
    g.check()
    assert torch.equal(plain.X[0], torch.cat(sp.X, 0))
    assert torch.equal(plain.dZ[0], torch.cat(sp.dZ, 0))
    plain.step()
    Zc = [torch.empty_like(z) for z in sp.Z]
    dXc = [torch.empty_like(x) for x in sp.dX]
    g2 = GuardBands()
    holder = type("H", (), {})()
    holder.Zc, holder.dXc = Zc, dXc
    g2.guard(holder, ["Zc", "dXc"])
    binding.tpmlp_sp_scatter(sp.dims, plain.Z[0], w.hidden, holder.Zc)
    binding.tpmlp_sp_scatter(sp.dims, plain.dX[0], w.hidden, holder.dXc)
    assert binding.tpmlp_sync_check() == binding.TPMLP_OK
    g2.check()
    _assert_bitwise(holder.Zc, sp.Z, "Z")
    _assert_bitwise(holder.dXc, sp.dX, "dX")
