"""GEMMs run as clusters of two CTA pairs that share each B box by TMA multicast
(tpmlp_set_b_multicast): full parity of the block against the fp64 oracle,
and every output bitwise equal to the single-pair launch (the tail split off
on both sides, since a split tile sums its products in another order).

Mode 2 forces the clusters onto every GEMM with at least two tiles in M, so
the small cases below exercise them: an odd M-tile count (the second pair of
the last cluster tile computes on zero-filled rows and stores nothing),
ragged edges, token chunks, several groups and several cluster tiles per
cluster.
"""
import os

import pytest
import torch

import oracle
from parity import compare_full
from tensor_transformer_mlp_gemm_gb300.inputs import (column_shards, custom, make_inputs,
                                                      row_shards)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup(gpu):
    oracle.set_threads(len(os.sched_getaffinity(0)))
    from tensor_transformer_mlp_gemm_gb300.build import build
    build()
    yield


def _step(w, inputs, multicast):
    from tensor_transformer_mlp_gemm_gb300 import binding
    from tensor_transformer_mlp_gemm_gb300.block import DeviceBlock
    binding.tpmlp_set_split_min_kblocks(0)
    binding.tpmlp_set_b_multicast(multicast)
    try:
        blk = DeviceBlock(w, inputs)
        blk.step()
        assert binding.tpmlp_sync_check() == binding.TPMLP_OK
    finally:
        binding.tpmlp_set_b_multicast(0)
        binding.tpmlp_set_split_min_kblocks(128)
    torch.cuda.synchronize()
    return blk


def _bitwise(a, b, what):
    if isinstance(a, list):
        for i, (x, y) in enumerate(zip(a, b)):
            _bitwise(x, y, f"{what}[{i}]")
        return
    assert torch.equal(a, b), what


@pytest.mark.parametrize("T,h,f,t,chunks", [
    (640, 264, 1032, 3, 1),     # 3 M-tiles (odd) in the token GEMMs, ragged N and K
    (1024, 512, 2048, 2, 2),    # token chunks
    (512, 256, 1024, 4, 4),     # token chunks, four shards
    (2048, 1024, 8192, 2, 1),   # several cluster tiles per cluster, 64-128 K steps
])
def test_multicast_full_and_bitwise(T, h, f, t, chunks):
    w = custom(T, h, f, t, sigma_w=0.05, seq_chunks=chunks)
    inputs = make_inputs(w, 21)
    mc = _step(w, inputs, 2)
    ref = oracle.forward_backward(inputs["X"], column_shards(inputs["A"], t), inputs["b1"],
                                  row_shards(inputs["B"], t), inputs["b2"], inputs["dZ"])
    compare_full(mc, ref)
    single = _step(w, inputs, 0)
    for name in ("Z", "dX", "dA", "dB", "db1", "db2"):
        _bitwise(getattr(mc, name), getattr(single, name), name)


def test_multicast_mode1_bitwise():
    """Mode 1 (clusters only where they fill their waves) on a layer big enough
    for it to pick them: the same results as single pairs."""
    w = custom(2048, 2048, 16384, 2, sigma_w=0.02)
    inputs = make_inputs(w, 22)
    mc = _step(w, inputs, 1)
    single = _step(w, inputs, 0)
    for name in ("Z", "dX", "dA", "dB", "db1", "db2"):
        _bitwise(getattr(mc, name), getattr(single, name), name)
