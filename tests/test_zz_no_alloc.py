"""The no-allocation column-sum entry point (tpmlp_column_sums_noalloc).

It serves callers that cannot allocate device memory (a library running
inside another runtime's memory pool, a loop that forbids allocation once it
has started) by keeping its partial sums in a fixed 4 MiB array inside the
library instead of a caller-provided workspace.

Checked here, each on two calls in a row (the second call runs on whatever
the first left in the shared array):
  * against the fp64 oracle's column sums of the same bf16 input, at the
    bias-gradient shapes, at 65536 columns, at a column count that is not a
    multiple of the 64-column strip, at ragged row counts, and at the
    2^20-column limit of the array;
  * against the bias gradients tpmlp_backward computes with its
    caller-allocated workspace, within the parity gate;
  * sizes beyond the array and misaligned columns are rejected before any
    launch; an empty batch gives zeros.

The entry point caps its row splits so that the partial sums fit the array
(splits x cols <= 2^20).  The split plan asks for about 16 x SMs / (cols / 64)
splits (at most one per 128 rows, at most 64), so on this GPU (152 SMs) splits x
cols stays below 16 x 152 x 64 + cols and the cap never binds; the cases above
run split counts from 1 to 64 (1 at 2^20 columns, 3 at 4096 x 65536, 23 at
3001 x 1000, 32 at 4096 x 1024, 64 at 65536 x 1000).

This file is collected last on purpose and also passes when run alone.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from parity import gate

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup(gpu):
    oracle.set_threads(len(os.sched_getaffinity(0)))
    from tensor_transformer_mlp_gemm_gb300.build import build
    build()
    yield


def _twice_against_oracle(src, what):
    """Two calls in a row on the same input, each against the oracle's fp64
    column sums; the two results are also bitwise equal."""
    from tensor_transformer_mlp_gemm_gb300 import binding
    rows, cols = src.shape
    ref = oracle.db2(src.cpu())
    outs = []
    for call in range(2):
        out = torch.full((cols,), float("nan"), dtype=torch.float32, device=src.device)
        assert binding.tpmlp_column_sums_noalloc(src, rows, cols, out) == binding.TPMLP_OK
        assert binding.tpmlp_sync_check() == binding.TPMLP_OK
        gate(f"{what}, call {call}", out.cpu(), ref)
        outs.append(out)
    assert torch.equal(outs[0], outs[1]), f"{what}: the second call differs from the first"


@pytest.mark.parametrize("rows,cols", [
    (4096, 1024),      # db2 of the small GPT-layer workload
    (4096, 65536),     # wider than 16384 columns
    (3001, 1000),      # columns not a multiple of the 64-column strip, ragged rows
    (65536, 1000),     # the deepest row split the plan makes
    (7, 24),           # fewer rows than one warp's slots
])
def test_noalloc_matches_oracle(gpu, rows, cols):
    g = torch.Generator("cpu").manual_seed(rows * 7919 + cols)
    src = torch.randn(rows, cols, generator=g).to(torch.bfloat16).to(gpu)
    _twice_against_oracle(src, f"{rows}x{cols}")


def test_noalloc_at_the_array_limit(gpu):
    cols = 1 << 20
    g = torch.Generator("cpu").manual_seed(5)
    src = torch.randn(256, cols, generator=g).to(torch.bfloat16).to(gpu)
    _twice_against_oracle(src, "256x2^20")


def test_noalloc_column_sums_match_backward(gpu):
    from tensor_transformer_mlp_gemm_gb300 import binding
    from tensor_transformer_mlp_gemm_gb300.block import DeviceBlock
    from tensor_transformer_mlp_gemm_gb300.inputs import custom, make_inputs

    # 4096 rows: the rows are split across CTAs, so the partial-sum scratch is used
    w = custom(4096, 1024, 4096, 2)
    blk = DeviceBlock(w, make_inputs(w, 21))
    blk.step()
    assert binding.tpmlp_sync_check() == binding.TPMLP_OK
    T, h, fi = w.tokens, w.hidden, w.ffn // w.t
    dY = blk.saved()["dY"]

    out = torch.empty(h, dtype=torch.float32, device=gpu)
    out1 = torch.empty(fi, dtype=torch.float32, device=gpu)
    for call in range(2):
        out.fill_(float("nan"))
        assert binding.tpmlp_column_sums_noalloc(blk.dZ[0], T, h, out) == binding.TPMLP_OK
        assert binding.tpmlp_sync_check() == binding.TPMLP_OK
        gate(f"db2, call {call}", out.cpu(), blk.db2.cpu())
        for i in range(w.t):
            out1.fill_(float("nan"))
            assert binding.tpmlp_column_sums_noalloc(dY[i], T, fi, out1) == binding.TPMLP_OK
            assert binding.tpmlp_sync_check() == binding.TPMLP_OK
            gate(f"db1 shard {i}, call {call}", out1.cpu(), blk.db1[i * fi:(i + 1) * fi].cpu())


def test_noalloc_rejects_and_empty(gpu):
    from tensor_transformer_mlp_gemm_gb300 import binding
    src = torch.zeros(16, 64, dtype=torch.bfloat16, device=gpu)
    out = torch.full((64,), 7.0, dtype=torch.float32, device=gpu)
    # sizes beyond the static scratch and columns that are not whole 16-byte
    # vectors are rejected before any launch
    assert binding.tpmlp_column_sums_noalloc(src, 1, (1 << 20) + 8, out) == \
        binding.TPMLP_ERR_UNSUPPORTED
    assert binding.tpmlp_column_sums_noalloc(src, 16, 12, out) == binding.TPMLP_ERR_UNSUPPORTED
    assert binding.tpmlp_column_sums_noalloc(src, -1, 64, out) == binding.TPMLP_ERR_INVALID_ARG
    # no rows: the sums are zero
    assert binding.tpmlp_column_sums_noalloc(src, 0, 64, out) == binding.TPMLP_OK
    assert binding.tpmlp_sync_check() == binding.TPMLP_OK
    assert torch.count_nonzero(out) == 0
