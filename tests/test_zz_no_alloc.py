"""The no-allocation column-sum entry point (tpmlp_column_sums_noalloc).

It serves callers that cannot allocate device memory, by keeping its
partial sums in a static array inside the library.  Its output must match the
bias gradients that tpmlp_backward computes with its caller-allocated
workspace, within the parity tolerance, on two calls in a row (the second
call runs on whatever the first left in the shared array).  This file is
collected last on purpose and must also pass when run alone.
"""
import pytest
import torch

from parity import gate

pytestmark = pytest.mark.gpu


def test_noalloc_column_sums_match_backward(gpu):
    from tensor_transformer_mlp_gemm_gb300.build import build
    build()
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

    # sizes beyond the static scratch are rejected before any launch
    big = (1 << 20) + 8
    assert binding.tpmlp_column_sums_noalloc(blk.dZ[0], 1, big, out) == \
        binding.TPMLP_ERR_UNSUPPORTED
    assert binding.tpmlp_column_sums_noalloc(blk.dZ[0], T, 12, out) == \
        binding.TPMLP_ERR_UNSUPPORTED
