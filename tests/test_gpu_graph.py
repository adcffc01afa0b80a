"""A whole forward + backward step of each component captured once in a CUDA
graph and replayed: the library's calls enqueue kernels and asynchronous
memsets only (no allocation, no synchronisation), so a step is capturable, and
a replay gives the same bits as the eager step."""
import pytest
import torch

from tensor_transformer_mlp_gemm_gb300.inputs import (LINEAR_WORKLOADS, WORKLOADS, custom,
                                                      make_inputs, make_linear_inputs,
                                                      make_sp_inputs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup(gpu):
    from tensor_transformer_mlp_gemm_gb300.build import build
    build()
    yield


def _capture_and_compare(obj, outputs):
    """Run obj.step() eagerly, snapshot outputs, zero them, replay a captured
    step, compare bitwise."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        obj.step(s)   # warm-up outside the capture (first-call set-up)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    want = [t.clone() for t in outputs()]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        obj.step(torch.cuda.current_stream())
    for t in outputs():
        t.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    from tensor_transformer_mlp_gemm_gb300 import binding
    assert binding.tpmlp_sync_check() == binding.TPMLP_OK
    for a, b in zip(outputs(), want):
        assert torch.equal(a, b)


def test_block_step_graph():
    from tensor_transformer_mlp_gemm_gb300.block import DeviceBlock
    w = custom(333, 264, 1032, 3)
    blk = DeviceBlock(w, make_inputs(w, 0))
    _capture_and_compare(blk, lambda: blk.Z + blk.dX + blk.dA + blk.dB + [blk.db1, blk.db2])


def test_sequence_parallel_block_step_graph():
    from tensor_transformer_mlp_gemm_gb300.block import DeviceBlock
    w = WORKLOADS["small_gpt"]
    blk = DeviceBlock(w, make_inputs(w, 1))
    _capture_and_compare(blk, lambda: blk.Z + blk.dX + blk.dA + [blk.db2])


@pytest.mark.parametrize("name", ["qkv_tiny", "attn_out_tiny"])
def test_linear_step_graph(name):
    from tensor_transformer_mlp_gemm_gb300.linear import DeviceLinear
    w = LINEAR_WORKLOADS[name]
    lay = DeviceLinear(w, make_linear_inputs(w, 0))
    _capture_and_compare(lay, lambda: lay.Y + lay.dX + lay.dW + [lay.db])


def test_sp_layer_step_graph():
    from tensor_transformer_mlp_gemm_gb300.sp import DeviceSPLayer
    w = custom(512, 256, 1024, 4, seq_chunks=4)
    lay = DeviceSPLayer(w, make_sp_inputs(w, 0))
    _capture_and_compare(lay, lambda: lay.Out + lay.dX + lay.dA + [lay.dgamma, lay.dbeta])
