"""The guard-band checker the GPU parity tests wrap around every output
(tests/guard.py), exercised on the CPU: a clean buffer passes, and a planted
write one element past either end of a buffer, or into an input, is caught."""
import pytest
import torch

from guard import MARGIN, SENTINEL, GuardBands


class _Layer:
    def __init__(self):
        self.Z = [torch.zeros(5, 24, dtype=torch.bfloat16), torch.zeros(5, 24, dtype=torch.bfloat16)]
        self.db = torch.zeros(24, dtype=torch.float32)
        self.X = torch.ones(5, 24, dtype=torch.bfloat16)


def _guarded():
    lay, g = _Layer(), GuardBands()
    g.guard(lay, ["Z", "db"])
    g.watch_inputs(lay, ["X"])
    return lay, g


def test_guarded_views_keep_shape_dtype_and_alignment():
    lay, g = _guarded()
    assert lay.Z[1].shape == (5, 24) and lay.Z[1].dtype == torch.bfloat16
    assert lay.db.shape == (24,) and lay.db.dtype == torch.float32
    for x in lay.Z + [lay.db]:
        assert x.data_ptr() % 256 == 0
        assert torch.all(x.view(torch.uint8) == SENTINEL)  # contents start as the sentinel


def test_clean_writes_pass():
    lay, g = _guarded()
    for z in lay.Z:
        z.fill_(3.0)
    lay.db.copy_(torch.arange(24, dtype=torch.float32))
    g.check()


@pytest.mark.parametrize("which,where", [(0, "after"), (1, "before"), (2, "after")])
def test_planted_overrun_is_caught(which, where):
    lay, g = _guarded()
    name, raw, start, n = g._bufs[which]
    assert start >= MARGIN and raw.numel() - start - n >= MARGIN
    # a store one element past the end (or just before the start) of the buffer
    if where == "after":
        raw[start + n] = 0
    else:
        raw[start - 1] = 0
    with pytest.raises(AssertionError) as e:
        g.check()
    assert name in str(e.value) and where in str(e.value)


def test_far_overrun_and_modified_input_are_caught():
    lay, g = _guarded()
    name, raw, start, n = g._bufs[2]
    raw[-1] = 0  # the last byte of the trailing band
    lay.X[2, 3] = 7.0
    with pytest.raises(AssertionError) as e:
        g.check()
    msg = str(e.value)
    assert "db" in msg and "input X[0] was modified" in msg
