"""The parity gate itself (tests/parity.py), on the CPU: the bf16 half spacing
it allows on top of the stated bound, and what it accepts and rejects."""
import numpy as np
import pytest
import torch

from parity import MAX_ABS, bf16_half_spacing, gate, measure


def test_half_spacing_of_bf16():
    r = np.array([0.0, 1.0, 1.5, -1.99, 2.0, 8.0, 16.0, 31.9, 32.0, 0.75])
    want = np.array([0.0, 2.0 ** -8, 2.0 ** -8, 2.0 ** -8, 2.0 ** -7, 2.0 ** -5, 2.0 ** -4,
                     2.0 ** -4, 2.0 ** -3, 2.0 ** -9])
    assert np.array_equal(bf16_half_spacing(r), want)
    # the spacing is that of torch's bf16: rounding never moves a value by more
    x = torch.linspace(-40.0, 40.0, 100001, dtype=torch.float64)
    err = (x.to(torch.bfloat16).double() - x).abs().numpy()
    assert np.all(err <= bf16_half_spacing(x.numpy()) * (1 + 1e-12))
    assert err.max() > 0.9 * 2.0 ** -3  # values above 32 do round by almost 0.125


def test_gate_accepts_rounding_and_rejects_more():
    ref = np.array([20.03125 + 0.06, 1.0, -3.0])           # RMS > 1: bound 3e-2 * RMS
    rms = float(np.sqrt(np.mean(ref * ref)))
    got = torch.tensor(ref, dtype=torch.float64).to(torch.bfloat16)
    gate("rounded", got, ref)                              # bf16 rounding alone passes
    bad = ref.copy()
    bad[1] += MAX_ABS * rms * 1.01                          # beyond the bound where spacing is small
    with pytest.raises(AssertionError):
        gate("off", torch.tensor(bad, dtype=torch.float64).to(torch.bfloat16), ref)
    # fp32 outputs get no rounding allowance
    m = measure(torch.tensor(ref + 0.5 * MAX_ABS * rms, dtype=torch.float32), ref)
    assert m["max_excess"] == pytest.approx(m["max_abs"])
