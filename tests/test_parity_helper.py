"""The GPU tests' comparison rule (tests/parity.py) on planted CPU cases:
within 2e-2 of the oracle rounded to the dtype, a one-step flip allowed only
where the dtype's grid step is wider than 2e-2, and only rarely."""
import numpy as np
import pytest
import torch

from parity import compare


class _Round:
    """Stand-in for the oracle module's round_to (the values below are
    already on the bf16 grid, so rounding them is the identity)."""
    @staticmethod
    def round_to(x, code):
        return np.asarray(torch.tensor(x).to(torch.bfloat16).double().numpy())


def _case(vals, gpu_vals):
    ref = np.array(vals, dtype=np.float64).reshape(1, -1)
    g = torch.tensor(np.array(gpu_vals, dtype=np.float32).reshape(1, -1)).to(torch.bfloat16)
    return g, ref


def test_small_error_passes():
    g, ref = _case([1.0] * 2000, [1.0078125] + [1.0] * 1999)  # one bf16 step at 1.0: 0.0078
    compare("x", g, ref, _Round)


def test_one_step_flip_where_grid_is_wide_passes():
    g, ref = _case([5.0] * 2000, [5.03125] + [5.0] * 1999)  # one step at [4, 8): 0.03125 > 2e-2
    compare("x", g, ref, _Round)


def test_two_step_error_fails():
    g, ref = _case([5.0] * 2000, [5.0625] + [5.0] * 1999)
    with pytest.raises(AssertionError):
        compare("x", g, ref, _Round)


def test_large_error_where_grid_is_fine_fails():
    g, ref = _case([1.0] * 2000, [1.03125] + [1.0] * 1999)  # 0.031 > 2e-2 at a 0.0078 grid
    with pytest.raises(AssertionError):
        compare("x", g, ref, _Round)


def test_many_flips_fail():
    g, ref = _case([5.0] * 1000, [5.03125] * 10 + [5.0] * 990)  # 1 % of the elements
    with pytest.raises(AssertionError):
        compare("x", g, ref, _Round)
