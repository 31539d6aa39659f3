"""The tolerance helper reads the 1e-2 bar at the bf16 output's resolution; pin its grid
spacing against torch's own bf16 numbers and its effect on a one-step miss."""
import numpy as np
import torch

from helpers import BF16_TOL, bf16_step, max_err


def test_bf16_step_is_the_gap_to_the_next_bf16_number():
    x = torch.tensor([0.3, 0.999, 1.0, 1.5, 2.0, 2.0107, 3.99, 4.0, 7.5, 100.0, 1e-3], dtype=torch.float32)
    b = x.to(torch.bfloat16)
    nxt = (b.view(torch.int16) + 1).view(torch.bfloat16)
    gap = (nxt.double() - b.double()).numpy()
    assert np.array_equal(bf16_step(b.double().numpy()), gap)


def test_max_err_counts_only_the_step_beyond_the_bar():
    assert abs(max_err(np.array([0.30]), np.array([0.305]), label="helper pin") - 0.005) < 1e-15   # |ref| < 2: plain
    one_step = max_err(np.array([2.0]), np.array([2.0107]), label="helper pin")                      # one step off at 2
    assert one_step <= BF16_TOL
    two_steps = max_err(np.array([2.0]), np.array([2.03]), label="helper pin")                       # two steps off
    assert two_steps > BF16_TOL
    assert max_err(np.array([np.nan]), np.array([1.0]), label="helper pin") == float("inf")
