"""The parity gate's own arithmetic (CPU): half a bf16 step at each magnitude,
and the out error with the final bf16 rounding taken out."""
import numpy as np
import torch

from helpers import OUT_TOL, bf16_half_step, out_err


def test_half_step_is_the_largest_rounding_error_of_bf16():
    rng = np.random.default_rng(0)
    # fp32 values, rounded once to bf16 (as the kernels round their fp32 results)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-8, 8, 200000))).astype(np.float32)
    xb = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    x = x.astype(np.float64)
    err = np.abs(xb - x)
    hs = bf16_half_step(x)
    assert np.all(err <= hs * (1 + 1e-12))
    assert np.max(err / hs) > 0.99  # and it is reached
    assert bf16_half_step(3.0) == 2.0 ** -7 and bf16_half_step(5.0) == 2.0 ** -6
    assert bf16_half_step(1.0) == 2.0 ** -8


def test_out_err_removes_only_the_final_rounding():
    ref = np.array([-2.24582, 0.5, 6.0])
    # the nearest-but-one bf16 value of -2.24582 after a 0.004 computation error
    assert out_err(np.array([-2.234375, 0.5, 6.0]), ref) < OUT_TOL
    # a bf16 value more than the gate beyond the rounding is caught at any
    # magnitude: 0.3 -> 0.3125 (step 2^-8 there), 2.5 -> 2.53125 (step 2^-6),
    # 5.0 -> 5.0625 (step 2^-5)
    for r, g in ((0.3, 0.3125), (2.5, 2.53125), (5.0, 5.0625)):
        assert float(torch.tensor(g).to(torch.bfloat16)) == g
        assert out_err(np.array([g]), np.array([r])) > OUT_TOL
    assert out_err(np.array([np.nan]), np.array([1.0])) == np.inf
    assert out_err(np.array([-np.inf]), np.array([-np.inf])) == 0.0
