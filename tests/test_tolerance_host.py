"""The bf16 store allowance of the parity tolerance (CPU): half the bf16 spacing at |x| bounds
round-to-nearest-even to bf16, tightly, and bf16-stored values are recognised."""
import numpy as np
import torch

import gpu_util as U


def test_half_spacing_bounds_bf16_rounding_tightly():
    rng = np.random.default_rng(7)
    # fp32 inputs: the kernels round fp32 values to bf16 once (torch's fp64 -> bf16 conversion
    # goes through fp32, a double rounding that can exceed half a spacing by a hair)
    x = np.concatenate([rng.normal(0, s, 20000) for s in (1e-3, 1.0, 30.0, 1e4)]).astype(np.float32)
    r = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    x = x.astype(np.float64)
    err = np.abs(r - x)
    allow = U.bf16_half_spacing(x)
    assert np.all(err <= allow * (1 + 1e-12))
    assert np.max(err / allow) > 0.99          # the bound is reached, not loose


def test_stored_as_bf16():
    x = torch.randn(1000, dtype=torch.float64)
    assert U.stored_as_bf16(x.to(torch.bfloat16).to(torch.float64).numpy())
    assert not U.stored_as_bf16(x.to(torch.float32).to(torch.float64).numpy())
