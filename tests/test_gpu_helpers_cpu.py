"""The GPU tests' comparison helper, checked on the CPU: the bf16 half-ulp
allowance equals torch's own bf16 rounding bound, no looser."""

import numpy as np
import torch

from gpu_helpers import bf16_half_ulp


def test_half_ulp_bounds_torch_bf16_rounding_tightly():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(200000) * s for s in (1e-3, 0.3, 1.0, 3.0, 40.0)])
    r = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).double().numpy()
    err = np.abs(r - x.astype(np.float32).astype(np.float64))
    hu = bf16_half_ulp(x)
    assert np.all(err <= hu * (1 + 1e-6))
    # tight: values just below a rounding midpoint get close to the bound
    assert np.max(err / hu) > 0.99
    # hand values: 8 significant bits
    assert bf16_half_ulp(np.array([1.0]))[0] == 2.0 ** -8
    assert bf16_half_ulp(np.array([2.5]))[0] == 2.0 ** -7
    assert bf16_half_ulp(np.array([-4.0]))[0] == 2.0 ** -6
    assert bf16_half_ulp(np.array([0.0]))[0] == 0.0
