"""GPU parity of the adaLN-single timestep map (td_timestep_table) against the fp64 oracle."""

import numpy as np
import pytest
import torch

import block_diffusion_lm_denoise_b300 as td
import oracle
from block_diffusion_lm_denoise_b300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d,T", [(256, 16), (4096, 16), (64, 37), (8, 1)])
def test_timestep_table_matches_oracle(cuda_device, d, T):
    w = synth.normal((6 * d, 256), 1 / 16, 77, "w_t", cuda_device, torch.float32)
    b = synth.normal((6 * d,), 0.02, 77, "b_t", cuda_device, torch.float32)
    phi = td.td_timestep_table(w, b, T)
    torch.cuda.synchronize()
    assert td.td_device_error() == 0
    ref = oracle.timestep_table(w, b, T).astype(np.float32).astype(np.float64)
    got = phi.cpu().numpy().astype(np.float64)
    # both sides sum in double precision and round to float once: equal, except where the
    # two double sums (different orders) straddle a float rounding boundary, one step apart
    step = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    assert (np.abs(got - ref) <= step).all()
    assert (got == ref).mean() >= 0.999
