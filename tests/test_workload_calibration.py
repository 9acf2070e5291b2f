"""The synthetic workloads' defining properties, checked with the fp64 oracle on the host
(no GPU): the mid-size single step's hidden-state scale makes about 30 % of its masked
positions clear gamma = 0.8, and the decode workload's calibrated LM-head scale commits
several positions per sequence in its first step while the plain scale commits none by
threshold. The constants come from the calibration scripts in tests/golden/, which call only
the oracle."""

import importlib.util
import os

import numpy as np

from block_diffusion_lm_denoise_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    spec = importlib.util.spec_from_file_location(name, os.path.join(GOLDEN, name + ".py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_mid_step_scale_clears_gamma_for_about_30_percent():
    cal = _load("calibrate_mid_scale")
    f = cal.masked_fraction_above(synth.MID_STEP_H_SCALE)
    assert 0.25 <= f <= 0.35, f
