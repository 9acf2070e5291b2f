"""Failure detection on the GPU without a fault: a bounded wait that runs out ends with an
error code the host reads (and the context stays usable), and a corrupt input is flagged."""

import ctypes
import time

import pytest
import torch

import block_diffusion_lm_denoise_b300 as td
from block_diffusion_lm_denoise_b300 import synth

pytestmark = pytest.mark.gpu


def test_a_wait_that_nothing_completes_gives_up_with_an_error_code(cuda_device):
    assert td.td_device_error() == 0
    t0 = time.perf_counter()
    td.td_check_bounded_wait(50000)          # 50 ms
    code = ctypes.c_int(0)
    status = td.lib().td_device_error(ctypes.byref(code))   # synchronises
    el = time.perf_counter() - t0
    assert code.value == 0x300 and status == 6              # TD_ERR_DEVICE_TIMEOUT
    assert 0.045 <= el < 1.5, el
    # the context is still usable: a normal call runs and leaves no error
    B, S, Hq, Hkv, D, L = 1, 16, 4, 1, 64, 64
    q = synth.normal((B, S, Hq, D), 1.0, 3, "q", cuda_device)
    kb = synth.normal((B, S, Hkv, D), 1.0, 3, "kb", cuda_device)
    vb = synth.normal((B, S, Hkv, D), 1.0, 3, "vb", cuda_device)
    kc = synth.normal((B, Hkv, L, D), 1.0, 3, "kc", cuda_device)
    vc = synth.normal((B, Hkv, L, D), 1.0, 3, "vc", cuda_device)
    dims = td.make_dims(B=B, S=S, d=64, Hq=Hq, Hkv=Hkv, D=D, V=8, Lmax=L, n_layers=1)
    o = td.td_block_attention(dims, q, kb, vb, kc, vc)
    assert td.td_device_error() == 0 and torch.isfinite(o.float()).all()


def test_limits_of_the_diagnostic_are_checked():
    with pytest.raises(td.TdError):
        td.td_check_bounded_wait(0)
    with pytest.raises(td.TdError):
        td.td_check_bounded_wait(3_000_000)


def test_a_token_outside_the_vocabulary_is_flagged_and_read_as_mask(cuda_device):
    wl = synth.tiny_step(cuda_device)
    dm = wl.dims
    tokens = wl.tokens.clone()
    masked = wl.masked.clone()
    masked[0, 3] = 0
    tokens[0, 3] = dm.V + 5                  # neither a vocabulary id nor [MASK]
    conf, _, _, _ = td.td_denoise_step(dm.as_dict(), wl.layers, wl.w_lm, wl.phi_table[0], 1,
                                       wl.T, wl.gamma, tokens, masked, emb=synth.normal(
                                           (dm.V + 1, dm.d), 1.0, 5, "emb", cuda_device),
                                       pos=synth.normal((dm.S, dm.d), 1.0, 5, "pos",
                                                        cuda_device))
    assert td.td_device_error() == 0x500
    assert torch.isfinite(conf).all()
