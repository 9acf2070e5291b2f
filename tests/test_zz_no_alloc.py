"""td_lmhead_commit_static: the LM head + commit for callers that cannot allocate device
memory (for example a plugin whose host framework owns all device memory through its own
pool, or a loop that must not call cudaMalloc / cudaFree because they can synchronise the
device). It uses a fixed scratch array inside the library instead of a caller workspace.

This file is collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test. It passes alone in a fresh process as well.
"""

import ctypes

import pytest
import torch

import block_diffusion_lm_denoise_b300 as td
import oracle
from block_diffusion_lm_denoise_b300 import synth
from parity_util import CONF_TOL, compare_commit

pytestmark = pytest.mark.gpu


def _case(dev, M, S, V, d, seed):
    B = M // S
    w = synth.normal((V, d), 0.02, seed, "w_lm", dev)
    temp = synth.uniform((M, 1), 0.2, 2.0, seed, "temp", dev)
    h = (synth.normal((M, d), 1.0, seed, "h", dev, torch.float32) / temp).to(torch.bfloat16)
    masked = synth.bernoulli((B, S), 0.8, seed, "m", dev).to(torch.uint8)
    tokens = torch.where(masked.bool(), torch.full((B, S), V, dtype=torch.int32, device=dev),
                         synth.integers((B, S), V, seed, "t", dev))
    return h, w, tokens, masked


def _call_static(dims, h, w, gamma, tokens, masked, conf, pred, ncom, done):
    lib = td.lib()
    st = lib.td_lmhead_commit_static(ctypes.byref(dims), h.data_ptr(), w.data_ptr(), gamma, 0,
                                     tokens.data_ptr(), masked.data_ptr(), conf.data_ptr(),
                                     pred.data_ptr(), ncom.data_ptr(), done.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.td_status_string(st).decode()


# the last case is the largest row count whose partials fit the 16 MiB scratch at this
# vocabulary: 3 * 2720 * 512 * 4 + 256 bytes
@pytest.mark.parametrize("M,S,V,d", [(256, 16, 4096, 512), (1024, 16, 131072, 4096),
                                     (2720, 16, 131072, 4096)])
def test_static_scratch_matches_workspace_entry_twice(cuda_device, M, S, V, d):
    gamma = 0.8
    h, w, tokens0, masked0 = _case(cuda_device, M, S, V, d, seed=31)
    dims = td.make_dims(B=M // S, S=S, d=d, Hq=1, Hkv=1, D=64, V=V, Lmax=0, n_layers=0)
    # the existing entry point, with a caller workspace
    t_ref, m_ref = tokens0.clone(), masked0.clone()
    c_ref, p_ref, n_ref, d_ref = td.td_lmhead_commit(dims, h, w, gamma, False, t_ref, m_ref)
    torch.cuda.synchronize()
    # the fixed-scratch entry point, two calls in a row from the same starting state
    for _ in range(2):
        tok, msk = tokens0.clone(), masked0.clone()
        conf = torch.full_like(c_ref, -1.0)
        pred = torch.full_like(p_ref, -1)
        ncom = torch.full_like(n_ref, -1)
        done = torch.full_like(d_ref, -1)
        _call_static(dims, h, w, gamma, tok, msk, conf, pred, ncom, done)
        torch.cuda.synchronize()
        assert td.td_device_error() == 0
        assert (conf - c_ref).abs().max().item() <= CONF_TOL
        assert torch.equal(pred, p_ref)
        assert torch.equal(tok, t_ref) and torch.equal(msk, m_ref)
        assert torch.equal(ncom, n_ref) and torch.equal(done, d_ref)
    # and against the fp64 oracle on three sampled sequences
    B = M // S
    seqs = sorted({0, B // 2, B - 1})
    rows = [b * S + i for b in seqs for i in range(S)]
    c, p, gap, _ = oracle.lmhead_confidence(h, w, rows=rows)
    nb = len(seqs)
    m0 = masked0[seqs].cpu().numpy().astype(bool)
    tok_o, msk_o, _, _ = oracle.commit(c.reshape(nb, S), p.reshape(nb, S),
                                       tokens0[seqs].cpu().numpy(), m0, gamma, False)
    compare_commit(dict(conf=c.reshape(nb, S), pred=p.reshape(nb, S), gap=gap.reshape(nb, S),
                        tokens=tok_o, masked=msk_o),
                   dict(conf=conf[seqs].cpu().numpy(), pred=pred[seqs].cpu().numpy(),
                        tokens=tok[seqs].cpu().numpy(), masked=msk[seqs].cpu().numpy()),
                   m0, gamma)


def test_static_scratch_rejects_problems_beyond_its_size(cuda_device):
    # 4096 rows x 512 vocabulary tiles x 12 bytes > 16 MiB: refused, nothing launched
    dims = td.make_dims(B=256, S=16, d=4096, Hq=1, Hkv=1, D=64, V=131072, Lmax=0, n_layers=0)
    x = torch.zeros(16, dtype=torch.uint8, device=cuda_device)
    p = x.data_ptr()
    st = td.lib().td_lmhead_commit_static(ctypes.byref(dims), p, p, 0.8, 0, p, p, p, p, p, p,
                                          None)
    assert st == 2   # TD_ERR_WORKSPACE
