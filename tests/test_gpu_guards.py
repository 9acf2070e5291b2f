"""Out-of-bounds writes and odd shapes, without a memory checker: every buffer an entry point
writes sits between poisoned guard bands that must be intact afterwards, and the whole step is
compared with the oracle at odd shapes (S = 1 / 4 / 32, B = 1, empty or ragged context,
head_dim 64 / 128, several tiles with a ragged tail)."""

import math

import numpy as np
import pytest
import torch

import block_diffusion_lm_denoise_b300 as td
from block_diffusion_lm_denoise_b300 import synth
from parity_util import stacked_step_parity

pytestmark = pytest.mark.gpu

GUARD = 4096       # bytes of poison on each side (a multiple of 256 keeps the alignment)
POISON = 0xA5


class Guarded:
    """A device tensor of the given shape and dtype inside a poisoned byte buffer."""

    def __init__(self, shape, dtype, device, fill=None):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((GUARD + n + GUARD,), POISON, dtype=torch.uint8, device=device)
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def intact(self):
        return bool((self.raw[:GUARD] == POISON).all() and (self.raw[-GUARD:] == POISON).all())


def _model(seed, dm, device):
    layers = [synth._layer(seed, l, dm, 1 / math.sqrt(dm.d), 1 / math.sqrt(dm.Hq * dm.D), 1.0,
                           device) for l in range(dm.n_layers)]
    w_lm = synth.normal((dm.V, dm.d), 0.05, seed, "w_lm", device)
    emb = synth.normal((dm.V + 1, dm.d), 1.0, seed, "emb", device)
    pos = synth.normal((dm.S, dm.d), 1.0, seed, "pos", device)
    phi = synth.phi_table(16, dm.d, seed, device)
    return layers, w_lm, emb, pos, phi


SHAPES = [
    # B, S, Hq, Hkv, D, Lmax, ctx_len
    (1, 1, 4, 1, 64, 0, None),                 # one token, no context
    (2, 4, 8, 2, 64, 130, [130, 5]),           # tiny block, ragged context past one tile
    (1, 32, 32, 2, 128, 257, None),            # S = 32: 512 query rows per KV head
    (3, 16, 32, 2, 128, 383, [383, 0, 129]),   # SM pairs, three tiles, empty and ragged
    (2, 64, 8, 2, 128, 200, [200, 63]),        # the largest block, S = 64
    (1, 48, 32, 2, 128, 129, None),            # S = 48: 96-row chunks on SM pairs
    (37, 16, 8, 2, 64, 100, None),             # B*S = 592: the GEMMs on SM pairs with a
                                               # ragged last row pair, V = 1000: a ragged
                                               # last vocabulary tile
]


@pytest.mark.parametrize("B,S,Hq,Hkv,D,Lmax,ctx", SHAPES)
def test_step_at_odd_shapes_writes_only_its_outputs_and_matches_oracle(cuda_device, B, S, Hq,
                                                                       Hkv, D, Lmax, ctx):
    dm = synth.Dims(B=B, S=S, d=256, Hq=Hq, Hkv=Hkv, D=D, V=1000, Lmax=Lmax, n_layers=2)
    layers, w_lm, emb, pos, phi = _model(101, dm, cuda_device)
    masked0 = synth.bernoulli((B, S), 0.7, 101, "m", cuda_device).to(torch.uint8)
    masked0[:, 0] = 1
    tok0 = torch.where(masked0.bool(), torch.full((B, S), dm.V, dtype=torch.int32,
                                                  device=cuda_device),
                       synth.integers((B, S), dm.V, 101, "tok", cuda_device))
    g_tok = Guarded((B, S), torch.int32, cuda_device, tok0)
    g_msk = Guarded((B, S), torch.uint8, cuda_device, masked0)
    g_conf = Guarded((B, S), torch.float32, cuda_device)
    g_pred = Guarded((B, S), torch.int32, cuda_device)
    g_ncom = Guarded((B,), torch.int32, cuda_device)
    g_done = Guarded((1,), torch.int32, cuda_device)
    nws = td.td_workspace_size(dm.as_dict(), td.TD_FN_DENOISE_STEP)
    g_ws = Guarded((max(256, nws),), torch.uint8, cuda_device)
    ctx_t = None if ctx is None else torch.tensor(ctx, dtype=torch.int32, device=cuda_device)
    td.td_denoise_step(dm.as_dict(), layers, w_lm, phi[1], 2, 16, 0.8, g_tok.t, g_msk.t,
                       emb=emb, pos=pos, ctx_len=ctx_t, conf=g_conf.t, pred=g_pred.t,
                       n_committed=g_ncom.t, all_done=g_done.t, ws=g_ws.t)
    torch.cuda.synchronize()
    assert td.td_device_error() == 0
    for g in (g_tok, g_msk, g_conf, g_pred, g_ncom, g_done, g_ws):
        assert g.intact()
    stacked_step_parity(dm.as_dict(), layers, w_lm, phi[1], 2, 16, 0.8, tok0, masked0,
                        dict(conf=g_conf.t.cpu().numpy(), pred=g_pred.t.cpu().numpy(),
                             tokens=g_tok.t.cpu().numpy(), masked=g_msk.t.cpu().numpy()),
                        emb=emb, pos=pos, ctx_len=ctx)


def test_attention_lmhead_and_append_write_only_their_outputs(cuda_device):
    B, S, Hq, Hkv, D, Lmax, V, d = 3, 16, 32, 2, 128, 300, 4096, 512
    dims = td.make_dims(B=B, S=S, d=d, Hq=Hq, Hkv=Hkv, D=D, V=V, Lmax=Lmax, n_layers=1)
    q = synth.normal((B, S, Hq, D), 1.0, 7, "q", cuda_device)
    kb = synth.normal((B, S, Hkv, D), 1.0, 7, "kb", cuda_device)
    vb = synth.normal((B, S, Hkv, D), 1.0, 7, "vb", cuda_device)
    kc = Guarded((B, Hkv, Lmax, D), torch.bfloat16, cuda_device,
                 synth.normal((B, Hkv, Lmax, D), 1.0, 7, "kc", cuda_device))
    vc = Guarded((B, Hkv, Lmax, D), torch.bfloat16, cuda_device,
                 synth.normal((B, Hkv, Lmax, D), 1.0, 7, "vc", cuda_device))
    o = Guarded((B, S, Hq, D), torch.bfloat16, cuda_device)
    lse = Guarded((B, S, Hq), torch.float32, cuda_device)
    aws = Guarded((max(256, td.td_workspace_size(dims, td.TD_FN_BLOCK_ATTENTION)),),
                  torch.uint8, cuda_device)
    ctx = torch.tensor([300, 17, 150], dtype=torch.int32, device=cuda_device)
    td.td_block_attention(dims, q, kb, vb, kc.t, vc.t, ctx, o=o.t, lse=lse.t, ws=aws.t)
    # the LM head + commit with every buffer guarded
    M = B * S
    h = synth.normal((M, d), 1.0, 7, "h", cuda_device)
    w = synth.normal((V, d), 0.3, 7, "w", cuda_device)
    tok = Guarded((B, S), torch.int32, cuda_device, torch.full((B, S), V, dtype=torch.int32))
    msk = Guarded((B, S), torch.uint8, cuda_device, torch.ones((B, S), dtype=torch.uint8))
    conf = Guarded((B, S), torch.float32, cuda_device)
    pred = Guarded((B, S), torch.int32, cuda_device)
    ncom = Guarded((B,), torch.int32, cuda_device)
    done = Guarded((1,), torch.int32, cuda_device)
    lws = Guarded((max(256, td.td_workspace_size(dims, td.TD_FN_LMHEAD_COMMIT)),), torch.uint8,
                  cuda_device)
    td.td_lmhead_commit(dims, h, w, 0.8, False, tok.t, msk.t, conf=conf.t, pred=pred.t,
                        n_committed=ncom.t, all_done=done.t, ws=lws.t)
    # a cache append at the end of the capacity of one sequence
    ctx2 = torch.tensor([284, 0, 100], dtype=torch.int32, device=cuda_device)
    new = [(synth.normal((B, S, Hkv, D), 1.0, 7, "kn", cuda_device),
            synth.normal((B, S, Hkv, D), 1.0, 7, "vn", cuda_device))]
    lay = dict(wqkv=h, wo=h, ada_E=torch.zeros(16, device=cuda_device), k_ctx=kc.t, v_ctx=vc.t)
    td.td_kv_append(dims, [lay], new, ctx2)
    torch.cuda.synchronize()
    assert td.td_device_error() == 0
    for g in (kc, vc, o, lse, aws, tok, msk, conf, pred, ncom, done, lws):
        assert g.intact()
    assert ctx2.cpu().tolist() == [300, 16, 116]


def test_lmhead_on_sm_pairs_with_ragged_rows_and_vocabulary(cuda_device):
    # 592 rows: the last 256-row pair tile holds 80 live rows; V = 1000: the last 256-column
    # vocabulary tile holds 232 columns. Every written buffer is guarded; sampled rows in
    # every row tile, the ragged one included, match the oracle.
    import oracle
    from parity_util import compare_commit
    B, S, d, V = 37, 16, 512, 1000
    M = B * S
    dims = td.make_dims(B=B, S=S, d=d, Hq=8, Hkv=2, D=64, V=V, Lmax=0, n_layers=0)
    h = synth.normal((M, d), 1.0, 13, "h", cuda_device)
    w = synth.normal((V, d), 0.2, 13, "w", cuda_device)
    t0 = torch.full((B, S), V, dtype=torch.int32)
    tok = Guarded((B, S), torch.int32, cuda_device, t0)
    msk = Guarded((B, S), torch.uint8, cuda_device, torch.ones((B, S), dtype=torch.uint8))
    conf = Guarded((B, S), torch.float32, cuda_device)
    pred = Guarded((B, S), torch.int32, cuda_device)
    ncom = Guarded((B,), torch.int32, cuda_device)
    done = Guarded((1,), torch.int32, cuda_device)
    lws = Guarded((max(256, td.td_workspace_size(dims, td.TD_FN_LMHEAD_COMMIT)),), torch.uint8,
                  cuda_device)
    td.td_lmhead_commit(dims, h, w, 0.8, False, tok.t, msk.t, conf=conf.t, pred=pred.t,
                        n_committed=ncom.t, all_done=done.t, ws=lws.t)
    torch.cuda.synchronize()
    assert td.td_device_error() == 0
    for g in (tok, msk, conf, pred, ncom, done, lws):
        assert g.intact()
    seqs = [0, 15, 16, 31, 32, 36]          # rows 0.., 240.., 256.., 496.., 512.., 576..591
    rows = [b * S + i for b in seqs for i in range(S)]
    c_ref, p_ref, gap, _ = oracle.lmhead_confidence(h, w, rows=rows)
    nb = len(seqs)
    tok_ref, msk_ref, _, _ = oracle.commit(c_ref.reshape(nb, S), p_ref.reshape(nb, S),
                                           t0[seqs].numpy(), np.ones((nb, S), bool), 0.8, False)
    compare_commit(dict(conf=c_ref.reshape(nb, S), pred=p_ref.reshape(nb, S),
                        gap=gap.reshape(nb, S), tokens=tok_ref, masked=msk_ref),
                   dict(conf=conf.t[seqs].cpu().numpy(), pred=pred.t[seqs].cpu().numpy(),
                        tokens=tok.t[seqs].cpu().numpy(), masked=msk.t[seqs].cpu().numpy()),
                   np.ones((nb, S), bool), 0.8)
