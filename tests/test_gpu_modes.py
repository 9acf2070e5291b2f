"""GPU parity of the mode variants and of multi-block generation against the fp64 oracle:
the left-to-right commit rule (the mock-AR reading), the context-cache append, and several
blocks decoded in a row with the cache growing between them."""

import math

import numpy as np
import pytest
import torch

import block_diffusion_lm_denoise_b300 as td
import oracle
from block_diffusion_lm_denoise_b300 import synth
from parity_util import attention_close, compare_commit, first_masked, stacked_step_parity

pytestmark = pytest.mark.gpu

L2R = td.TD_COMMIT_LEFT_TO_RIGHT


def _np(t):
    return oracle.as_f64(t)


def test_lmhead_left_to_right_commits_the_lowest_masked_position(cuda_device):
    M, S, V, d = 64, 16, 2048, 256
    h = synth.normal((M, d), 1.0, 31, "h", cuda_device)
    w = synth.normal((V, d), 0.3, 31, "w", cuda_device)
    B = M // S
    masked = synth.bernoulli((B, S), 0.6, 31, "m", cuda_device).to(torch.uint8)
    masked[0] = 0                                   # a finished sequence stays untouched
    tokens = torch.where(masked.bool(), torch.full((B, S), V, dtype=torch.int32, device=cuda_device),
                         synth.integers((B, S), V, 31, "t", cuda_device))
    t0, m0 = tokens.clone(), masked.clone()
    dims = td.make_dims(B=B, S=S, d=d, Hq=1, Hkv=1, D=64, V=V, Lmax=0, n_layers=0)
    conf, pred, ncom, done = td.td_lmhead_commit(dims, h, w, 0.0, False, tokens, masked, rule=L2R)
    torch.cuda.synchronize()
    assert td.td_device_error() == 0
    c, p, gap, _ = oracle.lmhead_confidence(h, w)
    tok_ref, msk_ref, n_ref, _ = oracle.commit(c.reshape(B, S), p.reshape(B, S), t0.cpu().numpy(),
                                               m0.cpu().numpy().astype(bool), 0.0, False,
                                               rule=oracle.RULE_LEFT_TO_RIGHT)
    compare_commit(dict(conf=c.reshape(B, S), pred=p.reshape(B, S), gap=gap.reshape(B, S),
                        tokens=tok_ref, masked=msk_ref),
                   dict(conf=conf.cpu().numpy(), pred=pred.cpu().numpy(),
                        tokens=tokens.cpu().numpy(), masked=masked.cpu().numpy()),
                   m0.cpu().numpy(), 0.0)
    assert list(ncom.cpu().numpy()) == list(n_ref) and n_ref[0] == 0 and (n_ref[1:] == 1).all()


def _small_model(seed, dm, cuda_device, w_scale=0.05):
    layers = [synth._layer(seed, l, dm, 1 / math.sqrt(dm.d), 1 / math.sqrt(dm.Hq * dm.D), 1.0,
                           cuda_device) for l in range(dm.n_layers)]
    w_lm = synth.normal((dm.V, dm.d), w_scale, seed, "w_lm", cuda_device)
    emb = synth.normal((dm.V + 1, dm.d), 1.0, seed, "emb", cuda_device)
    pos = synth.normal((dm.S, dm.d), 1.0, seed, "pos", cuda_device)
    phi = synth.phi_table(dm.S, dm.d, seed, cuda_device)
    return layers, w_lm, emb, pos, phi


@pytest.mark.parametrize("D", [64, 128])
def test_denoise_step_left_to_right_evaluates_one_row_per_sequence(cuda_device, D):
    dm = synth.Dims(B=3, S=16, d=256, Hq=8, Hkv=2, D=D, V=1024, Lmax=100, n_layers=2)
    layers, w_lm, emb, pos, phi = _small_model(41, dm, cuda_device)
    masked = synth.bernoulli((dm.B, dm.S), 0.5, 41, "m", cuda_device).to(torch.uint8)
    masked[1] = 0
    tokens = torch.where(masked.bool(), torch.full((dm.B, dm.S), dm.V, dtype=torch.int32,
                                                   device=cuda_device),
                         synth.integers((dm.B, dm.S), dm.V, 41, "tok", cuda_device))
    ctx = torch.tensor([100, 37, 0], dtype=torch.int32, device=cuda_device)
    t0, m0 = tokens.clone(), masked.clone()
    conf, pred, ncom, done = td.td_denoise_step(dm.as_dict(), layers, w_lm, phi[4], 5, 16, 0.8,
                                                tokens, masked, emb=emb, pos=pos, ctx_len=ctx,
                                                rule=L2R)
    torch.cuda.synchronize()
    assert td.td_device_error() == 0
    r = oracle.denoise_step(dm.as_dict(), layers, phi[4], w_lm, t0.cpu().numpy(),
                            m0.cpu().numpy().astype(bool), 0.8, 5, 16, emb=emb, pos=pos,
                            ctx_len=[100, 37, 0], rule=oracle.RULE_LEFT_TO_RIGHT)
    m0n = m0.cpu().numpy().astype(bool)
    compare_commit(r, dict(conf=conf.cpu().numpy(), pred=pred.cpu().numpy(),
                           tokens=tokens.cpu().numpy(), masked=masked.cpu().numpy()),
                   m0n, 0.8, step=True, evaluated=first_masked(m0n))
    assert list(ncom.cpu().numpy()) == [int(m0n[b].any()) for b in range(dm.B)]


def test_decode_block_left_to_right_takes_s_steps_in_order(cuda_device):
    dm = synth.Dims(B=2, S=8, d=256, Hq=8, Hkv=2, D=128, V=1024, Lmax=130, n_layers=2)
    layers, w_lm, emb, pos, phi = _small_model(43, dm, cuda_device)
    tokens = torch.full((dm.B, dm.S), dm.V, dtype=torch.int32, device=cuda_device)
    masked = torch.ones((dm.B, dm.S), dtype=torch.uint8, device=cuda_device)
    steps = td.td_decode_block(dm.as_dict(), layers, emb, pos, w_lm, phi, dm.S, 0.0, tokens,
                               masked, rule=L2R)
    torch.cuda.synchronize()
    assert td.td_device_error() == 0
    assert steps == dm.S and not masked.any()
    tok_ref, msk_ref, steps_ref, recs = oracle.decode_block(
        dm.as_dict(), [{k: v.cpu() for k, v in L.items()} for L in layers], phi.cpu(),
        w_lm.cpu(), emb.cpu(), pos.cpu(), 0.0, dm.S, trace=True, rule=oracle.RULE_LEFT_TO_RIGHT)
    assert steps_ref == dm.S
    # ids are compared up to the first step whose committed position has a near-tie argmax
    # (top-2 logit gap under 1e-4): from there on the two runs may legitimately differ
    got = tokens.cpu().numpy()
    for t, rec in enumerate(recs):
        if (rec["gap"][:, t] < 1e-4).any():
            break
        assert np.array_equal(got[:, t], tok_ref[:, t]), t


@pytest.mark.parametrize("form", [td.TD_GRAPH_CONDITIONAL, td.TD_GRAPH_FLAT])
def test_decode_block_resumes_a_stopped_loop(cuda_device, form):
    # a block decoded for three steps through td_denoise_step and then handed to the loop at
    # t_start = 4 ends exactly like the loop run from step 1 (the graph built for t_start = 4
    # holds steps 4..T only); a block with nothing masked takes no step
    dm = synth.Dims(B=3, S=16, d=256, Hq=8, Hkv=2, D=128, V=1024, Lmax=64, n_layers=2)
    layers, w_lm, emb, pos, phi = _small_model(47, dm, cuda_device, w_scale=0.08)
    ctx = torch.tensor([64, 20, 0], dtype=torch.int32, device=cuda_device)
    ws = td.workspace(dm.as_dict(), td.TD_FN_DECODE_BLOCK, cuda_device)

    def fresh():
        return (torch.full((dm.B, dm.S), dm.V, dtype=torch.int32, device=cuda_device),
                torch.ones((dm.B, dm.S), dtype=torch.uint8, device=cuda_device))

    td.td_decode_graph_form(form)
    try:
        tf, mf = fresh()
        steps_full = td.td_decode_block(dm.as_dict(), layers, emb, pos, w_lm, phi, dm.S, 0.8,
                                        tf, mf, ctx_len=ctx, ws=ws)
        torch.cuda.synchronize()
        assert td.td_device_error() == 0 and not mf.any()
        assert steps_full > 3, steps_full
        tp, mp = fresh()
        for t in range(1, 4):
            td.td_denoise_step(dm.as_dict(), layers, w_lm, phi[t - 1], t, dm.S, 0.8, tp, mp,
                               emb=emb, pos=pos, ctx_len=ctx, ws=ws)
        steps_rest = td.td_decode_block(dm.as_dict(), layers, emb, pos, w_lm, phi, dm.S, 0.8,
                                        tp, mp, t_start=4, ctx_len=ctx, ws=ws)
        torch.cuda.synchronize()
        assert td.td_device_error() == 0 and not mp.any()
        assert td.td_decode_graph_form() == form
        assert steps_rest == steps_full - 3
        assert torch.equal(tp, tf)
        # nothing masked on entry: no step runs and the block is left as it is
        steps_none = td.td_decode_block(dm.as_dict(), layers, emb, pos, w_lm, phi, dm.S, 0.8,
                                        tp, mp, ctx_len=ctx, ws=ws)
        torch.cuda.synchronize()
        assert steps_none == 0 and torch.equal(tp, tf)
    finally:
        td.td_decode_graph_form(td.TD_GRAPH_CONDITIONAL)


def test_kv_append_matches_oracle_and_flags_overflow(cuda_device):
    B, S, Hkv, D, Lmax, n_layers = 3, 16, 2, 128, 70, 2
    dm = td.make_dims(B=B, S=S, d=256, Hq=8, Hkv=Hkv, D=D, V=64, Lmax=Lmax, n_layers=n_layers)
    layers, new = [], []
    for l in range(n_layers):
        layers.append(dict(wqkv=torch.zeros(16, dtype=torch.bfloat16, device=cuda_device),
                           wo=torch.zeros(16, dtype=torch.bfloat16, device=cuda_device),
                           ada_E=torch.zeros(16, device=cuda_device),
                           k_ctx=synth.normal((B, Hkv, Lmax, D), 1.0, 51, f"k{l}", cuda_device),
                           v_ctx=synth.normal((B, Hkv, Lmax, D), 1.0, 51, f"v{l}", cuda_device)))
        new.append((synth.normal((B, S, Hkv, D), 1.0, 51, f"kn{l}", cuda_device),
                    synth.normal((B, S, Hkv, D), 1.0, 51, f"vn{l}", cuda_device)))
    start = [20, 54, 60]          # the last one would pass Lmax = 70
    ctx = torch.tensor(start, dtype=torch.int32, device=cuda_device)
    before = [(L["k_ctx"].clone(), L["v_ctx"].clone()) for L in layers]
    td.td_kv_append(dm, layers, new, ctx)
    torch.cuda.synchronize()
    assert td.td_device_error() == 0x600
    for l in range(n_layers):
        k2, v2, ln, ovf = oracle.kv_append(before[l][0], before[l][1], start, new[l][0], new[l][1])
        assert np.array_equal(_np(layers[l]["k_ctx"]), k2)
        assert np.array_equal(_np(layers[l]["v_ctx"]), v2)
        assert list(ovf) == [False, False, True]
    assert ctx.cpu().tolist() == [36, 70, 60]


def test_three_blocks_with_the_cache_growing_between_them(cuda_device):
    # multi-block generation: decode a block, append the context tower's keys / values of the
    # committed block (a seeded per-token stand-in for that tower), decode the next block.
    # Every step is compared with the oracle fed the GPU's state before that step (stage by
    # stage: layers, then LM head and commit on the GPU's final hidden state), so a near-tie
    # decision (excluded by the shared rules) cannot hide later mismatches.
    dm = synth.Dims(B=3, S=16, d=256, Hq=8, Hkv=2, D=128, V=2048, Lmax=90 + 3 * 16,
                    n_layers=2)
    layers, w_lm, emb, pos, phi = _small_model(61, dm, cuda_device, w_scale=0.08)
    # stand-in context tower: per layer a table token -> (k, v) rows [V + 1, Hkv, D]
    ktab = [synth.normal((dm.V + 1, dm.Hkv, dm.D), 1.0, 61, f"ktab{l}", cuda_device)
            for l in range(dm.n_layers)]
    vtab = [synth.normal((dm.V + 1, dm.Hkv, dm.D), 1.0, 61, f"vtab{l}", cuda_device)
            for l in range(dm.n_layers)]
    ctx = torch.tensor([90, 12, 0], dtype=torch.int32, device=cuda_device)
    cpu_layers = [{k: v.cpu() for k, v in L.items()} for L in layers]
    ctx_ref = [90, 12, 0]
    ws = td.workspace(dm.as_dict(), td.TD_FN_DECODE_BLOCK, cuda_device)
    for blk in range(3):
        tokens = torch.full((dm.B, dm.S), dm.V, dtype=torch.int32, device=cuda_device)
        masked = torch.ones((dm.B, dm.S), dtype=torch.uint8, device=cuda_device)
        # step by step through td_denoise_step, each step checked against the oracle
        tk, mk = tokens.clone(), masked.clone()
        for t in range(1, dm.S + 1):
            t_before, m_before = tk.clone(), mk.clone()
            conf, pred, ncom, done = td.td_denoise_step(dm.as_dict(), layers, w_lm, phi[t - 1],
                                                        t, dm.S, 0.8, tk, mk, emb=emb, pos=pos,
                                                        ctx_len=ctx, ws=ws)
            torch.cuda.synchronize()
            stacked_step_parity(dm.as_dict(), layers, w_lm, phi[t - 1], t, dm.S, 0.8, t_before,
                                m_before, dict(conf=conf.cpu().numpy(), pred=pred.cpu().numpy(),
                                               tokens=tk.cpu().numpy(),
                                               masked=mk.cpu().numpy()),
                                emb=emb, pos=pos, ctx_len=ctx_ref)
            if int(done.item()):
                break
        # the loop entry point reproduces the step-by-step run bit for bit
        steps = td.td_decode_block(dm.as_dict(), layers, emb, pos, w_lm, phi, dm.S, 0.8, tokens,
                                   masked, ctx_len=ctx, ws=ws)
        torch.cuda.synchronize()
        assert td.td_device_error() == 0 and not masked.any() and steps == t
        assert torch.equal(tokens, tk), blk
        if blk == 0:
            # the flat form of the loop graph (finished steps launch and return at once)
            # decodes the same block in the same number of steps
            assert td.td_decode_graph_form() == td.TD_GRAPH_CONDITIONAL
            tf = torch.full_like(tokens, dm.V)
            mf = torch.ones_like(masked)
            td.td_decode_graph_form(td.TD_GRAPH_FLAT)
            try:
                steps_f = td.td_decode_block(dm.as_dict(), layers, emb, pos, w_lm, phi, dm.S,
                                             0.8, tf, mf, ctx_len=ctx, ws=ws)
                torch.cuda.synchronize()
                assert td.td_decode_graph_form() == td.TD_GRAPH_FLAT
            finally:
                td.td_decode_graph_form(td.TD_GRAPH_CONDITIONAL)
            assert steps_f == steps and torch.equal(tf, tokens) and not mf.any()
        # grow the caches with the committed block (the same tokens on both sides)
        tok = tokens.long()
        new = [(ktab[l][tok].contiguous(), vtab[l][tok].contiguous()) for l in range(dm.n_layers)]
        td.td_kv_append(dm.as_dict(), layers, new, ctx)
        torch.cuda.synchronize()
        assert td.td_device_error() == 0
        for l in range(dm.n_layers):
            k2, v2, ln, ovf = oracle.kv_append(cpu_layers[l]["k_ctx"], cpu_layers[l]["v_ctx"],
                                               ctx_ref, new[l][0], new[l][1])
            assert np.array_equal(_np(layers[l]["k_ctx"]), k2)
            assert np.array_equal(_np(layers[l]["v_ctx"]), v2)
            cpu_layers[l]["k_ctx"] = torch.from_numpy(k2).to(torch.bfloat16)
            cpu_layers[l]["v_ctx"] = torch.from_numpy(v2).to(torch.bfloat16)
        ctx_ref = [c + dm.S for c in ctx_ref]
        assert ctx.cpu().tolist() == ctx_ref


@pytest.mark.parametrize("Hq,D", [(8, 64), (32, 128)])
def test_denoise_step_rotary_variant_matches_oracle(cuda_device, Hq, D):
    # Hq = 32, D = 128 runs the SM-pair attention, Hq = 8, D = 64 the single-SM one
    theta = 10000.0
    dm = synth.Dims(B=3, S=16, d=256, Hq=Hq, Hkv=2, D=D, V=1024, Lmax=150, n_layers=2)
    layers, w_lm, emb, pos, phi = _small_model(71, dm, cuda_device)
    masked = synth.bernoulli((dm.B, dm.S), 0.7, 71, "m", cuda_device).to(torch.uint8)
    tokens = torch.where(masked.bool(), torch.full((dm.B, dm.S), dm.V, dtype=torch.int32,
                                                   device=cuda_device),
                         synth.integers((dm.B, dm.S), dm.V, 71, "tok", cuda_device))
    ctx = torch.tensor([150, 61, 0], dtype=torch.int32, device=cuda_device)
    t0, m0 = tokens.clone(), masked.clone()
    conf, pred, ncom, done = td.td_denoise_step(dm.as_dict(), layers, w_lm, phi[2], 3, 16, 0.8,
                                                tokens, masked, emb=emb, pos=pos, ctx_len=ctx,
                                                rope_theta=theta)
    torch.cuda.synchronize()
    assert td.td_device_error() == 0
    cpu_layers = [{k: v.cpu() for k, v in L.items()} for L in layers]
    m0n = m0.cpu().numpy().astype(bool)
    stacked_step_parity(dm.as_dict(), layers, w_lm, phi[2], 3, 16, 0.8, t0, m0,
                        dict(conf=conf.cpu().numpy(), pred=pred.cpu().numpy(),
                             tokens=tokens.cpu().numpy(), masked=masked.cpu().numpy()),
                        emb=emb, pos=pos, ctx_len=[150, 61, 0], rope_theta=theta)
    # the rotation changes the result: the same step without it differs
    r = oracle.denoise_step(dm.as_dict(), cpu_layers, phi[2].cpu(), w_lm.cpu(), t0.cpu().numpy(),
                            m0n, 0.8, 3, 16, emb=emb.cpu(), pos=pos.cpu(), ctx_len=[150, 61, 0],
                            rope_theta=theta)
    r0 = oracle.denoise_step(dm.as_dict(), cpu_layers, phi[2].cpu(), w_lm.cpu(), t0.cpu().numpy(),
                             m0n, 0.8, 3, 16, emb=emb.cpu(), pos=pos.cpu(), ctx_len=[150, 61, 0])
    assert np.abs(r0["conf"] - r["conf"]).max() > 1e-4
    # the loop entry point with the variant reproduces step-by-step calls bit for bit
    tk = torch.full((dm.B, dm.S), dm.V, dtype=torch.int32, device=cuda_device)
    mk = torch.ones((dm.B, dm.S), dtype=torch.uint8, device=cuda_device)
    tb, mb = tk.clone(), mk.clone()
    for t in range(1, dm.S + 1):
        _, _, _, dn = td.td_denoise_step(dm.as_dict(), layers, w_lm, phi[t - 1], t, dm.S, 0.8,
                                         tk, mk, emb=emb, pos=pos, ctx_len=ctx, rope_theta=theta)
        if int(dn.item()):
            break
    steps = td.td_decode_block(dm.as_dict(), layers, emb, pos, w_lm, phi, dm.S, 0.8, tb, mb,
                               ctx_len=ctx, rope_theta=theta)
    torch.cuda.synchronize()
    assert steps == t and torch.equal(tb, tk) and not mb.any()


# ------------------------------------------------------------------------------ paged cache

def _page_pool(cache, page_table, n_pages):
    """A pool [n_pages, Hkv, 128, D] holding the contiguous cache [B, Hkv, Lmax, D] at the
    pages page_table[b, t] (other pages and rows past Lmax: zeros)."""
    B, Hkv, Lmax, D = cache.shape
    pool = torch.zeros((n_pages, Hkv, 128, D), dtype=cache.dtype, device=cache.device)
    for b in range(B):
        for t in range((Lmax + 127) // 128):
            rows = min(128, Lmax - 128 * t)
            pool[int(page_table[b, t]), :, :rows] = cache[b, :, 128 * t:128 * t + rows]
    return pool


def _shuffled_pages(B, max_pages, n_pages, seed, device):
    perm = synth.integers((n_pages,), 1 << 30, seed, "perm", "cpu").argsort()[: B * max_pages]
    return perm.reshape(B, max_pages).to(torch.int32).to(device)


@pytest.mark.parametrize("Hq,D", [(32, 128), (8, 64)])
def test_paged_attention_equals_contiguous_and_oracle(cuda_device, Hq, D):
    B, S, Hkv, Lmax = 3, 16, 2, 400
    ctx = [400, 130, 0]
    q = synth.normal((B, S, Hq, D), 1.0, 81, "q", cuda_device)
    kb = synth.normal((B, S, Hkv, D), 1.0, 81, "kb", cuda_device)
    vb = synth.normal((B, S, Hkv, D), 1.0, 81, "vb", cuda_device)
    kc = synth.normal((B, Hkv, Lmax, D), 1.0, 81, "kc", cuda_device)
    vc = synth.normal((B, Hkv, Lmax, D), 1.0, 81, "vc", cuda_device)
    max_pages, n_pages = 4, 17
    pt = _shuffled_pages(B, max_pages, n_pages, 81, cuda_device)
    kp, vp = _page_pool(kc, pt.cpu(), n_pages), _page_pool(vc, pt.cpu(), n_pages)
    ctx_t = torch.tensor(ctx, dtype=torch.int32, device=cuda_device)
    dims = td.make_dims(B=B, S=S, d=64, Hq=Hq, Hkv=Hkv, D=D, V=8, Lmax=Lmax, n_layers=1)
    o_c = td.td_block_attention(dims, q, kb, vb, kc, vc, ctx_t)
    o_p = td.td_block_attention(dims, q, kb, vb, kp, vp, ctx_t, page_table=pt, n_pages=n_pages)
    torch.cuda.synchronize()
    assert td.td_device_error() == 0
    assert torch.equal(o_c, o_p)
    o_ref, _ = oracle.block_attention(q, kb, vb, kc, vc, ctx)
    ok, worst = attention_close(_np(o_p), o_ref)
    assert ok, worst


def test_paged_append_and_step_equal_the_contiguous_layout(cuda_device):
    dm = synth.Dims(B=3, S=16, d=256, Hq=32, Hkv=2, D=128, V=1024, Lmax=300, n_layers=2)
    layers, w_lm, emb, pos, phi = _small_model(91, dm, cuda_device)
    max_pages, n_pages = 3, 11
    pt = _shuffled_pages(dm.B, max_pages, n_pages, 91, cuda_device)
    paged = [dict(L, k_ctx=_page_pool(L["k_ctx"], pt.cpu(), n_pages),
                  v_ctx=_page_pool(L["v_ctx"], pt.cpu(), n_pages)) for L in layers]
    start = [120, 250, 0]
    ctx_c = torch.tensor(start, dtype=torch.int32, device=cuda_device)
    ctx_p = ctx_c.clone()
    new = [(synth.normal((dm.B, dm.S, dm.Hkv, dm.D), 1.0, 91, f"kn{l}", cuda_device),
            synth.normal((dm.B, dm.S, dm.Hkv, dm.D), 1.0, 91, f"vn{l}", cuda_device))
           for l in range(dm.n_layers)]
    before = [(L["k_ctx"].cpu(), L["v_ctx"].cpu()) for L in layers]
    td.td_kv_append(dm.as_dict(), layers, new, ctx_c)
    td.td_kv_append(dm.as_dict(), paged, new, ctx_p, page_table=pt, n_pages=n_pages)
    torch.cuda.synchronize()
    assert td.td_device_error() == 0
    assert torch.equal(ctx_c, ctx_p) and ctx_p.cpu().tolist() == [s + dm.S for s in start]
    for l in range(dm.n_layers):
        k2, v2, _, _ = oracle.kv_append(before[l][0], before[l][1], start, new[l][0], new[l][1])
        ref_pool = _page_pool(torch.from_numpy(k2).to(torch.bfloat16), pt.cpu(), n_pages)
        assert torch.equal(paged[l]["k_ctx"].cpu(), ref_pool)
        assert torch.equal(layers[l]["k_ctx"].cpu(), torch.from_numpy(k2).to(torch.bfloat16))
    # one denoise step on either layout gives the same bits
    outs = []
    for lays, kw in ((layers, {}), (paged, dict(page_table=pt, n_pages=n_pages))):
        tk = torch.full((dm.B, dm.S), dm.V, dtype=torch.int32, device=cuda_device)
        mk = torch.ones((dm.B, dm.S), dtype=torch.uint8, device=cuda_device)
        conf, pred, _, _ = td.td_denoise_step(dm.as_dict(), lays, w_lm, phi[0], 1, 16, 0.8, tk,
                                              mk, emb=emb, pos=pos, ctx_len=ctx_c, **kw)
        outs.append((conf.clone(), pred.clone(), tk.clone(), mk.clone()))
    torch.cuda.synchronize()
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_paged_attention_at_full_size_is_bit_identical_to_contiguous(cuda_device):
    # the bench's attention shape: 64 sequences x 2 KV heads x 8192 keys, pages shuffled
    wl = synth.attention_sweep(8192, cuda_device, B=64)
    lay = wl.layers[0]
    dm = wl.dims
    B, Hkv, L, D = lay["k_ctx"].shape
    T = L // 128
    perm = synth.integers((B * T,), 1 << 30, 123, "perm", "cpu").argsort().to(cuda_device)
    page_table = perm.reshape(B, T).to(torch.int32)

    def pool_of(cache):
        tiles = cache.view(B, Hkv, T, 128, D).permute(0, 2, 1, 3, 4).reshape(B * T, Hkv, 128, D)
        pool = torch.empty_like(tiles)
        pool[perm] = tiles
        return pool

    kp, vp = pool_of(lay["k_ctx"]), pool_of(lay["v_ctx"])
    ctx = torch.tensor([L - 37 * b for b in range(B)], dtype=torch.int32, device=cuda_device)
    o_c = td.td_block_attention(dm.as_dict(), lay["q"], lay["k_blk"], lay["v_blk"], lay["k_ctx"],
                                lay["v_ctx"], ctx)
    o_p = td.td_block_attention(dm.as_dict(), lay["q"], lay["k_blk"], lay["v_blk"], kp, vp, ctx,
                                page_table=page_table, n_pages=B * T)
    torch.cuda.synchronize()
    assert td.td_device_error() == 0
    assert torch.equal(o_c, o_p)



def test_decode_loops_from_four_threads_match_one_thread(cuda_device):
    # Four host threads run the block decode loop at once, each on its own stream with its
    # own state and workspace (so each captures a graph of its own): every result equals the
    # one of the same loop run alone, and repeated calls (cached graphs) agree too.
    import threading
    dm = synth.Dims(B=2, S=16, d=256, Hq=8, Hkv=2, D=128, V=2048, Lmax=100, n_layers=2)
    layers, w_lm, emb, pos, phi = _small_model(71, dm, cuda_device, w_scale=0.08)
    ctx = torch.tensor([100, 41], dtype=torch.int32, device=cuda_device)

    def state():
        return dict(tokens=torch.full((dm.B, dm.S), dm.V, dtype=torch.int32, device=cuda_device),
                    masked=torch.ones((dm.B, dm.S), dtype=torch.uint8, device=cuda_device),
                    ws=td.workspace(dm.as_dict(), td.TD_FN_DECODE_BLOCK, cuda_device),
                    outs=td._outs(dm.B, dm.S, cuda_device, None, None, None, None),
                    stream=torch.cuda.Stream(cuda_device))

    def decode(st):
        with torch.cuda.stream(st["stream"]):   # ordered before the loop on its stream
            st["tokens"].fill_(dm.V)
            st["masked"].fill_(1)
        c, p, n, a = st["outs"]
        return td.td_decode_block(dm.as_dict(), layers, emb, pos, w_lm, phi, dm.S, 0.8,
                                  st["tokens"], st["masked"], ctx_len=ctx, conf=c, pred=p,
                                  n_committed=n, all_done=a, ws=st["ws"], stream=st["stream"])

    alone = state()
    steps_ref = decode(alone)
    tokens_ref = alone["tokens"].clone()
    assert td.td_device_error() == 0 and not alone["masked"].any()

    states = [state() for _ in range(4)]
    results, errors = [None] * 4, []

    def worker(i):
        try:
            runs = []
            for _ in range(3):
                steps = decode(states[i])
                runs.append((steps, states[i]["tokens"].clone(), states[i]["masked"].clone()))
            results[i] = runs
        except Exception as e:   # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    torch.cuda.synchronize()
    assert not errors, errors
    assert td.td_device_error() == 0
    for runs in results:
        assert runs is not None
        for steps, tokens, masked in runs:
            assert steps == steps_ref
            assert torch.equal(tokens, tokens_ref)
            assert not masked.any()
