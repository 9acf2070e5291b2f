"""Pins of the fp64 oracle against facts that do not come from the oracle itself:
closed forms, library routines for special cases, invariants of the method stated on the
pages, hand-derived golden cases and brute force on tiny inputs. CPU only.

A plausible slip in the oracle (a dropped 1/sqrt(D), a wrong GQA index, x W instead of
x W^T, a strict instead of inclusive threshold, a highest- instead of lowest-index tie
break, a missing gate, a sign) makes at least one of these fail.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from block_diffusion_lm_denoise_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def bf16_exact(shape, scale=1.0):
    """Random values that are exactly representable in bf16 (via torch's own rounding)."""
    x = torch.from_numpy(rng.standard_normal(shape) * scale).float().to(torch.bfloat16)
    return x.double().numpy()


# ----------------------------------------------------------------------------- bf16

def test_bf16_round_matches_torch_conversion():
    x = rng.standard_normal(200000).astype(np.float32) * np.float32(3.0)
    x = np.concatenate([x, np.float32([1.0 + 2**-8, 1.0 + 3 * 2**-8, -1.0 - 2**-8, 0.0,
                                        2.0**-100, 65504.0, 1e30])])
    ours = oracle.bf16_round(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    assert np.array_equal(ours, ref)


def test_bf16_round_ties_to_even_closed_form():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties go to the even mantissa (1.0)
    assert oracle.bf16_round(1.0 + 2**-8) == 1.0
    # 1 + 3*2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: even is 1 + 2^-6
    assert oracle.bf16_round(1.0 + 3 * 2**-8) == 1.0 + 2**-6
    # just above the tie rounds up
    assert oracle.bf16_round(1.0 + 2**-8 + 2**-30) == 1.0 + 2**-7


def test_bf16_round_is_not_a_double_rounding_through_float32():
    # a value whose fp32 rounding lands exactly on a bf16 tie; the direct rounding must not
    x = 1.0 + 2**-8 + 2**-40          # fp32(x) == 1 + 2^-8 (a tie), true value is above it
    assert oracle.bf16_round(x) == 1.0 + 2**-7


# ----------------------------------------------------------------------------- LayerNorm / adaLN

def test_layernorm_matches_torch_layer_norm_without_affine():
    h = rng.standard_normal((7, 96)) * 3 + 1.5
    ours = oracle.layer_norm(h)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(h), (96,), eps=oracle.LN_EPS).numpy()
    assert np.allclose(ours, ref, rtol=0, atol=1e-12)


def test_layernorm_moments_closed_form():
    h = rng.standard_normal((5, 128)) * 2.0
    x = oracle.layer_norm(h)
    var = h.var(axis=1)
    assert np.allclose(x.mean(axis=1), 0.0, atol=1e-12)
    # population variance of the output is var / (var + eps) exactly
    assert np.allclose(x.var(axis=1), var / (var + oracle.LN_EPS), rtol=1e-12)


def test_adaln_zero_modulation_is_plain_layernorm_rounded():
    d = 64
    h = bf16_exact((4, d))
    E = np.zeros((6, d)); phi = np.zeros((6, d))
    assert np.array_equal(oracle.adaln_modulate(h, E, phi), oracle.bf16_round(oracle.layer_norm(h)))


def test_adaln_constant_row_gives_shift_exactly():
    # a constant row has zero variance: x_hat = 0, so x_mod = bf16(shift)
    d = 32
    h = np.full((1, d), 0.75)
    E = np.zeros((6, d)); phi = np.zeros((6, d))
    E[0] = np.linspace(-1, 1, d); phi[0] = 0.125; E[1] = 5.0
    out = oracle.adaln_modulate(h, E, phi)
    assert np.array_equal(out[0], oracle.bf16_round(E[0] + 0.125))


def test_adaln_scale_and_shift_roles():
    # scale multiplies (1 + scale); shift adds: with x_hat = +-1 rows the result is closed form
    d = 2
    h = np.array([[1.0, -1.0]])                # mean 0, var 1 -> x_hat = [1, -1]/sqrt(1+eps)
    E = np.zeros((6, d)); phi = np.zeros((6, d))
    E[1] = [1.0, 1.0]                          # scale = 1 -> factor 2
    E[0] = [0.5, 0.5]                          # shift
    r = 1.0 / math.sqrt(1.0 + oracle.LN_EPS)
    assert np.array_equal(oracle.adaln_modulate(h, E, phi)[0],
                          oracle.bf16_round(np.array([2 * r + 0.5, -2 * r + 0.5])))


def test_zero_gate_leaves_hidden_state_bitwise():
    d, HD = 32, 16
    h = bf16_exact((3, d)); o = bf16_exact((3, HD)); wo = bf16_exact((d, HD))
    assert np.array_equal(oracle.oproj_gated_residual(h, o, wo, np.zeros(d)), h)


def test_gated_residual_uses_wo_transposed_and_gate():
    # W_o stored [d, Hq*D]: with W_o = identity padding, o W_o^T copies o into h's slots
    d, HD = 4, 4
    h = np.array([[1.0, 2.0, 3.0, 4.0]])
    o = np.array([[0.5, 0.25, -1.0, 2.0]])
    wo = np.eye(4)[[1, 0, 2, 3]]               # row n picks o[:, perm[n]]
    gate = np.array([1.0, 2.0, 0.0, -1.0])
    expect = oracle.bf16_round(h + gate * np.array([[0.25, 0.5, -1.0, 2.0]]))
    assert np.array_equal(oracle.oproj_gated_residual(h, o, wo, gate), expect)


def test_qkv_split_and_transposed_weight_convention():
    Hq, Hkv, D = 2, 1, 4
    d = 8
    N = (Hq + 2 * Hkv) * D                      # 16 output columns
    x = bf16_exact((3, d))
    w = np.zeros((N, d))
    # q columns 0..7 copy x[:, 0..7]; k columns copy x[:, 0..3] * 2; v columns x[:, 4..7] * -1
    for n in range(8):
        w[n, n] = 1.0
    for n in range(4):
        w[8 + n, n] = 2.0
        w[12 + n, 4 + n] = -1.0
    q, k, v = oracle.qkv_project(x, w, Hq, Hkv, D)
    assert np.array_equal(q.reshape(3, 8), x)
    assert np.array_equal(k.reshape(3, 4), 2 * x[:, :4])
    assert np.array_equal(v.reshape(3, 4), -x[:, 4:])


# ----------------------------------------------------------------------------- attention

def _att(q, kb, vb, kc, vc, ctx_len=None):
    return oracle.block_attention(q, kb, vb, kc, vc, ctx_len)


def test_attention_single_key_returns_its_value_exactly():
    # L = 0 and S = 1: one key, weight 1, output = v exactly
    D = 8
    q = bf16_exact((1, 1, 2, D)); kb = bf16_exact((1, 1, 1, D)); vb = bf16_exact((1, 1, 1, D))
    kc = np.zeros((1, 1, 0, D)); vc = np.zeros((1, 1, 0, D))
    o, lse = _att(q, kb, vb, kc, vc)
    assert np.array_equal(o[0, 0, 0], vb[0, 0, 0]) and np.array_equal(o[0, 0, 1], vb[0, 0, 0])
    s = q[0, 0, :, :] @ kb[0, 0, 0] / math.sqrt(D)
    assert np.allclose(lse[0, 0], s, atol=1e-15)


def test_attention_equal_keys_average_values():
    B, S, Hq, Hkv, D, L = 1, 3, 2, 1, 16, 5
    key = bf16_exact((D,))
    q = bf16_exact((B, S, Hq, D))
    kb = np.broadcast_to(key, (B, S, Hkv, D)).copy()
    kc = np.broadcast_to(key, (B, Hkv, L, D)).copy()
    vb = bf16_exact((B, S, Hkv, D)); vc = bf16_exact((B, Hkv, L, D))
    o, lse = _att(q, kb, vb, kc, vc)
    mean = (vc[0, 0].sum(0) + vb[0, :, 0].sum(0)) / (L + S)
    for i in range(S):
        for h in range(Hq):
            assert np.allclose(o[0, i, h], mean, atol=1e-14)
            s = q[0, i, h] @ key / math.sqrt(D)
            assert np.isclose(lse[0, i, h], s + math.log(L + S), atol=1e-13)


def test_attention_two_keys_logistic_weights_and_sqrt_d_scale():
    # D = 4, q = (a,0,0,0), key0 = (a,0,0,0), key1 = 0: scores (a^2/2, 0)
    D, a = 4, 1.5
    q = np.zeros((1, 1, 1, D)); q[0, 0, 0, 0] = a
    kc = np.zeros((1, 1, 1, D)); kc[0, 0, 0, 0] = a
    kb = np.zeros((1, 1, 1, D))
    vc = np.zeros((1, 1, 1, D)); vc[0, 0, 0, 1] = 1.0
    vb = np.zeros((1, 1, 1, D)); vb[0, 0, 0, 2] = 1.0
    o, _ = _att(q, kb, vb, kc, vc)
    w0 = 1.0 / (1.0 + math.exp(-a * a / 2.0))
    assert np.allclose(o[0, 0, 0], [0.0, w0, 1.0 - w0, 0.0], atol=1e-15)


def test_attention_gqa_groups_are_consecutive():
    # every value of KV head g equals g + 1: query head h must read (h // G) + 1
    B, S, Hq, Hkv, D, L = 2, 4, 8, 2, 8, 6
    q = bf16_exact((B, S, Hq, D)); kb = bf16_exact((B, S, Hkv, D)); kc = bf16_exact((B, Hkv, L, D))
    vb = np.zeros((B, S, Hkv, D)); vc = np.zeros((B, Hkv, L, D))
    for g in range(Hkv):
        vb[:, :, g, :] = g + 1.0
        vc[:, g, :, :] = g + 1.0
    o, _ = _att(q, kb, vb, kc, vc)
    G = Hq // Hkv
    for h in range(Hq):
        assert np.allclose(o[:, :, h, :], h // G + 1.0, atol=1e-14)


def test_attention_context_beyond_ctx_len_is_ignored_and_block_is_bidirectional():
    B, S, Hq, Hkv, D, L = 2, 4, 4, 2, 16, 9
    q = bf16_exact((B, S, Hq, D)); kb = bf16_exact((B, S, Hkv, D)); vb = bf16_exact((B, S, Hkv, D))
    kc = bf16_exact((B, Hkv, L, D)); vc = bf16_exact((B, Hkv, L, D))
    ctx = [5, 0]
    o1, l1 = _att(q, kb, vb, kc, vc, ctx)
    kc2 = kc.copy(); vc2 = vc.copy()
    kc2[0, :, 5:] = 100.0; vc2[0, :, 5:] = -7.0; kc2[1] = 3.0; vc2[1] = 9.0
    o2, l2 = _att(q, kb, vb, kc2, vc2, ctx)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # bidirectional inside the block: position 0 sees position S-1's value
    vb3 = vb.copy(); vb3[:, S - 1] += 1.0
    o3, _ = _att(q, kb, vb3, kc, vc, ctx)
    assert not np.allclose(o3[:, 0], o1[:, 0])


def test_attention_key_permutation_invariance_and_lse_merge_identity():
    B, S, Hq, Hkv, D, L = 1, 3, 2, 1, 8, 7
    q = bf16_exact((B, S, Hq, D)); kb = bf16_exact((B, S, Hkv, D)); vb = bf16_exact((B, S, Hkv, D))
    kc = bf16_exact((B, Hkv, L, D)); vc = bf16_exact((B, Hkv, L, D))
    o, lse = _att(q, kb, vb, kc, vc)
    perm = rng.permutation(L)
    o_p, lse_p = _att(q, kb, vb, kc[:, :, perm], vc[:, :, perm])
    assert np.allclose(o, o_p, atol=1e-14) and np.allclose(lse, lse_p, atol=1e-13)
    # the joint softmax equals the log-sum-exp merge of a block-only softmax (oracle with an
    # empty context) and a context-only softmax written out with einsum here
    empty = np.zeros((B, Hkv, 0, D))
    o_b, l_b = _att(q, kb, vb, empty, empty)
    kr = np.repeat(kc, Hq // Hkv, axis=1)
    vr = np.repeat(vc, Hq // Hkv, axis=1)
    scores = np.einsum("bshd,bhld->bshl", q, kr) / math.sqrt(D)
    l_c = np.log(np.exp(scores).sum(-1))
    o_c = np.einsum("bshl,bhld->bshd", np.exp(scores - l_c[..., None]), vr)
    m = np.logaddexp(l_c, l_b)
    merged = np.exp(l_c - m)[..., None] * o_c + np.exp(l_b - m)[..., None] * o_b
    assert np.allclose(merged, o, atol=1e-13) and np.allclose(m, lse, atol=1e-13)


# ----------------------------------------------------------------------------- LM head

def test_attention_matches_torch_sdpa_with_concatenated_keys_and_repeated_kv_heads():
    # the library routine, in fp64, on the keys ctx[:L_b] ++ block with each KV head
    # repeated for its G = Hq / Hkv consecutive query heads; lse from torch.logsumexp
    import torch
    gen = np.random.default_rng(17)
    B, S, Hq, Hkv, D, Lmax = 3, 5, 6, 2, 16, 9
    q = gen.standard_normal((B, S, Hq, D)); kb = gen.standard_normal((B, S, Hkv, D))
    vb = gen.standard_normal((B, S, Hkv, D))
    kc = gen.standard_normal((B, Hkv, Lmax, D)); vc = gen.standard_normal((B, Hkv, Lmax, D))
    ctx = [9, 0, 4]
    o, lse = oracle.block_attention(q, kb, vb, kc, vc, ctx)
    G = Hq // Hkv
    for b in range(B):
        L = ctx[b]
        keys = torch.cat([torch.from_numpy(kc[b, :, :L]), torch.from_numpy(kb[b]).transpose(0, 1)],
                         dim=1)                                  # [Hkv, L + S, D]
        vals = torch.cat([torch.from_numpy(vc[b, :, :L]), torch.from_numpy(vb[b]).transpose(0, 1)],
                         dim=1)
        keys = keys.repeat_interleave(G, dim=0)                  # [Hq, L + S, D]
        vals = vals.repeat_interleave(G, dim=0)
        qq = torch.from_numpy(q[b]).transpose(0, 1)              # [Hq, S, D]
        ref = torch.nn.functional.scaled_dot_product_attention(qq, keys, vals)
        assert np.allclose(o[b], ref.transpose(0, 1).numpy(), rtol=1e-12, atol=1e-12)
        sc = qq @ keys.transpose(1, 2) / math.sqrt(D)
        assert np.allclose(lse[b], torch.logsumexp(sc, dim=-1).transpose(0, 1).numpy(),
                           rtol=1e-12, atol=1e-12)


def test_lmhead_zero_weights_give_uniform_confidence_exactly():
    V, d = 1024, 64
    h = bf16_exact((3, d))
    conf, pred, gap, zmax = oracle.lmhead_confidence(h, np.zeros((V, d)), chunk=100)
    assert np.all(conf == 1.0 / V) and np.all(pred == 0) and np.all(gap == 0)


def test_lmhead_matches_scipy_softmax_on_a_small_case():
    from scipy.special import softmax
    V, d = 300, 24
    h = bf16_exact((5, d)); w = bf16_exact((V, d), 0.3)
    conf, pred, gap, zmax = oracle.lmhead_confidence(h, w, chunk=64)
    z = h @ w.T
    p = softmax(z, axis=1)
    assert np.allclose(conf, p.max(axis=1), rtol=1e-12)
    assert np.array_equal(pred, z.argmax(axis=1))
    zs = np.sort(z, axis=1)
    assert np.allclose(gap, zs[:, -1] - zs[:, -2], atol=1e-12)


def test_lmhead_planted_rows_and_lowest_id_ties_across_chunks():
    V, d = 1000, 32
    w = bf16_exact((V, d), 0.05)
    w[700] = w[123]                              # exact duplicate of a later-chunk row
    h = np.stack([w[123] * 4.0, w[456] * 4.0])
    conf, pred, gap, _ = oracle.lmhead_confidence(h, w, chunk=128)
    assert pred[0] == 123 and gap[0] == 0.0     # tie between 123 and 700: lowest id
    assert pred[1] == 456 and gap[1] > 0.0


# ----------------------------------------------------------------------------- commit rule

def test_commit_rule_golden_cases():
    with open(os.path.join(GOLDEN, "commit_rule.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        # confidences are held in float32 on both sides; the threshold is float32 too
        conf = np.float32(c["conf"]).astype(np.float64)[None]
        tok, msk, n, com = oracle.commit(conf, np.array(c["pred"])[None], np.array(c["tokens"])[None],
                                         np.array(c["masked"], bool)[None], c["gamma"], c["force_all"])
        assert list(np.nonzero(com[0])[0]) == c["expect_committed"], c["name"]
        assert list(tok[0]) == c["expect_tokens"], c["name"]
        assert n[0] == len(c["expect_committed"])


def test_commit_gamma_at_most_one_over_v_commits_everything():
    V = 1024
    conf = np.full((2, 16), 1.0 / V)             # the minimum possible max-probability
    masked = np.ones((2, 16), bool)
    _, msk, n, _ = oracle.commit(conf, np.zeros((2, 16), int), np.full((2, 16), V), masked,
                                 np.float32(2.0**-10), False)
    assert not msk.any() and list(n) == [16, 16]


def test_commit_monotone_in_gamma_and_never_reverts():
    for _ in range(50):
        conf = rng.uniform(0, 1, (3, 16))
        masked = rng.uniform(size=(3, 16)) < 0.7
        g1, g2 = sorted(rng.uniform(0, 1, 2))
        tok = np.where(masked, 999, 5)
        _, m1, _, c1 = oracle.commit(conf, np.arange(48).reshape(3, 16), tok, masked, g1, False)
        _, m2, _, c2 = oracle.commit(conf, np.arange(48).reshape(3, 16), tok, masked, g2, False)
        for b in range(3):
            if (conf[b][masked[b]] >= np.float32(g2)).any():
                assert set(np.nonzero(c2[b])[0]) <= set(np.nonzero(c1[b])[0])
            if masked[b].any():
                assert c1[b].sum() >= 1                 # at least one commit per step
        assert not (m1 & ~masked).any()                # committed stays committed


# ----------------------------------------------------------------------------- whole step / loop

def _tiny(seed=0, Lmax=8, n_layers=2, S=4, B=2, V=64):
    dm = synth.Dims(B=B, S=S, d=64, Hq=4, Hkv=2, D=64, V=V, Lmax=Lmax, n_layers=n_layers)
    layers = [synth._layer(seed, l, dm, 1 / 8, 1 / 16, 1.0, "cpu") for l in range(n_layers)]
    w_lm = synth.normal((V, dm.d), 0.3, seed, "w_lm")
    emb = synth.normal((V + 1, dm.d), 1.0, seed, "emb")
    pos = synth.normal((S, dm.d), 1.0, seed, "pos")
    phi = synth.phi_table(S, dm.d, seed)
    return dm, layers, w_lm, emb, pos, phi


def test_decode_loop_invariants_and_gamma_above_one_takes_s_steps():
    dm, layers, w_lm, emb, pos, phi = _tiny()
    d = dm.as_dict()
    T = dm.S
    tok, msk, steps, rec = oracle.decode_block(d, layers, phi, w_lm, emb, pos, 1.5, T, trace=True)
    assert steps == dm.S and not msk.any()
    for r in rec:
        assert list(r["n_committed"]) == [1] * dm.B        # fallback only: one per step
    # gamma <= 1/V: everything commits at step 1
    tok2, msk2, steps2, _ = oracle.decode_block(d, layers, phi, w_lm, emb, pos,
                                                 1.0 / dm.V, T)
    assert steps2 == 1 and not msk2.any()
    # invariants at the operating point: >= 1 per step, no revert, <= S steps
    tok3, msk3, steps3, rec3 = oracle.decode_block(d, layers, phi, w_lm, emb, pos, 0.8, T, trace=True)
    assert steps3 <= dm.S and not msk3.any()
    prev = np.ones((dm.B, dm.S), bool)
    prev_tok = np.full((dm.B, dm.S), dm.V)
    for r in rec3:
        assert all(n >= 1 for n, live in zip(r["n_committed"], prev.any(1)) if live)
        assert not (r["masked"] & ~prev).any()
        assert np.array_equal(r["tokens"][~prev], prev_tok[~prev])
        prev, prev_tok = r["masked"], r["tokens"]


def test_identical_rows_commit_lowest_position_first():
    # without the position stand-in every [MASK] row is identical at step 1
    dm, layers, w_lm, emb, pos, phi = _tiny(B=1)
    r = oracle.denoise_step(dm.as_dict(), layers, phi[0], w_lm,
                            np.full((1, dm.S), dm.V), np.ones((1, dm.S), bool), 1.5, 1, dm.S,
                            emb=emb, pos=torch.zeros_like(pos))
    assert np.all(r["conf"] == r["conf"][0, 0])
    assert list(np.nonzero(r["committed"][0])[0]) == [0]


def test_decode_loop_resume_matches_uninterrupted_run():
    dm, layers, w_lm, emb, pos, phi = _tiny(seed=5)
    d = dm.as_dict()
    tok, msk, steps, rec = oracle.decode_block(d, layers, phi, w_lm, emb, pos, 1.5, dm.S, trace=True)
    k = 2
    t_k, m_k = rec[k - 1]["tokens"], rec[k - 1]["masked"]
    tok2, msk2, steps2, _ = oracle.decode_block(d, layers, phi, w_lm, emb, pos, 1.5, dm.S,
                                                 tokens=t_k, masked=m_k, t_start=k + 1)
    assert np.array_equal(tok, tok2) and steps2 == steps - k


def test_sequences_are_independent():
    dm, layers, w_lm, emb, pos, phi = _tiny(seed=7, B=3)
    d = dm.as_dict()
    tok, _, _, _ = oracle.decode_block(d, layers, phi, w_lm, emb, pos, 0.8, dm.S)
    for b in range(3):
        lay_b = [dict(l, k_ctx=l["k_ctx"][b:b + 1], v_ctx=l["v_ctx"][b:b + 1]) for l in layers]
        tb, _, _, _ = oracle.decode_block(dict(d, B=1), lay_b, phi, w_lm, emb, pos, 0.8, dm.S)
        assert np.array_equal(tb[0], tok[b])


def test_brute_force_step_on_tiny_inputs():
    # one layer, everything recomputed with explicit per-element loops (no matrix routines)
    dm, layers, w_lm, emb, pos, phi = _tiny(seed=3, B=1, n_layers=1, Lmax=3, S=2, V=16)
    lay = {k: oracle.as_f64(v) for k, v in layers[0].items()}
    d, Hq, Hkv, D, S, L = dm.d, dm.Hq, dm.Hkv, dm.D, dm.S, dm.Lmax
    ph = oracle.as_f64(phi[0])
    tokens = np.array([[dm.V, 3]])
    ef, pf = oracle.as_f64(emb), oracle.as_f64(pos)
    h = np.array([[oracle.bf16_round(ef[tokens[0, i], c] + pf[i, c]) for c in range(dm.d)]
                  for i in range(S)])
    m = lay["ada_E"] + ph
    xm = np.zeros_like(h)
    for r in range(S):
        mu = sum(h[r]) / d
        var = sum((x - mu) ** 2 for x in h[r]) / d
        for c in range(d):
            xm[r, c] = oracle.bf16_round((h[r, c] - mu) / math.sqrt(var + 1e-6) * (1 + m[1, c]) + m[0, c])
    N = (Hq + 2 * Hkv) * D
    y = np.array([[oracle.bf16_round(sum(xm[r, c] * lay["wqkv"][n, c] for c in range(d)))
                   for n in range(N)] for r in range(S)])
    o = np.zeros((S, Hq * D))
    for i in range(S):
        for hh in range(Hq):
            g = hh // (Hq // Hkv)
            keys = [lay["k_ctx"][0, g, j] for j in range(L)] + [y[s, Hq * D + g * D: Hq * D + (g + 1) * D] for s in range(S)]
            vals = [lay["v_ctx"][0, g, j] for j in range(L)] + [y[s, (Hq + Hkv) * D + g * D: (Hq + Hkv) * D + (g + 1) * D] for s in range(S)]
            qv = y[i, hh * D:(hh + 1) * D]
            sc = [sum(qv[e] * kk[e] for e in range(D)) / math.sqrt(D) for kk in keys]
            mx = max(sc)
            ws = [math.exp(s_ - mx) for s_ in sc]
            tot = sum(ws)
            for e in range(D):
                o[i, hh * D + e] = oracle.bf16_round(sum(w_ * vv[e] for w_, vv in zip(ws, vals)) / tot)
    hn = np.array([[oracle.bf16_round(h[r, c] + m[2, c] * sum(o[r, k] * lay["wo"][c, k] for k in range(Hq * D)))
                    for c in range(d)] for r in range(S)])
    r = oracle.denoise_step(dm.as_dict() | {"B": 1}, layers, phi[0], w_lm, tokens,
                            np.array([[True, False]]), 0.8, 1, 16, emb=emb, pos=pos)
    # fp64 summation order differs (BLAS vs these loops) by ~1e-16 relative, far below a
    # bf16 step, so every storage point rounds the same way
    assert np.array_equal(r["h_final"], hn)
    wl = oracle.as_f64(w_lm)
    z = [[sum(hn[rr, c] * wl[v, c] for c in range(d)) for v in range(dm.V)] for rr in range(S)]
    for rr in range(S):
        zm = max(z[rr])
        cf = 1.0 / sum(math.exp(zz - zm) for zz in z[rr])
        assert abs(cf - r["conf"][0, rr]) < 1e-6
        assert z[rr].index(zm) == r["pred"][0, rr]


def test_embed_gathers_token_rows_and_adds_the_position_of_the_block_slot():
    # two sequences, so a position indexed by sequence instead of block slot would show;
    # the [MASK] id V reads the extra last row of the table
    V, S, d = 5, 3, 4
    rng = np.random.default_rng(8)
    emb = rng.standard_normal((V + 1, d))
    pos = rng.standard_normal((S, d))
    tokens = np.array([[V, 0, 4], [2, V, 2]])
    h = oracle.embed(tokens, emb, pos)
    assert h.shape == (2 * S, d)
    for b in range(2):
        for i in range(S):
            for c in range(d):
                assert h[b * S + i, c] == oracle.bf16_round(emb[tokens[b, i], c] + pos[i, c])
    # the sum is rounded once: bf16(e + p), not bf16(e) + bf16(p)
    e1 = np.zeros((V + 1, 1)); e1[0, 0] = 1.0
    p1 = np.array([[2.0 ** -9], [0.0], [0.0]])
    assert oracle.embed(np.array([[0, 1, 1]]), e1, p1)[0, 0] == oracle.bf16_round(1.0 + 2.0 ** -9)


# ----------------------------------------------------------------------------- mock-AR reading

def test_commit_left_to_right_golden_cases():
    with open(os.path.join(GOLDEN, "commit_left_to_right.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        conf = np.float32(c["conf"]).astype(np.float64)[None]
        tok, msk, n, com = oracle.commit(conf, np.array(c["pred"])[None], np.array(c["tokens"])[None],
                                         np.array(c["masked"], bool)[None], c["gamma"], c["force_all"],
                                         rule=oracle.RULE_LEFT_TO_RIGHT)
        assert list(np.nonzero(com[0])[0]) == c["expect_committed"], c["name"]
        assert list(tok[0]) == c["expect_tokens"], c["name"]
        assert n[0] == len(c["expect_committed"])


def test_left_to_right_decode_commits_positions_in_order_one_per_step():
    dm = synth.Dims(B=2, S=6, d=64, Hq=2, Hkv=1, D=64, V=50, Lmax=5, n_layers=1)
    L = synth._layer(3, 0, dm, 1 / 8, 1 / 8, 1.0, "cpu")
    emb = synth.normal((dm.V + 1, dm.d), 1.0, 3, "emb")
    pos = synth.normal((dm.S, dm.d), 1.0, 3, "pos")
    w = synth.normal((dm.V, dm.d), 0.3, 3, "w")
    phi = synth.phi_table(dm.S, dm.d, 3)
    _, _, steps, recs = oracle.decode_block(dm.as_dict(), [L], phi, w, emb, pos, 0.0, dm.S,
                                            trace=True, rule=oracle.RULE_LEFT_TO_RIGHT)
    # gamma = 0 would commit everything at once under the confidence rule; here one per step
    assert steps == dm.S
    for t, r in enumerate(recs):
        assert list(r["n_committed"]) == [1, 1]
        assert np.array_equal(np.nonzero(r["committed"][0])[0], [t])
        assert np.array_equal(np.nonzero(r["committed"][1])[0], [t])
        assert np.array_equal(r["tokens"][:, t], r["pred"][:, t])


# ----------------------------------------------------------------------------- cache growth

def test_kv_append_extends_the_attention_context_by_the_block():
    # attention over the grown cache equals a softmax written out here over
    # (old context rows) ++ (appended block rows) ++ (block keys)
    B, S, Hq, Hkv, D, Lmax = 2, 3, 4, 2, 16, 12
    q = bf16_exact((B, S, Hq, D)); kb = bf16_exact((B, S, Hkv, D)); vb = bf16_exact((B, S, Hkv, D))
    kc = bf16_exact((B, Hkv, Lmax, D)); vc = bf16_exact((B, Hkv, Lmax, D))
    kn = bf16_exact((B, S, Hkv, D)); vn = bf16_exact((B, S, Hkv, D))
    ctx = [5, 0]
    k2, v2, ln, ovf = oracle.kv_append(kc, vc, ctx, kn, vn)
    assert list(ln) == [8, 3] and not ovf.any()
    o, _ = oracle.block_attention(q, kb, vb, k2, v2, ln)
    G = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            g = h // G
            keys = np.concatenate([kc[b, g, :ctx[b]], kn[b, :, g], kb[b, :, g]])
            vals = np.concatenate([vc[b, g, :ctx[b]], vn[b, :, g], vb[b, :, g]])
            sc = q[b, :, h] @ keys.T / math.sqrt(D)
            w = np.exp(sc - sc.max(axis=1, keepdims=True))
            ref = (w / w.sum(axis=1, keepdims=True)) @ vals
            assert np.allclose(o[b, :, h], ref, atol=1e-13)
    # rows outside the appended window are untouched
    assert np.array_equal(k2[0, :, :5], kc[0, :, :5]) and np.array_equal(k2[0, :, 8:], kc[0, :, 8:])


def test_kv_append_overflow_leaves_the_sequence_unchanged():
    B, S, Hkv, D, Lmax = 2, 4, 1, 8, 10
    kc = bf16_exact((B, Hkv, Lmax, D)); vc = bf16_exact((B, Hkv, Lmax, D))
    kn = bf16_exact((B, S, Hkv, D)); vn = bf16_exact((B, S, Hkv, D))
    k2, v2, ln, ovf = oracle.kv_append(kc, vc, [7, 6], kn, vn)
    assert list(ovf) == [True, False] and list(ln) == [7, 10]
    assert np.array_equal(k2[0], kc[0]) and np.array_equal(v2[0], vc[0])
    assert np.array_equal(k2[1, 0, 6:10], kn[1, :, 0])


# ----------------------------------------------------------------------------- rotary variant

def test_rope_is_a_rotation_and_identity_at_position_zero():
    x = rng.standard_normal((5, 3, 64))
    pos = np.array([0, 1, 7, 1000, 32767])
    y = oracle.rope_rotate(x, pos, 10000.0)
    assert np.array_equal(y[0], x[0])                                  # angle 0
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
    # pair 0 turns by exactly pos radians (theta**0 = 1): closed form for one pair
    a = float(pos[2])
    assert np.allclose(y[2, :, 0], x[2, :, 0] * math.cos(a) - x[2, :, 1] * math.sin(a))
    assert np.allclose(y[2, :, 1], x[2, :, 0] * math.sin(a) + x[2, :, 1] * math.cos(a))
    # the last pair's frequency is theta**(-(D-2)/D)
    f = 10000.0 ** (-(64 - 2) / 64)
    assert np.allclose(y[3, :, 62], x[3, :, 62] * math.cos(1000 * f) - x[3, :, 63] * math.sin(1000 * f))


def test_rope_scores_depend_only_on_relative_position():
    # q . k after rotating both depends on p_q - p_k only (computed here with einsum)
    q = rng.standard_normal((1, 1, 32)); k = rng.standard_normal((1, 1, 32))
    s1 = np.einsum("rhd,rhd->", oracle.rope_rotate(q, [100], 500.0), oracle.rope_rotate(k, [90], 500.0))
    s2 = np.einsum("rhd,rhd->", oracle.rope_rotate(q, [13], 500.0), oracle.rope_rotate(k, [3], 500.0))
    s3 = np.einsum("rhd,rhd->", oracle.rope_rotate(q, [13], 500.0), oracle.rope_rotate(k, [4], 500.0))
    assert abs(s1 - s2) < 1e-12 and abs(s1 - s3) > 1e-6


def test_block_positions_follow_the_context():
    dims = dict(B=2, S=3, Lmax=50)
    assert list(oracle.block_positions(dims, [7, 0])) == [7, 8, 9, 0, 1, 2]
    assert list(oracle.block_positions(dims)) == [50, 51, 52, 50, 51, 52]


# ------------------------------------------------------------------------------ timestep map

def test_timestep_embedding_at_zero_and_unit_pair_norms():
    # tau = 0: every cosine is 1 and every sine 0 (closed form of the definition)
    e0 = oracle.timestep_embedding(0.0)[0]
    assert np.array_equal(e0[:128], np.ones(128)) and np.array_equal(e0[128:], np.zeros(128))
    # any tau: each (cos, sin) pair has unit length, so the embedding's squared norm is 128
    e = oracle.timestep_embedding(np.array([0.0625, 0.3, 1.0]))
    pairs = e[:, :128] ** 2 + e[:, 128:] ** 2
    assert np.allclose(pairs, 1.0, atol=1e-15)


def test_timestep_embedding_frequencies_as_complex_exponentials():
    # e[j] + i e[128 + j] = exp(i 1000 tau 10000^(-j/128)): the lowest index turns fastest (one
    # radian per 1/1000 of tau), the last slowest; checked against numpy's complex exponential
    tau = np.array([0.125, 0.5, 0.9375])
    e = oracle.timestep_embedding(tau)
    j = np.arange(128)
    z = np.exp(1j * 1000.0 * tau[:, None] * 10000.0 ** (-j[None, :] / 128.0))
    assert np.allclose(e[:, :128], z.real, atol=1e-12)
    assert np.allclose(e[:, 128:], z.imag, atol=1e-12)
    # j = 0 at tau = pi / 2000: cos = 0, sin = 1
    q = oracle.timestep_embedding(math.pi / 2000.0)[0]
    assert abs(q[0]) < 1e-15 and abs(q[128] - 1.0) < 1e-15


def test_timestep_table_rows_steps_and_bias():
    d, T = 8, 4
    rng = np.random.default_rng(5)
    W = rng.standard_normal((6 * d, 256))
    b = rng.standard_normal(6 * d)
    phi = oracle.timestep_table(W, b, T)
    assert phi.shape == (T, 6, d)
    # zero weights: every step's vector is the bias, laid out as 6 rows of d
    assert np.array_equal(oracle.timestep_table(np.zeros_like(W), b, T),
                          np.broadcast_to(b.reshape(6, d), (T, 6, d)))
    # step t uses tau = t / T; a one-hot weight column reads one embedding feature
    Wj = np.zeros_like(W)
    Wj[3 * d + 5, 200] = 1.0           # row 3 (of 6), column 5 <- feature 200 = sin(s w_72)
    got = oracle.timestep_table(Wj, np.zeros(6 * d), T)[:, 3, 5]
    want = [math.sin(1000.0 * t / T * 10000.0 ** (-72 / 128.0)) for t in range(1, T + 1)]
    assert np.allclose(got, want, atol=1e-12)
    # linear in (W, b)
    W2 = rng.standard_normal((6 * d, 256))
    b2 = rng.standard_normal(6 * d)
    lhs = oracle.timestep_table(W + 2.0 * W2, b + 2.0 * b2, T)
    rhs = phi + 2.0 * oracle.timestep_table(W2, b2, T)
    assert np.allclose(lhs, rhs, atol=1e-10)
