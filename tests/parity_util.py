"""Comparison rules shared by the GPU parity tests.

Tolerances (bf16 inputs, fp32 accumulation on the GPU, fp64 in the oracle):
  - attention output: per query row, ||o_gpu - o_ref||_2 <= 1e-2 ||o_ref||_2 and every
    element within 1e-2 * max|o_ref row| (the 1e-2 relative bar for attention outputs);
  - confidences: |conf_gpu - conf_ref| <= 2e-3;
  - token ids and commit masks: bit-exact, except positions whose oracle confidence lies
    within 1e-5 of gamma or whose top-2 logit gap is under 1e-4 (reported, excluded). A
    sequence whose commit decision rests on such a position (a near-threshold masked
    position, or a fallback whose two best masked confidences are within 1e-5) is excluded
    whole, since its whole commit set may legitimately differ.
Exclusions are decided from the oracle's values.
"""

from __future__ import annotations

import numpy as np

CONF_TOL = 2e-3
GAMMA_BAND = 1e-5
GAP_BAND = 1e-4
ATTN_REL = 1e-2


def attention_close(o_gpu: np.ndarray, o_ref: np.ndarray):
    """o_* [..., D]; returns (ok, worst row-relative L2 error)."""
    g = o_gpu.reshape(-1, o_gpu.shape[-1]).astype(np.float64)
    r = o_ref.reshape(-1, o_ref.shape[-1]).astype(np.float64)
    err = np.linalg.norm(g - r, axis=1)
    ref = np.linalg.norm(r, axis=1)
    rel = err / np.maximum(ref, 1e-30)
    elem = np.abs(g - r) <= ATTN_REL * np.abs(r).max(axis=1, keepdims=True) + 1e-30
    return bool((rel <= ATTN_REL).all() and elem.all()), float(rel.max())


def excluded_sequences(conf_ref, gap_ref, masked_before, gamma: float,
                       band: float = GAMMA_BAND):
    """Sequences whose commit set may legitimately differ (see module doc); `band` is the
    distance under which two confidences (or a confidence and gamma) count as tied."""
    conf_ref = np.asarray(conf_ref, np.float64)
    g = float(np.float32(gamma))
    B, S = conf_ref.shape
    ex = np.zeros(B, bool)
    for b in range(B):
        m = np.asarray(masked_before[b], bool)
        if not m.any():
            continue
        near = np.abs(conf_ref[b] - g) < band
        if (near & m).any():
            ex[b] = True
            continue
        if not (conf_ref[b][m] >= g).any():
            c = np.sort(conf_ref[b][m])[::-1]
            if len(c) > 1 and c[0] - c[1] < band:
                ex[b] = True
    return ex


def compare_commit(ref: dict, gpu: dict, masked_before, gamma: float, step: bool = False,
                   evaluated=None, tie_extra=None, conf_band: float = GAMMA_BAND):
    """ref: oracle outputs (conf, pred, gap, tokens, masked); gpu: numpy arrays of the same.
    step=True: the GPU side is a denoise step, which evaluates the LM head only on the rows
    that can commit (by default those masked when the step starts; `evaluated` overrides)
    and reports conf 0, pred -1 on the others.
    Returns a report dict; raises AssertionError on a mismatch outside the exclusions."""
    conf_ref = np.asarray(ref["conf"], np.float64)
    gap = np.asarray(ref["gap"], np.float64)
    conf_gpu = np.asarray(gpu["conf"], np.float64)
    pred_gpu = np.asarray(gpu["pred"])
    if evaluated is None:
        evaluated = np.asarray(masked_before, bool) if step else np.ones(conf_ref.shape, bool)
    evaluated = np.asarray(evaluated, bool)
    if step:
        assert (conf_gpu[~evaluated] == 0).all() and (pred_gpu[~evaluated] == -1).all(), \
            "rows committed before the step must read conf 0, pred -1"
    dconf = np.where(evaluated, np.abs(conf_gpu - conf_ref), 0.0)
    assert dconf.max(initial=0.0) <= CONF_TOL, f"conf error {dconf.max()}"
    ex_seq = excluded_sequences(conf_ref, gap, masked_before, gamma, conf_band)
    tie_pos = gap < GAP_BAND
    if tie_extra is not None:
        tie_pos = tie_pos | np.asarray(tie_extra, bool)
    pred_bad = (pred_gpu != np.asarray(ref["pred"])) & ~tie_pos & evaluated
    assert not pred_bad.any(), f"pred mismatch at {np.argwhere(pred_bad)[:8]}"
    mk_bad = (np.asarray(gpu["masked"], bool) != np.asarray(ref["masked"], bool))
    mk_bad[ex_seq] = False
    assert not mk_bad.any(), f"commit-mask mismatch at {np.argwhere(mk_bad)[:8]}"
    tok_bad = (np.asarray(gpu["tokens"]) != np.asarray(ref["tokens"])) & ~tie_pos
    tok_bad[ex_seq] = False
    assert not tok_bad.any(), f"token mismatch at {np.argwhere(tok_bad)[:8]}"
    return dict(max_conf_err=float(dconf.max()), excluded_sequences=int(ex_seq.sum()),
                tie_positions=int(tie_pos.sum()))


def first_masked(masked) -> np.ndarray:
    """The lowest-index masked position of each sequence, as a mask."""
    m = np.asarray(masked, bool)
    out = np.zeros_like(m)
    for b in range(m.shape[0]):
        idx = np.nonzero(m[b])[0]
        if len(idx):
            out[b, idx[0]] = True
    return out


def bf16_ulp(x) -> np.ndarray:
    """Spacing of bfloat16 values at |x| (8 significant bits); 2**-133 at zero."""
    a = np.abs(np.asarray(x, np.float64))
    return np.where(a > 0, np.exp2(np.floor(np.log2(np.maximum(a, 2.0**-126))) - 7), 2.0**-133)


def layer_close(h_gpu, h_ref, o_ref, wo, gate):
    """One layer's output on identical inputs. h_* [rows, d]; o_ref [rows, Hq*D] (the
    oracle's bf16 attention output); wo [d, Hq*D]; gate [d].

    Bound per element n of a row: the GPU's h_n may differ from the oracle's by its own
    rounding (two bf16 steps of the result: the storage point, plus a binade edge) and by what
    the attention bar allows through the gated output projection: with the row's attention
    output within 1e-2 of the oracle's in L2 norm, |delta(o . wo[n])| <= 1e-2 ||o||_2
    ||wo[n]||_2 (Cauchy-Schwarz), times |gate_n|. Also at most 10 % of the elements may differ
    by more than one bf16 step (a systematic error would move most of them).
    Returns (ok, worst ratio to the bound, fraction beyond one step)."""
    import oracle
    g = oracle.as_f64(h_gpu)
    r = oracle.as_f64(h_ref)
    o = oracle.as_f64(o_ref)
    w = oracle.as_f64(wo)
    bound = 2.0 * bf16_ulp(r) + ATTN_REL * np.abs(oracle.as_f64(gate))[None, :] * \
        np.linalg.norm(o, axis=1)[:, None] * np.linalg.norm(w, axis=1)[None, :]
    err = np.abs(g - r)
    beyond = float((err > bf16_ulp(r)).mean())
    worst = float((err / bound).max(initial=0.0))
    return bool(worst <= 1.0 and beyond <= 0.10), worst, beyond


def stacked_step_parity(dims, layers, w_lm, phi_t, t, T, gamma, tokens0, masked0, got,
                        h=None, emb=None, pos=None, ctx_len=None, rule=0,
                        rope_theta=0.0, seqs=None, page_table=None, n_pages=0,
                        end_to_end=True, cpu_layers=None, attn_precision=0):
    """Parity of one denoise step of stacked layers, at the bands of the acceptance rule.

    A stacked step feeds each layer's bf16 output to the next, and a GPU (fp32 accumulation)
    and the fp64 oracle round a few of those values to neighbouring bf16 numbers; the next
    layer carries such a difference on. So the step is checked stage by stage on identical
    inputs:
      1. the hidden state after every layer: the GPU's chained one-layer steps (their final
         state equals the whole step's bit for bit) against the oracle's layer fed the GPU's
         previous state (layer_close); the embedding bit for bit;
      2. conf / pred / tokens / masked of the step against the oracle's LM head and commit
         rule on the GPU's final hidden state: ids and commit masks bit-exact outside the
         exclusion bands, conf within 2e-3 (compare_commit);
      3. (end_to_end) conf of the oracle's whole step from the same inputs within 2e-3
         (end_to_end="report": computed and returned, not asserted).
    dims: dict; layers: GPU layer dicts; tokens0 / masked0: the state before the step (GPU
    tensors); got: the step's outputs (conf, pred, tokens, masked as numpy arrays). seqs: the
    sequences the oracle checks (default all); cpu_layers: oracle_layers(layers, seqs, ...)
    when the caller already has it. Returns a report dict."""
    import torch

    import block_diffusion_lm_denoise_b300 as td
    import oracle

    B, S, d = dims["B"], dims["S"], dims["d"]
    n_layers = dims["n_layers"]
    seqs = list(range(B)) if seqs is None else list(seqs)
    rows = [b * S + i for b in seqs for i in range(S)]
    dev = w_lm.device
    sub = dict(dims, B=len(seqs))
    ctx_sub = None if ctx_len is None else [int(ctx_len[b]) for b in seqs]
    if cpu_layers is None:
        cpu_layers = oracle_layers(layers, seqs, page_table, dims["Lmax"])

    def step(lays, h_in, out):
        dm = dict(dims, n_layers=len(lays))
        tk, mk = tokens0.clone(), masked0.clone()
        ctx_t = None if ctx_len is None else torch.as_tensor(ctx_len, dtype=torch.int32,
                                                               device=dev)
        return td.td_denoise_step(dm, lays, w_lm, phi_t, t, T, gamma, tk, mk, h=h_in,
                                  emb=None if h_in is not None else emb,
                                  pos=None if h_in is not None else pos, ctx_len=ctx_t,
                                  rule=rule, rope_theta=rope_theta, page_table=page_table,
                                  n_pages=n_pages, h_out=out, attn_precision=attn_precision)

    # the whole step again, reporting its final hidden state: same outputs as without
    h_final = torch.empty((B * S, d), dtype=torch.bfloat16, device=dev)
    c2, p2, _, _ = step(layers, h, h_final)
    torch.cuda.synchronize()
    assert np.array_equal(c2.cpu().numpy(), got["conf"]), "h_out changed conf"
    assert np.array_equal(p2.cpu().numpy(), got["pred"]), "h_out changed pred"
    # 1. the input of the first layer, then layer by layer
    if h is None:
        h_prev = torch.empty_like(h_final)
        step([], None, h_prev)
        torch.cuda.synchronize()
        tok_np = tokens0.cpu().numpy()
        ref0 = oracle.embed(tok_np[seqs], emb, pos.cpu())   # rows gathered on the device
        assert np.array_equal(oracle.as_f64(h_prev.cpu()[rows]), ref0), "embedding differs"
    else:
        h_prev = h
    worst_layer, beyond_layer = 0.0, 0.0
    for k in range(n_layers):
        h_k = torch.empty_like(h_final)
        step([layers[k]], h_prev, h_k)
        torch.cuda.synchronize()
        lay = cpu_layers[k]
        h_ref, o_ref = oracle.layer_forward(oracle.as_f64(h_prev.cpu()[rows]), lay, phi_t.cpu(),
                                            sub, ctx_sub, rope_theta)
        _, _, gate = oracle.adaln_vectors(lay["ada_E"], phi_t.cpu())
        ok, worst, beyond = layer_close(h_k.cpu()[rows], h_ref,
                                        o_ref.reshape(len(rows), -1), lay["wo"], gate)
        assert ok, (k, worst, beyond)
        worst_layer, beyond_layer = max(worst_layer, worst), max(beyond_layer, beyond)
        h_prev = h_k
    assert torch.equal(h_prev, h_final) if n_layers else True, "chained layers differ from the step"
    # 2. LM head and commit rule on the GPU's final hidden state
    m0 = masked0.cpu().numpy().astype(bool)[seqs]
    t0 = tokens0.cpu().numpy()[seqs]
    nb = len(seqs)
    evaluated = first_masked(m0) if (rule == 1 and t != T) else m0
    # logits only of the rows the step evaluates (the others read conf 0, pred -1)
    c, p, gap = np.zeros((nb, S)), np.full((nb, S), -1), np.full((nb, S), np.inf)
    ev = np.argwhere(evaluated)
    if len(ev):
        ce, pe, ge, _ = oracle.lmhead_confidence(h_final.cpu()[rows], w_lm,
                                                 rows=[b * S + i for b, i in ev])
        c[evaluated], p[evaluated], gap[evaluated] = ce, pe, ge
    tok_ref, msk_ref, _, _ = oracle.commit(c, p, t0, m0, gamma, t == T, rule=rule)
    rep = compare_commit(dict(conf=c, pred=p, gap=gap, tokens=tok_ref, masked=msk_ref),
                         {k: np.asarray(v)[seqs] for k, v in got.items()}, m0, gamma,
                         step=True, evaluated=evaluated)
    rep.update(layer_worst_ratio=worst_layer, layer_beyond_one_step=beyond_layer)
    if not end_to_end:
        return rep
    # 3. the oracle's own step from the same inputs: confidences within the bar
    r = oracle.denoise_step(sub, cpu_layers, phi_t.cpu(), w_lm, t0, m0, gamma, t, T,
                            h=None if h is None else h.cpu()[rows],
                            emb=emb,
                            pos=None if pos is None else pos.cpu(), ctx_len=ctx_sub,
                            rule=rule, rope_theta=rope_theta)
    dconf = np.where(evaluated, np.abs(np.asarray(got["conf"])[seqs] - r["conf"]), 0.0)
    if end_to_end != "report":
        assert dconf.max(initial=0.0) <= CONF_TOL, f"end-to-end conf error {dconf.max()}"
    pred_diff = int(((np.asarray(got["pred"])[seqs] != r["pred"]) & evaluated).sum())
    rep.update(end_to_end_conf_err=float(dconf.max(initial=0.0)),
               end_to_end_pred_differences=pred_diff)
    return rep


def oracle_layers(layers, seqs, page_table=None, Lmax=0):
    """Host copies of the GPU layer dicts for the oracle: weights whole, context caches only
    for the sequences `seqs` (selected on the device, contiguous layout)."""
    import torch
    out = []
    for L in layers:
        lay = {}
        for n, v in L.items():
            if n in ("k_ctx", "v_ctx"):
                if page_table is not None:
                    lay[n] = _unpage(v, page_table, seqs, Lmax)
                else:
                    idx = torch.tensor(seqs, dtype=torch.long, device=v.device)
                    lay[n] = v.index_select(0, idx).cpu()
            else:
                lay[n] = v.cpu()
        out.append(lay)
    return out


def _unpage(pool, page_table, seqs, Lmax):
    """The contiguous [len(seqs), Hkv, Lmax, D] cache of the given sequences, read from a page
    pool [n_pages, Hkv, 128, D] through the page table [B, max_pages] (CPU tensors)."""
    import torch
    pool = pool.cpu()
    pt = page_table.cpu()
    n_tiles = (Lmax + 127) // 128
    out = []
    for b in seqs:
        tiles = [pool[int(pt[b, j])] for j in range(n_tiles)]
        out.append(torch.cat(tiles, dim=1)[:, :Lmax])
    return torch.stack(out)
