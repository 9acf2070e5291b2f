"""Plain fp64 CPU oracle of the TwoTower block-diffusion denoise step.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import, call or execute this
module: only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
use it. It shares no code with the CUDA library (no kernels, headers, helpers or tables);
both sides read the same seeded input tensors and nothing else.

What it computes, step by step, in the order of the pages and in fp64 on the same bf16 /
fp32 input values the GPU reads. The pages only describe the method in prose:

  [chathome] "NVIDIA、Nemotron-Labs-TwoTowerを公開：凍結された自己回帰バックボーン上に構築
             されたオープンウェイト拡散言語モデル" (news.chathome.org)
             - inference paragraph ("推論では…"): the context tower yields a per-layer KV
               cache; the denoiser attends bidirectionally inside the block and causally to
               past clean blocks; each denoiser layer cross-attends to the matching context
               layer; the diffusion timestep modulates each layer through adaLN-single.
             - generation paragraph ("生成はブロックごとに…"): a block starts as S [MASK]
               tokens, is refined over T steps and committed; several tokens commit per step
               early in the refinement, where AR decoding commits exactly one.
             - evaluation paragraph ("2×H100 GPUでのBF16評価では…"): confidence masking with
               threshold gamma = 0.8 and block size S = 16; lower gamma commits more tokens
               per step.
  [aiboss]   "Nemotron-Labs-TwoTower - NVIDIAのオープンソースデュアルタワーアーキテクチャ
             普及言語モデル" (aiboss88.com), section "技術原理": the denoiser uses
             bidirectional block attention plus cross-attention to the context tower.

Readings taken where the pages are silent (each is listed with its reason in the design
notes of the repository):
  R1 adaLN-single: m = E_l + phi(t), rows (shift, scale, gate); a non-affine LayerNorm with
     population variance and eps = 1e-6; x_mod = LN(h) * (1 + scale) + shift; the attention
     output enters the residual stream as h + gate * (o W_o).
  R2 one joint softmax per query row over context keys and block keys; no mask (the cache
     holds only past tokens; the block is bidirectional); the cached K/V are used as-is.
  R3 GQA groups are consecutive: query head h reads KV head h // (Hq / Hkv).
  R4 no positional rotation by default; the decode loop adds a synthetic position table to
     the embedding as a stand-in for the order information of the out-of-scope Mamba layers.
     A rotary variant (rope_theta > 0) rotates the block's q and k at their absolute
     positions ctx_len + i, interleaved pairs, before their bf16 rounding.
  R5 [MASK] is token id V, outside the LM head's V outputs.
  R6 conf = max softmax probability; pred = lowest id among the maxima; commit set
     {masked i : conf_i >= gamma}; if empty while something is masked, the lowest-index
     masked position of maximal conf; at t == T every masked position commits.
  R7 bf16 storage points: x_mod (Q1), q/k/v (Q2), attention output (Q3), the updated
     hidden state (Q4), and the embedding sum; every other value stays in fp64 here.
  R19 the timestep map of adaLN-single (optional; the step itself takes phi(t) as input):
     phi(t) = W_t e(t / T) + b_t, e the 256-wide sinusoidal embedding of 1000 t / T.
"""

from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

LN_EPS = 1e-6


# ----------------------------------------------------------------------------------------
# Number format
# ----------------------------------------------------------------------------------------

def bf16_round(x) -> np.ndarray:
    """Round fp64 values to the nearest bfloat16 value (ties to even), returned as fp64.

    bfloat16 keeps 8 significant bits and the binary32 exponent range. Written from that
    definition with frexp/rint (no float32 intermediate, so no double rounding). Finite
    values only; magnitudes below 2**-126 are not needed by this oracle.
    """
    x = np.asarray(x, dtype=np.float64)
    mant, expo = np.frexp(x)                  # x = mant * 2**expo, 0.5 <= |mant| < 1
    scaled = np.ldexp(mant, 8)                # 8 significant bits before the point
    rounded = np.rint(scaled)                 # round half to even
    return np.ldexp(rounded, expo - 8)


def as_f64(t) -> np.ndarray:
    """A torch tensor (bf16 / fp32 / int) or array as an fp64 numpy array (exact)."""
    if hasattr(t, "detach"):
        t = t.detach().to("cpu")
        if str(t.dtype) in ("torch.bfloat16", "torch.float16"):
            t = t.float()
        t = t.numpy()
    return np.asarray(t, dtype=np.float64)


# ----------------------------------------------------------------------------------------
# adaLN-single ([chathome] inference paragraph; reading R1)
# ----------------------------------------------------------------------------------------

def adaln_vectors(E, phi):
    """m = E_l + phi(t) in fp64, returned as (shift, scale, gate) rows of length d."""
    m = as_f64(E) + as_f64(phi)
    return m[0], m[1], m[2]


TIMESTEP_DIM = 256        # width of the sinusoidal embedding of tau (R19)
TIMESTEP_SCALE = 1000.0   # tau in (0, 1] is embedded at 1000 tau (R19)


def timestep_embedding(tau) -> np.ndarray:
    """Sinusoidal embedding of the diffusion time tau = t / T (reading R19: the pages name
    adaLN-single but not its timestep map). With s = 1000 tau and frequencies
    w_j = 10000^(-j / 128), j = 0..127: e[j] = cos(s w_j), e[128 + j] = sin(s w_j).
    tau: scalar or [n]; returns [n, 256] (fp64)."""
    tau = np.atleast_1d(np.asarray(tau, dtype=np.float64))
    half = TIMESTEP_DIM // 2
    j = np.arange(half, dtype=np.float64)
    w = np.power(10000.0, -j / half)
    arg = (TIMESTEP_SCALE * tau)[:, None] * w[None, :]
    return np.concatenate([np.cos(arg), np.sin(arg)], axis=1)


def timestep_table(w_t, b_t, T: int) -> np.ndarray:
    """The shared adaLN-single vectors phi(t) for t = 1..T ([chathome] inference paragraph:
    the diffusion timestep modulates every layer through adaLN-single; reading R19):
    phi(t) = W_t e(t / T) + b_t with W_t [6d, 256] and b_t [6d] (fp32 parameters), computed
    in fp64 and returned as [T, 6, d] fp64 (the library stores it rounded to fp32)."""
    W = as_f64(w_t)
    b = as_f64(b_t)
    d6 = W.shape[0]
    tau = np.arange(1, T + 1, dtype=np.float64) / T
    e = timestep_embedding(tau)                                  # [T, 256]
    return (e @ W.T + b[None, :]).reshape(T, 6, d6 // 6)


def layer_norm(h) -> np.ndarray:
    """Non-affine LayerNorm of each row: (h - mean) / sqrt(population var + eps)."""
    h = as_f64(h)
    mu = h.mean(axis=-1, keepdims=True)
    var = ((h - mu) ** 2).mean(axis=-1, keepdims=True)
    return (h - mu) / np.sqrt(var + LN_EPS)


def adaln_modulate(h, E, phi) -> np.ndarray:
    """x_mod = bf16(LN(h) * (1 + scale) + shift)   [storage point Q1]."""
    shift, scale, _ = adaln_vectors(E, phi)
    return bf16_round(layer_norm(h) * (1.0 + scale) + shift)


# ----------------------------------------------------------------------------------------
# Projections
# ----------------------------------------------------------------------------------------

def rope_rotate(x, positions, theta: float) -> np.ndarray:
    """Rotary position embedding (a variant; the pages define no positional scheme, R4).

    x [rows, heads, D] fp64; positions [rows]. Interleaved pairs: for j < D/2 the pair
    (x[2j], x[2j+1]) is rotated by the angle pos * theta**(-2j/D):
      x'[2j]   = x[2j] cos a - x[2j+1] sin a
      x'[2j+1] = x[2j] sin a + x[2j+1] cos a
    """
    x = as_f64(x)
    D = x.shape[-1]
    j = np.arange(D // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * j / D)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]   # [rows, D/2]
    c = np.cos(ang)[:, None, :]
    sn = np.sin(ang)[:, None, :]
    x0 = x[..., 0::2]
    x1 = x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * sn
    out[..., 1::2] = x0 * sn + x1 * c
    return out


def qkv_project(x_mod, wqkv, Hq: int, Hkv: int, D: int, rope_pos=None, rope_theta: float = 0.0):
    """[q | k | v] = bf16(x_mod W_qkv), with W_qkv stored transposed as [(Hq+2Hkv)D, d].

    With rope_theta > 0, q and k are rotated (rope_rotate, positions rope_pos [rows]) before
    the rounding. Returns q [rows, Hq, D], k [rows, Hkv, D], v [rows, Hkv, D] (fp64 holding
    bf16 values, storage point Q2).
    """
    y = as_f64(x_mod) @ as_f64(wqkv).T
    rows = y.shape[0]
    q = y[:, : Hq * D].reshape(rows, Hq, D)
    k = y[:, Hq * D: (Hq + Hkv) * D].reshape(rows, Hkv, D)
    v = y[:, (Hq + Hkv) * D: (Hq + 2 * Hkv) * D].reshape(rows, Hkv, D)
    if rope_theta > 0:
        q = rope_rotate(q, rope_pos, rope_theta)
        k = rope_rotate(k, rope_pos, rope_theta)
    return bf16_round(q), bf16_round(k), bf16_round(v)


def oproj_gated_residual(h, o, wo, gate) -> np.ndarray:
    """h_new = bf16(h + gate * (o W_o)), W_o stored transposed as [d, Hq*D]  [Q4]."""
    o2 = as_f64(o).reshape(as_f64(h).shape[0], -1)
    return bf16_round(as_f64(h) + as_f64(gate) * (o2 @ as_f64(wo).T))


# ----------------------------------------------------------------------------------------
# Block attention ([chathome] inference paragraph; [aiboss] 技術原理; readings R2, R3)
# ----------------------------------------------------------------------------------------

def block_attention(q, k_blk, v_blk, k_ctx, v_ctx, ctx_len: Optional[Sequence[int]] = None):
    """Attention of every block query over (context keys of its KV head) ++ (block keys).

    q [B, S, Hq, D]; k_blk, v_blk [B, S, Hkv, D]; k_ctx, v_ctx [B, Hkv, Lmax, D];
    ctx_len: per-sequence valid context length (default Lmax).
    Returns (o, lse): o [B, S, Hq, D] in fp64 (unrounded), lse [B, S, Hq] = natural log of
    sum_j exp(score_j), scores = q . k_j / sqrt(D).
    """
    q = as_f64(q); k_blk = as_f64(k_blk); v_blk = as_f64(v_blk)
    k_ctx = as_f64(k_ctx); v_ctx = as_f64(v_ctx)
    B, S, Hq, D = q.shape
    Hkv = k_blk.shape[2]
    G = Hq // Hkv
    Lmax = k_ctx.shape[2]
    o = np.zeros((B, S, Hq, D))
    lse = np.zeros((B, S, Hq))
    for b in range(B):
        L = Lmax if ctx_len is None else int(ctx_len[b])
        for h in range(Hq):
            g = h // G
            keys = np.concatenate([k_ctx[b, g, :L, :], k_blk[b, :, g, :]], axis=0)
            vals = np.concatenate([v_ctx[b, g, :L, :], v_blk[b, :, g, :]], axis=0)
            scores = (q[b, :, h, :] @ keys.T) / math.sqrt(D)          # [S, L+S]
            smax = scores.max(axis=1, keepdims=True)
            w = np.exp(scores - smax)
            denom = w.sum(axis=1, keepdims=True)
            o[b, :, h, :] = (w / denom) @ vals
            lse[b, :, h] = (smax + np.log(denom))[:, 0]
    return o, lse


# ----------------------------------------------------------------------------------------
# LM head confidence ([chathome] evaluation paragraph; reading R6)
# ----------------------------------------------------------------------------------------

def lmhead_confidence(h, w_lm, rows: Optional[Sequence[int]] = None, chunk: int = 16384):
    """Per row: z = h_r W_lm^T in fp64 (never stored whole), then
    conf = max softmax(z) = 1 / sum_v exp(z_v - max z), pred = lowest argmax,
    gap = max z - second largest z (0 when the maximum is tied), zmax.

    h [R, d]; w_lm [V, d] (bf16 values). ``rows`` restricts the work to some rows.
    Vocabulary chunks are visited in increasing id order; the maximum and the lowest id
    attaining it are tracked exactly, the exponential sum is taken after the maximum is known.
    """
    h = as_f64(h)
    if rows is None:
        rows = range(h.shape[0])
    rows = list(rows)
    hs = h[rows]
    V = w_lm.shape[0]
    # pass 1: exact maximum, its lowest id and the runner-up value
    zmax = np.full(len(rows), -np.inf)
    pred = np.zeros(len(rows), dtype=np.int64)
    second = np.full(len(rows), -np.inf)
    for v0 in range(0, V, chunk):
        z = hs @ as_f64(w_lm[v0: v0 + chunk]).T                    # [R, c]
        cmax = z.max(axis=1)
        carg = z.argmax(axis=1)                                     # first occurrence
        # runner-up inside the chunk: max after removing one copy of the chunk maximum
        zc = z.copy()
        zc[np.arange(len(rows)), carg] = -np.inf
        csec = zc.max(axis=1) if zc.shape[1] > 1 else np.full(len(rows), -np.inf)
        better = cmax > zmax
        # new runner-up = max(old max, chunk runner-up) if the chunk wins, else max(second, cmax)
        second = np.where(better, np.maximum(zmax, csec), np.maximum(second, cmax))
        pred = np.where(better, v0 + carg, pred)
        zmax = np.where(better, cmax, zmax)
    # pass 2: sum of exponentials relative to the maximum
    ssum = np.zeros(len(rows))
    for v0 in range(0, V, chunk):
        z = hs @ as_f64(w_lm[v0: v0 + chunk]).T
        ssum += np.exp(z - zmax[:, None]).sum(axis=1)
    conf = 1.0 / ssum
    gap = zmax - second
    return conf, pred, gap, zmax


# ----------------------------------------------------------------------------------------
# Commit rule ([chathome] generation + evaluation paragraphs; reading R6)
# ----------------------------------------------------------------------------------------

RULE_CONFIDENCE = 0       # mask-diffusion mode: confidence masking with threshold gamma
RULE_LEFT_TO_RIGHT = 1    # mock-AR reading: exactly one position per step, left to right


def commit(conf, pred, tokens, masked, gamma: float, force_all: bool,
           rule: int = RULE_CONFIDENCE):
    """Apply the commit rule to each sequence.

    conf [B, S] (fp64), pred [B, S], tokens [B, S] int, masked [B, S] bool.
    gamma is the float32 threshold widened to fp64, so both sides compare with one number.
    rule RULE_CONFIDENCE: {masked i : conf_i >= gamma}, else the most confident masked
    position (lowest index on ties). rule RULE_LEFT_TO_RIGHT (the pages name a mock-AR mode
    without defining it; read as the AR order inside the block): the lowest-index masked
    position, whatever its confidence. force_all (step T) commits every masked position.
    Returns (tokens', masked', n_committed [B], committed [B, S] bool).
    """
    conf = np.asarray(conf, dtype=np.float64)
    tokens = np.array(tokens, dtype=np.int64, copy=True)
    masked = np.array(masked, dtype=bool, copy=True)
    g = float(np.float32(gamma))
    B, S = masked.shape
    committed = np.zeros((B, S), dtype=bool)
    for b in range(B):
        if force_all:
            chosen = [i for i in range(S) if masked[b, i]]
        elif rule == RULE_LEFT_TO_RIGHT:
            chosen = [i for i in range(S) if masked[b, i]][:1]
        else:
            chosen = [i for i in range(S) if masked[b, i] and conf[b, i] >= g]
            if not chosen and masked[b].any():
                best = max(conf[b, i] for i in range(S) if masked[b, i])
                chosen = [min(i for i in range(S) if masked[b, i] and conf[b, i] == best)]
        for i in chosen:
            tokens[b, i] = int(pred[b, i])
            masked[b, i] = False
            committed[b, i] = True
    return tokens, masked, committed.sum(axis=1), committed


# ----------------------------------------------------------------------------------------
# Whole step and block loop ([chathome] inference + generation paragraphs)
# ----------------------------------------------------------------------------------------

def embed(tokens, emb, pos) -> np.ndarray:
    """h0[b, i] = bf16(emb[tokens[b, i]] + pos[i]); returns [B*S, d]."""
    tokens = np.asarray(tokens)
    B, S = tokens.shape
    idx = tokens.reshape(-1).astype(np.int64)
    if hasattr(emb, "detach"):                      # gather the rows before widening
        import torch
        e = as_f64(emb[torch.from_numpy(idx).to(emb.device)])
    else:
        e = as_f64(np.asarray(emb)[idx])
    p = np.tile(as_f64(pos)[:S], (B, 1))
    return bf16_round(e + p)


def block_positions(dims, ctx_len=None) -> np.ndarray:
    """Absolute position of every block row b*S + i: ctx_len[b] + i (the block follows the
    context; default ctx_len = Lmax)."""
    B, S = dims["B"], dims["S"]
    L = np.full(B, dims["Lmax"]) if ctx_len is None else np.asarray(ctx_len)
    return (L[:, None] + np.arange(S)[None, :]).reshape(-1)


def layer_forward(h, layer, phi, dims, ctx_len=None, rope_theta: float = 0.0):
    """One denoiser attention layer on the block hidden state h [B*S, d] (bf16 values).

    layer: dict with wqkv, wo, ada_E, k_ctx, v_ctx (tensors or arrays; k_ctx/v_ctx may hold
    only the sequences in this call). rope_theta > 0 rotates the block's q and k at their
    absolute positions (the cached context keys are taken as already rotated by the context
    tower). Returns the new h and the attention output o.
    """
    B, S, Hq, Hkv, D = dims["B"], dims["S"], dims["Hq"], dims["Hkv"], dims["D"]
    _, _, gate = adaln_vectors(layer["ada_E"], phi)
    x_mod = adaln_modulate(h, layer["ada_E"], phi)
    q, k, v = qkv_project(x_mod, layer["wqkv"], Hq, Hkv, D,
                          rope_pos=block_positions(dims, ctx_len), rope_theta=rope_theta)
    o, _ = block_attention(q.reshape(B, S, Hq, D), k.reshape(B, S, Hkv, D),
                           v.reshape(B, S, Hkv, D), layer["k_ctx"], layer["v_ctx"], ctx_len)
    o = bf16_round(o)                                                   # [Q3]
    return oproj_gated_residual(h, o.reshape(B * S, Hq * D), layer["wo"], gate), o


def denoise_step(dims, layers, phi_t, w_lm, tokens, masked, gamma, t, T,
                 h=None, emb=None, pos=None, ctx_len=None, rule: int = RULE_CONFIDENCE,
                 rope_theta: float = 0.0):
    """One denoising step: embed (if h is None), every layer, LM head, commit.

    Returns a dict with conf, pred, gap, tokens, masked, n_committed, committed, h_final.
    """
    B, S = dims["B"], dims["S"]
    if h is None:
        h = embed(tokens, emb, pos)
    else:
        h = as_f64(h)
    for layer in layers:
        h, _ = layer_forward(h, layer, phi_t, dims, ctx_len, rope_theta)
    conf, pred, gap, zmax = lmhead_confidence(h, w_lm)
    conf = conf.reshape(B, S); pred = pred.reshape(B, S); gap = gap.reshape(B, S)
    tok2, msk2, ncom, committed = commit(conf, pred, tokens, masked, gamma, force_all=(t == T),
                                         rule=rule)
    return dict(conf=conf, pred=pred, gap=gap, zmax=zmax.reshape(B, S), tokens=tok2,
                masked=msk2, n_committed=ncom, committed=committed, h_final=h)


def decode_block(dims, layers, phi_table, w_lm, emb, pos, gamma, T, tokens=None, masked=None,
                 t_start: int = 1, ctx_len=None, trace: bool = False,
                 rule: int = RULE_CONFIDENCE, rope_theta: float = 0.0):
    """Block decode loop: starting from all [MASK] (or a given state), run steps
    t = t_start..T, stop after the first step that leaves nothing masked.

    Returns (tokens, masked, steps_taken, per-step records if trace).
    """
    B, S, V = dims["B"], dims["S"], dims["V"]
    if tokens is None:
        tokens = np.full((B, S), V, dtype=np.int64)
        masked = np.ones((B, S), dtype=bool)
    tokens = np.array(tokens, dtype=np.int64, copy=True)
    masked = np.array(masked, dtype=bool, copy=True)
    steps = 0
    records = []
    for t in range(t_start, T + 1):
        if not masked.any():
            break
        r = denoise_step(dims, layers, phi_table[t - 1], w_lm, tokens, masked, gamma, t, T,
                         emb=emb, pos=pos, ctx_len=ctx_len, rule=rule, rope_theta=rope_theta)
        tokens, masked = r["tokens"], r["masked"]
        steps += 1
        if trace:
            records.append(r)
        if not masked.any():
            break
    return tokens, masked, steps, records


# ----------------------------------------------------------------------------------------
# Context cache growth ([chathome] generation paragraph: once a block is committed, the
# context tower takes it in and the next block attends to it)
# ----------------------------------------------------------------------------------------

def kv_append(k_ctx, v_ctx, ctx_len, k_new, v_new):
    """Append one committed block's keys / values to a layer's context cache.

    k_ctx, v_ctx [B, Hkv, Lmax, D]; ctx_len [B]; k_new, v_new [B, S, Hkv, D] (the context
    tower's keys / values of the block, token-major as a projection yields them).
    Row ctx_len[b] + i of head g receives token i of head g. Sequences whose cache would
    overflow (ctx_len[b] + S > Lmax) are left unchanged and reported.
    Returns (k_ctx', v_ctx', ctx_len', overflow [B] bool); inputs are not modified.
    """
    k = np.array(as_f64(k_ctx), copy=True)
    v = np.array(as_f64(v_ctx), copy=True)
    kn = as_f64(k_new)
    vn = as_f64(v_new)
    B, Hkv, Lmax, D = k.shape
    S = kn.shape[1]
    ln = np.array(ctx_len, dtype=np.int64, copy=True)
    overflow = np.zeros(B, dtype=bool)
    for b in range(B):
        L = int(ln[b])
        if L < 0 or L + S > Lmax:
            overflow[b] = True
            continue
        for g in range(Hkv):
            k[b, g, L:L + S, :] = kn[b, :, g, :]
            v[b, g, L:L + S, :] = vn[b, :, g, :]
        ln[b] = L + S
    return k, v, ln, overflow
