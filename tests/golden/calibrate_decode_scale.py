"""Calibration of the block decode loop's LM-head weight scale (synth.DECODE_W_LM_SIGMA).

The decode workload is meant to commit several tokens per step early in a block, as the pages
describe for confidence masking at gamma = 0.8, rather than fall back to one commit per step
throughout. Its logits therefore use the sharpness of the mid-size single step (about 30 % of
the masked positions clear gamma = 0.8 there): this script runs the fp64 oracle (and nothing
else) on the first denoise step of the seeded decode workload, on a few of its sequences, for
each candidate standard deviation of W_lm, and prints the fraction of positions whose
confidence clears 0.8. The candidate closest to 30 % is the stored constant.

Usage: python tests/golden/calibrate_decode_scale.py [sigma ...]
"""

from __future__ import annotations

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from block_diffusion_lm_denoise_b300 import synth  # noqa: E402

TARGET = 0.30
SEQS = [0, 21, 42, 63]


def first_step_fraction(sigma: float, seqs=SEQS) -> float:
    """Fraction of the positions of the given sequences whose oracle confidence is >= 0.8 in
    step 1 of the decode workload with W_lm ~ N(0, sigma^2) (all positions are [MASK])."""
    wl = synth.decode_loop("cpu", kv_rows=seqs, w_lm_sigma=sigma, emb_rows=[synth.DECODE_V])
    dm = wl.dims
    d = dict(dm.as_dict(), B=len(seqs))
    # every position holds [MASK] (id V): the embedding table needs only that row, which
    # emb_rows placed at index 0
    tokens = np.zeros((len(seqs), dm.S), dtype=np.int64)
    masked = np.ones((len(seqs), dm.S), bool)
    r = oracle.denoise_step(d, wl.layers, wl.phi_table[0], wl.w_lm, tokens, masked, wl.gamma,
                            1, wl.T, emb=wl.emb, pos=wl.pos)
    return float((r["conf"] >= wl.gamma).mean())


def main(argv):
    sigmas = [float(x) for x in argv] or [0.06, 0.08, 0.085, 0.09, 0.10]
    best = None
    for s in sigmas:
        f = first_step_fraction(s)
        print(f"W_lm sigma {s:.3f}: fraction of positions with conf >= 0.8 at step 1 = {f:.3f}",
              flush=True)
        if best is None or abs(f - TARGET) < abs(best[1] - TARGET):
            best = (s, f)
    print(f"closest to {TARGET:.0%}: sigma {best[0]} ({best[1]:.3f})")


if __name__ == "__main__":
    main(sys.argv[1:])
