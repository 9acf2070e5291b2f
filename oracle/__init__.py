"""fp64 CPU oracle of the TwoTower denoise step (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package. See ``td_oracle`` for the method, its sources and its readings.
"""

from .td_oracle import (  # noqa: F401
    LN_EPS,
    RULE_CONFIDENCE,
    RULE_LEFT_TO_RIGHT,
    adaln_modulate,
    adaln_vectors,
    as_f64,
    bf16_round,
    block_attention,
    block_positions,
    commit,
    decode_block,
    denoise_step,
    embed,
    kv_append,
    layer_forward,
    layer_norm,
    lmhead_confidence,
    oproj_gated_residual,
    qkv_project,
    rope_rotate,
    timestep_embedding,
    timestep_table,
)
