"""fp64 CPU oracle for selected-block attention (test infrastructure only).

Importable only by the tests, the smoke check and the bench's CPU-baseline arm.
Parity: every function is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (closed forms, brute force, library routines,
invariants and a hand-worked example); none is "parity unpinned".
"""

from .bsa_oracle import (  # noqa: F401
    NEAR_TIE_REL,
    apply_rope,
    attention,
    attention_backward,
    attention_rows,
    attention_tile,
    causal_prefix_attention,
    boundary_gap,
    cdiv,
    default_scale,
    dense_indices,
    is_near_tie,
    keep_count,
    kv_geometry,
    pool_means,
    rope_then_select,
    rotate_half,
    round_to_bf16,
    select_blocks,
    tile_keys,
    topk_lowest_index,
)
