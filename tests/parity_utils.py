"""Helpers for the GPU parity tests: run the CUDA path through the binding,
run the oracle on the same bf16 bits, and compare (selection exactly up to
near-ties, attention within the stated tolerances)."""

from __future__ import annotations

import math
from typing import Iterable, Optional

import numpy as np
import torch

from oracle import bsa_oracle as O

# Tolerances for bf16 unit-normal inputs (attention outputs against the fp64
# oracle): max abs 2e-2, mean abs 2e-3, LSE abs 1e-2.
OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
LSE_ABS = 1e-2


def to_f32_np(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> float32 numpy (exact)."""
    return t.detach().float().cpu().numpy()


def compare_selection(gpu_idx: np.ndarray, gpu_cnt: np.ndarray, ref: dict) -> dict:
    """Counts must match exactly everywhere; index lists must match exactly on
    every row that is not a near-tie.  Returns statistics."""
    cnt_ref = ref["counts"]
    assert gpu_cnt.shape == cnt_ref.shape
    mism_cnt = np.argwhere(gpu_cnt != cnt_ref)
    assert mism_cnt.size == 0, f"count mismatch at {mism_cnt[:5].tolist()}"
    B, H, nQ = cnt_ref.shape
    bad, near, near_differs = 0, 0, 0
    first_bad = None
    for b in range(B):
        for h in range(H):
            for qb in range(nQ):
                c = int(cnt_ref[b, h, qb])
                same = np.array_equal(gpu_idx[b, h, qb, :c], ref["indices"][b, h, qb, :c])
                if ref["near_tie"][b, h, qb]:
                    near += 1
                    near_differs += 0 if same else 1
                elif not same:
                    bad += 1
                    if first_bad is None:
                        first_bad = (b, h, qb)
    assert bad == 0, f"{bad} rows with different index sets (first {first_bad})"
    return dict(rows=B * H * nQ, near_ties=near, near_ties_differing=near_differs)


def check_structure(gpu_idx: np.ndarray, gpu_cnt: np.ndarray, prefix: int, seq_lens, bq: int, bk: int):
    """Every row: prefix blocks first, strictly ascending, in range."""
    B, H, nQ = gpu_cnt.shape
    for b in range(B):
        geo = O.kv_geometry(prefix, seq_lens[b], bk)
        npb, nkv = geo["n_prefix_blocks"], geo["n_kv_valid"]
        for h in range(H):
            for qb in range(nQ):
                c = int(gpu_cnt[b, h, qb])
                if qb * bq >= seq_lens[b]:
                    assert c == 0
                    continue
                row = gpu_idx[b, h, qb, :c]
                assert (row[:npb] == np.arange(npb)).all()
                assert (np.diff(row) > 0).all()
                assert row.min() >= 0 and row.max() < nkv


def compare_attention(out_gpu: np.ndarray, lse_gpu: np.ndarray, out_ref: np.ndarray, lse_ref: np.ndarray,
                      seq_lens, tiles: Optional[Iterable[tuple]] = None, bq: int = None) -> dict:
    """Elementwise comparison over the rows the oracle computed (non-NaN)."""
    B, Sq, Hq, d = out_ref.shape
    mask = ~np.isnan(out_ref[..., 0])              # [B, Sq, Hq]
    assert mask.any()
    o_g = out_gpu[mask].astype(np.float64)
    o_r = out_ref[mask]
    assert np.isfinite(o_g).all(), "non-finite GPU output"
    err = np.abs(o_g - o_r)
    lmask = ~np.isnan(lse_ref)                     # [B, Hq, Sq]
    lg, lr = lse_gpu[lmask].astype(np.float64), lse_ref[lmask]
    inf_r = np.isneginf(lr)
    assert (np.isneginf(lg) == inf_r).all(), "-inf LSE rows differ"
    lerr = np.abs(lg[~inf_r] - lr[~inf_r]) if (~inf_r).any() else np.zeros(1)
    stats = dict(out_max_abs=float(err.max()), out_mean_abs=float(err.mean()),
                 lse_max_abs=float(lerr.max()), rows=int(mask.sum()))
    assert stats["out_max_abs"] <= OUT_MAX_ABS, stats
    assert stats["out_mean_abs"] <= OUT_MEAN_ABS, stats
    assert stats["lse_max_abs"] <= LSE_ABS, stats
    # padded rows: exactly 0 / -inf
    for b, L in enumerate(seq_lens):
        if L < Sq:
            assert (out_gpu[b, L:] == 0).all()
            assert np.isneginf(lse_gpu[b, :, L:]).all()
    return stats


def sample_tiles(B: int, Hq: int, nQb: int, seq_lens, bq: int, n_random: int, seed: int = 0):
    """Every head x {first, middle, last real} query block + random tiles, plus
    padded blocks of each request."""
    rng = np.random.default_rng(seed)
    tiles = set()
    for b in range(B):
        nqv = O.cdiv(seq_lens[b], bq)
        for h in range(Hq):
            for qb in {0, nqv // 2, nqv - 1}:
                tiles.add((b, h, qb))
        if nqv < nQb:
            tiles.add((b, int(rng.integers(Hq)), nqv))
            tiles.add((b, int(rng.integers(Hq)), nQb - 1))
    for _ in range(n_random):
        b = int(rng.integers(B))
        tiles.add((b, int(rng.integers(Hq)), int(rng.integers(O.cdiv(seq_lens[b], bq)))))
    return sorted(tiles)
