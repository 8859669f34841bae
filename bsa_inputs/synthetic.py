"""Seeded synthetic Q/K/V for selected-block attention workloads.

The shapes stand in for the video-latent attention layers that the pages
measure end to end (Cosmos3-Nano 720p/189 frames in "[Core] Add Cosmos3
attention strategy PoC", Test Result; MiniMax H3 1280x736/192 frames in
"[Model] Add MiniMax H3 attention strategy PoC"; Cosmos3-Edge 832x480x121 in
mstar PR 927).  No dataset, prompt or weight is involved: every tensor is
drawn from a seeded torch.Generator.

Layout follows the per-sequence ``[seq, heads, head_dim]`` tensors of
``cosmos_parallel.py`` (``cosmos3_cp_attention``) with a leading batch axis:
Q ``[B, Sq, Hq, d]``, K/V ``[B, Skv, Hkv, d]`` with ``Skv = prefix + Sq``.
Key position ``t < prefix`` is the understanding/text stream, key position
``prefix + i`` is generation token ``i`` (the generation pathway attends
``cat(und, gen)``).

Value recipes
-------------
* ``iid``: every element N(0, 1), drawn in fp32 and rounded to bf16 once.
* ``block``: generation token ``i`` at latent position ``(f, y, x)`` of the
  config's ``(F, Y, X)`` grid gets ``mu[f, y // 8, x // 8] + 0.5 * eps`` with
  ``mu ~ N(0, 1)`` per (frame, 8x8 patch tile, KV head, channel) and
  ``eps ~ N(0, 1)``.  Q heads of a GQA group and their K head share ``mu``
  (so block means carry locality); V has its own ``mu``.  Prefix K/V rows are
  i.i.d. N(0, 1).  Each batch element draws its own ``mu``.
* Padding rows (query rows ``>= L_b``, key rows ``>= prefix + L_b``) are set to
  ``pad_fill`` (NaN in tests to prove they are never read into real results).

Draw order per batch element: ``mu_qk``, ``mu_v`` (block recipe only), Q
noise, K noise, V noise.  Per-head keep ratios come from a separate CPU
generator so that they are identical whatever device the tensors are made on.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence, Tuple

import torch


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    prefix: int
    lens: Tuple[int, ...]          # real generation length per batch element
    block_q: int
    block_k: int
    keep: object                   # float, or ("uniform", lo, hi) drawn per query head
    recipe: str = "iid"            # "iid" or "block"
    grid: Optional[Tuple[int, int, int]] = None   # (frames, rows, cols) of the latent
    seed: int = 0
    description: str = ""

    @property
    def Sq(self) -> int:
        return max(self.lens)

    @property
    def Skv(self) -> int:
        return self.prefix + self.Sq


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def derived_sizes(cfg: Config) -> dict:
    """Padded sizes and block counts of a config (pure shape arithmetic)."""
    return dict(
        Sq=cfg.Sq,
        Skv=cfg.Skv,
        nQb=_cdiv(cfg.Sq, cfg.block_q),
        nKb=_cdiv(cfg.Skv, cfg.block_k),
        G=cfg.Hq // cfg.Hkv,
    )


# The five workloads, plus smaller cases that the oracle finishes in seconds
# while still spanning several tiles, GQA/MQA/MHA and ragged tails.
CONFIGS = {
    "tiny": Config(
        "tiny", B=1, Hq=4, Hkv=2, d=64, prefix=256, lens=(1024,), block_q=64,
        block_k=64, keep=0.25, recipe="iid", seed=1001,
        description="tiny GQA d64, 64x64 blocks, keep 25%"),
    "480p_dense": Config(
        "480p_dense", B=1, Hq=24, Hkv=8, d=128, prefix=512, lens=(48360,),
        block_q=256, block_k=128, keep=1.0, recipe="iid", grid=(31, 30, 52),
        seed=1002, description="480p latent (31x30x52), dense pass"),
    "480p_75": Config(
        "480p_75", B=1, Hq=24, Hkv=8, d=128, prefix=512, lens=(48360,),
        block_q=256, block_k=128, keep=0.25, recipe="block", grid=(31, 30, 52),
        seed=1003, description="480p latent (31x30x52), keep 25%"),
    "720p_75": Config(
        "720p_75", B=1, Hq=32, Hkv=8, d=128, prefix=1024, lens=(172800,),
        block_q=256, block_k=128, keep=0.25, recipe="block", grid=(48, 45, 80),
        seed=1004, description="720p latent (48x45x80), keep 25%"),
    "1280x736_ragged": Config(
        "1280x736_ragged", B=2, Hq=24, Hkv=24, d=128, prefix=512,
        lens=(176640, 150000), block_q=256, block_k=128,
        keep=("uniform", 0.10, 0.50), recipe="block", grid=(48, 46, 80),
        seed=1005, description="1280x736 latent (48x46x80), 2 ragged requests, per-head keep"),
    "480p_75_64x64": Config(
        "480p_75_64x64", B=1, Hq=24, Hkv=8, d=128, prefix=512, lens=(48360,),
        block_q=64, block_k=64, keep=0.25, recipe="block", grid=(31, 30, 52),
        seed=1006, description="480p latent, Hopper 64x64 geometry at d128, keep 25%"),
    # --- small parity cases (oracle in seconds; several tiles + ragged tails) ---
    "small_gqa": Config(
        "small_gqa", B=2, Hq=4, Hkv=2, d=128, prefix=256, lens=(1900, 1333),
        block_q=256, block_k=128, keep=0.3, recipe="block", grid=(4, 24, 24),
        seed=2001, description="2 ragged requests, GQA 2, 256x128 blocks"),
    "small_mqa_d64": Config(
        "small_mqa_d64", B=1, Hq=3, Hkv=1, d=64, prefix=100, lens=(777,),
        block_q=64, block_k=64, keep=0.4, recipe="iid", seed=2002,
        description="MQA, prefix not a multiple of the block, d64"),
    "small_mha_perhead": Config(
        "small_mha_perhead", B=2, Hq=3, Hkv=3, d=128, prefix=0, lens=(1024, 700),
        block_q=128, block_k=128, keep=("uniform", 0.1, 0.5), recipe="block",
        grid=(2, 16, 32), seed=2003,
        description="MHA, no prefix, per-head keep, 128x128 blocks"),
    "small_64x64_d128": Config(
        "small_64x64_d128", B=1, Hq=2, Hkv=1, d=128, prefix=128, lens=(640,),
        block_q=64, block_k=64, keep=0.25, recipe="iid", seed=2004,
        description="Hopper 64x64 geometry at d128"),
}

# The configs named by the workload description, in order (tiny, 480p dense,
# 480p 75%, 720p 75%, 1280x736 ragged).
WORKLOAD_CONFIGS = ("tiny", "480p_dense", "480p_75", "720p_75", "1280x736_ragged")


def keep_ratios(cfg: Config) -> list:
    """Keep ratio per query head (length 1 when shared), as float32 values."""
    if isinstance(cfg.keep, tuple):
        _, lo, hi = cfg.keep
        g = torch.Generator(device="cpu").manual_seed(cfg.seed + 7)
        r = lo + (hi - lo) * torch.rand(cfg.Hq, generator=g, dtype=torch.float32)
        return [float(x) for x in r]
    return [float(torch.tensor(cfg.keep, dtype=torch.float32))]


def _tile_ids(L: int, grid: Tuple[int, int, int]) -> Tuple[torch.Tensor, Tuple[int, int, int]]:
    F, Y, X = grid
    if L > F * Y * X:
        raise ValueError(f"length {L} exceeds the latent grid {grid}")
    t = torch.arange(L, dtype=torch.int64)
    f = t // (Y * X)
    y = (t // X) % Y
    x = t % X
    ty, tx = _cdiv(Y, 8), _cdiv(X, 8)
    return (f * ty + y // 8) * tx + x // 8, (F, ty, tx)


def make_inputs(cfg: Config, device="cpu", pad_fill: float = 0.0,
                lens: Optional[Sequence[int]] = None) -> dict:
    """Draw Q, K, V (bf16) for ``cfg`` on ``device``.

    Returns a dict with ``q``, ``k``, ``v``, ``seq_lens`` (python ints),
    ``keep_ratio`` (python floats holding float32 values) and the config.
    """
    device = torch.device(device)
    lens = tuple(cfg.lens if lens is None else lens)
    B, Hq, Hkv, d, P = cfg.B, cfg.Hq, cfg.Hkv, cfg.d, cfg.prefix
    Sq = max(lens)
    Skv = P + Sq
    G = Hq // Hkv
    gen = torch.Generator(device=device).manual_seed(cfg.seed)
    bf = torch.bfloat16
    q = torch.empty(B, Sq, Hq, d, dtype=bf, device=device)
    k = torch.empty(B, Skv, Hkv, d, dtype=bf, device=device)
    v = torch.empty(B, Skv, Hkv, d, dtype=bf, device=device)
    for b in range(B):
        L = lens[b]
        if cfg.recipe == "block":
            tid, (F, ty, tx) = _tile_ids(L, cfg.grid)
            tid = tid.to(device)
            n_tiles = F * ty * tx
            mu_qk = torch.randn(n_tiles, Hkv, d, generator=gen, device=device)
            mu_v = torch.randn(n_tiles, Hkv, d, generator=gen, device=device)
            # Q: chunks of rows keep the fp32 transient small at 720p.
            eq = torch.randn(L, Hq, d, generator=gen, device=device)
            for s0 in range(0, L, 32768):
                s1 = min(L, s0 + 32768)
                m = mu_qk[tid[s0:s1]].repeat_interleave(G, dim=1)
                q[b, s0:s1] = (m + 0.5 * eq[s0:s1]).to(bf)
            del eq
            ek = torch.randn(P + L, Hkv, d, generator=gen, device=device)
            k[b, :P] = ek[:P].to(bf)
            k[b, P:P + L] = (mu_qk[tid] + 0.5 * ek[P:]).to(bf)
            del ek
            ev = torch.randn(P + L, Hkv, d, generator=gen, device=device)
            v[b, :P] = ev[:P].to(bf)
            v[b, P:P + L] = (mu_v[tid] + 0.5 * ev[P:]).to(bf)
            del ev
        elif cfg.recipe == "iid":
            q[b, :L] = torch.randn(L, Hq, d, generator=gen, device=device).to(bf)
            k[b, :P + L] = torch.randn(P + L, Hkv, d, generator=gen, device=device).to(bf)
            v[b, :P + L] = torch.randn(P + L, Hkv, d, generator=gen, device=device).to(bf)
        else:
            raise ValueError(f"unknown recipe {cfg.recipe}")
        if L < Sq:
            q[b, L:] = pad_fill
        if P + L < Skv:
            k[b, P + L:] = pad_fill
            v[b, P + L:] = pad_fill
    return dict(q=q, k=k, v=v, seq_lens=list(lens), keep_ratio=keep_ratios(cfg), cfg=cfg)
