"""fp64 CPU oracle for selected-block attention.  TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the bench's CPU-baseline arm may import
this module.  The product path (the CUDA library and its binding) never calls
it, and it shares no code with that path: it is plain numpy in float64,
written from the pages' description of the method, slow and direct on purpose.

What the method computes (sources, by page title and section):

* "[Core] Add shared block-sparse attention adapters with FlashAttention-4"
  (vllm-omni PR 8335), Purpose: a selector produces per-query-head KV block
  indices and counts, an adapter executes exactly that selection; the shared
  layer keeps a protected KV prefix, pads a single document at its end, keeps
  the native MHA/MQA/GQA head mapping and block geometry, and never falls back
  to dense attention.  Target sparsity 75%; blocks 64x64 (Hopper) or 256x128
  (Blackwell), query x key.
* ``cosmos_parallel.py`` (diffusers Cosmos 3 example), ``cosmos3_cp_attention``:
  generation queries attend, non-causally, over ``cat(und, gen)`` keys and
  values; ``_repeat_kv_heads``: query head ``i`` pairs with KV head
  ``i // repeats``; ``build_gen_key_mask``: padded key positions get the most
  negative value so real queries ignore them.
* mstar PR 927, "What the review checked": default softmax scale
  ``head_dim ** -0.5``.

How the selector scores blocks is not on the pages.  The readings used here
(all listed with the design notes) are: mean-pool Q and K over the valid rows
of each block, score a (query block, key block) pair by the dot product of
the two means, keep per row the ``k_h = min(N, ceil(r_h * N))`` best
non-prefix valid key blocks under the order (score descending, block index
ascending), force every prefix block in, and write the indices ascending.
LSE is the natural-log log-sum-exp of the scaled logits.  Padded query rows
and rows that see no key get output 0 and LSE -inf.

Precision: every value is converted to float64 before any arithmetic; inputs
are the bf16 bit patterns the GPU receives.
"""

from __future__ import annotations

import math
from typing import Iterable, Optional, Sequence

import numpy as np

NEAR_TIE_REL = 1e-4   # relative gap below which a selection boundary is a near-tie


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


# ---------------------------------------------------------------------------
# Geometry of the concatenated key sequence
# ---------------------------------------------------------------------------

def kv_geometry(prefix_len: int, gen_len: int, block_k: int) -> dict:
    """Key blocks of one request.

    Keys are ``cat(und, gen)`` (cosmos_parallel.py, ``cosmos3_cp_attention``):
    positions ``[0, prefix_len)`` are the protected understanding/text prefix
    (PR 8335, Purpose: "protected KV prefixes"), positions
    ``[prefix_len, prefix_len + gen_len)`` are generation tokens, and anything
    after is suffix padding.  Key blocks tile this sequence from position 0;
    a block that holds any prefix position is a prefix block.
    """
    n_valid_keys = prefix_len + gen_len
    n_kv_valid = cdiv(n_valid_keys, block_k)
    n_prefix_blocks = cdiv(prefix_len, block_k)
    return dict(
        n_valid_keys=n_valid_keys,
        n_kv_valid=n_kv_valid,
        n_prefix_blocks=min(n_prefix_blocks, n_kv_valid),
        n_candidates=max(0, n_kv_valid - n_prefix_blocks),
    )


def keep_count(ratio: float, n_candidates: int) -> int:
    """``k = min(N, ceil(r * N))`` evaluated in float64.

    PR 8335 (Purpose) and PR 8583 (Test Result) speak only of a "75% target
    sparsity"; keeping the ceiling of the kept fraction keeps at least one
    block whenever ``r > 0`` and makes ``r = 1`` the dense pass.
    """
    if n_candidates <= 0:
        return 0
    r = float(ratio)
    if r <= 0.0:
        return 0
    return int(min(n_candidates, math.ceil(r * float(n_candidates))))


# ---------------------------------------------------------------------------
# Selector: pooling, scoring, top-k with the prefix forced in
# ---------------------------------------------------------------------------

def pool_means(x: np.ndarray, n_valid: int, block: int) -> np.ndarray:
    """Mean of the valid rows of each block.

    ``x`` is one request's ``[S, H, d]`` tensor (float64).  Block ``j`` covers
    rows ``[j*block, (j+1)*block)``; only rows ``< n_valid`` are averaged
    (suffix padding is not data; PR 8335, Purpose).  A block with no valid
    row gets NaN.  Returns ``[H, ceil(S/block), d]``.
    """
    S, H, d = x.shape
    nb = cdiv(S, block)
    out = np.full((H, nb, d), np.nan, dtype=np.float64)
    for j in range(nb):
        r0 = j * block
        r1 = min((j + 1) * block, n_valid, S)
        if r1 <= r0:
            continue
        out[:, j, :] = np.asarray(x[r0:r1], dtype=np.float64).mean(axis=0)
    return out


def topk_lowest_index(scores: np.ndarray, k: int) -> np.ndarray:
    """Positions of the ``k`` best scores; ties go to the lower position.

    The order is (score descending, position ascending), a total order, so the
    result is unique.  Returned ascending.
    """
    n = scores.shape[0]
    # lexsort: last key is the primary one -> (-score ascending, position ascending)
    order = np.lexsort((np.arange(n), -np.asarray(scores, dtype=np.float64)))
    return np.sort(order[:k]).astype(np.int64)


def boundary_gap(scores: np.ndarray, k: int) -> Optional[tuple]:
    """(k-th best, (k+1)-th best) scores, or None when there is no boundary."""
    n = scores.shape[0]
    if k <= 0 or k >= n:
        return None
    s = np.sort(scores)[::-1]
    return float(s[k - 1]), float(s[k])


def is_near_tie(scores: np.ndarray, k: int, rel: float = NEAR_TIE_REL) -> bool:
    """True when the k-th and (k+1)-th best scores differ by <= rel (relative).

    At such a boundary an fp32 GPU score and this fp64 score may legitimately
    rank the two blocks differently, so the row's index set is not unique.
    """
    g = boundary_gap(scores, k)
    if g is None:
        return False
    a, b = g
    return abs(a - b) <= rel * max(abs(a), abs(b))


def select_blocks(q: np.ndarray, k: np.ndarray, prefix_len: int,
                  seq_lens: Sequence[int], block_q: int, block_k: int,
                  keep_ratio: Sequence[float]) -> dict:
    """Per-query-head selected KV block lists (PR 8335, Purpose: "the selector
    produces per-query-head block indices/counts").

    ``q``: ``[B, Sq, Hq, d]``, ``k``: ``[B, Skv, Hkv, d]`` (any float dtype; used
    as float64).  ``keep_ratio`` has one value or one per query head.

    Returns ``indices`` ``[B, Hq, nQb, nKb]`` (entries past ``count`` are -1),
    ``counts`` ``[B, Hq, nQb]``, ``near_tie`` ``[B, Hq, nQb]`` (bool),
    ``scores`` ``[B, Hq, nQb, nKb]`` (NaN where not a candidate) and ``k``
    ``[B, Hq]`` (kept non-prefix blocks per valid row).
    """
    q = np.asarray(q)          # converted to float64 block by block
    k = np.asarray(k)
    B, Sq, Hq, d = q.shape
    _, Skv, Hkv, _ = k.shape
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    nQb, nKb = cdiv(Sq, block_q), cdiv(Skv, block_k)
    ratios = list(keep_ratio)
    if len(ratios) == 1:
        ratios = ratios * Hq
    if len(ratios) != Hq:
        raise ValueError("keep_ratio needs 1 or Hq values")
    indices = np.full((B, Hq, nQb, nKb), -1, dtype=np.int64)
    counts = np.zeros((B, Hq, nQb), dtype=np.int64)
    near = np.zeros((B, Hq, nQb), dtype=bool)
    scores_all = np.full((B, Hq, nQb, nKb), np.nan)
    kk = np.zeros((B, Hq), dtype=np.int64)
    for b in range(B):
        L = int(seq_lens[b])
        geo = kv_geometry(prefix_len, L, block_k)
        npb, nkv = geo["n_prefix_blocks"], geo["n_kv_valid"]
        ncand = nkv - npb
        qbar = pool_means(q[b], L, block_q)                  # [Hq, nQb, d]
        kbar = pool_means(k[b], geo["n_valid_keys"], block_k)  # [Hkv, nKb, d]
        n_q_valid = cdiv(L, block_q)
        for h in range(Hq):
            kh = keep_count(ratios[h], ncand)
            kk[b, h] = kh
            hk = h // G        # _repeat_kv_heads: query head i pairs with KV head i // G
            # block scores of every valid query block against the candidates
            S = qbar[h, :n_q_valid, :] @ kbar[hk, npb:nkv, :].T
            for qb in range(n_q_valid):
                s = S[qb]
                scores_all[b, h, qb, npb:nkv] = s
                chosen = topk_lowest_index(s, kh) + npb
                row = np.concatenate([np.arange(npb, dtype=np.int64), chosen])
                counts[b, h, qb] = row.shape[0]
                indices[b, h, qb, :row.shape[0]] = row
                near[b, h, qb] = is_near_tie(s, kh)
    return dict(indices=indices, counts=counts, near_tie=near, scores=scores_all, k=kk)


# ---------------------------------------------------------------------------
# Attention over the selected blocks
# ---------------------------------------------------------------------------

def attention_rows(qrows: np.ndarray, keys: np.ndarray, vals: np.ndarray,
                   scale: float):
    """Softmax attention of ``qrows`` [n, d] over ``keys``/``vals`` [m, d].

    ``z = (q . k) * scale``, ``out = sum softmax(z) v``, ``lse = log sum exp z``
    (natural log).  With no key at all: out 0, lse -inf.
    """
    n, d = qrows.shape
    if keys.shape[0] == 0:
        return np.zeros((n, vals.shape[1])), np.full(n, -np.inf)
    z = (qrows @ keys.T) * scale
    m = z.max(axis=1, keepdims=True)
    p = np.exp(z - m)
    l = p.sum(axis=1, keepdims=True)
    out = (p @ vals) / l
    lse = (m + np.log(l))[:, 0]
    return out, lse


def tile_keys(idx_row: Iterable[int], n_valid_keys: int, block_k: int) -> np.ndarray:
    """Key positions covered by the selected blocks, minus suffix padding."""
    pos = []
    for kb in idx_row:
        r0 = int(kb) * block_k
        r1 = min((int(kb) + 1) * block_k, n_valid_keys)
        if r1 > r0:
            pos.append(np.arange(r0, r1, dtype=np.int64))
    if not pos:
        return np.zeros(0, dtype=np.int64)
    return np.concatenate(pos)


def attention_tile(q: np.ndarray, k: np.ndarray, v: np.ndarray, b: int, h: int,
                   qb: int, idx_row, prefix_len: int, seq_len: int,
                   block_q: int, block_k: int, scale: float):
    """Output rows of one work tile (request b, query head h, query block qb).

    Returns (out [rows, d], lse [rows], row0): rows are every query position of
    the block inside the padded length; rows ``>= seq_len`` are padding and
    get 0 / -inf.
    """
    Sq = q.shape[1]
    Hq, Hkv = q.shape[2], k.shape[2]
    hk = h // (Hq // Hkv)
    r0 = qb * block_q
    r1 = min((qb + 1) * block_q, Sq)
    dv = v.shape[3]
    out = np.zeros((r1 - r0, dv))
    lse = np.full(r1 - r0, -np.inf)
    rv = min(r1, seq_len)
    if rv > r0:
        pos = tile_keys(idx_row, prefix_len + seq_len, block_k)
        qq = np.asarray(q[b, r0:rv, h, :], dtype=np.float64)
        kk = np.asarray(k[b, pos, hk, :], dtype=np.float64)
        vv = np.asarray(v[b, pos, hk, :], dtype=np.float64)
        o, l = attention_rows(qq, kk, vv, scale)
        out[: rv - r0] = o
        lse[: rv - r0] = l
    return out, lse, r0


def default_scale(d: int) -> float:
    """Softmax scale ``head_dim ** -0.5`` (mstar PR 927, review notes)."""
    return 1.0 / math.sqrt(d)


def dense_indices(prefix_len: int, seq_lens: Sequence[int], Sq: int, Skv: int,
                  block_q: int, block_k: int, Hq: int):
    """Index lists of the dense pass: every valid key block, for every valid
    query block (sparsity 0 runs through the same attention)."""
    B = len(seq_lens)
    nQb, nKb = cdiv(Sq, block_q), cdiv(Skv, block_k)
    idx = np.full((B, Hq, nQb, nKb), -1, dtype=np.int64)
    cnt = np.zeros((B, Hq, nQb), dtype=np.int64)
    for b, L in enumerate(seq_lens):
        nkv = kv_geometry(prefix_len, L, block_k)["n_kv_valid"]
        for qb in range(cdiv(L, block_q)):
            idx[b, :, qb, :nkv] = np.arange(nkv)
            cnt[b, :, qb] = nkv
    return idx, cnt


def attention(q, k, v, indices, counts, prefix_len: int, seq_lens: Sequence[int],
              block_q: int, block_k: int, scale: Optional[float] = None,
              tiles: Optional[Iterable[tuple]] = None):
    """Selected-block attention forward.

    ``indices`` ``[B, Hq, nQb, nKb]`` / ``counts`` ``[B, Hq, nQb]`` as written by
    the selector; the adapter attends exactly the listed blocks (PR 8335,
    Purpose).  ``tiles``: iterable of (b, h, qb) to compute (default all);
    entries not computed are NaN.

    Returns out ``[B, Sq, Hq, d]`` and lse ``[B, Hq, Sq]`` (float64).
    """
    q = np.asarray(q)
    B, Sq, Hq, d = q.shape
    dv = np.asarray(v).shape[3]
    if scale is None or scale <= 0:
        scale = default_scale(d)
    nQb = cdiv(Sq, block_q)
    out = np.full((B, Sq, Hq, dv), np.nan)
    lse = np.full((B, Hq, Sq), np.nan)
    if tiles is None:
        tiles = [(b, h, qb) for b in range(B) for h in range(Hq) for qb in range(nQb)]
    for (b, h, qb) in tiles:
        c = int(counts[b, h, qb])
        row = indices[b, h, qb, :c]
        o, l, r0 = attention_tile(q, k, v, b, h, qb, row, prefix_len, int(seq_lens[b]),
                                  block_q, block_k, scale)
        out[b, r0:r0 + o.shape[0], h, :] = o
        lse[b, h, r0:r0 + o.shape[0]] = l
    return out, lse


# ---------------------------------------------------------------------------
# Understanding stream: causal self-attention over the prefix
# ---------------------------------------------------------------------------

def causal_prefix_attention(q_und, k, v, prefix_len: int, scale: Optional[float] = None):
    """Causal self-attention of the understanding (prefix) stream.

    cosmos_parallel.py, ``cosmos3_cp_attention``: the understanding pathway
    self-attends causally over the full understanding sequence (``is_causal``
    with equal query and key lengths).  Query row i of ``q_und`` ``[B, P, Hq, d]``
    attends key positions ``0..i`` of ``k``/``v`` (``[B, >=P, Hkv, d]``; only the
    first P rows are understanding keys), reading KV head h // (Hq/Hkv).

    Returns out ``[B, P, Hq, d]`` and lse ``[B, Hq, P]`` (float64).
    """
    q_und = np.asarray(q_und)
    B, P, Hq, d = q_und.shape
    Hkv = np.asarray(k).shape[2]
    G = Hq // Hkv
    if scale is None or scale <= 0:
        scale = default_scale(d)
    out = np.zeros((B, P, Hq, np.asarray(v).shape[3]))
    lse = np.full((B, Hq, P), -np.inf)
    for b in range(B):
        for h in range(Hq):
            qq = np.asarray(q_und[b, :, h, :], dtype=np.float64)
            kk = np.asarray(k[b, :P, h // G, :], dtype=np.float64)
            vv = np.asarray(v[b, :P, h // G, :], dtype=np.float64)
            for i in range(P):
                o, l = attention_rows(qq[i:i + 1], kk[:i + 1], vv[:i + 1], scale)
                out[b, i, h] = o[0]
                lse[b, h, i] = l[0]
    return out, lse


# ---------------------------------------------------------------------------
# Rotary prologue (applied before selection and attention)
# ---------------------------------------------------------------------------

def round_to_bf16(x) -> np.ndarray:
    """float64/float32 -> nearest bf16 value (ties to even), returned as float64.

    IEEE round-to-nearest-even on the float32 bit pattern: add 0x7FFF plus the
    lowest kept bit, clear the 16 dropped bits.  NaN stays NaN."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) & 0xFFFF0000).astype(np.uint32).view(np.float32)
    r = np.where(np.isnan(f), np.float32(np.nan), r)
    return r.astype(np.float64)


def rotate_half(x: np.ndarray) -> np.ndarray:
    """Half-split rotation of the last axis: (x1, x2) -> (-x2, x1).

    cosmos_parallel.py imports ``_rotate_half`` from the Cosmos 3 transformer
    without printing it; this is the conventional half-split form that name
    denotes (first half paired with the second half)."""
    d = x.shape[-1]
    return np.concatenate([-x[..., d // 2:], x[..., : d // 2]], axis=-1)


def apply_rope(x, cos, sin) -> np.ndarray:
    """``x * cos + rotate_half(x) * sin`` (cosmos_parallel.py,
    ``_project_qkv_with_rope``), in float64.

    ``x``: ``[B, S, H, d]``; ``cos``/``sin``: ``[S, d]`` per position, shared by
    every head (the ``unsqueeze(1)`` over heads) and every request."""
    x = np.asarray(x, dtype=np.float64)
    c = np.asarray(cos, dtype=np.float64)[None, :, None, :]
    s = np.asarray(sin, dtype=np.float64)[None, :, None, :]
    return x * c + rotate_half(x) * s


def rope_then_select(q, k, cos_q, sin_q, cos_k, sin_k, prefix_len, seq_lens, block_q, block_k,
                     keep_ratio) -> dict:
    """The selector run on rotated Q and K: RoPE in float64, rounded to bf16
    (the precision the attention reads), then ``select_blocks``.  Returns the
    selection dict plus ``q_rot`` and ``k_rot`` (the rounded tensors)."""
    q_rot = round_to_bf16(apply_rope(q, cos_q, sin_q))
    k_rot = round_to_bf16(apply_rope(k, cos_k, sin_k))
    sel = select_blocks(q_rot, k_rot, prefix_len, seq_lens, block_q, block_k, keep_ratio)
    sel["q_rot"] = q_rot
    sel["k_rot"] = k_rot
    return sel


# ---------------------------------------------------------------------------
# Backward pass of the selected-block attention
# ---------------------------------------------------------------------------

def attention_backward(q, k, v, out, dout, lse, indices, counts, prefix_len: int,
                       seq_lens: Sequence[int], block_q: int, block_k: int,
                       scale: Optional[float] = None, tiles: Optional[Iterable[tuple]] = None):
    """Gradients of the selected-block attention forward with respect to Q, K, V.

    For every real query row i of tile (b, h, qb) and every key position j it
    attends (the listed blocks' real keys, KV head h // G), with the stored
    LSE of the forward:
        P_ij = exp(scale * q_i.k_j - lse_i),   D_i = sum_c dO_ic O_ic,
        dV_j += P_ij dO_i,   dS_ij = P_ij (dO_i.v_j - D_i),
        dQ_i += scale * dS_ij k_j,   dK_j += scale * dS_ij q_i.
    dK/dV of a KV head sum over every query head of its group and every query
    block that listed the key's block; keys nobody listed, padded keys and
    padded query rows get zero gradients.  Returns dq [B, Sq, Hq, d],
    dk, dv [B, Skv, Hkv, d] (float64).  ``tiles``: iterable of (b, h, qb) to
    process (default all); dQ of those tiles is then complete, while dK/dV
    hold only their contributions.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    out = np.asarray(out, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    B, Sq, Hq, d = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    if scale is None or scale <= 0:
        scale = default_scale(d)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    nQb = cdiv(Sq, block_q)
    if tiles is None:
        tiles = [(b, h, qb) for b in range(B) for h in range(Hq) for qb in range(nQb)]
    for (b, h, qb) in tiles:
        L = int(seq_lens[b])
        hk = h // G
        r0, r1 = qb * block_q, min((qb + 1) * block_q, L)
        if r1 <= r0:
            continue
        c = int(counts[b, h, qb])
        pos = tile_keys(indices[b, h, qb, :c], prefix_len + L, block_k)
        if pos.size == 0:
            continue
        qq, oo, gg = q[b, r0:r1, h], out[b, r0:r1, h], dout[b, r0:r1, h]
        kk, vv = k[b, pos, hk], v[b, pos, hk]
        p_ = np.exp((qq @ kk.T) * scale - lse[b, h, r0:r1, None])
        D = (gg * oo).sum(axis=1, keepdims=True)
        dv[b, pos, hk] += p_.T @ gg
        ds = p_ * (gg @ vv.T - D)
        dq[b, r0:r1, h] += scale * ds @ kk
        dk[b, pos, hk] += scale * ds.T @ qq
    return dq, dk, dv
