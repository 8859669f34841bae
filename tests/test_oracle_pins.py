"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test ties one oracle function to a closed form, a brute-force search, a
library routine (torch SDPA / logsumexp), an invariant of the mathematics, or
the hand-worked example in ``tests/golden/hand_worked.json``.  The last group
plants mistakes in copies of the oracle and checks that a pin catches each.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import bsa_oracle as O
from bsa_inputs import CONFIGS, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def f64(t):
    return t.float().numpy().astype(np.float64)


# ---------------------------------------------------------------- geometry ---

@pytest.mark.parametrize("P,L,bk,nkv,npb", [
    (512, 48360, 128, 382, 4),      # 480p: 48,872 keys, last block 104 keys
    (1024, 172800, 128, 1358, 8),   # 720p
    (512, 176640, 128, 1384, 4),    # 1280x736 request 0
    (512, 150000, 128, 1176, 4),    # 1280x736 request 1 (ragged)
    (256, 1024, 64, 20, 4),         # tiny
    (100, 777, 64, 14, 2),          # prefix straddles a block
    (0, 700, 128, 6, 0),            # no prefix
])
def test_kv_geometry_closed_form(P, L, bk, nkv, npb):
    g = O.kv_geometry(P, L, bk)
    assert g["n_kv_valid"] == nkv
    assert g["n_prefix_blocks"] == npb
    assert g["n_candidates"] == nkv - npb
    assert g["n_valid_keys"] == P + L


@pytest.mark.parametrize("r,N,k", [
    (0.25, 16, 4), (0.25, 378, 95), (0.25, 1350, 338), (1.0, 1350, 1350),
    (0.0, 10, 0), (0.5, 10, 5), (0.31, 10, 4), (0.5, 0, 0), (1e-9, 7, 1),
    # float32(0.3) = 0.300000011920929 > 0.3, so ceil(3.0000001) = 4: the ratio
    # is a float32 value converted exactly to float64, not a decimal 0.3.
    (0.3, 10, 4),
])
def test_keep_count_closed_form(r, N, k):
    assert O.keep_count(np.float32(r), N) == k


# ----------------------------------------------------------------- pooling ---

def test_pool_means_closed_form_ramp_and_padding():
    # rows x[t] = t (every head/channel); block means of an arithmetic ramp are
    # the midpoints; rows past n_valid (NaN here) never enter a mean.
    S, H, d, blk, nv = 11, 2, 3, 4, 9
    x = np.repeat(np.arange(S, dtype=np.float64)[:, None, None], H, 1).repeat(d, 2)
    x[nv:] = np.nan
    m = O.pool_means(x, nv, blk)
    assert m.shape == (H, 3, d)
    np.testing.assert_array_equal(m[:, 0], 1.5)
    np.testing.assert_array_equal(m[:, 1], 5.5)
    np.testing.assert_array_equal(m[:, 2], 8.0)    # only row 8 is valid
    m2 = O.pool_means(x, 8, blk)
    assert np.isnan(m2[:, 2]).all()                # no valid row -> NaN


def test_pool_means_permutation_invariant():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((16, 2, 5))
    p = np.concatenate([rng.permutation(8), 8 + rng.permutation(8)])
    np.testing.assert_allclose(O.pool_means(x, 16, 8), O.pool_means(x[p], 16, 8), rtol=0, atol=1e-15)


# ------------------------------------------------------------------- top-k ---

def _brute_topk(scores, k):
    """Best k-subset by integer score sum; among equal sums the lexicographically
    smallest sorted index tuple (the same as 'lower index wins' at ties)."""
    best = None
    for sub in itertools.combinations(range(len(scores)), k):
        key = (-sum(scores[i] for i in sub), sub)
        if best is None or key < best:
            best = key
    return np.array(best[1] if best else (), dtype=np.int64)


def test_topk_bruteforce_subsets():
    rng = np.random.default_rng(1)
    for trial in range(300):
        n = int(rng.integers(1, 10))
        k = int(rng.integers(0, n + 1))
        s = rng.integers(-3, 4, size=n)          # small integers: many exact ties
        got = O.topk_lowest_index(s.astype(np.float64), k)
        np.testing.assert_array_equal(got, _brute_topk(list(s), k))


def test_near_tie_flag():
    s = np.array([3.0, 1.0, 1.00005, 0.0])
    assert O.is_near_tie(s, 2)          # 2nd and 3rd best within 1e-4 relative
    assert not O.is_near_tie(s, 1)
    assert not O.is_near_tie(s, 4)      # no boundary when every block is kept
    assert O.is_near_tie(np.array([2.0, 2.0]), 1)


# ---------------------------------------------------------------- selector ---

def _tiny(cfg="tiny", **kw):
    inp = make_inputs(CONFIGS[cfg], "cpu", pad_fill=float("nan"), **kw)
    return inp, f64(inp["q"]), f64(inp["k"]), f64(inp["v"])


def test_selector_keep_one_is_dense_closed_form():
    inp, q, k, v = _tiny("small_gqa")
    c = inp["cfg"]
    sel = O.select_blocks(q, k, c.prefix, inp["seq_lens"], c.block_q, c.block_k, [1.0])
    for b, L in enumerate(inp["seq_lens"]):
        nkv = O.cdiv(c.prefix + L, c.block_k)
        nqv = O.cdiv(L, c.block_q)
        assert (sel["counts"][b, :, :nqv] == nkv).all()
        assert (sel["counts"][b, :, nqv:] == 0).all()
        for h in range(c.Hq):
            for qb in range(nqv):
                np.testing.assert_array_equal(sel["indices"][b, h, qb, :nkv], np.arange(nkv))


def test_selector_tiny_counts_and_structure():
    inp, q, k, v = _tiny()
    c = inp["cfg"]
    sel = O.select_blocks(q, k, c.prefix, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    # 20 key blocks, 4 of them prefix, keep ceil(0.25*16)=4 -> count 8 everywhere
    assert (sel["counts"] == 8).all()
    idx = sel["indices"][..., :8]
    assert (idx[..., :4] == np.arange(4)).all()
    assert (np.diff(idx, axis=-1) > 0).all()
    assert ((idx >= 0) & (idx < 20)).all()


def test_selector_matches_bruteforce_on_tiny():
    """Every row of the tiny case: the kept set is the best-sum k-subset of the
    candidate blocks, with scores recomputed here by explicit loops."""
    inp, q, k, v = _tiny("small_mqa_d64")
    c = inp["cfg"]
    L, P = inp["seq_lens"][0], c.prefix
    sel = O.select_blocks(q, k, P, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    nkv = O.cdiv(P + L, c.block_k)
    npb = O.cdiv(P, c.block_k)
    kk = O.keep_count(inp["keep_ratio"][0], nkv - npb)
    for h in range(c.Hq):
        for qb in range(O.cdiv(L, c.block_q)):
            rows = range(qb * c.block_q, min((qb + 1) * c.block_q, L))
            qbar = [sum(q[0, r, h, e] for r in rows) / len(rows) for e in range(c.d)]
            sc = []
            for kb in range(npb, nkv):
                keys = range(kb * c.block_k, min((kb + 1) * c.block_k, P + L))
                kbar = [sum(k[0, t, 0, e] for t in keys) / len(keys) for e in range(c.d)]
                sc.append(sum(a * b for a, b in zip(qbar, kbar)))
            # distinct real scores: the best-sum subset is the top-k set
            order = sorted(range(len(sc)), key=lambda j: -sc[j])
            want = sorted(j + npb for j in order[:kk])
            got = sel["indices"][0, h, qb, npb:npb + kk]
            if not sel["near_tie"][0, h, qb]:
                np.testing.assert_array_equal(got, want)
            np.testing.assert_array_equal(sel["indices"][0, h, qb, :npb], np.arange(npb))


def test_selector_tie_rule_duplicated_blocks():
    # K blocks 5 and 9 identical (and the q block means point at them): equal
    # scores, keep 1 -> the lower index wins.
    rng = np.random.default_rng(3)
    bk, d, P, L = 4, 8, 4, 40
    q = rng.standard_normal((1, L, 1, d))
    k = rng.standard_normal((1, P + L, 1, d)) * 0.01
    k[0, 5 * bk:6 * bk] = 3.0
    k[0, 9 * bk:10 * bk] = 3.0
    q[:] = np.abs(q) + 1.0
    sel = O.select_blocks(q, k, P, [L], 8, bk, [np.float32(0.05)])  # N=10 -> k=ceil(0.5)=1
    for qb in range(5):
        assert sel["counts"][0, 0, qb] == 2
        np.testing.assert_array_equal(sel["indices"][0, 0, qb, :2], [0, 5])


def test_selector_prefix_forced_even_when_worst():
    inp, q, k, v = _tiny()
    c = inp["cfg"]
    P = c.prefix
    # make the prefix keys score as low as possible for every query block
    qm = q[0, : inp["seq_lens"][0]].mean(axis=0)          # [Hq, d]
    k2 = k.copy()
    for hk in range(c.Hkv):
        k2[0, :P, hk, :] = -1e3 * qm[hk * (c.Hq // c.Hkv)]
    sel = O.select_blocks(q, k2, P, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    npb = P // c.block_k
    assert (sel["indices"][..., :npb] == np.arange(npb)).all()
    assert (sel["scores"][..., :npb] != sel["scores"][..., :npb]).all()   # never scored


def test_golden_hand_worked_selection():
    g = json.load(open(GOLDEN))
    for case in ("selection", "tie"):
        e = g[case]
        sel = O.select_blocks(np.array(e["q"], float), np.array(e["k"], float), e["prefix_len"],
                              e["seq_lens"], e["block_q"], e["block_k"],
                              [np.float32(x) for x in e["keep_ratio"]])
        np.testing.assert_array_equal(sel["counts"], e["expect_counts"])
        c = e["expect_counts"][0][0][0]
        np.testing.assert_array_equal(sel["indices"][..., :c], e["expect_indices"])


# --------------------------------------------------------------- attention ---

def test_golden_hand_worked_attention():
    e = json.load(open(GOLDEN))["attention"]
    out, lse = O.attention_rows(np.array([e["q"]]), np.array(e["keys"]), np.array(e["vals"]), e["scale"])
    np.testing.assert_allclose(out[0], e["expect_out"], rtol=1e-14)
    np.testing.assert_allclose(lse[0], e["expect_lse"], rtol=1e-14)


def _sdpa_dense(q, k, v, P, seq_lens, scale):
    """torch CPU fp64 SDPA per request with the additive padded-key mask
    (cosmos_parallel.py build_gen_key_mask semantics) and explicit GQA repeat."""
    B, Sq, Hq, d = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Sq, Hq, v.shape[3]))
    lse = np.full((B, Hq, Sq), -np.inf)
    for b in range(B):
        L = seq_lens[b]
        qt = torch.from_numpy(q[b, :L]).permute(1, 0, 2)            # [Hq, L, d]
        kt = torch.from_numpy(np.nan_to_num(k[b])).permute(1, 0, 2).repeat_interleave(G, 0)
        vt = torch.from_numpy(np.nan_to_num(v[b])).permute(1, 0, 2).repeat_interleave(G, 0)
        mask = torch.zeros(k.shape[1], dtype=torch.float64)
        mask[P + L:] = float("-inf")
        o = torch.nn.functional.scaled_dot_product_attention(
            qt, kt, vt, attn_mask=mask.view(1, 1, -1), scale=scale)
        z = (qt @ kt.transpose(1, 2)) * scale + mask
        out[b, :L] = o.permute(1, 0, 2).numpy()
        lse[b, :, :L] = torch.logsumexp(z, dim=-1).numpy()
    return out, lse


@pytest.mark.parametrize("cfg", ["tiny", "small_gqa", "small_mqa_d64"])
def test_dense_attention_matches_torch_sdpa(cfg):
    inp, q, k, v = _tiny(cfg)
    c = inp["cfg"]
    idx, cnt = O.dense_indices(c.prefix, inp["seq_lens"], c.Sq, c.Skv, c.block_q, c.block_k, c.Hq)
    out, lse = O.attention(q, k, v, idx, cnt, c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    ro, rl = _sdpa_dense(q, k, v, c.prefix, inp["seq_lens"], 1 / math.sqrt(c.d))
    np.testing.assert_allclose(out, ro, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, rl, rtol=0, atol=1e-12)


def test_sparse_attention_matches_masked_sdpa():
    """Selected-block attention equals dense SDPA with a boolean mask that
    allows exactly the listed blocks' valid keys."""
    inp, q, k, v = _tiny("small_gqa")
    c = inp["cfg"]
    sel = O.select_blocks(q, k, c.prefix, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    out, lse = O.attention(q, k, v, sel["indices"], sel["counts"], c.prefix, inp["seq_lens"],
                           c.block_q, c.block_k)
    G = c.Hq // c.Hkv
    scale = 1 / math.sqrt(c.d)
    for b, L in enumerate(inp["seq_lens"]):
        for h in range(c.Hq):
            allow = np.zeros((L, c.Skv), dtype=bool)
            for qb in range(O.cdiv(L, c.block_q)):
                r0, r1 = qb * c.block_q, min((qb + 1) * c.block_q, L)
                for kb in sel["indices"][b, h, qb, :sel["counts"][b, h, qb]]:
                    allow[r0:r1, kb * c.block_k:(kb + 1) * c.block_k] = True
            allow[:, c.prefix + L:] = False
            qt = torch.from_numpy(q[b, :L, h])[None]
            kt = torch.from_numpy(np.nan_to_num(k[b, :, h // G]))[None]
            vt = torch.from_numpy(np.nan_to_num(v[b, :, h // G]))[None]
            o = torch.nn.functional.scaled_dot_product_attention(
                qt, kt, vt, attn_mask=torch.from_numpy(allow)[None], scale=scale)[0]
            z = (qt[0] @ kt[0].T) * scale
            z[~torch.from_numpy(allow)] = float("-inf")
            np.testing.assert_allclose(out[b, :L, h], o.numpy(), rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[b, h, :L], torch.logsumexp(z, -1).numpy(), rtol=0, atol=1e-12)


def test_gqa_equals_mha_with_repeated_kv():
    inp, q, k, v = _tiny("small_gqa")
    c = inp["cfg"]
    G = c.Hq // c.Hkv
    sel = O.select_blocks(q, k, c.prefix, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    a = O.attention(q, k, v, sel["indices"], sel["counts"], c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    kr, vr = np.repeat(k, G, axis=2), np.repeat(v, G, axis=2)
    sel2 = O.select_blocks(q, kr, c.prefix, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    np.testing.assert_array_equal(sel["indices"], sel2["indices"])
    b = O.attention(q, kr, vr, sel2["indices"], sel2["counts"], c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_mqa_equals_mha_with_repeated_kv():
    inp, q, k, v = _tiny("small_mqa_d64")
    c = inp["cfg"]
    sel = O.select_blocks(q, k, c.prefix, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    a = O.attention(q, k, v, sel["indices"], sel["counts"], c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    kr, vr = np.repeat(k, c.Hq, axis=2), np.repeat(v, c.Hq, axis=2)
    b = O.attention(q, kr, vr, sel["indices"], sel["counts"], c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    np.testing.assert_array_equal(a[0], b[0])


def test_rows_sum_to_one():
    inp, q, k, v = _tiny()
    c = inp["cfg"]
    sel = O.select_blocks(q, k, c.prefix, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    ones = np.ones_like(v)
    out, _ = O.attention(q, k, ones, sel["indices"], sel["counts"], c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-13)


def test_dropped_blocks_do_not_matter():
    inp, q, k, v = _tiny("small_gqa")
    c = inp["cfg"]
    sel = O.select_blocks(q, k, c.prefix, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    a = O.attention(q, k, v, sel["indices"], sel["counts"], c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    # blocks that no (b, hk) row of head group hk selects may change freely
    k2, v2 = k.copy(), v.copy()
    G = c.Hq // c.Hkv
    rng = np.random.default_rng(5)
    for b in range(c.B):
        for hk in range(c.Hkv):
            used = set()
            for h in range(hk * G, (hk + 1) * G):
                for qb in range(sel["counts"].shape[2]):
                    used.update(sel["indices"][b, h, qb, :sel["counts"][b, h, qb]].tolist())
            for kb in range(O.cdiv(c.Skv, c.block_k)):
                if kb not in used:
                    sl = slice(kb * c.block_k, (kb + 1) * c.block_k)
                    k2[b, sl, hk] = rng.standard_normal(k2[b, sl, hk].shape) * 100
                    v2[b, sl, hk] = rng.standard_normal(v2[b, sl, hk].shape) * 100
    assert not np.array_equal(np.nan_to_num(k), np.nan_to_num(k2))
    bres = O.attention(q, k2, v2, sel["indices"], sel["counts"], c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    np.testing.assert_array_equal(a[0], bres[0])
    np.testing.assert_array_equal(a[1], bres[1])


def test_padding_garbage_and_padded_rows():
    inp, q, k, v = _tiny("small_gqa")
    c = inp["cfg"]
    # inputs carry NaN in every padded row
    assert np.isnan(q[1, inp["seq_lens"][1]:]).all()
    sel = O.select_blocks(q, k, c.prefix, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    out, lse = O.attention(q, k, v, sel["indices"], sel["counts"], c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    L1 = inp["seq_lens"][1]
    assert np.isfinite(out[1, :L1]).all() and np.isfinite(lse[1, :, :L1]).all()
    assert (out[1, L1:] == 0).all() and np.isneginf(lse[1, :, L1:]).all()
    # 1e4 garbage instead of NaN gives the same real rows
    q3, k3, v3 = q.copy(), k.copy(), v.copy()
    for arr, start in ((q3, L1), (k3, c.prefix + L1), (v3, c.prefix + L1)):
        arr[1, start:] = 1e4
    sel3 = O.select_blocks(q3, k3, c.prefix, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    np.testing.assert_array_equal(sel3["indices"], sel["indices"])
    o3, l3 = O.attention(q3, k3, v3, sel["indices"], sel["counts"], c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    np.testing.assert_array_equal(o3, out)
    np.testing.assert_array_equal(l3, lse)


def test_lse_closed_form_identical_keys():
    # every key equal: logits all c = (q.k)*scale -> lse = c + ln(n), out = mean(V)
    rng = np.random.default_rng(7)
    d, n = 16, 37
    qr = rng.standard_normal((3, d))
    kr = np.tile(rng.standard_normal(d), (n, 1))
    vr = rng.standard_normal((n, d))
    out, lse = O.attention_rows(qr, kr, vr, 0.25)
    np.testing.assert_allclose(lse, (qr @ kr[0]) * 0.25 + math.log(n), rtol=1e-13)
    np.testing.assert_allclose(out, np.tile(vr.mean(0), (3, 1)), rtol=1e-12, atol=1e-13)


def test_lse_consistency_identity():
    # exp(lse) * out == sum_j exp(z_j) v_j
    rng = np.random.default_rng(8)
    qr, kr, vr = rng.standard_normal((4, 8)), rng.standard_normal((9, 8)), rng.standard_normal((9, 8))
    out, lse = O.attention_rows(qr, kr, vr, 0.3)
    z = qr @ kr.T * 0.3
    np.testing.assert_allclose(np.exp(lse)[:, None] * out, np.exp(z) @ vr, rtol=1e-12)


def test_zero_count_row_is_zero_and_neginf():
    out, lse = O.attention_rows(np.ones((2, 4)), np.zeros((0, 4)), np.zeros((0, 4)), 1.0)
    assert (out == 0).all() and np.isneginf(lse).all()


# ------------------------------------------------------ planted mistakes ---

def test_planted_wrong_head_mapping_is_caught(monkeypatch):
    inp, q, k, v = _tiny("small_gqa")
    c = inp["cfg"]
    idx, cnt = O.dense_indices(c.prefix, inp["seq_lens"], c.Sq, c.Skv, c.block_q, c.block_k, c.Hq)
    good = O.attention_tile

    def wrong(q, k, v, b, h, qb, *a, **kw):          # h % Hkv instead of h // G
        G = q.shape[2] // k.shape[2]
        return good(q, k, v, b, (h % k.shape[2]) * G, qb, *a, **kw)
    monkeypatch.setattr(O, "attention_tile", wrong)
    out, _ = O.attention(q, k, v, idx, cnt, c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    ro, _ = _sdpa_dense(q, k, v, c.prefix, inp["seq_lens"], 1 / math.sqrt(c.d))
    assert np.nanmax(np.abs(out - ro)) > 1e-3


def test_planted_reversed_tie_rule_is_caught(monkeypatch):
    e = json.load(open(GOLDEN))["tie"]
    monkeypatch.setattr(O, "topk_lowest_index",
                        lambda s, k: np.sort(np.lexsort((-np.arange(len(s)), -s))[:k]))
    sel = O.select_blocks(np.array(e["q"], float), np.array(e["k"], float), e["prefix_len"],
                          e["seq_lens"], e["block_q"], e["block_k"], [np.float32(0.25)])
    assert not np.array_equal(sel["indices"][..., :2], e["expect_indices"])


def test_planted_missing_scale_is_caught():
    e = json.load(open(GOLDEN))["attention"]
    out, lse = O.attention_rows(np.array([e["q"]]) * 2, np.array(e["keys"]), np.array(e["vals"]), 1.0)
    assert abs(lse[0] - e["expect_lse"]) > 1e-3


def test_planted_dropped_prefix_is_caught(monkeypatch):
    e = json.load(open(GOLDEN))["selection"]
    good = O.kv_geometry
    monkeypatch.setattr(O, "kv_geometry", lambda P, L, bk: good(0, P + L, bk))
    sel = O.select_blocks(np.array(e["q"], float), np.array(e["k"], float), e["prefix_len"],
                          e["seq_lens"], e["block_q"], e["block_k"], [np.float32(0.5)])
    c = sel["counts"][0, 0, 0]
    assert c != 3 or not np.array_equal(sel["indices"][0, 0, :, :3], e["expect_indices"][0][0])


# ------------------------------------------------ causal understanding pass ---

def test_causal_prefix_matches_torch_sdpa_is_causal():
    rng = np.random.default_rng(11)
    B, P, Hq, Hkv, d = 2, 37, 4, 2, 16
    q = rng.standard_normal((B, P, Hq, d))
    k = rng.standard_normal((B, P + 9, Hkv, d))     # rows past P are generation keys: never read
    v = rng.standard_normal((B, P + 9, Hkv, d))
    out, lse = O.causal_prefix_attention(q, k, v, P)
    for b in range(B):
        qt = torch.from_numpy(q[b]).permute(1, 0, 2)
        kt = torch.from_numpy(k[b, :P]).permute(1, 0, 2).repeat_interleave(2, 0)
        vt = torch.from_numpy(v[b, :P]).permute(1, 0, 2).repeat_interleave(2, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True)
        np.testing.assert_allclose(out[b], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
        z = (qt @ kt.transpose(1, 2)) / math.sqrt(d)
        z = z.masked_fill(torch.ones(P, P, dtype=torch.bool).triu(1), float("-inf"))
        np.testing.assert_allclose(lse[b], torch.logsumexp(z, -1).numpy(), rtol=0, atol=1e-12)


def test_causal_prefix_first_row_and_generation_keys_ignored():
    rng = np.random.default_rng(12)
    q = rng.standard_normal((1, 5, 1, 4))
    k = rng.standard_normal((1, 8, 1, 4))
    v = rng.standard_normal((1, 8, 1, 4))
    out, lse = O.causal_prefix_attention(q, k, v, 5, scale=0.5)
    # row 0 sees only key 0: output = v[0], lse = its logit
    np.testing.assert_allclose(out[0, 0, 0], v[0, 0, 0], rtol=1e-14)
    np.testing.assert_allclose(lse[0, 0, 0], 0.5 * q[0, 0, 0] @ k[0, 0, 0], rtol=1e-14)
    k2, v2 = k.copy(), v.copy()
    k2[0, 5:] = 1e6
    v2[0, 5:] = np.nan
    out2, lse2 = O.causal_prefix_attention(q, k2, v2, 5, scale=0.5)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)


# ------------------------------------------------------------ RoPE prologue ---

def _rope_tables(S, d, base=10000.0, offset=0):
    inv = base ** (-np.arange(0, d // 2) * 2.0 / d)
    ang = np.outer(np.arange(offset, offset + S), inv)             # [S, d/2]
    ang = np.concatenate([ang, ang], axis=1)                       # half-split layout
    return np.cos(ang), np.sin(ang)


def test_round_to_bf16_matches_torch():
    rng = np.random.default_rng(13)
    x = np.concatenate([rng.standard_normal(20000) * 10 ** rng.uniform(-6, 6, 20000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.0078125, 3.0e38, np.inf, -np.inf]])
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(O.round_to_bf16(x), want)
    assert np.isnan(O.round_to_bf16(np.array([np.nan]))).all()


def test_rope_identity_at_angle_zero():
    rng = np.random.default_rng(14)
    x = rng.standard_normal((2, 9, 3, 16))
    np.testing.assert_array_equal(O.apply_rope(x, np.ones((9, 16)), np.zeros((9, 16))), x)


def test_rope_preserves_pair_norms():
    rng = np.random.default_rng(15)
    x = rng.standard_normal((1, 11, 2, 32))
    c, s = _rope_tables(11, 32)
    y = O.apply_rope(x, c, s)
    n_x = x[..., :16] ** 2 + x[..., 16:] ** 2
    n_y = y[..., :16] ** 2 + y[..., 16:] ** 2
    np.testing.assert_allclose(n_y, n_x, rtol=1e-12)
    # quarter turn on every pair: (x1, x2) -> (-x2, x1)
    np.testing.assert_allclose(O.apply_rope(x, np.zeros((11, 32)), np.ones((11, 32))), O.rotate_half(x), rtol=0)


def test_rope_rotates_basis_vectors_counterclockwise():
    # Closed form of the half-split rotation by theta (channel i paired with
    # channel i + d/2): e_0 -> cos(t) e_0 + sin(t) e_{d/2} and
    # e_{d/2} -> -sin(t) e_0 + cos(t) e_{d/2}, i.e. (x1, x2) ->
    # (x1 cos - x2 sin, x2 cos + x1 sin), the direction of x*cos + rotate_half(x)*sin.
    d, t = 8, 0.3
    cos, sin = np.full((1, d), math.cos(t)), np.full((1, d), math.sin(t))
    for src, want in ((0, {0: math.cos(t), d // 2: math.sin(t)}),
                      (d // 2, {0: -math.sin(t), d // 2: math.cos(t)})):
        x = np.zeros((1, 1, 1, d))
        x[..., src] = 1.0
        expect = np.zeros(d)
        for ch, val in want.items():
            expect[ch] = val
        np.testing.assert_allclose(O.apply_rope(x, cos, sin)[0, 0, 0], expect, rtol=0, atol=1e-15)


def _check_rope_complex_rotation():
    """Half-split RoPE equals multiplying z = x1 + i*x2 (first half real, second
    half imaginary) by exp(i*theta) per channel pair: an identity of complex
    arithmetic, computed here with numpy's complex multiply."""
    rng = np.random.default_rng(31)
    S, d = 7, 16
    x = rng.standard_normal((1, S, 2, d))
    theta = rng.uniform(-np.pi, np.pi, (S, d // 2))
    cos = np.concatenate([np.cos(theta)] * 2, axis=1)
    sin = np.concatenate([np.sin(theta)] * 2, axis=1)
    w = (x[..., : d // 2] + 1j * x[..., d // 2:]) * np.exp(1j * theta)[None, :, None, :]
    want = np.concatenate([w.real, w.imag], axis=-1)
    return not np.allclose(O.apply_rope(x, cos, sin), want, rtol=0, atol=1e-12)


def test_rope_equals_complex_multiplication():
    assert not _check_rope_complex_rotation()


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(16)
    d = 64
    qv, kv = rng.standard_normal(d), rng.standard_normal(d)
    c, s = _rope_tables(40, d)
    q = np.tile(qv, (1, 40, 1, 1)).reshape(1, 40, 1, d)
    k = np.tile(kv, (1, 40, 1, 1)).reshape(1, 40, 1, d)
    qr, kr = O.apply_rope(q, c, s)[0, :, 0], O.apply_rope(k, c, s)[0, :, 0]
    for m, n in [(5, 2), (25, 22), (39, 36)]:                     # all offset 3
        np.testing.assert_allclose(qr[m] @ kr[n], qr[5] @ kr[2], rtol=1e-10)


def test_rope_then_select_uses_rounded_rotated_inputs():
    inp = make_inputs(CONFIGS["small_mqa_d64"], "cpu", pad_fill=0.0)
    c = inp["cfg"]
    q, k = f64(inp["q"]), f64(inp["k"])
    cq, sq = _rope_tables(c.Sq, c.d)
    ck, sk = _rope_tables(c.Skv, c.d)
    sel = O.rope_then_select(q, k, cq, sq, ck, sk, c.prefix, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    ref = O.select_blocks(O.round_to_bf16(O.apply_rope(q, cq, sq)), O.round_to_bf16(O.apply_rope(k, ck, sk)),
                          c.prefix, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    np.testing.assert_array_equal(sel["indices"], ref["indices"])
    # rotation changes the selection (the prologue matters)
    plain = O.select_blocks(q, k, c.prefix, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    assert not np.array_equal(plain["indices"], sel["indices"])


# ----------------------------------------------------------------- backward ---

def _torch_selected_attention(q, k, v, idx, cnt, P, lens, bq, bk, scale):
    """Autograd-able fp64 torch version (dense matmuls with a boolean mask of
    the listed blocks) for the gradient pin."""
    B, Sq, Hq, d = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    outs = []
    for b in range(B):
        L = lens[b]
        allow = torch.zeros(Hq, Sq, Skv, dtype=torch.bool)
        for h in range(Hq):
            for qb in range(O.cdiv(Sq, bq)):
                r0, r1 = qb * bq, min((qb + 1) * bq, L)
                for kb in idx[b, h, qb, :cnt[b, h, qb]]:
                    allow[h, r0:r1, kb * bk:(kb + 1) * bk] = True
        allow[:, :, P + L:] = False
        kr = k[b].repeat_interleave(G, dim=1).permute(1, 0, 2)
        vr = v[b].repeat_interleave(G, dim=1).permute(1, 0, 2)
        z = (q[b].permute(1, 0, 2) @ kr.transpose(1, 2)) * scale
        z = z.masked_fill(~allow, float("-inf"))
        p_ = torch.softmax(z, dim=-1).nan_to_num(0.0)
        outs.append((p_ @ vr).permute(1, 0, 2))
    return torch.stack(outs)


@pytest.mark.parametrize("cfg", ["small_gqa", "small_mqa_d64"])
def test_backward_matches_torch_autograd(cfg):
    inp, q, k, v = _tiny(cfg)
    c = inp["cfg"]
    q, k, v = (np.nan_to_num(x) for x in (q, k, v))
    sel = O.select_blocks(q, k, c.prefix, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    out, lse = O.attention(q, k, v, sel["indices"], sel["counts"], c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    rng = np.random.default_rng(21)
    dout = rng.standard_normal(out.shape)
    for b, L in enumerate(inp["seq_lens"]):
        dout[b, L:] = 0.0          # padded rows carry no gradient
    scale = 1 / math.sqrt(c.d)
    dq, dk, dv = O.attention_backward(q, k, v, out, dout, lse, sel["indices"], sel["counts"], c.prefix,
                                      inp["seq_lens"], c.block_q, c.block_k)
    qt, kt, vt = (torch.from_numpy(x).requires_grad_(True) for x in (q, k, v))
    ot = _torch_selected_attention(qt, kt, vt, sel["indices"], sel["counts"], c.prefix, inp["seq_lens"],
                                   c.block_q, c.block_k, scale)
    np.testing.assert_allclose(ot.detach().numpy()[~np.isnan(out)], out[~np.isnan(out)], rtol=0, atol=1e-12)
    ot.backward(torch.from_numpy(dout))
    np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=0, atol=1e-10)
    np.testing.assert_allclose(dk, kt.grad.numpy(), rtol=0, atol=1e-10)
    np.testing.assert_allclose(dv, vt.grad.numpy(), rtol=0, atol=1e-10)


def test_backward_finite_difference_tiny():
    rng = np.random.default_rng(22)
    B, Sq, Hq, Hkv, d, P, bq, bk = 1, 8, 2, 1, 4, 4, 4, 4
    q, k, v = rng.standard_normal((B, Sq, Hq, d)), rng.standard_normal((B, P + Sq, Hkv, d)), rng.standard_normal((B, P + Sq, Hkv, d))
    idx = np.array([[[[0, 2, -1], [0, 1, 2]], [[1, -1, -1], [0, 2, -1]]]])
    cnt = np.array([[[2, 3], [1, 2]]])
    w = rng.standard_normal((B, Sq, Hq, d))          # loss = sum(w * out)
    out, lse = O.attention(q, k, v, idx, cnt, P, [Sq], bq, bk)
    dq, dk, dv = O.attention_backward(q, k, v, out, w, lse, idx, cnt, P, [Sq], bq, bk)
    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(12):
            i = tuple(rng.integers(0, s) for s in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[i] += eps
            xm[i] -= eps
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            lp = (w * O.attention(args["q"], args["k"], args["v"], idx, cnt, P, [Sq], bq, bk)[0]).sum()
            args[name] = xm
            lm = (w * O.attention(args["q"], args["k"], args["v"], idx, cnt, P, [Sq], bq, bk)[0]).sum()
            assert abs((lp - lm) / (2 * eps) - g[i]) < 1e-6, (name, i)


# ------------------------------------------- planted mistakes, backward ---
# Each mutation is a plausible slip in the oracle's backward (a sign, a
# dropped scale, a wrong operand or head mapping, a transposed product); the
# mutant is built from the function's own source and must fail the torch
# autograd pin above.
BACKWARD_MUTATIONS = [
    ("ds = p_ * (gg @ vv.T - D)", "ds = p_ * (gg @ vv.T + D)"),
    ("dq[b, r0:r1, h] += scale * ds @ kk", "dq[b, r0:r1, h] += ds @ kk"),
    ("dk[b, pos, hk] += scale * ds.T @ qq", "dk[b, pos, hk] += ds.T @ qq"),
    ("dv[b, pos, hk] += p_.T @ gg", "dv[b, pos, hk] += p_.T @ oo"),
    ("dk[b, pos, hk] += scale * ds.T @ qq", "dk[b, pos, hk] += scale * ds.T @ gg"),
    ("hk = h // G", "hk = h % Hkv"),
    ("p_ = np.exp((qq @ kk.T) * scale - lse[b, h, r0:r1, None])", "p_ = np.exp((qq @ kk.T) - lse[b, h, r0:r1, None])"),
    ("dq[b, r0:r1, h] += scale * ds @ kk", "dq[b, r0:r1, h] += scale * (p_ * (gg @ vv.T)) @ kk"),  # D dropped in dQ
]


@pytest.mark.parametrize("old,new", BACKWARD_MUTATIONS)
def test_planted_backward_mistake_is_caught(old, new):
    import inspect
    src = inspect.getsource(O.attention_backward)
    assert old in src, old
    ns = dict(vars(O))
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    mutant = ns["attention_backward"]
    inp, q, k, v = _tiny("small_gqa")
    c = inp["cfg"]
    q, k, v = (np.nan_to_num(x) for x in (q, k, v))
    sel = O.select_blocks(q, k, c.prefix, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    out, lse = O.attention(q, k, v, sel["indices"], sel["counts"], c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    dout = np.random.default_rng(23).standard_normal(out.shape)
    for b, L in enumerate(inp["seq_lens"]):
        dout[b, L:] = 0.0
    grads = mutant(q, k, v, out, dout, lse, sel["indices"], sel["counts"], c.prefix, inp["seq_lens"], c.block_q,
                   c.block_k)
    qt, kt, vt = (torch.from_numpy(x).requires_grad_(True) for x in (q, k, v))
    ot = _torch_selected_attention(qt, kt, vt, sel["indices"], sel["counts"], c.prefix, inp["seq_lens"],
                                   c.block_q, c.block_k, 1 / math.sqrt(c.d))
    ot.backward(torch.from_numpy(dout))
    worst = max(np.abs(g - t.grad.numpy()).max() for g, t in zip(grads, (qt, kt, vt)))
    assert worst > 1e-6, (new, worst)


# -------------------------------------- planted mistakes, forward and selector ---
# Source mutations of the oracle's building blocks, each paired with the
# independent check that must expose it (the check passes on the unmodified
# oracle: see test_forward_mutation_checks_pass_on_the_oracle).

def _check_golden_attention():
    e = json.load(open(GOLDEN))["attention"]
    out, lse = O.attention_rows(np.array([e["q"]]), np.array(e["keys"]), np.array(e["vals"]), e["scale"])
    return not (np.allclose(out[0], e["expect_out"], rtol=1e-14, atol=0)
                and abs(lse[0] - e["expect_lse"]) <= 1e-14 * abs(e["expect_lse"]))


def _check_dense_sdpa_with_nan_padding():
    inp, q, k, v = _tiny("small_gqa")
    c = inp["cfg"]
    idx, cnt = O.dense_indices(c.prefix, inp["seq_lens"], c.Sq, c.Skv, c.block_q, c.block_k, c.Hq)
    out, lse = O.attention(q, k, v, idx, cnt, c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    ro, rl = _sdpa_dense(q, k, v, c.prefix, inp["seq_lens"], 1 / math.sqrt(c.d))
    real = ~np.isnan(ro)
    for b, L in enumerate(inp["seq_lens"]):
        real[b, L:] = False
    return not (np.allclose(out[real], ro[real], rtol=0, atol=1e-12))


def _check_pool_ramp_with_padding():
    S, H, d, blk, nv = 11, 2, 3, 4, 9
    x = np.repeat(np.arange(S, dtype=np.float64)[:, None, None], H, 1).repeat(d, 2)
    x[nv:] = np.nan
    m = O.pool_means(x, nv, blk)
    return not (np.array_equal(m[:, 0], np.full((H, d), 1.5)) and np.array_equal(m[:, 2], np.full((H, d), 8.0)))


def _check_keep_count_closed_form():
    return O.keep_count(np.float32(0.25), 378) != 95 or O.keep_count(np.float32(0.25), 1350) != 338


def _check_lists_ascending_and_golden():
    g = json.load(open(GOLDEN))["selection"]
    sel = O.select_blocks(np.array(g["q"], float), np.array(g["k"], float), g["prefix_len"], g["seq_lens"],
                          g["block_q"], g["block_k"], [np.float32(x) for x in g["keep_ratio"]])
    bad = not np.array_equal(sel["indices"][..., :3], g["expect_indices"])
    rng = np.random.default_rng(5)
    scores = rng.permutation(40).astype(float)
    got = O.topk_lowest_index(scores, 10)
    return bad or not np.array_equal(got, np.sort(np.argsort(-scores)[:10]))


def _check_gqa_selection_equals_repeated_kv():
    inp, q, k, v = _tiny("small_gqa")
    c = inp["cfg"]
    G = c.Hq // c.Hkv
    a = O.select_blocks(q, k, c.prefix, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    bsel = O.select_blocks(q, np.repeat(k, G, axis=2), c.prefix, inp["seq_lens"], c.block_q, c.block_k,
                           inp["keep_ratio"])
    return not (np.array_equal(a["counts"], bsel["counts"]) and np.array_equal(a["indices"], bsel["indices"]))


FORWARD_MUTATIONS = [
    ("attention_rows", "lse = (m + np.log(l))[:, 0]", "lse = (m + np.log2(l))[:, 0]", _check_golden_attention),
    ("attention_rows", "out = (p @ vals) / l", "out = (p @ vals)", _check_golden_attention),
    ("attention_rows", "p = np.exp(z - m)", "p = np.exp(z)", _check_golden_attention),
    ("tile_keys", "r1 = min((int(kb) + 1) * block_k, n_valid_keys)", "r1 = (int(kb) + 1) * block_k",
     _check_dense_sdpa_with_nan_padding),
    ("pool_means", "r1 = min((j + 1) * block, n_valid, S)", "r1 = min((j + 1) * block, S)",
     _check_pool_ramp_with_padding),
    ("keep_count", "math.ceil(r * float(n_candidates))", "math.floor(r * float(n_candidates))",
     _check_keep_count_closed_form),
    ("topk_lowest_index", "return np.sort(order[:k]).astype(np.int64)", "return order[:k].astype(np.int64)",
     _check_lists_ascending_and_golden),
    ("select_blocks", "hk = h // G ", "hk = h % Hkv ", _check_gqa_selection_equals_repeated_kv),
    # rotation direction: rotate_half turned the other way, and the sin term subtracted
    ("rotate_half", "return np.concatenate([-x[..., d // 2:], x[..., : d // 2]], axis=-1)",
     "return np.concatenate([x[..., d // 2:], -x[..., : d // 2]], axis=-1)", _check_rope_complex_rotation),
    ("apply_rope", "return x * c + rotate_half(x) * s", "return x * c - rotate_half(x) * s",
     _check_rope_complex_rotation),
]


def test_forward_mutation_checks_pass_on_the_oracle():
    for _, _, _, check in FORWARD_MUTATIONS:
        assert not check(), check.__name__


@pytest.mark.parametrize("fname,old,new,check", FORWARD_MUTATIONS,
                         ids=[f"{m[0]}:{i}" for i, m in enumerate(FORWARD_MUTATIONS)])
def test_planted_forward_mistake_is_caught(monkeypatch, fname, old, new, check):
    import inspect
    src = inspect.getsource(getattr(O, fname))
    assert old in src, old
    ns = dict(vars(O))
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    monkeypatch.setattr(O, fname, ns[fname])
    try:
        caught = check()
    except (IndexError, ValueError, FloatingPointError):
        caught = True                       # the pin's run breaks down: caught as well
    assert caught, (fname, new)
