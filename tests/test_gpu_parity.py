"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small cases compare every element; the five workload configs compare every
selection row and sampled attention tiles, in the launch configuration the
bench times.  Invariants that must hold bit for bit on the GPU (dense pass ==
keep 1, dropped blocks do not matter, NaN padding is never read, GQA == MHA
with repeated K/V, strided views) are checked directly.
"""

import math

import numpy as np
import pytest
import torch

import block_sparse_attention_bsa_gb300 as bsa
from bsa_inputs import CONFIGS, WORKLOAD_CONFIGS, make_inputs
from oracle import bsa_oracle as O
from parity_utils import (check_structure, compare_attention, compare_selection, sample_tiles,
                          to_f32_np)

pytestmark = pytest.mark.gpu

SMALL = ["tiny", "small_gqa", "small_mqa_d64", "small_mha_perhead", "small_64x64_d128"]


@pytest.fixture(scope="module", autouse=True)
def built():
    bsa.build()


def cuda_inputs(name, pad_fill=float("nan"), **kw):
    inp = make_inputs(CONFIGS[name], "cpu", pad_fill=pad_fill, **kw)
    for key in ("q", "k", "v"):
        inp[key] = inp[key].cuda()
    return inp


def run_select(inp, keep=None):
    c = inp["cfg"]
    idx, cnt = bsa.bsa_select(inp["q"], inp["k"], c.prefix, inp["seq_lens"], c.block_q, c.block_k,
                              inp["keep_ratio"] if keep is None else keep)
    bsa.bsa_device_status()
    return idx, cnt


def run_forward(inp, idx, cnt, q=None, k=None, v=None):
    c = inp["cfg"]
    out, lse = bsa.bsa_forward(inp["q"] if q is None else q, inp["k"] if k is None else k,
                               inp["v"] if v is None else v, idx, cnt, c.prefix, inp["seq_lens"],
                               c.block_q, c.block_k)
    bsa.bsa_device_status()
    return out, lse


@pytest.mark.parametrize("name", SMALL)
def test_select_parity_small(name):
    inp = cuda_inputs(name)
    c = inp["cfg"]
    idx, cnt = run_select(inp)
    ref = O.select_blocks(to_f32_np(inp["q"]), to_f32_np(inp["k"]), c.prefix, inp["seq_lens"],
                          c.block_q, c.block_k, inp["keep_ratio"])
    gi, gc = idx.cpu().numpy(), cnt.cpu().numpy()
    stats = compare_selection(gi, gc, ref)
    check_structure(gi, gc, c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    assert bsa.bsa_validate_indices(idx, cnt, c.B, c.Hq, c.Sq, c.Skv, c.prefix, inp["seq_lens"],
                                    c.block_q, c.block_k) == 0
    print(name, stats)


def oracle_lists(inp):
    """The oracle's selection as int32 numpy arrays (the lists both forwards attend)."""
    c = inp["cfg"]
    ref = O.select_blocks(to_f32_np(inp["q"]), to_f32_np(inp["k"]), c.prefix, inp["seq_lens"], c.block_q,
                          c.block_k, inp["keep_ratio"])
    return ref, ref["indices"].astype(np.int32), ref["counts"].astype(np.int32)


@pytest.mark.parametrize("name", SMALL)
def test_forward_parity_small(name):
    """The CUDA forward and the oracle's attention over the oracle's lists."""
    inp = cuda_inputs(name)
    c = inp["cfg"]
    _, ri, rc = oracle_lists(inp)
    out, lse = run_forward(inp, torch.from_numpy(ri).cuda(), torch.from_numpy(rc).cuda())
    q, k, v = (to_f32_np(inp[x]).astype(np.float64) for x in ("q", "k", "v"))
    o_ref, l_ref = O.attention(q, k, v, ri, rc, c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    stats = compare_attention(out.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, inp["seq_lens"])
    print(name, stats)


@pytest.mark.parametrize("name", ["small_gqa", "tiny", "small_64x64_d128"])
def test_dense_pass_equals_keep_one_and_oracle(name):
    inp = cuda_inputs(name)
    c = inp["cfg"]
    idx1, cnt1 = run_select(inp, keep=[1.0])
    o_null, l_null = run_forward(inp, None, None)
    o_k1, l_k1 = run_forward(inp, idx1, cnt1)
    assert torch.equal(o_null, o_k1)
    assert torch.equal(l_null, l_k1)
    q, k, v = (to_f32_np(inp[x]).astype(np.float64) for x in ("q", "k", "v"))
    di, dc = O.dense_indices(c.prefix, inp["seq_lens"], c.Sq, c.Skv, c.block_q, c.block_k, c.Hq)
    o_ref, l_ref = O.attention(q, k, v, di, dc, c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    compare_attention(o_null.float().cpu().numpy(), l_null.cpu().numpy(), o_ref, l_ref, inp["seq_lens"])


def test_dropped_blocks_leave_output_bitwise_unchanged():
    inp = cuda_inputs("small_gqa")
    c = inp["cfg"]
    idx, cnt = run_select(inp)
    out, lse = run_forward(inp, idx, cnt)
    gi, gc = idx.cpu().numpy(), cnt.cpu().numpy()
    G = c.Hq // c.Hkv
    k2, v2 = inp["k"].clone(), inp["v"].clone()
    gen = torch.Generator(device="cuda").manual_seed(9)
    changed = 0
    for b in range(c.B):
        for hk in range(c.Hkv):
            used = set()
            for h in range(hk * G, (hk + 1) * G):
                for qb in range(gc.shape[2]):
                    used.update(gi[b, h, qb, :gc[b, h, qb]].tolist())
            for kb in range(O.cdiv(c.Skv, c.block_k)):
                if kb not in used:
                    sl = slice(kb * c.block_k, (kb + 1) * c.block_k)
                    shape = k2[b, sl, hk].shape
                    k2[b, sl, hk] = (100 * torch.randn(shape, generator=gen, device="cuda")).bfloat16()
                    v2[b, sl, hk] = (100 * torch.randn(shape, generator=gen, device="cuda")).bfloat16()
                    changed += 1
    assert changed > 0
    out2, lse2 = run_forward(inp, idx, cnt, k=k2, v=v2)
    assert torch.equal(out, out2)
    assert torch.equal(lse, lse2)


@pytest.mark.parametrize("name", ["small_gqa", "small_64x64_d128"])
def test_forward_without_lse_writes_the_same_output(name):
    """lse = NULL (return_lse=False): the kernel skips the LSE stores and
    writes the same output bits."""
    inp = cuda_inputs(name)
    c = inp["cfg"]
    idx, cnt = run_select(inp)
    out, lse = run_forward(inp, idx, cnt)
    out2, lse2 = bsa.bsa_forward(inp["q"], inp["k"], inp["v"], idx, cnt, c.prefix, inp["seq_lens"], c.block_q,
                                 c.block_k, return_lse=False)
    bsa.bsa_device_status()
    assert lse2 is None
    assert torch.equal(out, out2)


def test_rows_sum_to_one():
    inp = cuda_inputs("small_gqa")
    idx, cnt = run_select(inp)
    ones = torch.ones_like(inp["v"])
    out, _ = run_forward(inp, idx, cnt, v=ones)
    for b, L in enumerate(inp["seq_lens"]):
        err = (out[b, :L].float() - 1).abs().max().item()
        assert err <= 2 ** -7, err


def test_nan_padding_is_never_read():
    a = cuda_inputs("small_gqa", pad_fill=float("nan"))
    z = cuda_inputs("small_gqa", pad_fill=0.0)
    ia, ca = run_select(a)
    iz, cz = run_select(z)
    assert torch.equal(ca, cz)
    for b in range(a["cfg"].B):
        for h in range(a["cfg"].Hq):
            for qb in range(ca.shape[2]):
                c = int(ca[b, h, qb])
                assert torch.equal(ia[b, h, qb, :c], iz[b, h, qb, :c])
    oa, la = run_forward(a, ia, ca)
    oz, lz = run_forward(z, iz, cz)
    assert torch.equal(oa, oz)
    assert torch.equal(la, lz)
    assert torch.isfinite(oa).all()


def test_gqa_matches_mha_with_repeated_kv_bitwise():
    inp = cuda_inputs("small_gqa")
    c = inp["cfg"]
    G = c.Hq // c.Hkv
    idx, cnt = run_select(inp)
    out, lse = run_forward(inp, idx, cnt)
    kr = inp["k"].repeat_interleave(G, dim=2).contiguous()
    vr = inp["v"].repeat_interleave(G, dim=2).contiguous()
    idx2, cnt2 = bsa.bsa_select(inp["q"], kr, c.prefix, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    assert torch.equal(cnt, cnt2)
    out2, lse2 = run_forward(inp, idx2, cnt2, k=kr, v=vr)
    assert torch.equal(out, out2)
    assert torch.equal(lse, lse2)


def test_strided_views_match_contiguous():
    inp = cuda_inputs("small_gqa", pad_fill=0.0)
    c = inp["cfg"]
    q, k, v = inp["q"], inp["k"], inp["v"]
    # packed buffers: Q inside [B, Sq, Hq + 8, d]; K/V inside one [B, Skv, 2, Hkv, d] tensor
    qp = torch.zeros(c.B, c.Sq, c.Hq + 8, c.d, dtype=torch.bfloat16, device="cuda")
    qp[:, :, 3:3 + c.Hq] = q
    kv = torch.stack([k, v], dim=2)
    qs, ks, vs = qp[:, :, 3:3 + c.Hq], kv[:, :, 0], kv[:, :, 1]
    assert not qs.is_contiguous() and not ks.is_contiguous()
    idx, cnt = run_select(inp)
    out, lse = run_forward(inp, idx, cnt)
    idx2, cnt2 = bsa.bsa_select(qs, ks, c.prefix, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    assert torch.equal(cnt, cnt2)
    out2, lse2 = run_forward(inp, idx2, cnt2, q=qs, k=ks, v=vs)
    assert torch.equal(out, out2)
    assert torch.equal(lse, lse2)


@pytest.mark.parametrize("name", ["tiny", "small_64x64_d128", "small_mha_perhead"])
def test_merged_small_query_blocks_match_per_block_lists(name):
    """64/128-row query blocks run 256 rows at a time over merged lists; each
    row must see exactly its own query block's list: compare against the
    oracle and against feeding one query block's list at a time (the other
    blocks' counts set to 0)."""
    inp = cuda_inputs(name, pad_fill=0.0)
    c = inp["cfg"]
    idx, cnt = run_select(inp)
    out, lse = run_forward(inp, idx, cnt)
    ratio = 256 // c.block_q
    for g in range(ratio):
        cnt_g = cnt.clone()
        keep = torch.zeros_like(cnt_g, dtype=torch.bool)
        keep[:, :, g::ratio] = True
        cnt_g[~keep] = 0
        out_g, lse_g = run_forward(inp, idx, cnt_g)
        for qb in range(g, cnt.shape[2], ratio):
            r0, r1 = qb * c.block_q, min((qb + 1) * c.block_q, c.Sq)
            # The merged list puts the blocks both 128-row halves selected
            # first, so a row's blocks come in another order than in a list
            # of its own query block alone (and 64-key blocks pair up
            # differently): the fp32 row sums are equal up to rounding.  A
            # row that saw another block's selection would differ by far more.
            assert torch.allclose(out[:, r0:r1].float(), out_g[:, r0:r1].float(), rtol=1e-2, atol=1e-3)
            assert torch.allclose(lse[:, :, r0:r1], lse_g[:, :, r0:r1], rtol=0, atol=1e-4)


@pytest.mark.parametrize("name", ["small_64x64_d128", "small_mqa_d64", "small_mha_perhead"])
def test_merged_lists_of_every_class_shape(name):
    """Hand-made lists that give the merged 256-row lists every shape the
    forward walks: one 128-row half with no block at all, halves with disjoint
    selections of odd sizes (a padding entry per class when 64-key blocks are
    paired), one half with blocks of its own past the other's (a tail one half
    walks alone), and blocks both halves share next to blocks of one half."""
    inp = cuda_inputs(name, pad_fill=float("nan"))
    c = inp["cfg"]
    nQb, nKb = -(-c.Sq // c.block_q), -(-c.Skv // c.block_k)
    per_half = 128 // c.block_q
    rng = np.random.default_rng(4242)
    idx = np.full((c.B, c.Hq, nQb, nKb), -1, np.int32)
    cnt = np.zeros((c.B, c.Hq, nQb), np.int32)
    for b, L in enumerate(inp["seq_lens"]):
        for h in range(c.Hq):
            for qb in range(-(-L // c.block_q)):
                kind = (qb // (2 * per_half) + h + b) % 4
                half = (qb % (2 * per_half)) // per_half
                if kind == 0:        # half 1 attends nothing
                    blocks = [] if half else rng.choice(nKb, min(5, nKb), replace=False)
                elif kind == 1:      # disjoint, 3 and 5 blocks
                    blocks = range(3) if half == 0 else range(nKb - 5, nKb)
                elif kind == 2:      # two shared blocks, half 0 has 7 more
                    blocks = [1, 2] + ([] if half else list(range(4, min(nKb, 11))))
                else:                # anything
                    blocks = rng.choice(nKb, int(rng.integers(1, nKb + 1)), replace=False)
                blocks = sorted(set(int(x) for x in blocks))
                idx[b, h, qb, :len(blocks)] = blocks
                cnt[b, h, qb] = len(blocks)
    out, lse = run_forward(inp, torch.from_numpy(idx).cuda(), torch.from_numpy(cnt).cuda())
    qf, kf, vf = (to_f32_np(inp[x]).astype(np.float64) for x in ("q", "k", "v"))
    o_ref, l_ref = O.attention(qf, kf, vf, idx, cnt, c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    stats = compare_attention(out.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, inp["seq_lens"])
    print(name, stats)


def test_keep_zero_without_prefix_gives_empty_rows():
    inp = cuda_inputs("small_mha_perhead")
    idx, cnt = run_select(inp, keep=[0.0])
    assert int(cnt.max()) == 0
    out, lse = run_forward(inp, idx, cnt)
    assert (out == 0).all()
    assert torch.isneginf(lse).all()


def test_validate_finds_corrupted_rows():
    inp = cuda_inputs("small_gqa")
    c = inp["cfg"]
    idx, cnt = run_select(inp)
    args = (c.B, c.Hq, c.Sq, c.Skv, c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    assert bsa.bsa_validate_indices(idx, cnt, *args) == 0
    bad = idx.clone()
    bad[0, 0, 0, 3] = bad[0, 0, 0, 2]            # not strictly ascending
    bad[0, 1, 1, 0] = 5                          # prefix block 0 missing
    bad[1, 2, 0, 4] = 10 ** 6                    # out of range
    assert bsa.bsa_validate_indices(bad, cnt, *args) == 3
    cnt2 = cnt.clone()
    cnt2[1, 0, -1] = 1                           # padded query block with a count
    assert bsa.bsa_validate_indices(idx, cnt2, *args) == 1


def test_out_of_range_indices_are_clamped_not_read():
    """Indices past the key blocks (and a count above nKb) are clamped by the
    kernel: the block reads as fully masked, nothing faults."""
    inp = cuda_inputs("small_gqa")
    c = inp["cfg"]
    idx, cnt = run_select(inp)
    bad = idx.clone()
    nkb = bad.shape[3]
    bad[0, 0, 0, cnt[0, 0, 0] - 1] = 10 ** 6
    cnt_big = cnt.clone()
    cnt_big[0, 1, 0] = nkb + 50
    run_forward(inp, bad, cnt_big)


# ------------------------------------------- causal understanding stream ---

@pytest.mark.parametrize("P,Hq,Hkv,d,bq,bk", [
    (700, 4, 2, 128, 256, 128),      # ragged last query and key blocks
    (1024, 8, 2, 128, 256, 128),     # the 720p workload's prefix length
    (333, 3, 1, 64, 64, 64),         # MQA, 64x64 geometry
    (512, 2, 2, 128, 128, 64),
])
def test_causal_prefix_parity(P, Hq, Hkv, d, bq, bk):
    g = torch.Generator(device="cpu").manual_seed(P * 7 + Hq)
    q = torch.randn(2, P, Hq, d, generator=g).bfloat16()
    k = torch.randn(2, P + 300, Hkv, d, generator=g).bfloat16()     # generation rows after P
    v = torch.randn(2, P + 300, Hkv, d, generator=g).bfloat16()
    k[:, P:] = float("nan")                                         # never read
    v[:, P:] = float("nan")
    out, lse = bsa.bsa_forward_causal(q.cuda(), k.cuda(), v.cuda(), bq, bk)
    bsa.bsa_device_status()
    o_ref, l_ref = O.causal_prefix_attention(q.float().numpy(), k.float().numpy(), v.float().numpy(), P)
    stats = compare_attention(out.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, [P, P])
    print("causal", P, Hq, Hkv, d, bq, bk, stats)


def test_causal_equals_dense_on_last_row():
    """The last understanding row sees every prefix key: it must equal a dense
    pass of that row over the prefix (a selected-block forward with P keys)."""
    g = torch.Generator(device="cpu").manual_seed(5)
    P, Hq, Hkv, d = 512, 2, 1, 128
    q = torch.randn(1, P, Hq, d, generator=g).bfloat16().cuda()
    k = torch.randn(1, P, Hkv, d, generator=g).bfloat16().cuda()
    v = torch.randn(1, P, Hkv, d, generator=g).bfloat16().cuda()
    out, lse = bsa.bsa_forward_causal(q, k, v, 256, 128)
    dense, dl = bsa.bsa_forward(q, k, v, None, None, 0, None, 256, 128)
    bsa.bsa_device_status()
    assert (out[0, -1].float() - dense[0, -1].float()).abs().max().item() <= 2 ** -8
    assert abs(lse[0, 0, -1].item() - dl[0, 0, -1].item()) <= 1e-5


# ------------------------------------------------- rotary prologue fused ---

def _tables(S, d, offset=0, base=10000.0):
    inv = base ** (-torch.arange(0, d // 2, dtype=torch.float64) * 2.0 / d)
    ang = torch.outer(torch.arange(offset, offset + S, dtype=torch.float64), inv)
    ang = torch.cat([ang, ang], dim=1)
    return ang.cos().float(), ang.sin().float()


@pytest.mark.parametrize("name", ["small_gqa", "small_mqa_d64", "small_mha_perhead"])
def test_select_rope_parity(name):
    inp = cuda_inputs(name, pad_fill=0.0)
    c = inp["cfg"]
    # understanding positions 0..P-1 for the prefix keys, generation positions after
    cq, sq = _tables(c.Sq, c.d, offset=c.prefix)
    ck, sk = _tables(c.Skv, c.d)
    q_out, k_out, idx, cnt = bsa.bsa_select_rope(inp["q"], inp["k"], cq.cuda(), sq.cuda(), ck.cuda(), sk.cuda(),
                                                 c.prefix, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    bsa.bsa_device_status()
    ref = O.rope_then_select(to_f32_np(inp["q"]), to_f32_np(inp["k"]), cq.numpy(), sq.numpy(), ck.numpy(),
                             sk.numpy(), c.prefix, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    # rotated tensors: the fp32 rotation differs from the fp64 one by fp32
    # rounding of the two products (absolute, ~1e-7 of the terms, which
    # matters where they cancel); after rounding both to bf16 they are at most
    # one bf16 ulp plus that apart, and almost always identical
    for got, want, x, cs, sn in ((q_out, ref["q_rot"], inp["q"], cq, sq), (k_out, ref["k_rot"], inp["k"], ck, sk)):
        g = got.float().cpu().numpy().astype(np.float64)
        xf = to_f32_np(x).astype(np.float64)
        terms = np.abs(xf) * np.abs(cs.numpy())[None, :, None, :] + \
            np.abs(O.rotate_half(xf)) * np.abs(sn.numpy())[None, :, None, :]
        tol = np.abs(want) * 2.0 ** -7 + terms * 2.0 ** -22
        assert (np.abs(g - want) <= tol).all(), float(np.max(np.abs(g - want) - tol))
        assert (g == want).mean() > 0.999
    stats = compare_selection(idx.cpu().numpy(), cnt.cpu().numpy(), ref)
    # fused == rotate first, then select on the rotated tensors (bit for bit)
    idx2, cnt2 = bsa.bsa_select(q_out, k_out, c.prefix, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    assert torch.equal(cnt, cnt2)
    for b in range(c.B):
        for h in range(c.Hq):
            for qb in range(cnt.shape[2]):
                n = int(cnt[b, h, qb])
                assert torch.equal(idx[b, h, qb, :n], idx2[b, h, qb, :n])
    print(name, stats)


def test_select_rope_in_place():
    inp = cuda_inputs("small_gqa", pad_fill=0.0)
    c = inp["cfg"]
    cq, sq = _tables(c.Sq, c.d, offset=c.prefix)
    ck, sk = _tables(c.Skv, c.d)
    q1, k1, i1, n1 = bsa.bsa_select_rope(inp["q"], inp["k"], cq.cuda(), sq.cuda(), ck.cuda(), sk.cuda(), c.prefix,
                                         inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    q, k = inp["q"].clone(), inp["k"].clone()
    q2, k2, i2, n2 = bsa.bsa_select_rope(q, k, cq.cuda(), sq.cuda(), ck.cuda(), sk.cuda(), c.prefix, inp["seq_lens"],
                                         c.block_q, c.block_k, inp["keep_ratio"], q_out=q, k_out=k)
    bsa.bsa_device_status()
    assert torch.equal(q1, q) and torch.equal(k1, k) and torch.equal(n1, n2)


# ----------------------------------------------------------- full size ---

def full_inputs(name):
    cfg = CONFIGS[name]
    return make_inputs(cfg, "cuda", pad_fill=float("nan"))


@pytest.mark.parametrize("name", list(WORKLOAD_CONFIGS) + ["480p_75_64x64"])
def test_workload_config_parity(name):
    inp = full_inputs(name)
    c = inp["cfg"]
    idx, cnt = run_select(inp)
    gi, gc = idx.cpu().numpy(), cnt.cpu().numpy()
    q32, k32 = to_f32_np(inp["q"]), to_f32_np(inp["k"])
    ref = O.select_blocks(q32, k32, c.prefix, inp["seq_lens"], c.block_q, c.block_k, inp["keep_ratio"])
    sel_stats = compare_selection(gi, gc, ref)
    check_structure(gi, gc, c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    if name == "480p_dense":
        out_g, lse_g = run_forward(inp, idx, cnt)
        o_null, l_null = run_forward(inp, None, None)
        assert torch.equal(o_null, out_g) and torch.equal(l_null, lse_g)
        del out_g, lse_g, o_null, l_null
    # the forward in the bench's launch configuration, over the oracle's lists
    ri, rc = ref["indices"].astype(np.int32), ref["counts"].astype(np.int32)
    out, lse = run_forward(inp, torch.from_numpy(ri).cuda(), torch.from_numpy(rc).cuda())
    tiles = sample_tiles(c.B, c.Hq, gc.shape[2], inp["seq_lens"], c.block_q, n_random=8, seed=c.seed)
    v32 = to_f32_np(inp["v"])
    o_ref, l_ref = O.attention(q32, k32, v32, ri, rc, c.prefix, inp["seq_lens"], c.block_q, c.block_k,
                               tiles=tiles)
    att = compare_attention(out.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, inp["seq_lens"])
    kept = gc.sum() / max(1, sum(O.cdiv(c.prefix + L, c.block_k) * O.cdiv(L, c.block_q)
                                 for L in inp["seq_lens"]) * c.Hq)
    print(name, sel_stats, att, f"tile keep fraction {kept:.4f}")
