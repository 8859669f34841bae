"""GPU parity of the backward pass (dQ, dK, dV) against the fp64 oracle.

Every input of the CUDA call comes from the seeded generators or the oracle:
the lists are the oracle's selection, ``out``/``lse`` the oracle's forward
(rounded to bf16 / fp32 as the forward stores them), ``dout`` a seeded draw.
Small cases compare every element; the 480p workload checks identities that
hold at any size (dK of a KV head sums to zero over its keys because each
row of dS sums to zero; dV sums to the summed dout of the rows its group
attends) plus sampled query tiles of dQ against the oracle.
"""

import numpy as np
import pytest
import torch

import block_sparse_attention_bsa_gb300 as bsa
from bsa_inputs import CONFIGS, make_inputs
from oracle import bsa_oracle as O
from parity_utils import to_f32_np

pytestmark = pytest.mark.gpu

# Relative tolerances of bf16 gradients against the fp64 oracle: P and dS are
# rounded to bf16 before their MMAs (unit roundoff 2^-8 each, random in sign)
# and the results are stored in bf16, so errors stay a few tenths of a percent
# of the tensor's scale (measured: dQ 0.42%, dK/dV 0.24%).
REL_FRO = 1e-2
REL_MAX = 3e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    bsa.build()


def seeded_dout(shape, seed, lens, pad_fill=float("nan")):
    g = torch.Generator().manual_seed(seed)
    d = torch.randn(shape, generator=g).to(torch.bfloat16)
    for b, L in enumerate(lens):
        d[b, L:] = pad_fill
    return d


def oracle_case(name, keep=None):
    """Inputs (CPU bf16 / numpy) and the oracle's selection, forward and backward."""
    inp = make_inputs(CONFIGS[name], "cpu", pad_fill=float("nan"))
    c = inp["cfg"]
    q, k, v = (to_f32_np(inp[x]).astype(np.float64) for x in ("q", "k", "v"))
    sel = O.select_blocks(to_f32_np(inp["q"]), to_f32_np(inp["k"]), c.prefix, inp["seq_lens"],
                          c.block_q, c.block_k, inp["keep_ratio"] if keep is None else keep)
    idx, cnt = sel["indices"].astype(np.int32), sel["counts"].astype(np.int32)
    o_ref, l_ref = O.attention(q, k, v, idx, cnt, c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    # what the forward stores: bf16 out (0 on padded rows), fp32 lse (-inf there)
    out_bf = torch.from_numpy(np.nan_to_num(o_ref, nan=0.0)).to(torch.bfloat16)
    lse32 = torch.from_numpy(np.where(np.isnan(l_ref), -np.inf, l_ref)).to(torch.float32)
    dout = seeded_dout(tuple(inp["q"].shape), c.seed + 11, inp["seq_lens"])
    dq, dk, dv = O.attention_backward(q, k, v, to_f32_np(out_bf), to_f32_np(dout), lse32.numpy(), idx, cnt,
                                      c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    return inp, idx, cnt, out_bf, lse32, dout, (dq, dk, dv)


def run_backward(inp, idx, cnt, out_bf, lse32, dout):
    c = inp["cfg"]
    dev = lambda t: t.cuda()
    res = bsa.bsa_backward(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]), dev(out_bf), dev(dout), dev(lse32),
                           dev(torch.from_numpy(idx)), dev(torch.from_numpy(cnt)), c.prefix, inp["seq_lens"],
                           c.block_q, c.block_k)
    bsa.bsa_device_status()
    return res


def compare_grad(name, g, r, real):
    """g: GPU bf16 tensor, r: fp64 oracle array, real: boolean mask [B, S] of rows that may be non-zero."""
    gn = g.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(gn).all(), f"{name}: non-finite values"
    mask = np.broadcast_to(real[:, :, None, None], gn.shape)
    assert (gn[~mask] == 0).all(), f"{name}: padded rows are not zero"
    err = np.abs(gn - r)
    scale = np.abs(r).max()
    rel_fro = np.linalg.norm(gn - r) / max(np.linalg.norm(r), 1e-30)
    rel_max = err.max() / max(scale, 1e-30)
    assert rel_fro <= REL_FRO and rel_max <= REL_MAX, (name, rel_fro, rel_max)
    return dict(rel_fro=float(rel_fro), rel_max=float(rel_max))


@pytest.mark.parametrize("name", ["small_gqa", "small_mha_perhead", "tiny", "small_mqa_d64", "small_64x64_d128"])
def test_backward_parity_small(name):
    inp, idx, cnt, out_bf, lse32, dout, (dq_r, dk_r, dv_r) = oracle_case(name)
    c = inp["cfg"]
    dq, dk, dv = run_backward(inp, idx, cnt, out_bf, lse32, dout)
    B, Sq, Skv = c.B, c.Sq, c.Skv
    real_q = np.arange(Sq)[None, :] < np.array(inp["seq_lens"])[:, None]
    real_k = np.arange(Skv)[None, :] < (c.prefix + np.array(inp["seq_lens"]))[:, None]
    stats = {n: compare_grad(n, g, r, m) for n, g, r, m in
             (("dq", dq, dq_r, real_q), ("dk", dk, dk_r, real_k), ("dv", dv, dv_r, real_k))}
    print(name, stats)


def test_backward_is_deterministic():
    inp, idx, cnt, out_bf, lse32, dout, _ = oracle_case("small_gqa")
    a = run_backward(inp, idx, cnt, out_bf, lse32, dout)
    b = run_backward(inp, idx, cnt, out_bf, lse32, dout)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_backward_strided_inputs_match_contiguous():
    """q, k, v, out and dout as views of packed buffers (16-byte aligned, not
    contiguous): the same gradient bits as contiguous copies."""
    inp, idx, cnt, out_bf, lse32, dout, _ = oracle_case("small_gqa")
    c = inp["cfg"]
    a = run_backward(inp, idx, cnt, out_bf, lse32, dout)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    qp = torch.zeros(c.B, c.Sq, 3, c.Hq, c.d, dtype=torch.bfloat16, device="cuda")  # q, out, dout side by side
    qp[:, :, 0], qp[:, :, 1], qp[:, :, 2] = q, out_bf.cuda(), dout.cuda()
    kv = torch.stack([k, v], dim=2)
    views = (qp[:, :, 0], kv[:, :, 0], kv[:, :, 1], qp[:, :, 1], qp[:, :, 2])
    assert not any(t.is_contiguous() for t in views)
    b = bsa.bsa_backward(*views, lse32.cuda(), torch.from_numpy(idx).cuda(), torch.from_numpy(cnt).cuda(),
                         c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    bsa.bsa_device_status()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_backward_dense_lists_match_oracle():
    """keep ratio 1: every valid key block of every row (the dense pass's lists)."""
    inp, idx, cnt, out_bf, lse32, dout, (dq_r, dk_r, dv_r) = oracle_case("small_gqa", keep=[1.0])
    c = inp["cfg"]
    dq, dk, dv = run_backward(inp, idx, cnt, out_bf, lse32, dout)
    real_q = np.arange(c.Sq)[None, :] < np.array(inp["seq_lens"])[:, None]
    real_k = np.arange(c.Skv)[None, :] < (c.prefix + np.array(inp["seq_lens"]))[:, None]
    compare_grad("dq", dq, dq_r, real_q)
    compare_grad("dk", dk, dk_r, real_k)
    compare_grad("dv", dv, dv_r, real_k)


def dq_rounding_bound(q, k, v, out, dout, lse, pos, rows, h, hk, scale):
    """Elementwise bound on |dQ_gpu - dQ_exact| for one tile from the kernel's
    roundings: dS is rounded to bf16 before the dS K product (unit roundoff
    2^-8 per element, summed in magnitude over the keys) and dQ is stored in
    bf16 (2^-8 of the value); everything else is fp32 with errors far below."""
    qq, kk, vv = q[rows, h], k[pos, hk], v[pos, hk]
    p_ = np.exp((qq @ kk.T) * scale - lse[h, rows, None])
    D = (dout[rows, h] * out[rows, h]).sum(axis=1, keepdims=True)
    ds = p_ * (dout[rows, h] @ vv.T - D)
    ref = scale * ds @ kk
    return 2.0 ** -8 * scale * (np.abs(ds) @ np.abs(kk)) + 2.0 ** -8 * np.abs(ref)


@pytest.mark.parametrize("name", ["480p_75", "480p_75_64x64"])
def test_backward_480p_identities_and_sampled_dq(name):
    """480p latent, keep 25%, the oracle's lists through the CUDA forward and
    backward: identities over all keys, and sampled dQ tiles against the
    oracle's backward of those tiles on the same out/lse (the oracle's
    forward of the tiles, written into the forward's buffers)."""
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, "cpu")
    L = inp["seq_lens"][0]
    G = cfg.Hq // cfg.Hkv
    sel = O.select_blocks(to_f32_np(inp["q"]), to_f32_np(inp["k"]), cfg.prefix, inp["seq_lens"],
                          cfg.block_q, cfg.block_k, inp["keep_ratio"])
    idx_h, cnt_h = sel["indices"].astype(np.int32), sel["counts"].astype(np.int32)
    dout_h = seeded_dout(tuple(inp["q"].shape), cfg.seed + 11, inp["seq_lens"], pad_fill=0.0)
    q, k, v, dout = (t.cuda() for t in (inp["q"], inp["k"], inp["v"], dout_h))
    idx, cnt = torch.from_numpy(idx_h).cuda(), torch.from_numpy(cnt_h).cuda()
    out, lse = bsa.bsa_forward(q, k, v, idx, cnt, cfg.prefix, inp["seq_lens"], cfg.block_q, cfg.block_k)
    # sampled tiles: the oracle's forward of those rows replaces the kernel's
    rng = np.random.default_rng(5)
    nQb = -(-cfg.Sq // cfg.block_q)
    tiles = [(0, int(rng.integers(cfg.Hq)), int(rng.integers(nQb))) for _ in range(6)]
    qf, kf, vf = (to_f32_np(inp[x]).astype(np.float64) for x in ("q", "k", "v"))
    o_ref, l_ref = O.attention(qf, kf, vf, idx_h, cnt_h, cfg.prefix, inp["seq_lens"], cfg.block_q,
                               cfg.block_k, tiles=tiles)
    o_bf = O.round_to_bf16(np.nan_to_num(o_ref, nan=0.0))
    l32 = np.where(np.isnan(l_ref), -np.inf, l_ref).astype(np.float32).astype(np.float64)
    for (_, h, qb) in tiles:
        r0, r1 = qb * cfg.block_q, min((qb + 1) * cfg.block_q, L)
        out[0, r0:r1, h] = torch.from_numpy(o_bf[0, r0:r1, h]).to(torch.bfloat16).cuda()
        lse[0, h, r0:r1] = torch.from_numpy(l32[0, h, r0:r1]).float().cuda()
    dq, dk, dv = bsa.bsa_backward(q, k, v, out, dout, lse, idx, cnt, cfg.prefix, inp["seq_lens"],
                                  cfg.block_q, cfg.block_k)
    bsa.bsa_device_status()
    # sum_j dK_j = scale * sum_i (sum_j dS_ij) q_i = 0
    dk_sum = dk.double().sum(dim=1)                                  # [B, Hkv, d]
    dk_abs = dk.double().abs().sum(dim=1)
    assert (dk_sum.abs() <= 1e-2 * dk_abs + 1e-3).all(), float((dk_sum.abs() / dk_abs).max())
    # sum_j dV_j = sum over the group's real rows of dout (every row's P sums to 1)
    dv_sum = dv.double().sum(dim=1)
    do_sum = dout.double().view(cfg.B, cfg.Sq, cfg.Hkv, G, cfg.d).sum(dim=(1, 3))
    tol = 1e-2 * dv.double().abs().sum(dim=1) + 1e-2
    assert ((dv_sum - do_sum).abs() <= tol).all(), float((dv_sum - do_sum).abs().max())
    assert torch.isfinite(dq.float()).all()
    doh = to_f32_np(dout_h).astype(np.float64)
    dq_ref, _, _ = O.attention_backward(qf, kf, vf, o_bf, doh, l32, idx_h, cnt_h, cfg.prefix,
                                        inp["seq_lens"], cfg.block_q, cfg.block_k, tiles=tiles)
    dqh = dq[0].float().cpu().numpy().astype(np.float64)
    scale = O.default_scale(cfg.d)
    for (_, h, qb) in tiles:
        r0, r1 = qb * cfg.block_q, min((qb + 1) * cfg.block_q, L)
        pos = O.tile_keys(idx_h[0, h, qb, :cnt_h[0, h, qb]], cfg.prefix + L, cfg.block_k)
        bound = dq_rounding_bound(qf[0], kf[0], vf[0], o_bf[0], doh[0], l32[0], pos, slice(r0, r1), h,
                                  h // G, scale)
        g, r = dqh[r0:r1, h], dq_ref[0, r0:r1, h]
        excess = np.abs(g - r) / (bound + 1e-6)
        rel = np.linalg.norm(g - r) / np.linalg.norm(r)
        print("tile", h, qb, "rel_fro", rel, "max err / bound", float(excess.max()))
        assert excess.max() <= 1.0, (h, qb, rel, float(excess.max()))


def elementwise_bounds(q, k, v, out, dout, lse, indices, counts, prefix_len, seq_lens, block_q, block_k):
    """Per-element bounds on |grad_gpu - grad_exact| from the kernels' roundings,
    accumulated tile by tile like the oracle's backward but over magnitudes:
      * dS (dQ, dK) and P^T (dV) rounded to bf16 before their MMAs:
        2^-8 sum |dS| |k| (dQ), 2^-8 scale sum |dS| |q| (dK), 2^-8 sum P |dO| (dV);
      * dP and D accumulated in fp32 over d <= 128 products (and the exponent
        argument likewise): 2^-16 per unit of sum_c |dO_c| (|v_c| + |O_c|), carried
        through P into dQ and dK;
      * the result stored in bf16: 2^-8 |grad|, added by the caller.
    Returns (bq, bk, bv) shaped like dq, dk, dv."""
    B, Sq, Hq, d = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    scale = O.default_scale(d)
    bq, bk, bv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    nQb = -(-Sq // block_q)
    for b in range(B):
        L = int(seq_lens[b])
        for h in range(Hq):
            hk = h // G
            for qb in range(nQb):
                r0, r1 = qb * block_q, min((qb + 1) * block_q, L)
                if r1 <= r0:
                    continue
                c = int(counts[b, h, qb])
                pos = O.tile_keys(indices[b, h, qb, :c], prefix_len + L, block_k)
                if pos.size == 0:
                    continue
                qq, oo, gg = q[b, r0:r1, h], out[b, r0:r1, h], dout[b, r0:r1, h]
                kk, vv = k[b, pos, hk], v[b, pos, hk]
                p_ = np.exp((qq @ kk.T) * scale - lse[b, h, r0:r1, None])
                D = (gg * oo).sum(axis=1, keepdims=True)
                ds = np.abs(p_ * (gg @ vv.T - D))
                w = p_ * (np.abs(gg) @ np.abs(vv).T + np.abs(gg * oo).sum(axis=1, keepdims=True))
                bq[b, r0:r1, h] += scale * (2.0 ** -8 * ds + 2.0 ** -16 * w) @ np.abs(kk)
                bk[b, pos, hk] += scale * (2.0 ** -8 * ds + 2.0 ** -16 * w).T @ np.abs(qq)
                bv[b, pos, hk] += 2.0 ** -8 * p_.T @ np.abs(gg)
    return bq, bk, bv


@pytest.mark.parametrize("name", ["small_gqa", "small_mha_perhead", "tiny", "small_mqa_d64", "small_64x64_d128"])
def test_backward_small_every_element_within_its_rounding_bound(name):
    """Every element of dQ, dK and dV on the small configurations lies within
    the bound its roundings allow (not only relative to the tensor's largest
    value), including the entries whose exact gradient is zero."""
    inp, idx, cnt, out_bf, lse32, dout, grads_r = oracle_case(name)
    c = inp["cfg"]
    grads = run_backward(inp, idx, cnt, out_bf, lse32, dout)
    q, k, v = (np.nan_to_num(to_f32_np(inp[x]).astype(np.float64)) for x in ("q", "k", "v"))
    bounds = elementwise_bounds(q, k, v, to_f32_np(out_bf).astype(np.float64),
                                np.nan_to_num(to_f32_np(dout).astype(np.float64)), lse32.numpy().astype(np.float64),
                                idx, cnt, c.prefix, inp["seq_lens"], c.block_q, c.block_k)
    for n, g, r, bnd in zip(("dq", "dk", "dv"), grads, grads_r, bounds):
        gn = g.float().cpu().numpy().astype(np.float64)
        tol = bnd + 2.0 ** -8 * np.abs(r) + 1e-7
        excess = np.abs(gn - r) / tol
        print(name, n, "max err / bound", float(excess.max()))
        assert excess.max() <= 1.0, (name, n, float(excess.max()), np.unravel_index(excess.argmax(), excess.shape))
