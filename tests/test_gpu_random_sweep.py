"""Seeded random sweep over the supported geometry (head dim 64/128, 64/128/
256-row query blocks, 64/128-key blocks), head mappings (MHA, GQA, MQA),
prefixes that are or are not block multiples, ragged lengths (including 0
and 1) and softmax scales (the default head_dim^-1/2 or an explicit one):
selector, forward and backward through the C ABI against the fp64 oracle on
the same bits.  The forward and backward run over the oracle's lists; the
backward's out/lse are the oracle's forward as the forward stores them.  A
second sweep does the same for the causal understanding pass.
"""

import numpy as np
import pytest
import torch

import block_sparse_attention_bsa_gb300 as bsa
from bsa_inputs.synthetic import Config, make_inputs
from oracle import bsa_oracle as O
from parity_utils import compare_attention, compare_selection, to_f32_np

pytestmark = pytest.mark.gpu

N_CASES = 40
N_CAUSAL = 16


def random_config(i: int) -> Config:
    rng = np.random.default_rng(9100 + i)
    d = int(rng.choice([64, 128]))
    bq = int(rng.choice([64, 128, 256]))
    bk = int(rng.choice([64, 128]))
    Hkv = int(rng.choice([1, 2, 3]))
    G = int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 4))
    prefix = int(rng.choice([0, bk, 2 * bk, int(rng.integers(1, 300))]))
    lens = tuple(int(x) for x in rng.choice([0, 1, int(rng.integers(2, 200)), int(rng.integers(200, 900))],
                                            size=B))
    if max(lens) == 0:
        lens = (int(rng.integers(1, 600)),) + lens[1:]
    keep = float(rng.choice([0.0, 0.2, 0.5, 1.0]))
    return Config(f"sweep{i}", B=B, Hq=Hkv * G, Hkv=Hkv, d=d, prefix=prefix, lens=lens, block_q=bq, block_k=bk,
                  keep=keep, recipe="iid", seed=9100 + i)


def case_scale(i: int) -> float:
    """Softmax scale of case i: 0 (the library default, head_dim^-1/2) or an
    explicit value; drawn from its own seed so the geometry draws stay put."""
    return float(np.random.default_rng(9700 + i).choice([0.0, 0.0, 0.05, 0.2]))


@pytest.fixture(scope="module", autouse=True)
def built():
    bsa.build()


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_geometry(i):
    cfg = random_config(i)
    inp = make_inputs(cfg, "cpu", pad_fill=float("nan"))
    lens = inp["seq_lens"]
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    idx, cnt = bsa.bsa_select(q, k, cfg.prefix, lens, cfg.block_q, cfg.block_k, inp["keep_ratio"])
    bsa.bsa_device_status()
    qf, kf, vf = (to_f32_np(inp[x]).astype(np.float64) for x in ("q", "k", "v"))
    ref = O.select_blocks(to_f32_np(inp["q"]), to_f32_np(inp["k"]), cfg.prefix, lens, cfg.block_q, cfg.block_k,
                          inp["keep_ratio"])
    compare_selection(idx.cpu().numpy(), cnt.cpu().numpy(), ref)
    ri, rc = ref["indices"].astype(np.int32), ref["counts"].astype(np.int32)
    ri_t, rc_t = torch.from_numpy(ri).cuda(), torch.from_numpy(rc).cuda()
    sc = case_scale(i)
    oscale = sc if sc > 0 else None
    out, lse = bsa.bsa_forward(q, k, v, ri_t, rc_t, cfg.prefix, lens, cfg.block_q, cfg.block_k, softmax_scale=sc)
    bsa.bsa_device_status()
    o_ref, l_ref = O.attention(qf, kf, vf, ri, rc, cfg.prefix, lens, cfg.block_q, cfg.block_k, scale=oscale)
    compare_attention(out.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, lens)
    out_bf = torch.from_numpy(np.nan_to_num(o_ref, nan=0.0)).to(torch.bfloat16)
    lse32 = torch.from_numpy(np.where(np.isnan(l_ref), -np.inf, l_ref)).to(torch.float32)
    dout = torch.randn(inp["q"].shape, generator=torch.Generator().manual_seed(cfg.seed + 11)).to(torch.bfloat16)
    for b, L in enumerate(lens):
        dout[b, L:] = float("nan")
    dq, dk, dv = bsa.bsa_backward(q, k, v, out_bf.cuda(), dout.cuda(), lse32.cuda(), ri_t, rc_t, cfg.prefix, lens,
                                  cfg.block_q, cfg.block_k, softmax_scale=sc)
    bsa.bsa_device_status()
    dq_r, dk_r, dv_r = O.attention_backward(qf, kf, vf, to_f32_np(out_bf), np.nan_to_num(to_f32_np(dout)),
                                            lse32.numpy(), ri, rc, cfg.prefix, lens, cfg.block_q, cfg.block_k,
                                            scale=oscale)
    for name, g, r in (("dq", dq, dq_r), ("dk", dk, dk_r), ("dv", dv, dv_r)):
        gn = g.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(gn).all(), (cfg, name)
        nr = np.linalg.norm(r)
        if nr == 0:
            # exact zero, e.g. a row whose only key gets P = 1 so that dS = dP - D = 0;
            # the GPU forms dP (MMA) and D (its own fp32 sum) in different orders
            assert np.abs(gn).max() <= 1e-4, (cfg, name, np.abs(gn).max())
            continue
        rel = np.linalg.norm(gn - r) / nr
        assert rel <= 1e-2 and np.abs(gn - r).max() <= 3e-2 * np.abs(r).max(), (cfg, name, rel)


@pytest.mark.parametrize("i", range(N_CAUSAL))
def test_random_causal_pass(i):
    """Causal understanding pass over random geometry, head mapping, batch,
    prefix length (down to one row) and scale, against the fp64 oracle."""
    rng = np.random.default_rng(9800 + i)
    d = int(rng.choice([64, 128]))
    bq = int(rng.choice([64, 128, 256]))
    bk = int(rng.choice([64, 128]))
    Hkv = int(rng.choice([1, 2, 3]))
    Hq = Hkv * int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 4))
    P = int(rng.choice([1, 2, 63, 64, 65, int(rng.integers(3, 900))]))
    sc = float(rng.choice([0.0, 0.0, 0.05, 0.2]))
    g = torch.Generator(device="cpu").manual_seed(9800 + i)
    q = torch.randn(B, P, Hq, d, generator=g).bfloat16()
    extra = int(rng.integers(0, 200))                     # generation rows after the prefix: never read
    k = torch.randn(B, P + extra, Hkv, d, generator=g).bfloat16()
    v = torch.randn(B, P + extra, Hkv, d, generator=g).bfloat16()
    k[:, P:] = float("nan")
    v[:, P:] = float("nan")
    out, lse = bsa.bsa_forward_causal(q.cuda(), k.cuda(), v.cuda(), bq, bk, softmax_scale=sc)
    bsa.bsa_device_status()
    o_ref, l_ref = O.causal_prefix_attention(q.float().numpy(), k.float().numpy(), v.float().numpy(), P,
                                             scale=sc if sc > 0 else None)
    compare_attention(out.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, [P] * B)
