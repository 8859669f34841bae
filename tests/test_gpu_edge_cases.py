"""Degenerate inputs through the CUDA selector, forward and backward, each
against the fp64 oracle on the same bits: an empty request in a batch, a
sequence shorter than one query block, keep ratio 0 with a protected prefix
(the lists hold the prefix blocks only), a prefix that is not a multiple of
the key block with ragged lengths, and batches of more requests than one
launch takes (8).  Inputs of the forward and backward
come from the oracle (its selection, its forward), never from the CUDA path.
"""

import numpy as np
import pytest
import torch

import block_sparse_attention_bsa_gb300 as bsa
from bsa_inputs.synthetic import Config, make_inputs
from oracle import bsa_oracle as O
from parity_utils import compare_attention, compare_selection, to_f32_np

pytestmark = pytest.mark.gpu

CASES = {
    "empty_request": Config("empty_request", B=2, Hq=4, Hkv=2, d=128, prefix=128, lens=(0, 300), block_q=256,
                            block_k=128, keep=0.5, recipe="iid", seed=3001),
    "short_d64_64x64": Config("short_d64_64x64", B=1, Hq=2, Hkv=1, d=64, prefix=0, lens=(37,), block_q=64,
                              block_k=64, keep=1.0, recipe="iid", seed=3002),
    "keep0_prefix": Config("keep0_prefix", B=1, Hq=3, Hkv=3, d=128, prefix=256, lens=(700,), block_q=128,
                           block_k=128, keep=0.0, recipe="iid", seed=3003),
    "odd_prefix_ragged": Config("odd_prefix_ragged", B=3, Hq=4, Hkv=1, d=64, prefix=100, lens=(333, 64, 1),
                                block_q=64, block_k=64, keep=0.35, recipe="iid", seed=3004),
    # more requests than one forward/backward launch takes (8): two launches
    "batch_11_two_launches": Config("batch_11_two_launches", B=11, Hq=4, Hkv=2, d=64, prefix=64,
                                    lens=(300, 0, 17, 256, 129, 1, 64, 200, 90, 333, 5), block_q=256,
                                    block_k=128, keep=0.4, recipe="iid", seed=3005),
    "batch_10_64x64": Config("batch_10_64x64", B=10, Hq=2, Hkv=1, d=128, prefix=100,
                             lens=(130, 64, 0, 1, 250, 65, 190, 7, 128, 99), block_q=64, block_k=64, keep=0.3,
                             recipe="iid", seed=3006),
    # head dim 128 with 128-key blocks (the CTA-pair kernel) over two launches
    "batch_9_pairs": Config("batch_9_pairs", B=9, Hq=4, Hkv=2, d=128, prefix=128,
                            lens=(520, 0, 1, 257, 256, 33, 700, 128, 255), block_q=256, block_k=128, keep=0.4,
                            recipe="iid", seed=3007),
}


@pytest.fixture(scope="module", autouse=True)
def built():
    bsa.build()


@pytest.mark.parametrize("name", list(CASES))
def test_edge_case_select_forward_backward(name):
    cfg = CASES[name]
    inp = make_inputs(cfg, "cpu", pad_fill=float("nan"))
    lens = inp["seq_lens"]
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    # selector against the oracle's selection
    idx, cnt = bsa.bsa_select(q, k, cfg.prefix, lens, cfg.block_q, cfg.block_k, inp["keep_ratio"])
    bsa.bsa_device_status()
    qf, kf, vf = (to_f32_np(inp[x]).astype(np.float64) for x in ("q", "k", "v"))
    ref = O.select_blocks(to_f32_np(inp["q"]), to_f32_np(inp["k"]), cfg.prefix, lens, cfg.block_q, cfg.block_k,
                          inp["keep_ratio"])
    compare_selection(idx.cpu().numpy(), cnt.cpu().numpy(), ref)
    if cfg.keep == 0.0:
        npb = O.kv_geometry(cfg.prefix, lens[0], cfg.block_k)["n_prefix_blocks"]
        assert (ref["counts"][0] == npb).all()
    # forward over the oracle's lists
    ri, rc = ref["indices"].astype(np.int32), ref["counts"].astype(np.int32)
    ri_t, rc_t = torch.from_numpy(ri).cuda(), torch.from_numpy(rc).cuda()
    out, lse = bsa.bsa_forward(q, k, v, ri_t, rc_t, cfg.prefix, lens, cfg.block_q, cfg.block_k)
    bsa.bsa_device_status()
    o_ref, l_ref = O.attention(qf, kf, vf, ri, rc, cfg.prefix, lens, cfg.block_q, cfg.block_k)
    on, ln = out.float().cpu().numpy(), lse.cpu().numpy()
    for b, L in enumerate(lens):                  # padded rows: exactly 0 and -inf
        assert (on[b, L:] == 0).all() and np.isneginf(ln[b, :, L:]).all()
    if any(L > 0 for L in lens):
        compare_attention(on, ln, o_ref, l_ref, lens)
    # backward on the oracle's forward (as stored: bf16 out, fp32 lse) and a seeded dout
    out_bf = torch.from_numpy(np.nan_to_num(o_ref, nan=0.0)).to(torch.bfloat16)
    lse32 = torch.from_numpy(np.where(np.isnan(l_ref), -np.inf, l_ref)).to(torch.float32)
    dout = torch.randn(inp["q"].shape, generator=torch.Generator().manual_seed(cfg.seed + 11)).to(torch.bfloat16)
    for b, L in enumerate(lens):
        dout[b, L:] = float("nan")                # padded rows are never read
    dq, dk, dv = bsa.bsa_backward(q, k, v, out_bf.cuda(), dout.cuda(), lse32.cuda(), ri_t, rc_t, cfg.prefix, lens,
                                  cfg.block_q, cfg.block_k)
    bsa.bsa_device_status()
    dq_r, dk_r, dv_r = O.attention_backward(qf, kf, vf, to_f32_np(out_bf), np.nan_to_num(to_f32_np(dout)),
                                            lse32.numpy(), ri, rc, cfg.prefix, lens, cfg.block_q, cfg.block_k)
    for name_, g, r in (("dq", dq, dq_r), ("dk", dk, dk_r), ("dv", dv, dv_r)):
        gn = g.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(gn).all(), name_
        nr = np.linalg.norm(r)
        if nr == 0:
            # exact zero (e.g. a row whose only key gets P = 1, so dS = dP - D = 0): the GPU
            # forms dP (MMA) and D (its own fp32 sum) in different orders, rounding-level values
            assert np.abs(gn).max() <= 1e-4, name_
        else:
            assert np.linalg.norm(gn - r) / nr <= 1e-2, (name_, np.linalg.norm(gn - r) / nr)
            assert np.abs(gn - r).max() <= 3e-2 * np.abs(r).max(), name_
    # an empty request has no gradient anywhere (no query row attends its keys)
    for b, L in enumerate(lens):
        if L == 0:
            assert (dq[b].float() == 0).all() and (dk[b].float() == 0).all() and (dv[b].float() == 0).all()
