"""The selector's tie rule on the GPU: among equal block scores the lower
block index wins (score descending, index ascending).  Key blocks that are
exact copies of each other have bitwise equal means, so their scores are
equal in fp32 on the GPU and in fp64 in the oracle alike.
"""

import numpy as np
import pytest
import torch

import block_sparse_attention_bsa_gb300 as bsa
from bsa_inputs.synthetic import Config, make_inputs
from oracle import bsa_oracle as O
from parity_utils import to_f32_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    bsa.build()


def select_both(cfg, k):
    inp = make_inputs(cfg, "cpu", pad_fill=0.0)
    q = inp["q"]
    idx, cnt = bsa.bsa_select(q.cuda(), k.cuda(), cfg.prefix, inp["seq_lens"], cfg.block_q, cfg.block_k,
                              inp["keep_ratio"])
    bsa.bsa_device_status()
    ref = O.select_blocks(to_f32_np(q), to_f32_np(k), cfg.prefix, inp["seq_lens"], cfg.block_q, cfg.block_k,
                          inp["keep_ratio"])
    return inp, idx.cpu().numpy(), cnt.cpu().numpy(), ref


@pytest.mark.parametrize("keep", [0.1, 0.37, 0.8])
def test_all_blocks_equal_pick_the_lowest_indices(keep):
    cfg = Config("ties_all", B=1, Hq=4, Hkv=2, d=128, prefix=256, lens=(2048,), block_q=256, block_k=128,
                 keep=keep, recipe="iid", seed=4001)
    inp = make_inputs(cfg, "cpu", pad_fill=0.0)
    k = inp["k"].clone()
    P = cfg.prefix
    for kb in range(1, (P + 2048) // 128):         # every generation key block = the first one
        if kb * 128 >= P:
            k[:, kb * 128:(kb + 1) * 128] = k[:, P:P + 128]
    _, gi, gc, ref = select_both(cfg, k)
    npb = P // 128
    N = (P + 2048) // 128 - npb
    kh = O.keep_count(inp["keep_ratio"][0], N)
    want = list(range(npb)) + list(range(npb, npb + kh))
    for h in range(cfg.Hq):
        for qb in range(gc.shape[2]):
            assert gc[0, h, qb] == npb + kh
            assert list(gi[0, h, qb, :npb + kh]) == want, (h, qb)
            assert list(ref["indices"][0, h, qb, :npb + kh]) == want


def test_duplicated_block_groups_follow_the_oracle_on_exact_ties():
    cfg = Config("ties_groups", B=2, Hq=6, Hkv=3, d=128, prefix=128, lens=(3000, 2500), block_q=256,
                 block_k=128, keep=0.3, recipe="iid", seed=4002)
    inp = make_inputs(cfg, "cpu", pad_fill=0.0)
    k = inp["k"].clone()
    rng = np.random.default_rng(4002)
    nkb = (cfg.prefix + 2500) // 128                 # blocks real in both requests
    for _ in range(6):                                 # groups of copies of one block
        src = int(rng.integers(1, nkb))
        for dst in rng.choice(np.arange(1, nkb), size=3, replace=False):
            k[:, int(dst) * 128:(int(dst) + 1) * 128] = k[:, src * 128:(src + 1) * 128]
    inp_, gi, gc, ref = select_both(cfg, k)
    assert (gc == ref["counts"]).all()
    exact_tie_rows = 0
    for b in range(cfg.B):
        for h in range(cfg.Hq):
            for qb in range(gc.shape[2]):
                c = int(gc[b, h, qb])
                if not ref["near_tie"][b, h, qb]:
                    assert (gi[b, h, qb, :c] == ref["indices"][b, h, qb, :c]).all(), (b, h, qb)
                    continue
                # a near-tie row whose boundary scores are exactly equal is decided by the
                # index rule alone, so it must match too
                sc = ref["scores"][b, h, qb]
                gap = O.boundary_gap(sc[~np.isnan(sc)], int(ref["k"][b, h]))
                if gap is not None and gap[0] == gap[1]:
                    exact_tie_rows += 1
                    assert (gi[b, h, qb, :c] == ref["indices"][b, h, qb, :c]).all(), (b, h, qb)
    print("rows decided by an exact tie at the boundary:", exact_tie_rows)
    assert exact_tie_rows > 0
