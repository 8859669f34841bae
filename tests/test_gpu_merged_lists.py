"""The merged 256-row lists that bsa_forward builds for 64- and 128-row query
blocks, read back from the caller's forward workspace and compared entry by
entry (integers: bit-exact) with a host rebuild from the selector's lists.

Format (bsa.h, bsa_forward_workspace_size): after the per-launch tile
counters and group orders, int32 [B, Hq, ceil(Sq/256), nKb + 3] entries
(key block | membership bit of each original query block << 24), int32
counts and int32 (steps of the half-0-only class, steps of the half-1-only
class) per row.  A row holds, in steps of per_step entries (two 64-key
blocks or one 128-key block): the blocks both 128-row halves selected, then
the blocks only one half selected, one step of half 0 and one of half 1 in
turn while both classes last, then the rest of the longer one; each class
ascending, and a class whose size is not a multiple of per_step ends with a
padding entry (the block past the end, no membership bit).
"""

import numpy as np
import pytest
import torch

import block_sparse_attention_bsa_gb300 as bsa
from bsa_inputs import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


def expected_rows(idx, cnt, nKb, block_q, block_k):
    """Host rebuild of every merged row: (entries, count, (c0, c1))."""
    B, Hq, nQb, _ = idx.shape
    ratio = 256 // block_q
    per_half = ratio // 2
    S = 2 if block_k == 64 else 1
    nSb = -(-nQb // ratio)
    out = {}
    for b in range(B):
        for h in range(Hq):
            for sb in range(nSb):
                member = {}
                for g in range(ratio):
                    qb = sb * ratio + g
                    if qb >= nQb:
                        continue
                    for kb in idx[b, h, qb, :max(0, min(int(cnt[b, h, qb]), nKb))]:
                        if 0 <= kb < nKb:
                            member[int(kb)] = member.get(int(kb), 0) | (1 << g)
                lo = (1 << per_half) - 1
                classes = [[], [], []]
                for kb in sorted(member):
                    m = member[kb]
                    h0, h1 = bool(m & lo), bool(m & ~lo)
                    classes[0 if (h0 and h1) else (1 if h0 else 2)].append(kb | (m << 24))
                steps = [-(-len(c) // S) for c in classes]
                for c in range(3):                      # pad each class to whole steps
                    classes[c] += [nKb] * (steps[c] * S - len(classes[c]))
                m_ = min(steps[1], steps[2])
                row = list(classes[0])
                for k in range(max(steps[1], steps[2])):
                    for c in (1, 2):
                        if k < steps[c] and (k < m_ or steps[c] > m_):
                            row += classes[c][k * S:(k + 1) * S]
                out[(b, h, sb)] = (row, S * sum(steps), (steps[1], steps[2]))
    return out


@pytest.mark.parametrize("name", ["tiny", "small_64x64_d128", "small_mqa_d64", "small_mha_perhead"])
def test_merged_lists_match_host_rebuild(name):
    bsa.build()
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, "cuda", pad_fill=0.0)
    q, k, v = inp["q"], inp["k"], inp["v"]
    idx, cnt = bsa.bsa_select(q, k, cfg.prefix, inp["seq_lens"], cfg.block_q, cfg.block_k, inp["keep_ratio"])
    B, Sq, Hq = q.shape[0], q.shape[1], q.shape[2]
    Skv = k.shape[1]
    need = bsa.bsa_forward_workspace_size(B, Hq, Sq, Skv, cfg.block_q, cfg.block_k)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    bsa.bsa_forward(q, k, v, idx, cnt, cfg.prefix, inp["seq_lens"], cfg.block_q, cfg.block_k, workspace=ws)
    bsa.bsa_device_status()
    # layout: the launch chunks' counters and orders (the size bsa_forward needs
    # for 256-row query blocks), then the lists, counts and class sizes, each
    # starting on a 256-byte boundary
    al = lambda x: (x + 255) // 256 * 256
    base = bsa.bsa_forward_workspace_size(B, Hq, Sq, Skv, 256, 128)
    nKb = -(-Skv // cfg.block_k)
    nSb = -(-Sq // 256)
    rows, stride = B * Hq * nSb, nKb + 3
    raw = ws.cpu().numpy()
    ents = raw[base:base + rows * stride * 4].view(np.int32).reshape(B, Hq, nSb, stride)
    o = base + al(rows * stride * 4)
    counts = raw[o:o + rows * 4].view(np.int32).reshape(B, Hq, nSb)
    o += al(rows * 4)
    cls = raw[o:o + rows * 8].view(np.int32).reshape(B, Hq, nSb, 2)
    exp = expected_rows(idx.cpu().numpy(), cnt.cpu().numpy(), nKb, cfg.block_q, cfg.block_k)
    for (b, h, sb), (row, n, c) in exp.items():
        assert counts[b, h, sb] == n, (b, h, sb)
        assert tuple(cls[b, h, sb]) == c, (b, h, sb)
        assert list(ents[b, h, sb, :n]) == row, (b, h, sb)
