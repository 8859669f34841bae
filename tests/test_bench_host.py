"""Host logic of bench.py (CPU): the FLOP and byte counts that the reported
TFLOP/s and roofline fractions divide by, the schedules' call counts, the
replica aggregation, the traffic lookup's source check and the verdicts of
the line's parity comparison."""

import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from bsa_inputs import CONFIGS, make_inputs  # noqa: E402
from oracle import bsa_oracle as O  # noqa: E402


def small_lists(name):
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, "cpu", pad_fill=0.0)
    sel = O.select_blocks(inp["q"].float().numpy(), inp["k"].float().numpy(), cfg.prefix, inp["seq_lens"],
                          cfg.block_q, cfg.block_k, inp["keep_ratio"])
    return cfg, inp["seq_lens"], sel["indices"], sel["counts"]


@pytest.mark.parametrize("name", ["small_gqa", "small_mqa_d64", "tiny"])
def test_exact_pair_flops_count_real_rows_and_keys(name):
    """4 d per (real query row, real listed key): counted key by key here."""
    cfg, lens, idx, cnt = small_lists(name)
    pairs = 0
    for b, L in enumerate(lens):
        real_keys = np.arange(cfg.prefix + L)
        for h in range(cfg.Hq):
            for qb in range(cnt.shape[2]):
                rows = len(range(qb * cfg.block_q, min((qb + 1) * cfg.block_q, L)))
                listed = set()
                for kb in idx[b, h, qb, :cnt[b, h, qb]]:
                    listed.update(range(kb * cfg.block_k, (kb + 1) * cfg.block_k))
                pairs += rows * len(listed.intersection(real_keys.tolist()))
    got = bench.valid_pair_flops(cnt, idx, lens, cfg.prefix, cfg.d, cfg.block_q, cfg.block_k)
    assert got == 4.0 * cfg.d * pairs
    # the tile-granular count is an upper bound that includes padded rows and keys
    assert bench.tile_flops(cnt, cfg.d, cfg.block_q, cfg.block_k) >= got


def test_tile_flops_and_algorithmic_bytes_of_the_720p_workload():
    """720p, keep 25 %: 21,600 work tiles x 346 listed blocks; every byte counted once."""
    cfg = CONFIGS["720p_75"]
    nQb = -(-cfg.Sq // cfg.block_q)
    assert (nQb, cfg.Hq) == (675, 32)
    counts = np.full((1, cfg.Hq, nQb), 346)
    assert bench.tile_flops(counts, cfg.d, cfg.block_q, cfg.block_k) == 4 * 128 * 256 * 128 * 21_600 * 346
    q_o = 2 * 172_800 * 32 * 128 * 2               # Q read, O written (bf16)
    kv = 2 * 173_824 * 8 * 128 * 2                 # K and V read (bf16)
    lse = 4 * 32 * 172_800                         # fp32 LSE written
    lists = 4 * 21_600 * 346                       # int32 list entries read
    assert bench.algorithmic_bytes(cfg, counts) == q_o + kv + lse + lists == 3_595_151_104


def test_replicas_aggregate_the_slowest_rank():
    assert bench.whole_job_tflops(1e12, 1, 1000.0) == pytest.approx(1.0)
    assert bench.whole_job_tflops(125.0e12, 4, 100.0) == pytest.approx(5000.0)


@pytest.mark.parametrize("name,arm,dense,sparse", [
    ("cosmos3", "dense", 35 * 36, 0),
    ("cosmos3", "mixed", 10 * 36 + 25 * 8, 25 * 28),      # 10 dense steps, then 28 of 36 layers sparse
    ("cosmos3", "all_sparse", 0, 35 * 36),
    ("h3", "dense", 50 * 48, 0),
    ("h3", "mixed", 20 * 48, 30 * 48),                    # the first 20 of 50 iterations dense
])
def test_schedule_arms_call_counts(name, arm, dense, sparse):
    sch = bench.SCHEDULES[name]
    is_dense = sch["arms"][arm]
    calls = [is_dense(s, l) for s in range(sch["steps"]) for l in range(sch["layers"])]
    assert sum(calls) == dense and len(calls) - sum(calls) == sparse


def test_traffic_is_reported_only_for_the_captured_sources(monkeypatch):
    cfg = CONFIGS["720p_75"]
    counts = np.zeros((1, 1, 1))
    monkeypatch.setitem(bench.FMHA_TRAFFIC, "sha", bench.fmha_source_sha())
    val, src = bench.fmha_traffic(cfg, counts)
    assert val == float(bench.FMHA_TRAFFIC["720p_75"]) and "ncu capture" in src
    assert bench.fmha_traffic(CONFIGS["tiny"], counts)[0] is None          # never captured
    monkeypatch.setitem(bench.FMHA_TRAFFIC, "sha", "0" * 16)
    val, src = bench.fmha_traffic(cfg, counts)
    assert val is None and "changed" in src


def test_bench_parity_verdicts_catch_planted_defects():
    """The CPU-baseline leg's comparison: the oracle's own bf16-stored results
    pass; a swapped list entry and a shifted output tile each fail."""
    import torch
    cfg = CONFIGS["small_gqa"]
    inp = make_inputs(cfg, "cpu", pad_fill=0.0)
    q, k, v = (inp[x].float().numpy().astype(np.float64) for x in ("q", "k", "v"))
    sel = O.select_blocks(inp["q"].float().numpy(), inp["k"].float().numpy(), cfg.prefix, inp["seq_lens"],
                          cfg.block_q, cfg.block_k, inp["keep_ratio"])
    idx = torch.from_numpy(sel["indices"].astype(np.int32))
    cnt = torch.from_numpy(sel["counts"].astype(np.int32))
    o, l = O.attention(q, k, v, sel["indices"], sel["counts"], cfg.prefix, inp["seq_lens"], cfg.block_q,
                       cfg.block_k)
    out = torch.from_numpy(np.nan_to_num(o)).bfloat16()
    lse = torch.from_numpy(np.where(np.isnan(l), -np.inf, l)).float()
    good = bench.cpu_baseline(inp, idx, cnt, out, lse, n_tiles_sample=64, budget_s=10, tiny=False)["parity"]
    assert good["selection"]["ok"] and good["attention"]["ok"], good
    bad_idx = idx.clone()
    bad_idx[0, 0, 1, 2], bad_idx[0, 0, 1, 3] = idx[0, 0, 1, 3], idx[0, 0, 1, 2]
    bad_out = out.clone()
    bad_out[0, :10, 0, :] += 0.5
    bad = bench.cpu_baseline(inp, bad_idx, cnt, bad_out, lse, n_tiles_sample=64, budget_s=10, tiny=False)["parity"]
    assert not bad["selection"]["ok"] and bad["selection"]["list_mismatches_outside_near_ties"] == 1
    assert not bad["attention"]["ok"]


def test_dense_tiles_and_schedule_arms():
    """Dense work counts every real query block against every key block with a
    real key; a schedule's attention time is its call counts x call times."""
    cfg = CONFIGS["480p_dense"]
    # 189 query blocks x 382 key blocks x 24 heads (the last blocks ragged)
    assert bench.dense_tiles(cfg.lens, cfg.prefix, cfg.Hq, cfg.block_q, cfg.block_k) == 189 * 382 * 24
    r = CONFIGS["1280x736_ragged"]
    assert bench.dense_tiles(r.lens, r.prefix, r.Hq, 256, 128) == (690 * 1384 + 586 * 1176) * 24
    arms = bench.schedule_arms("cosmos3", 4.0, 1.0)["arms"]
    assert arms["dense"]["attention_s"] == pytest.approx(35 * 36 * 4.0 / 1e3)
    assert arms["all_sparse"]["speedup_vs_dense"] == pytest.approx(4.0)
    mixed = (10 * 36 + 25 * 8) * 4.0 + 25 * 28 * 1.0
    assert arms["mixed"]["speedup_vs_dense"] == pytest.approx(35 * 36 * 4.0 / mixed)


def test_tiny_oracle_timing_runs_in_child_processes():
    t = bench.tiny_oracle_timing()
    assert t["one_core"]["threads"] == 1 and t["one_core"]["seconds"] > 0
    assert t["all_cores"]["threads"] == (os.cpu_count() or 1) and t["all_cores"]["tflops"] > 0


def test_workload_config_replaces_the_generation_length():
    assert bench.workload_config("720p_75") is CONFIGS["720p_75"]
    c = bench.workload_config("720p_75", 75000)
    assert c.name == "720p_75_L75000" and c.lens == (75000,)
    assert (c.Hq, c.Hkv, c.d, c.prefix, c.block_q, c.block_k) == (32, 8, 128, 1024, 256, 128)
    F, Y, X = c.grid
    assert (Y, X) == (45, 80) and F * Y * X >= 75000 > (F - 1) * Y * X
    inp = make_inputs(bench.workload_config("small_gqa", 500), "cpu")   # grid large enough for the recipe
    assert inp["q"].shape[1] == 500 and list(inp["seq_lens"]) == [500, 500]
    # a length that is not captured reports no traffic figure
    assert bench.fmha_traffic(c, np.zeros(1))[0] is None


def test_code_hash_ignores_comments_but_not_code():
    src = 'int f(int x) { // note\n  return x + 1; /* more */ }\nconst char* s = "// kept";\n'
    assert bench.strip_c_comments(src) == 'int f(int x) { \n  return x + 1;  }\nconst char* s = "// kept";\n'
    n = lambda x: " ".join(bench.strip_c_comments(x).split())
    assert n(src) == n(src.replace("// note", "// another note\n// and a line"))
    assert n(src) != n(src.replace("x + 1", "x + 2"))
