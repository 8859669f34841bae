"""Failure detection on the GPU, without any fault, trap or hang: the
bounded-wait timeout path, and outputs written in bounds only.

A one-thread kernel waits, with the attention kernels' bounded-wait code and a
short limit, for an mbarrier phase that nothing completes.  The wait gives up,
records the timeout in the device error word of its kernel family and exits;
``bsa_device_status`` must report it once (BSA_ERR_TIMEOUT), clear it, and the
context must keep working: a select + forward + backward afterwards still
matches the fp64 oracle.  Output and workspace buffers placed between
sentinel margins must come back with the margins unchanged.  With BSA_DEBUG
set, malformed index lists given to the forward or the backward are reported
by ``bsa_device_status`` (BSA_ERR_INVALID_INDICES); without it they are
clamped and never read out of bounds.
"""

import time

import numpy as np
import pytest
import torch

import block_sparse_attention_bsa_gb300 as bsa
from bsa_inputs import CONFIGS, make_inputs
from oracle import bsa_oracle as O
from parity_utils import compare_attention, compare_selection, to_f32_np

pytestmark = pytest.mark.gpu

TIMEOUT_STATUS = 6        # BSA_ERR_TIMEOUT


@pytest.fixture(scope="module", autouse=True)
def built():
    bsa.build()


@pytest.mark.parametrize("family", [0, 1])
def test_wait_that_gives_up_is_reported_once(family):
    bsa.bsa_device_status()                               # start from a clean error word
    limit_ns = 200_000_000
    t0 = time.perf_counter()
    bsa.bsa_debug_wait_probe(family, limit_ns)
    with pytest.raises(bsa.BsaError) as e:
        bsa.bsa_device_status()
    elapsed = time.perf_counter() - t0
    assert e.value.status == TIMEOUT_STATUS, str(e.value)
    assert ("forward" if family == 0 else "backward") in str(e.value)
    assert elapsed >= 0.9 * limit_ns * 1e-9               # the wait ran to its limit
    bsa.bsa_device_status()                               # reported once, then cleared


def test_context_keeps_working_after_timeouts():
    bsa.bsa_debug_wait_probe(0, 20_000_000)
    bsa.bsa_debug_wait_probe(1, 20_000_000)
    with pytest.raises(bsa.BsaError) as e:
        bsa.bsa_device_status()
    assert e.value.status == TIMEOUT_STATUS and "forward and backward" in str(e.value)
    bsa.bsa_device_status()
    cfg = CONFIGS["small_gqa"]
    inp = make_inputs(cfg, "cpu", pad_fill=float("nan"))
    lens = inp["seq_lens"]
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    idx, cnt = bsa.bsa_select(q, k, cfg.prefix, lens, cfg.block_q, cfg.block_k, inp["keep_ratio"])
    bsa.bsa_device_status()
    ref = O.select_blocks(to_f32_np(inp["q"]), to_f32_np(inp["k"]), cfg.prefix, lens, cfg.block_q, cfg.block_k,
                          inp["keep_ratio"])
    compare_selection(idx.cpu().numpy(), cnt.cpu().numpy(), ref)
    ri, rc = ref["indices"].astype(np.int32), ref["counts"].astype(np.int32)
    ri_t, rc_t = torch.from_numpy(ri).cuda(), torch.from_numpy(rc).cuda()
    out, lse = bsa.bsa_forward(q, k, v, ri_t, rc_t, cfg.prefix, lens, cfg.block_q, cfg.block_k)
    dout = torch.randn(q.shape, generator=torch.Generator(device="cuda").manual_seed(3), device="cuda").bfloat16()
    dq, dk, dv = bsa.bsa_backward(q, k, v, out, dout, lse, ri_t, rc_t, cfg.prefix, lens, cfg.block_q, cfg.block_k)
    bsa.bsa_device_status()
    qf, kf, vf = (to_f32_np(inp[x]).astype(np.float64) for x in ("q", "k", "v"))
    o_ref, l_ref = O.attention(qf, kf, vf, ri, rc, cfg.prefix, lens, cfg.block_q, cfg.block_k)
    compare_attention(out.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, lens)
    for g in (dq, dk, dv):
        assert torch.isfinite(g.float()).all()


def _canary(shape, dtype, fill, pad=4096):
    """A view of `shape` in the middle of a buffer whose margins hold `fill`."""
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * pad,), fill, dtype=dtype, device="cuda")
    return buf, buf[pad:pad + n].view(shape), pad


@pytest.mark.parametrize("name", ["small_gqa", "small_64x64_d128"])
def test_outputs_and_workspaces_are_written_in_bounds_only(name):
    """Every output and workspace buffer sits between sentinel margins; after
    select, forward and backward the margins are unchanged."""
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, "cpu", pad_fill=0.0)
    lens = inp["seq_lens"]
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    B, Sq, Hq, d = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    nQb, nKb = -(-Sq // cfg.block_q), -(-Skv // cfg.block_k)
    u8 = torch.uint8
    bufs = []

    def make(shape, dtype, fill):
        buf, view, pad = _canary(shape, dtype, fill)
        bufs.append((buf, pad, view.numel(), fill))
        return view

    idx = make((B, Hq, nQb, nKb), torch.int32, 0x7EADBEEF)
    cnt = make((B, Hq, nQb), torch.int32, 0x7EADBEEF)
    sws = make((bsa.bsa_select_workspace_size(B, Hq, Hkv, Sq, Skv, d, cfg.block_q, cfg.block_k),), u8, 0xA5)
    out = make((B, Sq, Hq, d), torch.bfloat16, 1536.0)
    lse = make((B, Hq, Sq), torch.float32, 4321.0)
    fws = make((max(16, bsa.bsa_forward_workspace_size(B, Hq, Sq, Skv, cfg.block_q, cfg.block_k)),), u8, 0xA5)
    dq = make((B, Sq, Hq, d), torch.bfloat16, 1536.0)
    dk = make((B, Skv, Hkv, d), torch.bfloat16, 1536.0)
    dv = make((B, Skv, Hkv, d), torch.bfloat16, 1536.0)
    bws = make((bsa.bsa_backward_workspace_size(B, Hq, Hkv, Sq, Skv, cfg.block_q, cfg.block_k),), u8, 0xA5)
    bsa.bsa_select(q, k, cfg.prefix, lens, cfg.block_q, cfg.block_k, inp["keep_ratio"], indices=idx, counts=cnt,
                   workspace=sws)
    bsa.bsa_forward(q, k, v, idx, cnt, cfg.prefix, lens, cfg.block_q, cfg.block_k, out=out, lse=lse, workspace=fws)
    dout = torch.randn(q.shape, generator=torch.Generator(device="cuda").manual_seed(5), device="cuda").bfloat16()
    bsa.bsa_backward(q, k, v, out, dout, lse, idx, cnt, cfg.prefix, lens, cfg.block_q, cfg.block_k, dq=dq, dk=dk,
                     dv=dv, workspace=bws)
    bsa.bsa_device_status()
    for buf, pad, n, fill in bufs:
        assert (buf[:pad] == fill).all() and (buf[pad + n:] == fill).all(), (buf.dtype, n)
    assert torch.isfinite(out.float()).all() and torch.isfinite(dq.float()).all()


INVALID_INDICES_STATUS = 5   # BSA_ERR_INVALID_INDICES


@pytest.fixture
def debug_env(monkeypatch):
    monkeypatch.setenv("BSA_DEBUG", "1")


def _lists_with_defects(cfg, idx, cnt):
    """Two malformed rows: one out of order, one with a block past the request's keys."""
    bad = idx.clone()
    c0 = int(cnt[0, 0, 0])
    assert c0 >= 2
    bad[0, 0, 0, 0], bad[0, 0, 0, 1] = idx[0, 0, 0, 1], idx[0, 0, 0, 0]
    c1 = int(cnt[0, 1, 0])
    bad[0, 1, 0, c1 - 1] = -(-cfg.Skv // cfg.block_k) + 5
    return bad


def test_debug_validation_reports_malformed_lists(debug_env):
    cfg = CONFIGS["small_gqa"]
    inp = make_inputs(cfg, "cuda", pad_fill=0.0)
    q, k, v, lens = inp["q"], inp["k"], inp["v"], inp["seq_lens"]
    idx, cnt = bsa.bsa_select(q, k, cfg.prefix, lens, cfg.block_q, cfg.block_k, inp["keep_ratio"])
    out, lse = bsa.bsa_forward(q, k, v, idx, cnt, cfg.prefix, lens, cfg.block_q, cfg.block_k)
    bsa.bsa_device_status()                               # the selector's lists are well formed
    bad = _lists_with_defects(cfg, idx, cnt)
    bsa.bsa_forward(q, k, v, bad, cnt, cfg.prefix, lens, cfg.block_q, cfg.block_k)
    with pytest.raises(bsa.BsaError) as e:
        bsa.bsa_device_status()
    assert e.value.status == INVALID_INDICES_STATUS and str(e.value).startswith("BSA_ERR_INVALID_INDICES: 2 ")
    bsa.bsa_device_status()                               # reported once
    dout = torch.randn(q.shape, generator=torch.Generator(device="cuda").manual_seed(1), device="cuda").bfloat16()
    bsa.bsa_backward(q, k, v, out, dout, lse, bad, cnt, cfg.prefix, lens, cfg.block_q, cfg.block_k)
    with pytest.raises(bsa.BsaError) as e:
        bsa.bsa_device_status()
    assert e.value.status == INVALID_INDICES_STATUS


def test_without_debug_malformed_lists_are_clamped_silently(monkeypatch):
    monkeypatch.delenv("BSA_DEBUG", raising=False)
    cfg = CONFIGS["small_gqa"]
    inp = make_inputs(cfg, "cuda", pad_fill=0.0)
    q, k, v, lens = inp["q"], inp["k"], inp["v"], inp["seq_lens"]
    idx, cnt = bsa.bsa_select(q, k, cfg.prefix, lens, cfg.block_q, cfg.block_k, inp["keep_ratio"])
    bad = _lists_with_defects(cfg, idx, cnt)
    out, _ = bsa.bsa_forward(q, k, v, bad, cnt, cfg.prefix, lens, cfg.block_q, cfg.block_k)
    bsa.bsa_device_status()                               # no validation: no report, no fault
    assert torch.isfinite(out.float()).all()
