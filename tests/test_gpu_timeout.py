"""The bounded-wait timeout path on the GPU, without any fault, trap or hang.

A one-thread kernel waits, with the attention kernels' bounded-wait code and a
short limit, for an mbarrier phase that nothing completes.  The wait gives up,
records the timeout in the device error word of its kernel family and exits;
``bsa_device_status`` must report it once (BSA_ERR_TIMEOUT), clear it, and the
context must keep working: a select + forward + backward afterwards still
matches the fp64 oracle.
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
