"""bsa_select_noalloc: the selector for callers that cannot allocate device
memory (a plugin whose host runtime owns every device allocation, or a
deployment with a fixed memory budget).  Its block means live in the
library's static device scratch instead of caller workspace.

Checked through the C ABI against bsa_select (workspace variant) on two
calls in a row with different problems, so the second call runs over the
first call's leftovers in the shared static array.  Index lists and counts
are integers: they must be identical.  This file is collected last on
purpose, so that a run stopping at the first failure has run everything else.
"""

import ctypes

import pytest
import torch

import block_sparse_attention_bsa_gb300 as bsa
from block_sparse_attention_bsa_gb300 import _lib
from bsa_inputs import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


def _desc(t):
    B, S, H, D = t.shape
    sb, ss, sh, _ = t.stride()
    return _lib.BsaTensor(t.data_ptr(), B, S, H, D, sb, ss, sh)


def _noalloc(lib, q, k, cfg, lens, keep, idx=None, cnt=None):
    nQb, nKb = -(-q.shape[1] // cfg.block_q), -(-k.shape[1] // cfg.block_k)
    if idx is None:
        idx = torch.full((q.shape[0], q.shape[2], nQb, nKb), -7, dtype=torch.int32, device="cuda")
    if cnt is None:
        cnt = torch.full((q.shape[0], q.shape[2], nQb), -7, dtype=torch.int32, device="cuda")
    qd, kd = _desc(q), _desc(k)
    keep_arr = (ctypes.c_float * len(keep))(*keep)
    lens_arr = (ctypes.c_int32 * len(lens))(*lens)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.bsa_select_noalloc(ctypes.byref(qd), ctypes.byref(kd), cfg.prefix, lens_arr, cfg.block_q,
                                cfg.block_k, keep_arr, len(keep), idx.data_ptr(), cnt.data_ptr(), stream)
    assert st == 0, lib.bsa_get_last_error().decode()
    return idx, cnt


@pytest.mark.parametrize("names", [("small_gqa", "1280x736_ragged"), ("480p_75", "tiny")])
def test_noalloc_select_matches_workspace_select_twice(names):
    bsa.build()
    lib = _lib.load()
    for name in names:
        cfg = CONFIGS[name]
        inp = make_inputs(cfg, "cuda", pad_fill=float("nan"))
        q, k = inp["q"], inp["k"]
        ref_idx, ref_cnt = bsa.bsa_select(q, k, cfg.prefix, inp["seq_lens"], cfg.block_q, cfg.block_k,
                                          inp["keep_ratio"])
        idx, cnt = _noalloc(lib, q, k, cfg, inp["seq_lens"], inp["keep_ratio"])
        bsa.bsa_device_status()
        assert torch.equal(cnt, ref_cnt), name
        for c in torch.unique(ref_cnt).tolist():
            rows = ref_cnt == c
            assert torch.equal(idx[rows][:, :c], ref_idx[rows][:, :c]), (name, c)


def test_noalloc_rejects_problems_above_the_static_scratch():
    bsa.build()
    lib = _lib.load()
    # 4 requests x 64 heads x 2048 query blocks x d128 fp32 means: far above 64 MiB.  The size
    # check runs before anything touches the (fake, never dereferenced) pointers.
    fake = 0x10000
    q = _lib.BsaTensor(fake, 4, 2048 * 64, 64, 128, 2048 * 64 * 64 * 128, 64 * 128, 128)
    k = _lib.BsaTensor(fake, 4, 2048 * 64, 64, 128, 2048 * 64 * 64 * 128, 64 * 128, 128)
    keep = (ctypes.c_float * 1)(0.25)
    st = lib.bsa_select_noalloc(ctypes.byref(q), ctypes.byref(k), 0, None, 64, 64, keep, 1, fake, fake, None)
    assert st == 2
    assert "static scratch" in lib.bsa_get_last_error().decode()


def test_noalloc_call_allocates_no_device_memory():
    """The defining property: once the first call on the device has looked up
    the scratch address, a call with the caller's buffers changes neither
    torch's allocator nor the device's free memory."""
    bsa.build()
    lib = _lib.load()
    cfg = CONFIGS["small_gqa"]
    inp = make_inputs(cfg, "cuda", pad_fill=float("nan"))
    q, k = inp["q"], inp["k"]
    idx, cnt = _noalloc(lib, q, k, cfg, inp["seq_lens"], inp["keep_ratio"])     # warm-up call
    # buffers for the second call exist before the measurement starts
    idx2, cnt2 = torch.full_like(idx, -7), torch.full_like(cnt, -7)
    torch.cuda.synchronize()
    allocated, free = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    _noalloc(lib, q, k, cfg, inp["seq_lens"], inp["keep_ratio"], idx=idx2, cnt=cnt2)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == allocated
    assert torch.cuda.mem_get_info()[0] == free
    bsa.bsa_device_status()
    assert torch.equal(cnt2, cnt) and torch.equal(idx2, idx)
