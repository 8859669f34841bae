"""The library's calls can be captured in a CUDA graph: with caller-provided
outputs and workspaces they only launch kernels (and one memset) on the given
stream, never synchronise or allocate.  A captured select + forward +
backward replays to the same bits as the eager calls, also after the inputs
are overwritten in place (the graph reads the buffers, not captured values).
"""

import pytest
import torch

import block_sparse_attention_bsa_gb300 as bsa
from bsa_inputs import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    bsa.build()


@pytest.mark.parametrize("name", ["small_gqa", "tiny"])
def test_select_forward_backward_replay_in_a_cuda_graph(name):
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, "cuda", pad_fill=0.0)
    q, k, v = inp["q"], inp["k"], inp["v"]
    lens, keep = inp["seq_lens"], inp["keep_ratio"]
    B, Sq, Hq, d = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    nQb, nKb = -(-Sq // cfg.block_q), -(-Skv // cfg.block_k)
    dev = q.device
    idx = torch.empty((B, Hq, nQb, nKb), dtype=torch.int32, device=dev)
    cnt = torch.empty((B, Hq, nQb), dtype=torch.int32, device=dev)
    sws = torch.empty(bsa.bsa_select_workspace_size(B, Hq, Hkv, Sq, Skv, d, cfg.block_q, cfg.block_k),
                      dtype=torch.uint8, device=dev)
    fws = torch.empty(max(256, bsa.bsa_forward_workspace_size(B, Hq, Sq, Skv, cfg.block_q, cfg.block_k)),
                      dtype=torch.uint8, device=dev)
    bws = torch.empty(bsa.bsa_backward_workspace_size(B, Hq, Hkv, Sq, Skv, cfg.block_q, cfg.block_k),
                      dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=dev)
    dout = torch.randn(q.shape, generator=torch.Generator(device=dev).manual_seed(7), device=dev).to(torch.bfloat16)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    stream = torch.cuda.Stream()

    def step():
        bsa.bsa_select(q, k, cfg.prefix, lens, cfg.block_q, cfg.block_k, keep, indices=idx, counts=cnt,
                       workspace=sws, stream=stream)
        bsa.bsa_forward(q, k, v, idx, cnt, cfg.prefix, lens, cfg.block_q, cfg.block_k, out=out, lse=lse,
                        workspace=fws, stream=stream)
        bsa.bsa_backward(q, k, v, out, dout, lse, idx, cnt, cfg.prefix, lens, cfg.block_q, cfg.block_k, dq=dq,
                         dk=dk, dv=dv, workspace=bws, stream=stream)

    with torch.cuda.stream(stream):
        step()                                   # eager (also sets the kernels' attributes once)
    stream.synchronize()
    bsa.bsa_device_status(stream)
    eager = [t.clone() for t in (idx, cnt, out, lse, dq, dk, dv)]
    for t in (out, lse, dq, dk, dv):
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    g.replay()
    torch.cuda.synchronize()
    bsa.bsa_device_status(stream)
    for a, b in zip(eager, (idx, cnt, out, lse, dq, dk, dv)):
        if a is eager[0]:                        # list entries past the count are unspecified
            continue
        assert torch.equal(a, b)
    for bb in range(B):
        for h in range(Hq):
            for qb in range(nQb):
                c = int(cnt[bb, h, qb])
                assert torch.equal(eager[0][bb, h, qb, :c], idx[bb, h, qb, :c])
    # new inputs in the same buffers: the replay recomputes from them
    q.mul_(-1)
    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    eager2 = [t.clone() for t in (out, lse, dq)]
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager2, (out, lse, dq)):
        assert torch.equal(a, b)
    assert not torch.equal(eager2[0], eager[2])
