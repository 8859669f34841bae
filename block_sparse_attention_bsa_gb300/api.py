"""Python binding of libbsa: argument marshalling only.

Each function has the name of the C entry point it calls (include/bsa.h) and
turns torch tensors into pointers, sizes and strides.  Every step of the
selector and of the attention runs in the library's CUDA kernels; there is no
other path, and a missing library or a non-CUDA tensor raises.
"""

from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import torch

from . import _lib

BLOCK_Q_SUPPORTED = (64, 128, 256)
BLOCK_K_SUPPORTED = (64, 128)


class BsaError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        self.status_name = _lib.STATUS_NAMES.get(status, str(status))
        super().__init__(f"{self.status_name}: {message}")


def _check(status: int):
    if status != 0:
        msg = _lib.load().bsa_get_last_error().decode(errors="replace")
        raise BsaError(status, msg)


def _desc(t: torch.Tensor, name: str) -> _lib.BsaTensor:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be bfloat16 (got {t.dtype})")
    if t.dim() != 4:
        raise ValueError(f"{name} must be 4-D [B, S, H, d] (got {tuple(t.shape)})")
    if t.stride(3) != 1:
        raise ValueError(f"{name} must have a contiguous last dim")
    B, S, H, D = t.shape
    sb, ss, sh, _ = t.stride()
    return _lib.BsaTensor(t.data_ptr(), B, S, H, D, sb, ss, sh)


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _i32_array(vals: Optional[Sequence[int]]):
    if vals is None:
        return None
    return (ctypes.c_int32 * len(vals))(*[int(x) for x in vals])


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def _check_buffer(name: str, t, shape, dtype, device) -> None:
    """Raises ValueError unless ``t`` is a contiguous tensor of exactly
    ``shape`` and ``dtype`` on ``device``.  The C ABI receives bare pointers
    and cannot see a buffer's size, so every caller-passed input list and
    output buffer is checked here, before anything is launched."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if (t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous()
            or t.device != torch.device(device)):
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)} on {device} "
                         f"(got {t.dtype}, {tuple(t.shape)}, contiguous={t.is_contiguous()}, {t.device})")


def _lists(indices, counts, B, Hq, nQb, nKb, device):
    """Index/count buffers for a selector call: new ones (indices start at -1)
    or the caller's, checked."""
    if indices is None:
        indices = torch.full((B, Hq, nQb, nKb), -1, dtype=torch.int32, device=device)
    if counts is None:
        counts = torch.empty((B, Hq, nQb), dtype=torch.int32, device=device)
    _check_buffer("indices", indices, (B, Hq, nQb, nKb), torch.int32, device)
    _check_buffer("counts", counts, (B, Hq, nQb), torch.int32, device)
    return indices, counts


def bsa_version() -> int:
    return _lib.load().bsa_version()


def bsa_get_last_error() -> str:
    return _lib.load().bsa_get_last_error().decode(errors="replace")


def bsa_select_workspace_size(B, Hq, Hkv, Sq, Skv, d, block_q, block_k) -> int:
    return int(_lib.load().bsa_select_workspace_size(B, Hq, Hkv, Sq, Skv, d, block_q, block_k))


def bsa_forward_workspace_size(B, Hq, Sq, Skv, block_q, block_k) -> int:
    return int(_lib.load().bsa_forward_workspace_size(B, Hq, Sq, Skv, block_q, block_k))


def _workspace(nbytes: int, device, given: Optional[torch.Tensor]) -> Optional[torch.Tensor]:
    if nbytes == 0:
        return given
    if given is not None:
        return given
    # torch's allocator returns 512-byte aligned blocks
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def bsa_select(q: torch.Tensor, k: torch.Tensor, prefix_len: int, seq_lens: Optional[Sequence[int]],
               block_q: int, block_k: int, keep_ratio, *, indices: Optional[torch.Tensor] = None,
               counts: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
               stream=None):
    """Selected key blocks per (request, query head, query block).

    Returns ``(indices [B, Hq, nQb, nKb] int32, counts [B, Hq, nQb] int32)``;
    entries of ``indices`` past a row's count are not written (new buffers
    start at -1).  ``keep_ratio``: a float or a sequence of 1 or Hq floats.
    """
    qd, kd = _desc(q, "q"), _desc(k, "k")
    B, Sq, Hq, d = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    nQb, nKb = _cdiv(Sq, block_q), _cdiv(Skv, block_k)
    if isinstance(keep_ratio, (int, float)):
        keep_ratio = [float(keep_ratio)]
    keep = (ctypes.c_float * len(keep_ratio))(*[float(x) for x in keep_ratio])
    indices, counts = _lists(indices, counts, B, Hq, nQb, nKb, q.device)
    need = bsa_select_workspace_size(B, Hq, Hkv, Sq, Skv, d, block_q, block_k)
    ws = _workspace(need, q.device, workspace)
    lib = _lib.load()
    st = lib.bsa_select(ctypes.byref(qd), ctypes.byref(kd), int(prefix_len), _i32_array(seq_lens),
                        int(block_q), int(block_k), keep, len(keep_ratio), indices.data_ptr(),
                        counts.data_ptr(), ws.data_ptr() if ws is not None else None,
                        ws.numel() if ws is not None else 0, _stream_ptr(stream))
    _check(st)
    return indices, counts


def bsa_select_rope(q: torch.Tensor, k: torch.Tensor, cos_q: torch.Tensor, sin_q: torch.Tensor,
                    cos_k: torch.Tensor, sin_k: torch.Tensor, prefix_len: int, seq_lens: Optional[Sequence[int]],
                    block_q: int, block_k: int, keep_ratio, *, q_out: Optional[torch.Tensor] = None,
                    k_out: Optional[torch.Tensor] = None, indices: Optional[torch.Tensor] = None,
                    counts: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None, stream=None):
    """Rotary prologue fused with the selector: returns ``(q_out, k_out,
    indices, counts)``; q_out/k_out are the rotated bf16 tensors (contiguous)
    to pass to bsa_forward.  cos/sin: fp32 CUDA tensors [S, d]."""
    qd, kd = _desc(q, "q"), _desc(k, "k")
    B, Sq, Hq, d = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    nQb, nKb = _cdiv(Sq, block_q), _cdiv(Skv, block_k)
    for name, t, rows in (("cos_q", cos_q, Sq), ("sin_q", sin_q, Sq), ("cos_k", cos_k, Skv), ("sin_k", sin_k, Skv)):
        if t.dtype != torch.float32 or tuple(t.shape) != (rows, d) or not t.is_contiguous() or t.device != q.device:
            raise ValueError(f"{name} must be a contiguous fp32 tensor [{rows}, {d}] on {q.device}")
    if isinstance(keep_ratio, (int, float)):
        keep_ratio = [float(keep_ratio)]
    keep = (ctypes.c_float * len(keep_ratio))(*[float(x) for x in keep_ratio])
    q_out = torch.empty((B, Sq, Hq, d), dtype=torch.bfloat16, device=q.device) if q_out is None else q_out
    k_out = torch.empty((B, Skv, Hkv, d), dtype=torch.bfloat16, device=q.device) if k_out is None else k_out
    _check_buffer("q_out", q_out, (B, Sq, Hq, d), torch.bfloat16, q.device)
    _check_buffer("k_out", k_out, (B, Skv, Hkv, d), torch.bfloat16, q.device)
    indices, counts = _lists(indices, counts, B, Hq, nQb, nKb, q.device)
    need = bsa_select_workspace_size(B, Hq, Hkv, Sq, Skv, d, block_q, block_k)
    ws = _workspace(need, q.device, workspace)
    st = _lib.load().bsa_select_rope(ctypes.byref(qd), ctypes.byref(kd), cos_q.data_ptr(), sin_q.data_ptr(),
                                     cos_k.data_ptr(), sin_k.data_ptr(), int(prefix_len), _i32_array(seq_lens),
                                     int(block_q), int(block_k), keep, len(keep_ratio), q_out.data_ptr(),
                                     k_out.data_ptr(), indices.data_ptr(), counts.data_ptr(),
                                     ws.data_ptr() if ws is not None else None,
                                     ws.numel() if ws is not None else 0, _stream_ptr(stream))
    _check(st)
    return q_out, k_out, indices, counts


def bsa_select_noalloc(q: torch.Tensor, k: torch.Tensor, prefix_len: int, seq_lens: Optional[Sequence[int]],
                       block_q: int, block_k: int, keep_ratio, *, indices: Optional[torch.Tensor] = None,
                       counts: Optional[torch.Tensor] = None, stream=None):
    """bsa_select without caller workspace: the block means go to the
    library's static device scratch (for callers that cannot allocate device
    memory).  Same results; calls that overlap on the GPU race on the scratch."""
    qd, kd = _desc(q, "q"), _desc(k, "k")
    B, Sq, Hq, d = q.shape
    nQb, nKb = _cdiv(Sq, block_q), _cdiv(k.shape[1], block_k)
    if isinstance(keep_ratio, (int, float)):
        keep_ratio = [float(keep_ratio)]
    keep = (ctypes.c_float * len(keep_ratio))(*[float(x) for x in keep_ratio])
    indices, counts = _lists(indices, counts, B, Hq, nQb, nKb, q.device)
    st = _lib.load().bsa_select_noalloc(ctypes.byref(qd), ctypes.byref(kd), int(prefix_len),
                                        _i32_array(seq_lens), int(block_q), int(block_k), keep,
                                        len(keep_ratio), indices.data_ptr(), counts.data_ptr(),
                                        _stream_ptr(stream))
    _check(st)
    return indices, counts


def bsa_forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, indices: Optional[torch.Tensor],
                counts: Optional[torch.Tensor], prefix_len: int, seq_lens: Optional[Sequence[int]],
                block_q: int, block_k: int, softmax_scale: float = 0.0, *,
                out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                return_lse: bool = True, workspace: Optional[torch.Tensor] = None, stream=None):
    """Attention over the listed key blocks (``indices=None``: dense pass).

    Returns ``(out [B, Sq, Hq, d] bf16, lse [B, Hq, Sq] fp32 or None)``.
    """
    qd, kd, vd = _desc(q, "q"), _desc(k, "k"), _desc(v, "v")
    B, Sq, Hq, d = q.shape
    if out is None:
        out = torch.empty((B, Sq, Hq, d), dtype=torch.bfloat16, device=q.device)
    _check_buffer("out", out, (B, Sq, Hq, d), torch.bfloat16, q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_buffer("lse", lse, (B, Hq, Sq), torch.float32, q.device)
    if (indices is None) != (counts is None):
        raise ValueError("indices and counts are given together (both None: the dense pass)")
    if indices is not None:
        _check_buffer("indices", indices, (B, Hq, _cdiv(Sq, block_q), _cdiv(k.shape[1], block_k)), torch.int32,
                      q.device)
        _check_buffer("counts", counts, (B, Hq, _cdiv(Sq, block_q)), torch.int32, q.device)
    need = bsa_forward_workspace_size(B, Hq, Sq, k.shape[1], block_q, block_k)
    ws = _workspace(need, q.device, workspace)
    lib = _lib.load()
    st = lib.bsa_forward(ctypes.byref(qd), ctypes.byref(kd), ctypes.byref(vd),
                         indices.data_ptr() if indices is not None else None,
                         counts.data_ptr() if counts is not None else None,
                         int(prefix_len), _i32_array(seq_lens), int(block_q), int(block_k),
                         float(softmax_scale), out.data_ptr(),
                         lse.data_ptr() if lse is not None else None,
                         ws.data_ptr() if ws is not None else None,
                         ws.numel() if ws is not None else 0, _stream_ptr(stream))
    _check(st)
    return out, lse


def bsa_forward_causal(q_und: torch.Tensor, k: torch.Tensor, v: torch.Tensor, block_q: int, block_k: int,
                       softmax_scale: float = 0.0, *, out: Optional[torch.Tensor] = None,
                       lse: Optional[torch.Tensor] = None, return_lse: bool = True,
                       workspace: Optional[torch.Tensor] = None, stream=None):
    """Causal self-attention of the understanding stream: row i of ``q_und``
    ``[B, P, Hq, d]`` attends key rows 0..i of ``k``/``v`` (only their first P
    rows are read).  Returns ``(out [B, P, Hq, d], lse [B, Hq, P] or None)``."""
    qd, kd, vd = _desc(q_und, "q_und"), _desc(k, "k"), _desc(v, "v")
    B, P, Hq, d = q_und.shape
    if out is None:
        out = torch.empty((B, P, Hq, d), dtype=torch.bfloat16, device=q_und.device)
    _check_buffer("out", out, (B, P, Hq, d), torch.bfloat16, q_und.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, P), dtype=torch.float32, device=q_und.device)
    if lse is not None:
        _check_buffer("lse", lse, (B, Hq, P), torch.float32, q_und.device)
    need = bsa_forward_workspace_size(B, Hq, P, k.shape[1], block_q, block_k)
    ws = _workspace(need, q_und.device, workspace)
    st = _lib.load().bsa_forward_causal(ctypes.byref(qd), ctypes.byref(kd), ctypes.byref(vd), int(block_q),
                                        int(block_k), float(softmax_scale), out.data_ptr(),
                                        lse.data_ptr() if lse is not None else None,
                                        ws.data_ptr() if ws is not None else None,
                                        ws.numel() if ws is not None else 0, _stream_ptr(stream))
    _check(st)
    return out, lse


def bsa_backward_workspace_size(B, Hq, Hkv, Sq, Skv, block_q, block_k) -> int:
    return int(_lib.load().bsa_backward_workspace_size(B, Hq, Hkv, Sq, Skv, block_q, block_k))


def bsa_backward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor, dout: torch.Tensor,
                 lse: torch.Tensor, indices: torch.Tensor, counts: torch.Tensor, prefix_len: int,
                 seq_lens: Optional[Sequence[int]], block_q: int, block_k: int, softmax_scale: float = 0.0, *,
                 dq: Optional[torch.Tensor] = None, dk: Optional[torch.Tensor] = None,
                 dv: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None, stream=None):
    """Gradients of ``bsa_forward`` with respect to q, k and v, given the
    forward's ``out`` and ``lse`` and the upstream gradient ``dout``.

    Returns ``(dq [B, Sq, Hq, d], dk [B, Skv, Hkv, d], dv [B, Skv, Hkv, d])``, bf16.
    """
    qd, kd, vd = _desc(q, "q"), _desc(k, "k"), _desc(v, "v")
    od, dod = _desc(out, "out"), _desc(dout, "dout")
    B, Sq, Hq, d = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    if dq is None:
        dq = torch.empty((B, Sq, Hq, d), dtype=torch.bfloat16, device=q.device)
    if dk is None:
        dk = torch.empty((B, Skv, Hkv, d), dtype=torch.bfloat16, device=q.device)
    if dv is None:
        dv = torch.empty((B, Skv, Hkv, d), dtype=torch.bfloat16, device=q.device)
    for name, t, shape in (("dq", dq, (B, Sq, Hq, d)), ("dk", dk, (B, Skv, Hkv, d)), ("dv", dv, (B, Skv, Hkv, d))):
        _check_buffer(name, t, shape, torch.bfloat16, q.device)
    _check_buffer("lse", lse, (B, Hq, Sq), torch.float32, q.device)
    _check_buffer("indices", indices, (B, Hq, _cdiv(Sq, block_q), _cdiv(Skv, block_k)), torch.int32, q.device)
    _check_buffer("counts", counts, (B, Hq, _cdiv(Sq, block_q)), torch.int32, q.device)
    need = bsa_backward_workspace_size(B, Hq, Hkv, Sq, Skv, block_q, block_k)
    ws = _workspace(need, q.device, workspace)
    st = _lib.load().bsa_backward(ctypes.byref(qd), ctypes.byref(kd), ctypes.byref(vd), ctypes.byref(od),
                                  ctypes.byref(dod), lse.data_ptr(), indices.data_ptr(), counts.data_ptr(),
                                  int(prefix_len), _i32_array(seq_lens), int(block_q), int(block_k),
                                  float(softmax_scale), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                  ws.data_ptr() if ws is not None else None,
                                  ws.numel() if ws is not None else 0, _stream_ptr(stream))
    _check(st)
    return dq, dk, dv


def bsa_validate_indices(indices: torch.Tensor, counts: torch.Tensor, B: int, Hq: int, Sq: int, Skv: int,
                         prefix_len: int, seq_lens: Optional[Sequence[int]], block_q: int, block_k: int,
                         require_prefix: bool = True, stream=None) -> int:
    """Number of malformed rows (synchronises the stream to read it)."""
    bad = torch.zeros(1, dtype=torch.int32, device=indices.device)
    lib = _lib.load()
    st = lib.bsa_validate_indices(indices.data_ptr(), counts.data_ptr(), B, Hq, Sq, Skv, int(prefix_len),
                                  _i32_array(seq_lens), block_q, block_k, 1 if require_prefix else 0,
                                  bad.data_ptr(), _stream_ptr(stream))
    _check(st)
    return int(bad.item())


def bsa_device_status(stream=None) -> None:
    """Synchronises and raises BsaError if a bounded device wait gave up."""
    _check(_lib.load().bsa_device_status(_stream_ptr(stream)))


def bsa_debug_wait_probe(family: int, limit_ns: int, stream=None) -> None:
    """Enqueues a one-thread kernel whose bounded mbarrier wait (the kernels'
    wait code, limit ``limit_ns``) runs out on purpose, so that the next
    ``bsa_device_status`` raises a timeout; ``family`` 0 is the forward side,
    1 the backward kernels.  For testing the timeout reporting path."""
    _check(_lib.load().bsa_debug_wait_probe(int(family), int(limit_ns), _stream_ptr(stream)))
