"""The C-ABI library loads, exports what include/bsa.h declares, and rejects
bad arguments on the host before anything reaches a GPU (CPU only).

Every call below fails host-side validation, so none of them launches a
kernel: they are safe with fake device pointers and without a GPU.
"""

import ctypes
import os
import re

import pytest

from block_sparse_attention_bsa_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load()


def declared_symbols():
    txt = open(os.path.join(ROOT, "include", "bsa.h")).read()
    return sorted(set(re.findall(r"BSA_API\s+[\w\s\*]+?\b(bsa_\w+)\s*\(", txt)))


def test_header_declares_the_expected_calls():
    assert declared_symbols() == sorted([
        "bsa_version", "bsa_get_last_error", "bsa_select_workspace_size", "bsa_select",
        "bsa_forward_workspace_size", "bsa_forward", "bsa_validate_indices", "bsa_device_status",
        "bsa_select_noalloc", "bsa_forward_causal", "bsa_select_rope",
        "bsa_backward_workspace_size", "bsa_backward", "bsa_debug_wait_probe",
    ])


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert set(declared_symbols()) == set(_lib.SIGNATURES)


def test_only_api_symbols_are_exported():
    build()
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.lib_path()], capture_output=True, text=True).stdout
    ours = sorted({l.split()[-1] for l in out.splitlines() if l.split() and l.split()[-1].startswith("bsa_")})
    assert ours == declared_symbols()


def test_version(lib):
    assert lib.bsa_version() == 100


FAKE = 0x10000   # 16-byte aligned, never dereferenced: every call below fails validation first


def T(B=1, S=512, H=4, D=128, sb=None, ss=None, sh=None, ptr=FAKE):
    sh = D if sh is None else sh
    ss = H * D if ss is None else ss
    sb = S * H * D if sb is None else sb
    return _lib.BsaTensor(ptr, B, S, H, D, sb, ss, sh)


def call_select(lib, q, k, prefix=0, lens=None, bq=256, bk=128, keep=(0.25,), n_keep=None,
                ind=FAKE, cnt=FAKE, ws=FAKE, ws_bytes=1 << 40):
    keep_arr = (ctypes.c_float * len(keep))(*keep)
    lens_arr = (ctypes.c_int32 * len(lens))(*lens) if lens is not None else None
    return lib.bsa_select(ctypes.byref(q) if q is not None else None, ctypes.byref(k), prefix, lens_arr,
                          bq, bk, keep_arr, len(keep) if n_keep is None else n_keep, ind, cnt, ws,
                          ws_bytes, None)


def call_forward(lib, q, k, v, prefix=0, lens=None, bq=256, bk=128, scale=0.0, out=FAKE, ws=None, ws_bytes=0):
    lens_arr = (ctypes.c_int32 * len(lens))(*lens) if lens is not None else None
    return lib.bsa_forward(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), None, None, prefix, lens_arr,
                           bq, bk, scale, out, None, ws, ws_bytes, None)


def err(lib):
    return lib.bsa_get_last_error().decode()


@pytest.mark.parametrize("case,status,needle", [
    ("null_q", 1, "q descriptor is NULL"),
    ("head_dim", 2, "head dim 96"),
    ("gqa", 1, "not a multiple of Hkv"),
    ("geometry", 2, "block geometry"),
    ("misaligned", 1, "16-byte aligned"),
    ("stride", 1, "multiples of 8"),
    ("seq_len", 1, "seq_lens[0]"),
    ("prefix_overflow", 1, "exceeds Skv"),
    ("neg_prefix", 1, "negative"),
    ("keep_range", 1, "outside [0, 1]"),
    ("n_keep", 1, "n_keep"),
    ("workspace_small", 3, "smaller than"),
    ("workspace_null", 3, "workspace is NULL"),
    ("workspace_align", 3, "256-byte aligned"),
    ("batch_mismatch", 1, "batch of q"),
])
def test_select_rejects_bad_arguments(lib, case, status, needle):
    q, k = T(H=4), T(H=2, S=512 + 256)
    kw = dict(prefix=256)
    if case == "null_q":
        q = None
    elif case == "head_dim":
        q, k = T(D=96), T(D=96, S=768)
    elif case == "gqa":
        q, k = T(H=3), T(H=2, S=768)
    elif case == "geometry":
        kw["bq"] = 96
    elif case == "misaligned":
        q = T(ptr=FAKE + 2)
    elif case == "stride":
        q = T(ss=4 * 128 + 4)
    elif case == "seq_len":
        kw["lens"] = [513]
    elif case == "prefix_overflow":
        kw["prefix"] = 300
    elif case == "neg_prefix":
        kw["prefix"] = -1
    elif case == "keep_range":
        kw["keep"] = (1.5,)
    elif case == "n_keep":
        kw["keep"] = (0.2, 0.3)
    elif case == "workspace_small":
        kw["ws_bytes"] = 16
    elif case == "workspace_null":
        kw["ws"] = None
    elif case == "workspace_align":
        kw["ws"] = FAKE + 16
    elif case == "batch_mismatch":
        k = T(B=2, H=2, S=768)
    st = call_select(lib, q, k, **kw)
    assert st == status, (case, st, err(lib))
    assert needle in err(lib), err(lib)


def test_select_workspace_size_formula(lib):
    # fp32 means of Q [B,Hq,nQb,d] and K [B,Hkv,nKb,d], each rounded up to 256 B
    B, Hq, Hkv, Sq, Skv, d, bq, bk = 1, 32, 8, 172800, 173824, 128, 256, 128
    want = ((B * Hq * 675 * d * 4 + 255) // 256) * 256 + ((B * Hkv * 1358 * d * 4 + 255) // 256) * 256
    assert lib.bsa_select_workspace_size(B, Hq, Hkv, Sq, Skv, d, bq, bk) == want
    assert lib.bsa_select_workspace_size(0, Hq, Hkv, Sq, Skv, d, bq, bk) == 0


@pytest.mark.parametrize("case,status,needle", [
    ("v_shape", 1, "v shape"),
    ("out_null", 1, "out is NULL"),
    ("out_align", 1, "out is not 16-byte aligned"),
    ("scale_nan", 1, "softmax_scale"),
    ("geometry", 2, "block geometry"),
])
def test_forward_rejects_bad_arguments(lib, case, status, needle):
    q, k, v = T(H=4), T(H=2, S=768), T(H=2, S=768)
    kw = dict(prefix=256)
    if case == "v_shape":
        v = T(H=2, S=700)
    elif case == "out_null":
        kw["out"] = None
    elif case == "out_align":
        kw["out"] = FAKE + 8
    elif case == "scale_nan":
        kw["scale"] = float("nan")
    elif case == "geometry":
        kw["bk"] = 256
    st = call_forward(lib, q, k, v, **kw)
    assert st == status, (case, st, err(lib))
    assert needle in err(lib), err(lib)


def test_forward_workspace_required(lib):
    q, k, v = T(H=4), T(H=2, S=768), T(H=2, S=768)
    need = lib.bsa_forward_workspace_size(1, 4, 512, 768, 256, 128)
    assert need == 256 + 256      # tile counter + group order (8 requests x 4 heads x 4 B, rounded)
    assert lib.bsa_forward_workspace_size(9, 4, 512, 768, 256, 128) == 2 * need   # two launch chunks of 8
    # 64-row query blocks: + merged lists [1, 4, 2 super-blocks, 12 key blocks + 3 padding entries]
    # int32, their counts and their class sizes (two int32 per row)
    m = lib.bsa_forward_workspace_size(1, 4, 512, 768, 64, 64)
    assert m == need + ((4 * 2 * 15 * 4 + 255) // 256) * 256 + 256 + 256
    st = call_forward(lib, q, k, v, prefix=256)
    assert st == 3 and "workspace is NULL" in err(lib)
    st = call_forward(lib, q, k, v, prefix=256, ws=FAKE, ws_bytes=need - 1)
    assert st == 3 and "smaller than" in err(lib)


def test_forward_counts_required_with_indices(lib):
    q, k, v = T(H=4), T(H=2, S=768), T(H=2, S=768)
    st = lib.bsa_forward(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), FAKE, None, 256, None, 256, 128,
                         0.0, FAKE, None, None, 0, None)
    assert st == 1 and "counts is NULL" in err(lib)


def test_validate_rejects_bad_sizes(lib):
    st = lib.bsa_validate_indices(FAKE, FAKE, 0, 4, 512, 768, 256, None, 256, 128, 1, FAKE, None)
    assert st == 1
    st = lib.bsa_validate_indices(None, FAKE, 1, 4, 512, 768, 256, None, 256, 128, 1, FAKE, None)
    assert st == 1


def test_python_binding_refuses_cpu_tensors():
    import torch
    import block_sparse_attention_bsa_gb300 as bsa
    q = torch.zeros(1, 256, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        bsa.bsa_select(q, q, 0, None, 64, 64, 0.5)
    with pytest.raises(ValueError, match="CUDA tensor"):
        bsa.bsa_forward(q, q, q, None, None, 0, None, 64, 64)


def test_binding_checks_caller_buffers_before_any_launch():
    """The C ABI sees bare pointers, so the binding checks every buffer a caller
    passes (shape, dtype, contiguity, device) on the host; a wrong one raises
    ValueError before anything is launched."""
    import torch
    from block_sparse_attention_bsa_gb300 import api
    dev = torch.device("cpu")
    good_i = torch.full((1, 4, 2, 6), -1, dtype=torch.int32)
    good_c = torch.zeros((1, 4, 2), dtype=torch.int32)
    i, c = api._lists(good_i, good_c, 1, 4, 2, 6, dev)
    assert i is good_i and c is good_c
    bad_lists = [torch.full((1, 4, 2, 5), -1, dtype=torch.int32),                 # row capacity short
                 good_i.to(torch.int64),                                           # wrong dtype
                 torch.full((1, 4, 6, 2), -1, dtype=torch.int32).transpose(2, 3)]  # not contiguous
    for bad in bad_lists:
        with pytest.raises(ValueError, match="indices"):
            api._lists(bad, good_c, 1, 4, 2, 6, dev)
    with pytest.raises(ValueError, match="counts"):
        api._lists(good_i, torch.zeros((1, 4, 3), dtype=torch.int32), 1, 4, 2, 6, dev)
    with pytest.raises(ValueError, match="q_out"):
        api._check_buffer("q_out", torch.zeros(1, 8, 4, 64, dtype=torch.float16), (1, 8, 4, 64), torch.bfloat16, dev)
    with pytest.raises(ValueError, match="on meta"):
        api._check_buffer("out", torch.zeros(1, 8, 4, 64, dtype=torch.bfloat16), (1, 8, 4, 64), torch.bfloat16,
                          torch.device("meta"))


def test_causal_rejects_bad_arguments(lib):
    q, k, v = T(H=4, S=512), T(H=2, S=400), T(H=2, S=400)
    st = lib.bsa_forward_causal(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), 256, 128, 0.0, FAKE, None,
                                None, 0, None)
    assert st == 1 and "exceeds Skv" in err(lib)          # understanding keys must cover P rows
    k, v = T(H=2, S=512), T(H=2, S=512)
    st = lib.bsa_forward_causal(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), 256, 128, 0.0, FAKE, None,
                                None, 0, None)
    assert st == 3 and "workspace is NULL" in err(lib)


def test_select_rope_rejects_missing_tables(lib):
    q, k = T(H=4), T(H=2, S=768)
    keep = (ctypes.c_float * 1)(0.25)
    st = lib.bsa_select_rope(ctypes.byref(q), ctypes.byref(k), None, FAKE, FAKE, FAKE, 256, None, 256, 128, keep, 1,
                             FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, None)
    assert st == 1 and "cos_q is NULL" in err(lib)
    st = lib.bsa_select_rope(ctypes.byref(q), ctypes.byref(k), FAKE, FAKE, FAKE + 4, FAKE, 256, None, 256, 128, keep, 1,
                             FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, None)
    assert st == 1 and "cos_k is not 16-byte aligned" in err(lib)
    st = lib.bsa_select_rope(ctypes.byref(q), ctypes.byref(k), FAKE, FAKE, FAKE, FAKE, 256, None, 96, 128, keep, 1,
                             FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, None)
    assert st == 2 and "block geometry" in err(lib)


def call_backward(lib, q, k, v, o=None, do=None, lse=FAKE, ind=FAKE, cnt=FAKE, prefix=0, lens=None, bq=256,
                  bk=128, scale=0.0, dq=FAKE, dk=FAKE, dv=FAKE, ws=FAKE, ws_bytes=1 << 40):
    o = q if o is None else o
    do = q if do is None else do
    lens_arr = (ctypes.c_int32 * len(lens))(*lens) if lens is not None else None
    return lib.bsa_backward(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.byref(o), ctypes.byref(do),
                            lse, ind, cnt, prefix, lens_arr, bq, bk, scale, dq, dk, dv, ws, ws_bytes, None)


@pytest.mark.parametrize("case,status,needle", [
    ("head_dim96", 2, "head dim 96"),
    ("block_q96", 2, "block geometry"),
    ("block_k256", 2, "block geometry"),
    ("dout_shape", 1, "dout shape"),
    ("out_shape", 1, "out shape"),
    ("no_indices", 1, "indices and counts are required"),
    ("no_lse", 1, "lse is NULL"),
    ("dq_null", 1, "must be non-NULL"),
    ("dk_align", 1, "16-byte aligned"),
    ("scale_inf", 1, "softmax_scale"),
    ("workspace_small", 3, "smaller than"),
])
def test_backward_rejects_bad_arguments(lib, case, status, needle):
    q, k, v = T(H=4), T(H=2, S=768), T(H=2, S=768)
    kw = dict(prefix=256)
    if case == "head_dim96":
        q, k, v = T(H=4, D=96), T(H=2, S=768, D=96), T(H=2, S=768, D=96)
    elif case == "block_q96":
        kw["bq"] = 96
    elif case == "block_k256":
        kw["bk"] = 256
    elif case == "dout_shape":
        kw["do"] = T(H=4, S=256)
    elif case == "out_shape":
        kw["o"] = T(H=2)
    elif case == "no_indices":
        kw["ind"] = None
    elif case == "no_lse":
        kw["lse"] = None
    elif case == "dq_null":
        kw["dq"] = None
    elif case == "dk_align":
        kw["dk"] = FAKE + 4
    elif case == "scale_inf":
        kw["scale"] = float("inf")
    elif case == "workspace_small":
        kw["ws_bytes"] = 1024
    st = call_backward(lib, q, k, v, **kw)
    assert st == status, (case, st, err(lib))
    assert needle in err(lib), err(lib)


def test_backward_workspace_size_formula(lib):
    # On 128 x 128 (query tile, key tile) pairs, each part rounded up to 256 B: per query tile 128
    # lse and 128 D values (fp32); 256 B of item counters; 4 mask bitmaps [B,Hkv,G*nQt,ceil(nKt/32)]
    # u32; dQ lists [B,Hq,nQt,nKt] + counts [B,Hq,nQt]; inverse counts [B,Hkv,nKt] and lists
    # [B,Hkv,nKt,G*nQt] int32.  The block geometry does not change the size.
    B, Hq, Hkv, Sq, Skv = 1, 32, 8, 172800, 173824
    r = lambda x: ((x + 255) // 256) * 256
    nQt, nKt, G = 1350, 1358, 4
    want = (r(B * Hq * nQt * 256 * 4) + 256 + r(4 * B * Hkv * G * nQt * 43 * 4) + r(B * Hq * nQt * nKt * 4)
            + r(B * Hq * nQt * 4) + r(B * Hkv * nKt * 4) + r(B * Hkv * nKt * G * nQt * 4))
    for bq, bk in ((256, 128), (64, 64), (128, 64)):
        assert lib.bsa_backward_workspace_size(B, Hq, Hkv, Sq, Skv, bq, bk) == want
    assert lib.bsa_backward_workspace_size(B, Hq, 5, Sq, Skv, 256, 128) == 0


def test_wait_probe_rejects_bad_arguments(lib):
    for fam, lim in ((2, 10 ** 8), (-1, 10 ** 8), (0, 999_999), (1, 10 ** 10 + 1)):
        st = lib.bsa_debug_wait_probe(fam, lim, None)
        assert st == 1, (fam, lim, st)                      # BSA_ERR_INVALID_ARG, nothing launched
        assert b"bsa_debug_wait_probe" in lib.bsa_get_last_error()


def test_product_package_never_touches_the_oracle():
    """The library and its binding import nothing from oracle/ (only the tests,
    the smoke check and the bench's CPU-baseline arm may)."""
    import subprocess
    import sys
    code = ("import sys, block_sparse_attention_bsa_gb300 as b; b.build(); "
            "from block_sparse_attention_bsa_gb300 import _lib; _lib.load(); "
            "print(any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules))")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip().splitlines()[-1] == "False"
    pkg = os.path.join(ROOT, "block_sparse_attention_bsa_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                assert "oracle" not in open(os.path.join(dirpath, f)).read(), f


def test_noalloc_reports_argument_errors_under_its_own_name(lib):
    """bsa_select_noalloc checks its arguments (under its own name) before it
    looks at the static scratch: an unsupported geometry is reported as such,
    not as a size problem."""
    q, k = T(H=4), T(H=2, S=768)
    keep = (ctypes.c_float * 1)(0.25)
    st = lib.bsa_select_noalloc(ctypes.byref(q), ctypes.byref(k), 256, None, 100, 128, keep, 1, FAKE, FAKE, None)
    assert st == 2 and err(lib).startswith("bsa_select_noalloc: block geometry")
    st = lib.bsa_select_noalloc(ctypes.byref(q), ctypes.byref(k), 256, None, 256, 128, keep, 1, None, FAKE, None)
    assert st == 1 and err(lib) == "bsa_select_noalloc: indices is NULL"
