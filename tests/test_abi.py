"""The C-ABI library builds, loads, and exports every entry point include/sageattn.h declares;
host-side validation returns the documented status before anything touches a GPU."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sageattn.h")


@pytest.fixture(scope="module")
def lib():
    from quantized_attention_mean_gb300 import build as b
    b.build()
    from quantized_attention_mean_gb300 import _lib
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(sage_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_api():
    names = declared_functions()
    for required in ("sage_attn", "sage_attn_varlen", "sage_attn_workspace_size",
                     "sage_attn_varlen_workspace_size", "sage_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported_and_bound(lib):
    from quantized_attention_mean_gb300._lib import SIGNATURES
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in SIGNATURES, name


def test_status_strings(lib):
    for code in range(13):
        s = lib.sage_status_string(code).decode()
        assert s.startswith("SAGE_")
    assert lib.sage_status_string(99).decode() == "unknown sage_status"


def test_workspace_size(lib):
    n = lib.sage_attn_workspace_size(2, 8, 8, 4096, 4096, 128, 1)
    # at least the INT8-in-fp16 codes of Q and K plus the E4M3 V^T
    assert n >= 2 * 8 * 4096 * 128 * (2 + 2 + 1)
    assert lib.sage_attn_workspace_size(1, 2, 2, 256, 256, 200, 1) == 0
    assert lib.sage_attn_workspace_size(1, 2, 2, 256, 256, 64, 7) == 0
    assert lib.sage_attn_varlen_workspace_size(16, 32, 32, 70000, 70000, 128, 1) > 0


def _call(lib, **over):
    from quantized_attention_mean_gb300._lib import SageTensor
    fake = 0x10000  # never dereferenced: validation fails or stops before any launch
    t = SageTensor(fake, (ctypes.c_int64 * 3)(2 * 256 * 64, 256 * 64, 64))
    a = dict(batch=1, hq=2, hkv=2, nq=256, nk=256, d=64, dtype=0, layout=0, causal=0, scale=0.0,
             lse=0, gran=1, acc=0, sk=1, sv=0, ws=fake * 16, wsb=1 << 40)
    a.update(over)
    return lib.sage_attn(ctypes.byref(t), ctypes.byref(t), ctypes.byref(t), ctypes.byref(t), None,
                         a["batch"], a["hq"], a["hkv"], a["nq"], a["nk"], a["d"], a["dtype"],
                         a["layout"], a["causal"], a["scale"], a["lse"], a["gran"], a["acc"],
                         a["sk"], a["sv"], ctypes.c_void_p(a["ws"]), a["wsb"], None)


def test_host_validation_statuses(lib):
    assert _call(lib, d=200) == 2          # SAGE_ERR_HEAD_DIM
    assert _call(lib, d=0) == 2
    assert _call(lib, dtype=4) == 3        # SAGE_ERR_DTYPE
    assert _call(lib, hq=3, hkv=2) == 5    # SAGE_ERR_GQA
    assert _call(lib, acc=3) == 8          # SAGE_ERR_UNSUPPORTED (pure fp16 accumulation)
    assert _call(lib, gran=5) == 1         # SAGE_ERR_INVALID_ARG
    assert _call(lib, layout=2) == 1
    assert _call(lib, lse=1) == 1          # return_lse without an lse buffer
    assert _call(lib, nk=0) == 1           # softmax over no keys
    assert _call(lib, nq=0) == 0           # empty query set: no-op
    assert _call(lib, batch=0) == 0
    assert _call(lib, wsb=16) == 6         # SAGE_ERR_WORKSPACE
    assert _call(lib, ws=0x10000 + 8) == 6 # misaligned workspace


def test_null_tensor_is_invalid(lib):
    assert lib.sage_attn(None, None, None, None, None, 1, 2, 2, 8, 8, 64, 0, 0, 0, 0.0, 0, 1, 0,
                         1, 0, None, 0, None) == 1


def test_merge_partials_host_validation(lib):
    from quantized_attention_mean_gb300._lib import SageTensor
    fake = 0x10000  # never dereferenced: validation fails before any launch
    t = SageTensor(fake, (ctypes.c_int64 * 3)(8 * 4 * 64, 4 * 64, 64))
    views = (SageTensor * 2)(t, t)
    lses = (ctypes.c_void_p * 2)(fake, fake)
    args = dict(outs=ctypes.cast(views, ctypes.c_void_p), lses=ctypes.cast(lses, ctypes.c_void_p),
                n=2, out=ctypes.byref(t), lse=ctypes.c_void_p(fake), B=1, H=2, N=3, d=64, dtype=0,
                layout=0)

    def call(**over):
        a = dict(args, **over)
        return lib.sage_merge_partials(a["outs"], a["lses"], a["n"], a["out"], a["lse"], a["B"],
                                       a["H"], a["N"], a["d"], a["dtype"], a["layout"], None)
    assert call(n=0) == 1
    assert call(n=17) == 1
    assert call(layout=5) == 1
    assert call(dtype=9) == 3
    assert call(d=129) == 2
    assert call(d=0) == 2
    assert call(B=0) == 0            # empty problem: nothing launched
    bad = SageTensor(fake + 1, (ctypes.c_int64 * 3)(64, 64, 64))
    assert call(out=ctypes.byref(bad)) == 4
    neg = SageTensor(fake, (ctypes.c_int64 * 3)(-64, 64, 64))
    assert call(out=ctypes.byref(neg)) == 4


def _varlen(lib, **over):
    from quantized_attention_mean_gb300._lib import SagePacked
    fake = 0x10000  # never dereferenced: validation fails or stops before any launch
    a = dict(qdata=fake, st=2 * 64, sh=64, cuq=fake, cuk=fake, batch=2, maxq=100, maxk=100,
             tq=150, tk=150, hq=2, hkv=2, d=64, dtype=0, causal=0, scale=0.0, lse=0, gran=1,
             acc=0, sk=1, sv=0, ws=fake * 16, wsb=1 << 40)
    a.update(over)
    t = SagePacked(a["qdata"], a["st"], a["sh"])
    ok = SagePacked(fake, 2 * 64, 64)
    return lib.sage_attn_varlen(ctypes.byref(t), ctypes.byref(ok), ctypes.byref(ok), ctypes.byref(ok),
                                None, ctypes.c_void_p(a["cuq"]), ctypes.c_void_p(a["cuk"]), a["batch"],
                                a["maxq"], a["maxk"], a["tq"], a["tk"], a["hq"], a["hkv"], a["d"],
                                a["dtype"], a["causal"], a["scale"], a["lse"], a["gran"], a["acc"],
                                a["sk"], a["sv"], ctypes.c_void_p(a["ws"]), a["wsb"], None)


def test_varlen_host_validation_statuses(lib):
    assert _varlen(lib, cuq=0) == 1               # null cu_seqlens_q
    assert _varlen(lib, cuk=0) == 1               # null cu_seqlens_k
    assert _varlen(lib, cuq=0x10000 + 2) == 1     # cu_seqlens not 4-byte aligned
    assert _varlen(lib, d=200) == 2               # SAGE_ERR_HEAD_DIM
    assert _varlen(lib, hq=3) == 5                # SAGE_ERR_GQA
    assert _varlen(lib, batch=-1) == 1
    assert _varlen(lib, tq=0) == 0                # no query tokens: no-op
    assert _varlen(lib, batch=0) == 0
    assert _varlen(lib, tk=0) == 1                # queries but no keys
    assert _varlen(lib, maxk=0) == 1
    assert _varlen(lib, qdata=0) == 1             # null tensor data
    assert _varlen(lib, qdata=0x10001) == 4       # SAGE_ERR_STRIDE: odd address
    assert _varlen(lib, st=-128) == 4             # negative token stride
    assert _varlen(lib, wsb=16) == 6              # SAGE_ERR_WORKSPACE
    assert _varlen(lib, lse=1) == 1               # return_lse without an lse buffer


def test_pv16_entry_host_validation(lib):
    from quantized_attention_mean_gb300._lib import SageTensor
    fake = 0x10000
    t = SageTensor(fake, (ctypes.c_int64 * 3)(2 * 256 * 64, 256 * 64, 64))

    def call(hq=2, hkv=2, d=64, wsb=1 << 40):
        return lib.sage_attn_qk_int8_pv_fp16(ctypes.byref(t), ctypes.byref(t), ctypes.byref(t),
                                             ctypes.byref(t), None, 1, hq, hkv, 256, 256, d, 0, 0, 0,
                                             0.0, 0, 1, 0, 1, 0, ctypes.c_void_p(fake * 16), wsb, None)
    assert call(d=129) == 2
    assert call(hq=3) == 5
    assert call(wsb=16) == 6


def test_dense_stride_statuses(lib):
    from quantized_attention_mean_gb300._lib import SageTensor
    fake = 0x10000
    good = SageTensor(fake, (ctypes.c_int64 * 3)(2 * 256 * 64, 256 * 64, 64))
    odd = SageTensor(fake + 1, (ctypes.c_int64 * 3)(2 * 256 * 64, 256 * 64, 64))
    neg = SageTensor(fake, (ctypes.c_int64 * 3)(2 * 256 * 64, -256 * 64, 64))
    for bad in (odd, neg):
        for pos in range(4):
            ts = [good] * 4
            ts[pos] = bad
            st = lib.sage_attn(*(ctypes.byref(x) for x in ts), None, 1, 2, 2, 256, 256, 64, 0, 0, 0,
                               0.0, 0, 1, 0, 1, 0, ctypes.c_void_p(fake * 16), 1 << 40, None)
            assert st == 4, (pos, st)                 # SAGE_ERR_STRIDE
