"""The C ABI without a GPU: the library loads, exports what include/fa.h
declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

import exact_attention_54_gb300 as fa
from exact_attention_54_gb300 import build as fabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")

OK, NULL, SHAPE, HEADDIM, DTYPE, ALIGN, SPLITS, SCALE = 0, -1, -2, -3, -4, -5, -6, -7


@pytest.fixture(scope="module")
def lib():
    fabuild.build()
    return fa.load_library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^FA_API\s+[\w\s\*]+?\b(fa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fa_fwd", "fa_fwd_varlen", "fa_decode_splitkv", "fa_splitkv_merge", "fa_check_device_error",
              "fa_status_string", "fa_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(fa.EXPORTED_SYMBOLS) <= set(declared_functions())


def test_only_the_abi_is_exported(lib):
    out = os.popen(f"nm -D --defined-only {fa.library_path()}").read()
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported == set(declared_functions()), exported


def test_status_strings_and_version(lib):
    for code in range(-13, 1):
        s = fa.fa_status_string(code)
        assert s and s != "unknown status"
    assert fa.fa_status_string(-1234) == "unknown status"
    assert lib.fa_version() == 200


# Fake device addresses: validation must fail before any of them is used.
A = 0x10000
MIS = 0x10008  # 8-byte aligned only


def _fwd(lib, q=A, k=A, v=A, o=A, lse=A, B=1, H=1, Sq=128, Sk=128, D=64, causal=0, scale=0.125, dtype=0):
    return lib.fa_fwd(q, k, v, o, lse, B, H, Sq, Sk, D, causal, scale, dtype, None)


def test_fwd_validation(lib):
    assert _fwd(lib, q=None) == NULL
    assert _fwd(lib, lse=None) == NULL
    assert _fwd(lib, dtype=2) == DTYPE
    assert _fwd(lib, D=96) == HEADDIM
    for d in (384, 768, 2048):  # Split-D serves 512 and 1024 only
        assert _fwd(lib, D=d) == HEADDIM, d
    for kw in ({"B": 0}, {"H": 0}, {"Sq": 0}, {"Sk": 0}, {"Sq": -5}, {"Sk": (1 << 30) + 1}):
        assert _fwd(lib, **kw) == SHAPE, kw
    assert _fwd(lib, B=1 << 16, H=1 << 16) == SHAPE  # B*H overflows 32-bit work indexing
    for s in (0.0, -1.0, float("inf"), float("nan")):
        assert _fwd(lib, scale=s) == SCALE
    assert _fwd(lib, q=MIS) == ALIGN
    assert _fwd(lib, o=MIS) == ALIGN
    assert _fwd(lib, lse=A + 2) == ALIGN


def _varlen(lib, q=A, k=A, v=A, o=A, lse=A, cq=A, ck=A, n=2, tq=10, tk=10, mx=8, H=2, D=128, causal=1,
            scale=0.1, dtype=1):
    return lib.fa_fwd_varlen(q, k, v, o, lse, cq, ck, n, tq, tk, mx, H, D, causal, scale, dtype, None)


def test_varlen_validation(lib):
    assert _varlen(lib, cq=None) == NULL
    assert _varlen(lib, ck=None) == NULL
    assert _varlen(lib, dtype=-1) == DTYPE
    assert _varlen(lib, D=32) == HEADDIM
    for kw in ({"n": 0}, {"tq": 0}, {"tk": 0}, {"mx": 0}, {"H": 0}):
        assert _varlen(lib, **kw) == SHAPE, kw
    assert _varlen(lib, scale=-0.5) == SCALE
    assert _varlen(lib, k=MIS) == ALIGN


def _split(lib, q=A, k=A, v=A, op=A, mp=A, lp=A, B=2, H=2, Sk=100, D=128, S=32, scale=0.1, dtype=1):
    return lib.fa_decode_splitkv(q, k, v, op, mp, lp, B, H, Sk, D, S, scale, dtype, None)


def test_decode_validation(lib):
    assert _split(lib, op=None) == NULL
    assert _split(lib, dtype=5) == DTYPE
    assert _split(lib, D=80) == HEADDIM
    assert _split(lib, Sk=0) == SHAPE
    assert _split(lib, S=0) == SPLITS
    assert _split(lib, S=101) == SPLITS  # more partitions than keys
    assert _split(lib, Sk=5000, S=1025) == SPLITS
    assert _split(lib, scale=0.0) == SCALE
    assert _split(lib, v=MIS) == ALIGN
    assert _split(lib, mp=A + 2) == ALIGN


def _paged(lib, q=A, kc=A, vc=A, bt=A, sl=A, op=A, mp=A, lp=A, B=2, H=2, D=128, nb=64, bs=16, mb=8, S=4,
           scale=0.1, dtype=1):
    return lib.fa_decode_paged_splitkv(q, kc, vc, bt, sl, op, mp, lp, B, H, D, nb, bs, mb, S, scale, dtype, None)


def test_paged_validation(lib):
    import ctypes as C
    vp, i, f = C.c_void_p, C.c_int, C.c_float
    lib.fa_decode_paged_splitkv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp]
    assert _paged(lib, bt=None) == NULL
    assert _paged(lib, sl=None) == NULL
    assert _paged(lib, dtype=3) == DTYPE
    assert _paged(lib, D=32) == HEADDIM
    for kw in ({"B": 0}, {"H": 0}, {"nb": 0}, {"mb": 0}, {"bs": 0}, {"bs": 24}, {"bs": 2048}):
        assert _paged(lib, **kw) == SHAPE, kw
    assert _paged(lib, S=0) == SPLITS
    assert _paged(lib, S=1025) == SPLITS
    assert _paged(lib, scale=float("nan")) == SCALE
    assert _paged(lib, kc=MIS) == ALIGN
    assert _paged(lib, bt=A + 2) == ALIGN


def _fused(lib, q=A, k=A, v=A, o=A, lse=A, op=A, mp=A, lp=A, cnt=A, B=2, H=2, Sk=100, D=128, S=32, scale=0.1,
           dtype=1):
    return lib.fa_decode_splitkv_fused(q, k, v, o, lse, op, mp, lp, cnt, B, H, Sk, D, S, scale, dtype, None)


def test_fused_decode_validation(lib):
    for kw in ("q", "o", "lse", "op", "cnt"):
        assert _fused(lib, **{kw: None}) == NULL, kw
    assert _fused(lib, dtype=4) == DTYPE
    assert _fused(lib, D=96) == HEADDIM
    assert _fused(lib, Sk=0) == SHAPE
    assert _fused(lib, S=0) == SPLITS
    assert _fused(lib, S=101) == SPLITS
    assert _fused(lib, scale=-1.0) == SCALE
    assert _fused(lib, o=MIS) == ALIGN
    assert _fused(lib, cnt=A + 2) == ALIGN
    assert _fused(lib, lse=A + 1) == ALIGN


def _paged_fused(lib, q=A, kc=A, vc=A, bt=A, sl=A, o=A, lse=A, op=A, mp=A, lp=A, cnt=A, B=2, H=2, D=128, nb=64, bs=16,
                 mb=8, S=4, scale=0.1, dtype=1):
    return lib.fa_decode_paged_splitkv_fused(q, kc, vc, bt, sl, o, lse, op, mp, lp, cnt, B, H, D, nb, bs, mb, S, scale,
                                             dtype, None)


def test_paged_fused_validation(lib):
    for kw in ("bt", "sl", "o", "lse", "cnt"):
        assert _paged_fused(lib, **{kw: None}) == NULL, kw
    assert _paged_fused(lib, dtype=2) == DTYPE
    assert _paged_fused(lib, D=256) == HEADDIM
    for kw in ({"nb": 0}, {"bs": 12}, {"mb": 0}):
        assert _paged_fused(lib, **kw) == SHAPE, kw
    assert _paged_fused(lib, S=2000) == SPLITS
    assert _paged_fused(lib, scale=float("inf")) == SCALE
    assert _paged_fused(lib, o=MIS) == ALIGN
    assert _paged_fused(lib, cnt=A + 1) == ALIGN


def _bwd(lib, q=A, k=A, v=A, o=A, do=A, lse=A, dq=A, dk=A, dv=A, ws=A, wsb=1 << 30, B=1, H=2, Sq=200, Sk=300,
         D=128, causal=1, scale=0.1, dtype=1):
    return lib.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, wsb, B, H, Sq, Sk, D, causal, scale, dtype, None)


def test_bwd_validation(lib):
    for kw in ("q", "o", "do", "lse", "dq", "dk", "dv", "ws"):
        assert _bwd(lib, **{kw: None}) == NULL, kw
    assert _bwd(lib, dtype=3) == DTYPE
    assert _bwd(lib, D=256) == HEADDIM
    for kw in ({"B": 0}, {"H": 0}, {"Sq": 0}, {"Sk": 0}):
        assert _bwd(lib, **kw) == SHAPE, kw
    assert _bwd(lib, scale=0.0) == SCALE
    assert _bwd(lib, dq=MIS) == ALIGN
    assert _bwd(lib, ws=MIS) == ALIGN
    need = lib.fa_bwd_workspace_bytes(1, 2, 200, 128)
    assert need == 4 * (2 * 200 * 128 + 2 * 2 * 256) + 16
    assert _bwd(lib, wsb=need - 4) == -12
    assert lib.fa_bwd_workspace_bytes(1, 2, 200, 96) == 0


def _bwd_varlen(lib, q=A, k=A, v=A, o=A, do=A, lse=A, dq=A, dk=A, dv=A, ws=A, wsb=1 << 30, cq=A, ck=A, nseq=3,
                Tq=500, Tk=600, mq=300, mk=320, H=2, D=128, causal=1, scale=0.1, dtype=1):
    return lib.fa_bwd_varlen(q, k, v, o, do, lse, dq, dk, dv, ws, wsb, cq, ck, nseq, Tq, Tk, mq, mk, H, D, causal,
                             scale, dtype, None)


def test_bwd_varlen_validation(lib):
    for kw in ("q", "k", "v", "o", "do", "lse", "dq", "dk", "dv", "ws", "cq", "ck"):
        assert _bwd_varlen(lib, **{kw: None}) == NULL, kw
    assert _bwd_varlen(lib, dtype=2) == DTYPE
    assert _bwd_varlen(lib, D=256) == HEADDIM
    for kw in ({"nseq": 0}, {"Tq": 0}, {"Tk": 0}, {"mq": 0}, {"mk": 0}, {"H": 0}, {"Tq": (1 << 30) + 1},
               {"nseq": 1 << 20, "H": 1 << 12}):
        assert _bwd_varlen(lib, **kw) == SHAPE, kw
    assert _bwd_varlen(lib, scale=-1.0) == SCALE
    for kw in ("q", "dk", "ws"):
        assert _bwd_varlen(lib, **{kw: MIS}) == ALIGN, kw
    assert _bwd_varlen(lib, cq=A + 2) == ALIGN
    need = lib.fa_bwd_varlen_workspace_bytes(500, 2, 128)
    assert need == 4 * (500 * 2 * 128 + 2 * 2 * 500) + 16
    assert _bwd_varlen(lib, wsb=need - 4) == -12
    assert lib.fa_bwd_varlen_workspace_bytes(500, 2, 80) == 0


def test_merge_validation(lib):
    m = lib.fa_splitkv_merge
    assert m(None, A, A, A, A, 2, 2, 128, 8, 1, None) == NULL
    assert m(A, A, A, A, A, 2, 2, 128, 8, 7, None) == DTYPE
    assert m(A, A, A, A, A, 2, 2, 100, 8, 1, None) == HEADDIM
    assert m(A, A, A, A, A, 0, 2, 128, 8, 1, None) == SHAPE
    assert m(A, A, A, A, A, 2, 2, 128, 0, 1, None) == SPLITS
    assert m(A, A, A, MIS, A, 2, 2, 128, 8, 1, None) == ALIGN


def test_withhold_setting_validation(lib):
    """The failure-path test setting takes no negative load and resets with (0, 0)."""
    assert lib.fa_test_withhold_load(-1, 0) == SHAPE
    assert lib.fa_test_withhold_load(0, 0) == 0


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        fa.load_library(os.path.join(tmp_path, "missing.so"))


def test_selftest_library_exports(lib):
    st = ctypes.CDLL(fabuild.SELFTEST_LIB)
    for n in ("fa_selftest_qk", "fa_selftest_pv", "fa_selftest_tn", "fa_selftest_ldmax", "fa_selftest_watchdog",
              "fa_selftest_empty_launch"):
        assert hasattr(st, n)
