"""The C ABI without a GPU: the library loads, exports every declared entry point,
and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

from exact_tiled_attention_fattn_gb300 import build as fbuild
from exact_tiled_attention_fattn_gb300 import fattn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fattn.h")

A = 0x100000  # a 16-byte aligned fake device address (never dereferenced: calls fail validation first)


@pytest.fixture(scope="module")
def lib():
    fbuild.build()
    return fattn.load_library()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fattn_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert names == sorted(fattn.SIGNATURES), "binding signatures must mirror include/fattn.h"
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == {"fattn_fwd", "fattn_fwd_block_sparse", "fattn_fwd_masked", "fattn_fwd_fp8",
                          "fattn_fwd_paged", "fattn_bwd",
                          "fattn_bwd_workspace_size", "fattn_decode_workspace_size",
                          "fattn_decode_paged",
                          "fattn_decode_paged_static", "fattn_merge_partials", "fattn_status_string",
                          "fattn_debug_read_status", "fattn_debug_set_wait_limit"}


def test_status_strings(lib):
    for code in range(7):
        s = lib.fattn_status_string(code)
        assert s and s.decode() != "unknown status"
    assert lib.fattn_status_string(99).decode() == "unknown status"


def _fwd(lib, q=A, k=A, v=A, o=A, lse=A, B=1, Hq=4, Hkv=2, N=128, d=128, causal=1, scale=0.1, cu=None, T=0,
         dtype=fattn.FATTN_BF16):
    return lib.fattn_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, causal, scale, cu, T, dtype, None)


def test_fwd_validation(lib):
    E = fattn
    assert _fwd(lib, q=None) == E.FATTN_ERR_INVALID_ARG
    assert _fwd(lib, o=None) == E.FATTN_ERR_INVALID_ARG
    assert _fwd(lib, Hq=3, Hkv=2) == E.FATTN_ERR_INVALID_ARG
    assert _fwd(lib, N=-1) == E.FATTN_ERR_INVALID_ARG
    assert _fwd(lib, B=-1) == E.FATTN_ERR_INVALID_ARG
    assert _fwd(lib, Hkv=0) == E.FATTN_ERR_INVALID_ARG
    assert _fwd(lib, q=A + 8) == E.FATTN_ERR_INVALID_ARG              # misaligned
    assert _fwd(lib, v=A + 2) == E.FATTN_ERR_INVALID_ARG
    assert _fwd(lib, lse=A + 2) == E.FATTN_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("nan")) == E.FATTN_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("inf")) == E.FATTN_ERR_INVALID_ARG
    assert _fwd(lib, dtype=7) == E.FATTN_ERR_INVALID_ARG
    assert _fwd(lib, d=96) == E.FATTN_ERR_UNSUPPORTED
    assert _fwd(lib, d=256) == E.FATTN_ERR_UNSUPPORTED
    assert _fwd(lib, T=-5, cu=A) == E.FATTN_ERR_INVALID_ARG
    # empty problems are valid and launch nothing
    assert _fwd(lib, B=0) == E.FATTN_OK
    assert _fwd(lib, N=0) == E.FATTN_OK
    assert _fwd(lib, cu=A, T=0, N=16) == E.FATTN_OK
    assert _fwd(lib, B=0, q=None, k=None, v=None, o=None) == E.FATTN_OK   # empty tensors carry no pointer


def _dec(lib, q=A, kc=A, vc=A, bt=A, sl=A, S=4, o=A, lse=A, B=2, Hq=8, Hkv=2, d=128, ps=16, maxp=8, pages=16,
         scale=0.1, ws=A, wsb=None):
    if wsb is None:
        wsb = lib.fattn_decode_workspace_size(B, Hq, d, S)
    return lib.fattn_decode_paged(q, kc, vc, bt, sl, S, o, lse, B, Hq, Hkv, d, ps, maxp, pages, scale, ws, wsb, None)


def test_decode_validation(lib):
    E = fattn
    assert _dec(lib, q=None) == E.FATTN_ERR_INVALID_ARG
    assert _dec(lib, bt=None) == E.FATTN_ERR_INVALID_ARG
    assert _dec(lib, S=0) == E.FATTN_ERR_INVALID_ARG
    assert _dec(lib, Hq=6, Hkv=4) == E.FATTN_ERR_INVALID_ARG
    assert _dec(lib, ps=0) == E.FATTN_ERR_INVALID_ARG
    assert _dec(lib, pages=0) == E.FATTN_ERR_INVALID_ARG
    assert _dec(lib, kc=A + 4) == E.FATTN_ERR_INVALID_ARG
    assert _dec(lib, bt=A + 2) == E.FATTN_ERR_INVALID_ARG
    assert _dec(lib, scale=float("nan")) == E.FATTN_ERR_INVALID_ARG
    assert _dec(lib, d=80) == E.FATTN_ERR_UNSUPPORTED
    assert _dec(lib, ws=None) == E.FATTN_ERR_WORKSPACE
    assert _dec(lib, wsb=lib.fattn_decode_workspace_size(2, 8, 128, 4) - 1) == E.FATTN_ERR_WORKSPACE
    assert _dec(lib, ws=A + 16) == E.FATTN_ERR_WORKSPACE                # workspace must be 256-byte aligned


def test_workspace_size_arithmetic(lib):
    B, Hq, d, S = 8, 32, 128, 64
    rows = B * Hq * S
    expect = (rows * 4 + 255) // 256 * 256 + (rows * d * 4 + 255) // 256 * 256 + ((1 + B * Hq) * 4 + 255) // 256 * 256
    assert lib.fattn_decode_workspace_size(B, Hq, d, S) == expect
    assert lib.fattn_decode_workspace_size(0, Hq, d, S) == 0
    assert lib.fattn_decode_workspace_size(B, Hq, d, 0) == 0


def test_merge_validation(lib):
    E = fattn
    f = lib.fattn_merge_partials
    assert f(None, A, A, A, 2, 4, 3, 128, E.FATTN_BF16, None) == E.FATTN_ERR_INVALID_ARG
    assert f(A, A, A, A, 0, 4, 3, 128, E.FATTN_BF16, None) == E.FATTN_ERR_INVALID_ARG
    assert f(A, A, A, A, 2, 4, 0, 128, E.FATTN_BF16, None) == E.FATTN_ERR_INVALID_ARG
    assert f(A + 4, A, A, A, 2, 4, 3, 128, E.FATTN_BF16, None) == E.FATTN_ERR_INVALID_ARG
    assert f(A, A, A, A, 2, 4, 3, 128, 5, None) == E.FATTN_ERR_INVALID_ARG
    assert f(A, A, A, A, 2, 4, 3, 6, E.FATTN_BF16, None) == E.FATTN_ERR_UNSUPPORTED
    assert f(A, A, A, A, 2, 4, 3, 1024, E.FATTN_FP32, None) == E.FATTN_ERR_UNSUPPORTED


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(fattn, "_lib", None)
    with pytest.raises(RuntimeError, match="libfattn.so not found"):
        fattn.load_library(str(tmp_path / "nope.so"))


def test_block_sparse_validation(lib):
    E = fattn
    f = lambda **kw: lib.fattn_fwd_block_sparse(kw.get("q", A), A, A, A, A, kw.get("B", 1), kw.get("Hq", 4), 2,
                                                kw.get("N", 256), kw.get("d", 128), 1, 0.1, kw.get("m", A),
                                                kw.get("mh", 1), None)
    assert f(m=None) == E.FATTN_ERR_INVALID_ARG
    assert f(mh=2) == E.FATTN_ERR_INVALID_ARG          # neither 1 nor Hq
    assert f(q=A + 8) == E.FATTN_ERR_INVALID_ARG
    assert f(d=80) == E.FATTN_ERR_UNSUPPORTED
    assert f(N=2048 * 128 + 1) == E.FATTN_ERR_UNSUPPORTED  # mask rows longer than 2048 blocks
    assert f(B=0, q=None, m=None) == E.FATTN_OK          # empty problem


def test_paged_prefill_validation(lib):
    E = fattn

    def f(**kw):
        g = lambda n, dflt: kw.get(n, dflt)
        return lib.fattn_fwd_paged(g("q", A), g("kc", A), A, g("bt", A), A, A, A, None, g("B", 2), g("Hq", 4),
                                   g("Hkv", 2), g("d", 128), g("P", 16), g("maxp", 8), g("pages", 64),
                                   g("Tq", 100), g("maxq", 64), 1, 0.1, None)
    assert f(bt=None) == E.FATTN_ERR_INVALID_ARG
    assert f(kc=A + 4) == E.FATTN_ERR_INVALID_ARG
    assert f(Hkv=3) == E.FATTN_ERR_INVALID_ARG
    assert f(pages=0) == E.FATTN_ERR_INVALID_ARG
    assert f(d=96) == E.FATTN_ERR_UNSUPPORTED
    assert f(P=8) == E.FATTN_ERR_UNSUPPORTED and f(P=48) == E.FATTN_ERR_UNSUPPORTED
    assert f(pages=(1 << 31) // 16) == E.FATTN_ERR_UNSUPPORTED    # pool rows past int32
    assert f(Tq=0, q=None, bt=None) == E.FATTN_OK                  # empty problem


def test_backward_validation(lib):
    E = fattn
    assert lib.fattn_bwd_workspace_size(2, 4, 300) == 2 * 2 * 4 * 384 * 4
    assert lib.fattn_bwd_workspace_size(0, 4, 300) == 0

    def f(**kw):
        g = lambda n, dflt: kw.get(n, dflt)
        return lib.fattn_bwd(g("q", A), A, A, A, A, A, A, A, A, g("B", 2), g("Hq", 4), g("Hkv", 2), g("N", 300),
                             g("d", 128), 1, 0.1, g("ws", A), g("wsb", 1 << 20), None)
    assert f(q=None) == E.FATTN_ERR_INVALID_ARG
    assert f(Hkv=3) == E.FATTN_ERR_INVALID_ARG
    assert f(d=96) == E.FATTN_ERR_UNSUPPORTED
    assert f(ws=None) == E.FATTN_ERR_WORKSPACE
    assert f(wsb=100) == E.FATTN_ERR_WORKSPACE
    assert f(ws=A + 16) == E.FATTN_ERR_WORKSPACE
    assert f(B=0, q=None) == E.FATTN_OK


def test_masked_validation(lib):
    E = fattn

    def f(**kw):
        g = lambda n, dflt: kw.get(n, dflt)
        return lib.fattn_fwd_masked(g("q", A), A, A, A, None, g("B", 2), 4, 2, g("N", 300), g("d", 128), 1, 0.1,
                                    g("m", A), g("sb", 0), g("sh", 0), g("ld", 304), None)
    assert f(m=None) == E.FATTN_ERR_INVALID_ARG
    assert f(m=A + 8) == E.FATTN_ERR_INVALID_ARG
    assert f(ld=296) == E.FATTN_ERR_INVALID_ARG          # shorter than N
    assert f(ld=302) == E.FATTN_ERR_INVALID_ARG          # not whole groups of 8
    assert f(sb=12) == E.FATTN_ERR_INVALID_ARG and f(sh=-8) == E.FATTN_ERR_INVALID_ARG
    assert f(d=96) == E.FATTN_ERR_UNSUPPORTED
    assert f(B=0, q=None, m=None) == E.FATTN_OK


def test_fp8_validation(lib):
    E = fattn

    def f(**kw):
        g = lambda n, dflt: kw.get(n, dflt)
        return lib.fattn_fwd_fp8(g("q", A), A, A, A, None, 2, 4, 2, 300, g("d", 128), 1, 0.1, g("qd", 0.01), 0.01,
                                 0.01, None)
    assert f(q=None) == E.FATTN_ERR_INVALID_ARG
    assert f(qd=0.0) == E.FATTN_ERR_INVALID_ARG and f(qd=float("nan")) == E.FATTN_ERR_INVALID_ARG
    assert f(d=64) == E.FATTN_ERR_UNSUPPORTED

