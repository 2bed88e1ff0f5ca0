"""The C-ABI library builds, loads and exports every symbol that include/attn.h
declares; host-side argument checks return their documented codes without
launching anything (no GPU needed: every case here fails validation first)."""
import ctypes
import os
import re

import pytest

import attention_flash_gqa_gb300 as attn
from attention_flash_gqa_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")

OK, INVALID, UNSUPPORTED, MISALIGNED, WORKSPACE = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return attn.load_library()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(declared_functions())
    assert {"attn_fwd", "attn_bwd", "attn_fwd_varlen", "attn_fwd_paged", "attn_decode_paged"} <= names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in attn.h but not exported"


def test_version_and_status_strings(lib):
    assert attn.load_library().attn_version() >= 100
    for code, name in attn.STATUS.items():
        assert attn.attn_status_string(code) == name
    assert attn.attn_status_string(99) == "ATTN_ERR_UNKNOWN"


def test_workspace_sizes(lib):
    assert attn.attn_workspace_size(attn.ATTN_OP_FWD, 2, 32, 4, 4096, 512) == 0
    ws = attn.attn_workspace_size(attn.ATTN_OP_BWD, 2, 32, 4, 4096, 512)
    rows = 2 * 4096
    assert ws >= rows * 32 * 512 * 4 + rows * 32 * 4
    assert ws % 256 == 0
    assert attn.attn_workspace_size(attn.ATTN_OP_BWD_VARLEN, 1, 32, 4, 18000, 512) >= 18000 * 32 * 513 * 4
    d = attn.attn_workspace_size(attn.ATTN_OP_DECODE_PAGED, 64, 32, 8, 0, 128)
    assert d >= 64 * 4 + 64 * 32 * 130 * 4
    # head_dim 256 with 16 KV heads: four blocks of 4 heads, each writing its own heads' partials
    d2 = attn.attn_workspace_size(attn.ATTN_OP_DECODE_PAGED, 64, 32, 16, 0, 256)
    assert d2 >= 65 * 4 + 64 * 32 * 260 * 4
    assert attn.attn_workspace_size(99, 1, 1, 1, 1, 256) == 0


A = 1 << 20  # a fake, 16-byte aligned "device" address: never dereferenced on these paths
P = ctypes.c_void_p


def fwd(lib, **kw):
    a = dict(q=A, k=A, v=A, o=A, lse=A, B=1, Hq=4, Hkv=2, S=128, D=256, scale=0.0625, causal=1, window=0)
    a.update(kw)
    return lib.attn_fwd(P(a["q"]), P(a["k"]), P(a["v"]), P(a["o"]), P(a["lse"]), a["B"], a["Hq"], a["Hkv"], a["S"],
                        a["D"], a["scale"], a["causal"], a["window"], None, 0, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), INVALID), (dict(lse=0), INVALID), (dict(B=-1), INVALID), (dict(S=-5), INVALID),
    (dict(Hq=0), INVALID), (dict(Hkv=0), INVALID), (dict(Hq=6, Hkv=4), INVALID),
    (dict(scale=0.0), INVALID), (dict(scale=-1.0), INVALID), (dict(scale=float("nan")), INVALID),
    (dict(scale=float("inf")), INVALID), (dict(window=-1), INVALID),
    (dict(causal=0), UNSUPPORTED), (dict(D=96), UNSUPPORTED), (dict(D=32), UNSUPPORTED), (dict(D=1024), UNSUPPORTED),
    (dict(q=A + 8), MISALIGNED), (dict(o=A + 2), MISALIGNED), (dict(lse=A + 4), MISALIGNED),
    (dict(B=0), OK), (dict(S=0), OK),
])
def test_fwd_argument_checks(lib, kw, code):
    assert fwd(lib, **kw) == code


def test_varlen_argument_checks(lib):
    f = lib.attn_fwd_varlen
    base = [P(A)] * 5 + [P(A), 3, 1000, 512, 4, 2, 512, 0.044, 1, 0, None, 0, None]
    def call(**over):
        args = list(base)
        names = ["q", "k", "v", "o", "lse", "cu", "nseq", "T", "maxlen", "Hq", "Hkv", "D", "scale", "causal", "window"]
        for key, val in over.items():
            args[names.index(key)] = val
        return f(*args)
    assert call(cu=None) == INVALID
    assert call(nseq=-1) == INVALID
    assert call(T=-1) == INVALID
    assert call(maxlen=-1) == INVALID
    assert call(Hq=5) == INVALID
    assert call(D=192) == UNSUPPORTED
    assert call(q=P(A + 4)) == MISALIGNED
    assert call(nseq=0) == OK


def test_bwd_argument_checks(lib):
    def call(ws=P(256 * 4096), wsb=1 << 40, cu=None, B=2, nseq=0, maxlen=0, dO=P(A), D=512, S=300):
        return lib.attn_bwd(P(A), P(A), P(A), P(A), P(A), dO, P(A), P(A), P(A), B, 8, 2, S, D, 0.044, 1, 0, cu,
                            nseq, maxlen, ws, wsb, None)
    assert call(dO=None) == INVALID
    assert call(ws=None) == WORKSPACE
    need = attn.attn_workspace_size(attn.ATTN_OP_BWD, 2, 8, 2, 300, 512)
    assert call(wsb=need - 1) == WORKSPACE
    assert call(ws=P(256 * 4096 + 16)) == MISALIGNED
    assert call(cu=P(A), B=2, nseq=1, maxlen=300) == INVALID  # packed layout wants B == 1
    assert call(D=96) == UNSUPPORTED
    assert call(B=0) == OK


def test_decode_argument_checks(lib):
    def call(B=4, Hq=32, Hkv=8, D=128, ps=16, maxp=8, npages=64, scale=0.088, window=0, ws=P(256 * 4096),
             wsb=1 << 30, bt=P(A), q=P(A)):
        return lib.attn_decode_paged(q, P(A), P(A), bt, P(A), P(A), P(A), B, Hq, Hkv, D, ps, maxp, npages, scale,
                                     window, ws, wsb, None)
    assert call(bt=None) == INVALID
    assert call(Hq=30) == INVALID
    assert call(scale=0.0) == INVALID
    assert call(B=-1) == INVALID
    assert call(window=-1) == INVALID
    assert call(D=64) == UNSUPPORTED
    assert call(D=512) == UNSUPPORTED
    assert call(D=256, Hq=64, Hkv=8) == UNSUPPORTED  # group of 8 at head_dim 256
    assert call(ps=32) == UNSUPPORTED
    assert call(Hkv=512, Hq=512) == UNSUPPORTED
    assert call(Hq=8 * 16, Hkv=8) == UNSUPPORTED  # group of 16
    assert call(B=5000) == UNSUPPORTED
    assert call(q=P(A + 8)) == MISALIGNED
    assert call(bt=P(A + 2)) == MISALIGNED
    assert call(ws=None) == WORKSPACE
    assert call(wsb=100) == WORKSPACE
    assert call(B=0) == OK


def test_prefill_paged_argument_checks(lib):
    def call(q=P(A), bt=P(A), cu=P(A), R=3, T=600, maxq=512, Hq=32, Hkv=4, D=512, ps=16, maxp=256, npages=4096,
             scale=0.044, causal=1, window=0):
        return lib.attn_fwd_paged(q, P(A), P(A), bt, P(A), cu, P(A), P(A), R, T, maxq, Hq, Hkv, D, ps, maxp, npages,
                                  scale, causal, window, None)
    assert call(bt=None) == INVALID
    assert call(cu=None) == INVALID
    assert call(R=-1) == INVALID
    assert call(T=-1) == INVALID
    assert call(Hq=30) == INVALID
    assert call(scale=float("nan")) == INVALID
    assert call(window=-2) == INVALID
    assert call(npages=0) == INVALID  # new tokens but no cache
    assert call(causal=0) == UNSUPPORTED
    assert call(D=96) == UNSUPPORTED
    assert call(ps=32) == UNSUPPORTED
    assert call(R=40000) == UNSUPPORTED  # 2 CTAs per (request, head) at D = 512
    assert call(q=P(A + 8)) == MISALIGNED
    assert call(cu=P(A + 2)) == MISALIGNED
    assert call(T=0) == OK
    assert call(R=0, q=None, bt=None, cu=None) == OK  # nothing to do: pointers may be NULL


def test_merge_lse_argument_checks(lib):
    def call(op=P(A), lp=P(A), o=P(A), l=P(A), n=4, B=1, S=100, H=8, D=512):
        return lib.attn_merge_lse(op, lp, o, l, n, B, S, H, D, None)
    assert call(n=0) == INVALID
    assert call(B=-1) == INVALID
    assert call(H=0) == INVALID
    assert call(op=None) == INVALID
    assert call(D=96) == UNSUPPORTED
    assert call(n=65) == UNSUPPORTED
    assert call(op=P(A + 8)) == MISALIGNED
    assert call(l=P(A + 2)) == MISALIGNED
    assert call(S=0, op=None, lp=None, o=None, l=None) == OK


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(attn, "_LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(attn, "_lib", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        attn.load_library()
