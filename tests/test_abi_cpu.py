"""C-ABI library: loads, exports every symbol spec_verify.h declares, and
rejects bad arguments on the host before any CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

import speculative_decoding_verification_54_gb300 as sv
from speculative_decoding_verification_54_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return sv.load()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_\w+)\s*\(", text)))


def test_header_declares_the_public_entry_points():
    names = declared_functions()
    for must in ("spec_verify_greedy", "spec_verify_sample", "spec_verify_workspace_bytes",
                 "spec_verify_status"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)
    assert set(declared_functions()) <= set(sv.EXPORTED) | {"spec_verify_error_string"}


def test_checked_build_exports_the_same_symbols():
    """The bounds-checked debug build (-DSPEC_CHECK_BOUNDS) loads and exports
    every declared entry point too."""
    path = _build.build(checked=True)
    chk = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(chk, name), name
    chk.spec_verify_error_string.restype = ctypes.c_char_p
    assert b"bounds" in chk.spec_verify_error_string(sv.SPEC_ERR_DEVICE_BOUNDS)


def test_version_and_error_strings(lib):
    assert sv.spec_verify_version() >= 100
    assert sv.error_string(sv.SPEC_OK) == "ok"
    assert "timed out" in sv.error_string(sv.SPEC_ERR_TIMEOUT)
    assert sv.error_string(12345) == "unknown error"


def test_workspace_bytes(lib):
    a = sv.spec_verify_workspace_bytes(32, 4, 262144)
    b = sv.spec_verify_workspace_bytes(64, 4, 262144)
    c = sv.spec_verify_workspace_bytes(32, 8, 262144)
    assert 0 < a < b and a < c and a % 256 == 0
    for bad in ((0, 4, 4096), (8, 0, 4096), (8, 32, 4096), (8, 4, 4100), (8, 4, 0)):
        with pytest.raises(sv.SpecVerifyError) as e:
            sv.spec_verify_workspace_bytes(*bad)
        assert e.value.code == sv.SPEC_ERR_INVALID_ARG


# Fake device addresses: validation must reject these without touching them.
A16, A8, WS = 0x10000, 0x10008, 0x20000


def _sample(lib, **kw):
    args = dict(t=A16, d=A16, dt=sv.SPEC_BF16, tok=A16, temp=A16, ua=A16, ur=A16, B=4, g=4,
                V=4096, out=A16, num=A16, dbg=None, ws=WS, wsb=1 << 30)
    args.update(kw)
    return lib.spec_verify_sample(args["t"], args["d"], args["dt"], args["tok"], args["temp"],
                                  args["ua"], args["ur"], args["B"], args["g"], args["V"],
                                  args["out"], args["num"], args["dbg"], args["ws"], args["wsb"],
                                  None)


def _greedy(lib, **kw):
    args = dict(t=A16, dt=sv.SPEC_F32, tok=A16, B=4, g=4, V=4096, out=A16, num=A16, ws=WS,
                wsb=1 << 30)
    args.update(kw)
    return lib.spec_verify_greedy(args["t"], args["dt"], args["tok"], args["B"], args["g"],
                                  args["V"], args["out"], args["num"], args["ws"], args["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(t=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(d=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(tok=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(temp=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(ua=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(ur=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(out=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(num=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(B=0), sv.SPEC_ERR_INVALID_ARG),
    (dict(g=0), sv.SPEC_ERR_INVALID_ARG),
    (dict(g=32), sv.SPEC_ERR_INVALID_ARG),
    (dict(V=4100), sv.SPEC_ERR_INVALID_ARG),
    (dict(V=0), sv.SPEC_ERR_INVALID_ARG),
    (dict(dt=7), sv.SPEC_ERR_UNSUPPORTED),
    (dict(t=A8), sv.SPEC_ERR_ALIGNMENT),
    (dict(d=A8), sv.SPEC_ERR_ALIGNMENT),
    (dict(dbg=A8), sv.SPEC_ERR_ALIGNMENT),
    (dict(ws=None), sv.SPEC_ERR_WORKSPACE),
    (dict(ws=WS + 16), sv.SPEC_ERR_WORKSPACE),
    (dict(wsb=1024), sv.SPEC_ERR_WORKSPACE),
])
def test_sample_rejects_bad_arguments_on_host(lib, kw, code):
    assert _sample(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(t=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(tok=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(g=40), sv.SPEC_ERR_INVALID_ARG),
    (dict(V=12), sv.SPEC_ERR_INVALID_ARG),
    (dict(dt=-1), sv.SPEC_ERR_UNSUPPORTED),
    (dict(t=A8), sv.SPEC_ERR_ALIGNMENT),
    (dict(wsb=10), sv.SPEC_ERR_WORKSPACE),
])
def test_greedy_rejects_bad_arguments_on_host(lib, kw, code):
    assert _greedy(lib, **kw) == code


def test_binding_fails_loudly_without_library(tmp_path):
    from speculative_decoding_verification_54_gb300 import binding
    saved = binding._lib
    binding._lib = None
    try:
        with pytest.raises(RuntimeError):
            binding.load(str(tmp_path / "missing.so"))
    finally:
        binding._lib = saved


def _lmhead(lib, **kw):
    args = dict(h=A16, w=A16, d=A16, tok=A16, temp=A16, ua=A16, ur=A16, B=64, g=4, V=262144,
                H=1536, out=A16, num=A16, dbg=None, ws=WS, wsb=1 << 20)
    args.update(kw)
    return lib.spec_verify_lmhead_sample(args["h"], args["w"], args["d"], args["tok"], args["temp"],
                                         args["ua"], args["ur"], args["B"], args["g"], args["V"],
                                         args["H"], args["out"], args["num"], args["dbg"], args["ws"],
                                         args["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(h=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(w=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(d=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(tok=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(ur=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(H=0), sv.SPEC_ERR_INVALID_ARG),
    (dict(H=1000), sv.SPEC_ERR_INVALID_ARG),
    (dict(V=262148), sv.SPEC_ERR_INVALID_ARG),
    (dict(g=0), sv.SPEC_ERR_INVALID_ARG),
    (dict(B=77), sv.SPEC_ERR_UNSUPPORTED),   # 77*5 = 385 verify rows > 384
    (dict(B=13, g=31), sv.SPEC_ERR_UNSUPPORTED),  # 13*32 = 416 rows
    (dict(h=A8), sv.SPEC_ERR_ALIGNMENT),
    (dict(w=A8), sv.SPEC_ERR_ALIGNMENT),
    (dict(d=A8), sv.SPEC_ERR_ALIGNMENT),
    (dict(dbg=A8), sv.SPEC_ERR_ALIGNMENT),
    (dict(ws=None), sv.SPEC_ERR_WORKSPACE),
    (dict(ws=WS + 64), sv.SPEC_ERR_WORKSPACE),
    (dict(wsb=1 << 20), sv.SPEC_ERR_WORKSPACE),  # the stored logits alone are 268 MB
])
def test_lmhead_rejects_bad_arguments_on_host(lib, kw, code):
    assert _lmhead(lib, **kw) == code


def test_lmhead_workspace_bytes(lib):
    plain = sv.spec_verify_workspace_bytes(64, 4, 262144)
    lm = sv.spec_verify_workspace_bytes(64, 4, 262144, 1536)
    # the lm_head workspace holds the plain one plus the stored fp32 rows j < gamma
    assert lm >= plain + 64 * 4 * 262144 * 4
    assert lm % 256 == 0
    for bad, code in (((64, 4, 262144, 100), sv.SPEC_ERR_INVALID_ARG),
                      ((80, 4, 262144, 1536), sv.SPEC_ERR_UNSUPPORTED)):
        with pytest.raises(sv.SpecVerifyError) as e:
            sv.spec_verify_workspace_bytes(*bad)
        assert e.value.code == code


def _multi(lib, **kw):
    args = dict(t=A16, dt=sv.SPEC_BF16, tok=A16, B=4, n=3, g=4, V=4096, out=A16, num=A16, ch=None, ws=WS,
                wsb=1 << 30)
    args.update(kw)
    return lib.spec_verify_greedy_multi(args["t"], args["dt"], args["tok"], args["B"], args["n"], args["g"],
                                        args["V"], args["out"], args["num"], args["ch"], args["ws"], args["wsb"],
                                        None)


@pytest.mark.parametrize("kw,code", [
    (dict(t=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(tok=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(out=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(n=0), sv.SPEC_ERR_INVALID_ARG),
    (dict(B=0), sv.SPEC_ERR_INVALID_ARG),
    (dict(B=20000, n=4), sv.SPEC_ERR_INVALID_ARG),   # B * n_cand > 65535
    (dict(g=32), sv.SPEC_ERR_INVALID_ARG),
    (dict(V=12), sv.SPEC_ERR_INVALID_ARG),
    (dict(dt=5), sv.SPEC_ERR_UNSUPPORTED),
    (dict(t=A8), sv.SPEC_ERR_ALIGNMENT),
    (dict(ws=None), sv.SPEC_ERR_WORKSPACE),
    (dict(wsb=4096), sv.SPEC_ERR_WORKSPACE),
])
def test_greedy_multi_rejects_bad_arguments_on_host(lib, kw, code):
    assert _multi(lib, **kw) == code


def _topkp(lib, **kw):
    args = dict(t=A16, d=A16, dt=sv.SPEC_BF16, tok=A16, temp=A16, ua=A16, ur=A16, B=4, g=4, V=4096, k=64,
                p=0.95, out=A16, num=A16, dbg=None, ws=WS, wsb=1 << 30)
    args.update(kw)
    return lib.spec_verify_sample_topkp(args["t"], args["d"], args["dt"], args["tok"], args["temp"], args["ua"],
                                        args["ur"], args["B"], args["g"], args["V"], args["k"], args["p"],
                                        args["out"], args["num"], args["dbg"], args["ws"], args["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(t=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(ur=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(k=0), sv.SPEC_ERR_INVALID_ARG),
    (dict(k=1025), sv.SPEC_ERR_INVALID_ARG),
    (dict(p=0.0), sv.SPEC_ERR_INVALID_ARG),
    (dict(p=1.5), sv.SPEC_ERR_INVALID_ARG),
    (dict(p=float("nan")), sv.SPEC_ERR_INVALID_ARG),
    (dict(V=4100), sv.SPEC_ERR_INVALID_ARG),
    (dict(dt=3), sv.SPEC_ERR_UNSUPPORTED),
    (dict(d=A8), sv.SPEC_ERR_ALIGNMENT),
    (dict(ws=WS + 8), sv.SPEC_ERR_WORKSPACE),
    (dict(wsb=4096), sv.SPEC_ERR_WORKSPACE),
])
def test_topkp_rejects_bad_arguments_on_host(lib, kw, code):
    assert _topkp(lib, **kw) == code


def test_topkp_workspace_bytes(lib):
    plain = sv.spec_verify_workspace_bytes(32, 4, 262144)
    out = ctypes.c_size_t(0)
    assert lib.spec_verify_topkp_workspace_bytes(32, 4, 262144, ctypes.byref(out)) == sv.SPEC_OK
    assert out.value >= plain + 32 * 9 * 2048 * 8      # the kept lists


def _head(lib, **kw):
    args = dict(h=A16, c=A16, w=A16, off=A16, o2t=A16, R=4, H=1536, V=262144, nc=2048, k=32, mc=8192,
                ot=A16, ol=A16, oc=A16, ws=WS, wsb=1 << 30)
    args.update(kw)
    return lib.spec_centroid_head(args["h"], args["c"], args["w"], args["off"], args["o2t"], args["R"], args["H"],
                                  args["V"], args["nc"], args["k"], args["mc"], args["ot"], args["ol"], args["oc"],
                                  args["ws"], args["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(h=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(off=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(H=1000), sv.SPEC_ERR_INVALID_ARG),
    (dict(H=2304), sv.SPEC_ERR_INVALID_ARG),
    (dict(nc=0), sv.SPEC_ERR_INVALID_ARG),
    (dict(nc=8193), sv.SPEC_ERR_INVALID_ARG),
    (dict(k=0), sv.SPEC_ERR_INVALID_ARG),
    (dict(k=257), sv.SPEC_ERR_INVALID_ARG),
    (dict(nc=16, k=17), sv.SPEC_ERR_INVALID_ARG),
    (dict(mc=8193), sv.SPEC_ERR_INVALID_ARG),
    (dict(R=0), sv.SPEC_ERR_INVALID_ARG),
    (dict(w=A8), sv.SPEC_ERR_ALIGNMENT),
    (dict(ws=WS + 8), sv.SPEC_ERR_WORKSPACE),
    (dict(wsb=1024), sv.SPEC_ERR_WORKSPACE),
])
def test_centroid_head_rejects_bad_arguments_on_host(lib, kw, code):
    assert _head(lib, **kw) == code


def _sparse(lib, **kw):
    args = dict(t=A16, dt=sv.SPEC_BF16, ct=A16, cl=A16, cc=A16, stride=8192, tok=A16, temp=A16, ua=A16, ur=A16,
                B=4, g=4, V=262144, out=A16, num=A16, dbg=None, ws=WS, wsb=1 << 30)
    args.update(kw)
    return lib.spec_verify_sample_sparse(args["t"], args["dt"], args["ct"], args["cl"], args["cc"], args["stride"],
                                         args["tok"], args["temp"], args["ua"], args["ur"], args["B"], args["g"],
                                         args["V"], args["out"], args["num"], args["dbg"], args["ws"], args["wsb"],
                                         None)


@pytest.mark.parametrize("kw,code", [
    (dict(t=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(ct=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(cc=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(stride=0), sv.SPEC_ERR_INVALID_ARG),
    (dict(g=0), sv.SPEC_ERR_INVALID_ARG),
    (dict(V=4100), sv.SPEC_ERR_INVALID_ARG),
    (dict(dt=3), sv.SPEC_ERR_UNSUPPORTED),
    (dict(t=A8), sv.SPEC_ERR_ALIGNMENT),
    (dict(ws=WS + 8), sv.SPEC_ERR_WORKSPACE),
    (dict(wsb=4096), sv.SPEC_ERR_WORKSPACE),
])
def test_sparse_rejects_bad_arguments_on_host(lib, kw, code):
    assert _sparse(lib, **kw) == code


def test_centroid_and_sparse_workspace_bytes(lib):
    out = ctypes.c_size_t(0)
    assert lib.spec_centroid_head_workspace_bytes(4, 2048, 32, ctypes.byref(out)) == sv.SPEC_OK
    assert out.value >= 4 * 2048 * 4 + 4 * 32 * 4 + 4 * 33 * 4
    assert lib.spec_centroid_head_workspace_bytes(4, 2048, 3000, ctypes.byref(out)) == sv.SPEC_ERR_INVALID_ARG
    # the score GEMM's K parts: while tiles (128 clusters) x row chunks (256
    # rows) are few, up to 8 partial sums per score; otherwise one
    def head_ws(R, nc):
        assert lib.spec_centroid_head_workspace_bytes(R, nc, 8, ctypes.byref(out)) == sv.SPEC_OK
        return out.value
    small = head_ws(128, 2048)           # 16 tiles x 1 chunk: split
    assert small >= 8 * 128 * 2048 * 4
    large = head_ws(64 * 256, 2048)      # 16 tiles x 64 chunks: no split
    assert 64 * 256 * 2048 * 4 <= large < 2 * 64 * 256 * 2048 * 4
    assert head_ws(4, 2048) >= 8 * 4 * 2048 * 4
    plain = sv.spec_verify_workspace_bytes(32, 4, 262144)
    assert lib.spec_verify_sparse_workspace_bytes(32, 4, 262144, ctypes.byref(out)) == sv.SPEC_OK
    assert out.value >= plain + 32 * 257 * 4     # per-chunk candidate offsets
