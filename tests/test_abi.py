"""The C ABI library: it builds, loads, exports every symbol include/kda.h
declares, and rejects bad arguments synchronously, before any launch (these
calls need no GPU)."""
import ctypes
import os
import re

import pytest

import gated_delta_rule_05_gb300 as kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    kda.build()
    return kda.lib()


def declared_functions():
    with open(os.path.join(ROOT, "include", "kda.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(kda.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(kda.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), name


def test_status_strings(lib):
    for code in range(5):
        assert kda.kda_status_string(code).startswith("KDA_")
    assert "UNKNOWN" in kda.kda_status_string(99)


def test_workspace_bytes(lib):
    assert kda.kda_prefill_workspace_bytes(0, 1, 128, 128) == 0
    assert kda.kda_prefill_workspace_bytes(1, 32, 128, 128) == 512
    assert kda.kda_prefill_workspace_bytes(64, 32, 128, 128) == 512
    assert kda.kda_prefill_workspace_bytes(65, 32, 128, 128) == 768


A = 0x10000            # a fake, 256-byte-aligned address: never dereferenced,
                       # because every call below fails validation first.
NULL = None


def prefill(lib, **kw):
    args = dict(q=A, k=A, v=A, g=A, b=A, S0=NULL, cu=NULL, N=1, T=64, H=2,
                dk=128, dv=128, dt=kda.KDA_BF16, o=A * 2, Sf=NULL, ws=A * 3,
                wsb=512, stream=NULL)
    args.update(kw)
    return lib.kda_prefill(*args.values())


def decode(lib, **kw):
    args = dict(q=A, k=A, v=A, g=A, b=A, S=A * 4, N=4, H=2, dk=128, dv=128,
                dt=kda.KDA_BF16, o=A * 2, stream=NULL)
    args.update(kw)
    return lib.kda_decode_step(*args.values())


@pytest.mark.parametrize("kw,code", [
    (dict(dk=96, dv=96), kda.KDA_ERR_UNSUPPORTED),
    (dict(dk=128, dv=64), kda.KDA_ERR_UNSUPPORTED),
    (dict(dt=7), kda.KDA_ERR_UNSUPPORTED),
    (dict(N=0), kda.KDA_ERR_INVALID_ARG),
    (dict(H=0), kda.KDA_ERR_INVALID_ARG),
    (dict(T=-1), kda.KDA_ERR_INVALID_ARG),
    (dict(N=2), kda.KDA_ERR_INVALID_ARG),           # N > 1 needs cu_seqlens
    (dict(q=NULL), kda.KDA_ERR_INVALID_ARG),
    (dict(b=NULL), kda.KDA_ERR_INVALID_ARG),
    (dict(q=A + 2), kda.KDA_ERR_INVALID_ARG),       # misaligned
    (dict(T=1 << 31), kda.KDA_ERR_INVALID_ARG),     # beyond 32-bit offsets
    (dict(S0=A * 8, Sf=A * 8 + 256), kda.KDA_ERR_INVALID_ARG),   # partial overlap
    (dict(ws=NULL), kda.KDA_ERR_WORKSPACE),
    (dict(wsb=100), kda.KDA_ERR_WORKSPACE),
    (dict(ws=A * 3 + 16), kda.KDA_ERR_WORKSPACE),   # not 256-byte aligned
])
def test_prefill_rejects(lib, kw, code):
    assert prefill(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(dk=48, dv=48), kda.KDA_ERR_UNSUPPORTED),
    (dict(dt=3), kda.KDA_ERR_UNSUPPORTED),
    (dict(N=0), kda.KDA_ERR_INVALID_ARG),
    (dict(S=NULL), kda.KDA_ERR_INVALID_ARG),
    (dict(o=NULL), kda.KDA_ERR_INVALID_ARG),
    (dict(v=A + 4), kda.KDA_ERR_INVALID_ARG),
    (dict(o=A * 4), kda.KDA_ERR_INVALID_ARG),       # o overlaps the state
])
def test_decode_rejects(lib, kw, code):
    assert decode(lib, **kw) == code


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import importlib
    monkeypatch.setattr(kda, "_lib", None)
    monkeypatch.setattr(kda, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        kda.lib()
    importlib.reload(kda)


def noalloc(lib, **kw):
    args = dict(q=A, k=A, v=A, g=A, b=A, S0=NULL, cu=NULL, N=1, T=64, H=2, dk=128, dv=128,
                dt=kda.KDA_BF16, o=A * 2, Sf=NULL, stream=NULL)
    args.update(kw)
    return lib.kda_prefill_noalloc(*args.values())


@pytest.mark.parametrize("kw,code", [
    (dict(N=4097, cu=A * 5), kda.KDA_ERR_WORKSPACE),     # beyond the fixed scratch
    (dict(N=0), kda.KDA_ERR_INVALID_ARG),
])
def test_noalloc_rejects(lib, kw, code):
    # both are rejected before the scratch array's address is looked up
    assert noalloc(lib, **kw) == code


def segmented(lib, **kw):
    args = dict(q=A, k=A, v=A, g=A, b=A, S0=NULL, T=64, H=2, dk=128, dv=128, dt=kda.KDA_BF16,
                o=A * 2, Sf=NULL, segments=2, ws=A * 3, wsb=512, stream=NULL)
    args.update(kw)
    return lib.kda_prefill_segmented(*args.values())


@pytest.mark.parametrize("kw,code", [
    (dict(q=NULL), kda.KDA_ERR_INVALID_ARG),
    (dict(dk=96, dv=96), kda.KDA_ERR_UNSUPPORTED),
    (dict(T=-1), kda.KDA_ERR_INVALID_ARG),
    (dict(ws=NULL), kda.KDA_ERR_WORKSPACE),
])
def test_segmented_rejects(lib, kw, code):
    # a single chunk cannot be cut: the call is kda_prefill, with its checks
    assert segmented(lib, **kw) == code
