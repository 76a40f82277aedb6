"""The C-ABI library builds, loads without a GPU, exports every entry point its header declares,
and rejects bad arguments on the host before touching the device (CPU only)."""
import ctypes
import os
import re

import pytest

import speculative_decoding_rejection_verify_gb300 as sv
from speculative_decoding_rejection_verify_gb300 import _build

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
HEADER = os.path.join(INCLUDE, "spec_verify.h")
HEADERS = [os.path.join(INCLUDE, f) for f in sorted(os.listdir(INCLUDE)) if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return sv.load()


def declared_functions(path=None):
    names = set()
    for h in ([path] if path else HEADERS):
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(spec_\w+)\s*\(", src, flags=re.M))
    return sorted(names)


def test_header_declares_the_entry_points():
    assert set(declared_functions(HEADER)) == set(sv.EXPORTS)
    assert set(declared_functions(os.path.join(INCLUDE, "spec_control.h"))) == set(sv.CONTROL_EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"


def test_workspace_sizes(lib):
    n = sv.workspace_bytes(1024, 4, 128256, sv.DTYPE_BF16, 0)
    nchunk = (128256 + 8191) // 8192
    assert n >= 1024 * 9 * nchunk * 8  # one (max, sum) pair per chunk of every row
    assert n % 256 == 0
    big = sv.workspace_bytes(256, 8, 152064, sv.DTYPE_F32, 50)
    assert big > sv.workspace_bytes(256, 8, 152064, sv.DTYPE_F32, 0)  # top-k candidates
    assert lib.spec_verify_workspace_bytes(-1, 4, 100, 0, 0) == 0
    assert lib.spec_verify_workspace_bytes(1, 17, 100, 0, 0) == 0
    assert lib.spec_verify_workspace_bytes(1, 4, 100, 7, 0) == 0
    assert lib.spec_verify_host_staging_bytes(8, 5, 32000, 1, 0, 0) > 8 * 11 * 32000 * 2


def _call(lib, B=1, K=4, V=100, T=1.0, top_k=0, p=1, q=1, draft=1, ua=1, ur=1, tok=1, n=1, dtype=0,
          ws=256, wsb=1 << 20):
    P = ctypes.c_void_p
    return lib.spec_verify(P(p) if p else None, P(q) if q else None, P(draft) if draft else None, None,
                           P(ua) if ua else None, P(ur) if ur else None, T, top_k,
                           P(tok) if tok else None, P(n) if n else None, None, B, K, V, dtype,
                           P(ws) if ws else None, wsb, None)


def test_host_side_validation(lib):
    # every case below is rejected before any CUDA call (the pointers are never dereferenced)
    assert _call(lib, B=-1) == 1
    assert _call(lib, V=0) == 1
    assert _call(lib, T=-0.5) == 1
    assert _call(lib, T=float("nan")) == 1
    assert _call(lib, top_k=-1) == 1
    assert _call(lib, K=17) == 2
    assert _call(lib, V=sv.MAX_V + 1) == 2
    assert _call(lib, dtype=5) == 2
    assert _call(lib, top_k=300, V=1000) == 2
    assert _call(lib, p=0) == 1
    assert _call(lib, q=0) == 1
    assert _call(lib, ua=0) == 1
    assert _call(lib, ur=0) == 1
    assert _call(lib, draft=0) == 1
    assert _call(lib, tok=0) == 1
    assert _call(lib, ws=0) == 4
    assert _call(lib, ws=128) == 4  # misaligned
    assert _call(lib, wsb=16) == 4  # too small
    assert _call(lib, B=0) == 0  # empty batch: nothing to do
    # greedy needs neither q nor the uniforms
    assert _call(lib, B=0, T=0.0, q=0, ua=0, ur=0) == 0


def _call_ex(lib, sampling, B=1, K=4, V=100, wsb=1 << 20):
    P = ctypes.c_void_p
    return lib.spec_verify_ex(P(1), P(1), P(1), None, P(1), P(1),
                              ctypes.byref(sampling) if sampling is not None else None, P(1), P(1), None,
                              B, K, V, 0, P(256), wsb, None)


def test_sampling_parameter_validation(lib):
    S = sv.SamplingStruct
    assert _call_ex(lib, None) == 1
    assert _call_ex(lib, S(1.0, 0.0, 0, 1.0)) == 1            # draft temperature 0 under T > 0
    assert _call_ex(lib, S(1.0, -1.0, 0, 1.0)) == 1
    assert _call_ex(lib, S(1.0, float("inf"), 0, 1.0)) == 1
    assert _call_ex(lib, S(1.0, 0.5, 0, 0.0)) == 1            # top_p must be > 0
    assert _call_ex(lib, S(1.0, 0.5, 0, float("nan"))) == 1
    assert _call_ex(lib, S(1.0, 0.5, -2, 0.9)) == 1
    assert _call_ex(lib, S(1.0, 0.5, 0, 0.9), B=0) == 0       # valid parameters, empty batch
    assert _call_ex(lib, S(0.0, 0.0, 0, 0.9), B=0) == 0       # greedy ignores T_q
    assert _call_ex(lib, S(1.0, 0.5, 0, 1.7), B=0) == 0       # top_p >= 1 is off


def test_status_strings(lib):
    for code in range(6):
        assert lib.spec_verify_status_string(code)
    assert lib.spec_verify_status_string(99) == b"unknown status"


def test_product_path_has_no_fallback(monkeypatch, tmp_path):
    """Without the compiled library the binding raises instead of computing anything itself."""
    import importlib
    monkeypatch.setattr(_build, "LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(sv, "_lib", None)
    with pytest.raises(RuntimeError):
        sv.load()
    importlib.reload(_build)


def test_package_does_not_import_the_oracle():
    root = os.path.dirname(os.path.abspath(sv.__file__))
    for dirpath, _, files in os.walk(root):
        for f in files:
            if f.endswith((".py", ".cu", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "oracle/" not in src, f
