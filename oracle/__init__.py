"""fp64 CPU oracle for the speculative-sampling verify step — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import this package.  The CUDA library never links or calls it, and the two
share no code: this wrapper loads ``liboracle.so`` built from ``oracle.c`` (plain C, double
precision) with ``gcc``.

What it computes is stated in ``oracle.c`` with the page passages it follows (cf-1.com §2.1-§2.2,
2kiu.com §2.2 and §7, gsyq.cn §3.1-§3.3).  Logits are passed as float32 arrays or as bf16 raw bits in
uint16 arrays; every value is widened exactly to double.

Parity unpinned (conventions, fixed by reading only): the top-k tie rule, the ascending-token-id
CDF order, and the 2^-24 uniform grid.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

DTYPE_F32 = 0
DTYPE_BF16 = 1

FLAG_RESIDUAL_ZERO = 1
FLAG_CDF_CLAMP = 2
FLAG_BAD_TOKEN = 4
FLAG_BAD_K = 8
FLAG_NONFINITE = 16
FLAG_TOPK_TIE = 32

# Flags the build uses: no fast-math and no FMA contraction, so x86 and Arm hosts agree.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-fno-fast-math"]


def build(out: str = _LIB, extra_flags: Optional[list] = None) -> str:
    """Compile oracle.c into a shared library (``extra_flags`` lets a test build a variant)."""
    cmd = ["gcc", *CFLAGS, *(extra_flags or []), _SRC, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _stale() -> bool:
    return (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)


_P = ctypes.c_void_p


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    i32, f32, f64 = ctypes.c_int, ctypes.c_float, ctypes.c_double
    lib.oracle_row_dist.argtypes = [_P, i32, i32, f64, i32, _P, _P]
    lib.oracle_row_dist.restype = i32
    lib.oracle_row_dist_ex.argtypes = [_P, i32, i32, f64, i32, f64, _P, _P]
    lib.oracle_row_dist_ex.restype = i32
    lib.oracle_decide.argtypes = [_P, _P, i32, i32, _P, _P, f64, _P, _P, _P, _P, _P, _P, _P, _P]
    lib.oracle_decide.restype = i32
    lib.oracle_verify.argtypes = [_P, _P, _P, _P, _P, _P, f32, i32, _P, _P, _P, _P, _P, _P, _P,
                                  _P, _P, i32, i32, i32, i32, i32]
    lib.oracle_verify.restype = i32
    lib.oracle_verify_ex.argtypes = [_P, _P, _P, _P, _P, _P, f32, f32, i32, f32, _P, _P, _P, _P, _P, _P,
                                     _P, _P, _P, _P, i32, i32, i32, i32, i32]
    lib.oracle_verify_ex.restype = i32
    lib.oracle_verify_cuts.argtypes = [_P, _P, _P, _P, _P, _P, f32, f32, i32, f32, _P, _P, _P, _P, _P, _P,
                                       _P, _P, _P, _P, _P, _P, i32, i32, i32, i32, i32]
    lib.oracle_verify_cuts.restype = i32
    lib.oracle_row_dist_at.argtypes = [_P, i32, i32, f64, i32, f64, f64, _P, _P]
    lib.oracle_row_dist_at.restype = i32
    lib.oracle_decide_multi.argtypes = [_P, _P, i32, i32, i32, _P, _P, f64, _P, _P, _P, _P, _P, _P]
    lib.oracle_decide_multi.restype = i32
    lib.oracle_verify_multi.argtypes = [_P, _P, _P, _P, _P, f32, f32, _P, _P, _P, _P, _P, _P, i32, i32, i32, i32,
                                        i32, i32]
    lib.oracle_verify_multi.restype = i32
    lib.oracle_decide_trials.argtypes = [_P, _P, i32, i32, i32, _P, _P, _P, _P, _P, _P, i32]
    lib.oracle_decide_trials.restype = i32
    return lib


_lib: Optional[ctypes.CDLL] = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library, or a variant at ``path``."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        if _stale():
            build()
        _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logits(a: np.ndarray):
    """(array, dtype code) for float32 logits or bf16 bits held in uint16."""
    if a.dtype == np.float32:
        return np.ascontiguousarray(a), DTYPE_F32
    if a.dtype == np.uint16:
        return np.ascontiguousarray(a), DTYPE_BF16
    raise TypeError(f"logits must be float32 or bf16 bits (uint16), got {a.dtype}")


def row_dist(z: np.ndarray, temperature: float, top_k: int = 0, top_p: float = 1.0, lib=None,
             cut: Optional[float] = None):
    """Normalised distribution of one logit row (temperature, then top-k, then top-p).

    Returns (P float64[V], info dict {m, lognorm, threshold, kept, threshold_p, nucleus_margin},
    flags).  top_p is taken as the float32 value the CUDA library receives.  ``cut``: a nucleus
    cut to take instead of finding one (keep the logits >= cut inside the top-k set)."""
    lib = lib or load()
    z, dt = _logits(z)
    V = z.shape[-1]
    P = np.empty(V, np.float64)
    info = np.empty(6, np.float64)
    fl = lib.oracle_row_dist_at(_ptr(z), dt, V, float(temperature), int(top_k), float(np.float32(top_p)),
                                float("nan") if cut is None else float(cut), _ptr(P), _ptr(info))
    return P, dict(m=info[0], lognorm=info[1], threshold=info[2], kept=info[3], threshold_p=info[4],
                   nucleus_margin=info[5]), int(fl)


def decide(P: np.ndarray, Q: np.ndarray, x, ua, ur: float, lib=None):
    """The verify decision of one request on fp64 distributions P [(K+1),V], Q [K,V].

    The uniforms are taken as float64 (the batch entry points take the float32 grid values)."""
    lib = lib or load()
    P = np.ascontiguousarray(P, np.float64)
    K = P.shape[0] - 1
    V = P.shape[1]
    Q = np.ascontiguousarray(Q, np.float64).reshape(K, V) if K > 0 else np.zeros((1, V))
    x = np.ascontiguousarray(x, np.int32).reshape(K)
    ua = np.ascontiguousarray(ua, np.float64).reshape(K)
    tok = np.empty(K + 1, np.int32)
    n = np.empty(1, np.int32)
    pd, qd, am = (np.empty(max(K, 1)) for _ in range(3))
    sm = np.empty(1)
    rm = np.empty(1)
    work = np.empty(V)
    fl = lib.oracle_decide(_ptr(P), _ptr(Q), V, K, _ptr(x), _ptr(ua), float(ur), _ptr(tok), _ptr(n),
                           _ptr(pd), _ptr(qd), _ptr(am), _ptr(sm), _ptr(rm), _ptr(work))
    return dict(tokens=tok, n_acc=int(n[0]), p_draft=pd[:K], q_draft=qd[:K], accept_margin=am[:K],
                sample_margin=float(sm[0]), residual_mass=float(rm[0]), flags=int(fl))


def decide_trials(P: np.ndarray, Q: np.ndarray, x: np.ndarray, ua: np.ndarray, ur: np.ndarray,
                  nthreads: int = 0, lib=None):
    """N independent decisions on one shared pair of distributions.

    x, ua: [N, K]; ur: [N].  Returns (tokens [N, K+1], n_acc [N], flags [N])."""
    lib = lib or load()
    P = np.ascontiguousarray(P, np.float64)
    K = P.shape[0] - 1
    V = P.shape[1]
    Q = np.ascontiguousarray(Q, np.float64) if K > 0 else np.zeros((1, V))
    N = ur.shape[0]
    x = np.ascontiguousarray(x, np.int32).reshape(N, K)
    ua = np.ascontiguousarray(ua, np.float32).reshape(N, K)
    ur = np.ascontiguousarray(ur, np.float32)
    tok = np.empty((N, K + 1), np.int32)
    n = np.empty(N, np.int32)
    fl = np.empty(N, np.int32)
    lib.oracle_decide_trials(_ptr(P), _ptr(Q), V, K, N, _ptr(x), _ptr(ua), _ptr(ur), _ptr(tok),
                             _ptr(n), _ptr(fl), nthreads or (os.cpu_count() or 1))
    return tok, n, fl


def verify(p: np.ndarray, q: Optional[np.ndarray], draft: np.ndarray, k_per_row: Optional[np.ndarray],
           ua: Optional[np.ndarray], ur: Optional[np.ndarray], temperature: float, top_k: int = 0,
           nthreads: int = 1, lib=None, draft_temperature: Optional[float] = None,
           top_p: float = 1.0, row_cut: Optional[np.ndarray] = None) -> dict:
    """The whole verify step on host arrays, same argument meaning as the CUDA ``spec_verify_ex``.

    p: [B, K_max+1, V], q: [B, K_max, V] (float32 or bf16-as-uint16; q may be None when
    temperature == 0), draft: [B, K_max] int32, k_per_row: [B] int32 or None, ua: [B, K_max],
    ur: [B] float32; draft_temperature None = temperature; top_p 1 = off.  ``row_cut``
    [B, 2*K_max+1] (optional): per row, NaN = find the nucleus, a value = take it as the nucleus
    cut.  Returns a dict of numpy outputs (tokens, n_acc, stats..., flags, nucleus_margin and
    row_cut [B, 2*K_max+1], the latter each row's smallest kept logit bound)."""
    lib = lib or load()
    p, dt = _logits(p)
    B, K1, V = p.shape
    K_max = K1 - 1
    if q is not None:
        q, dtq = _logits(q)
        assert dtq == dt and q.shape == (B, K_max, V)
    draft = np.ascontiguousarray(draft, np.int32).reshape(B, K_max)
    kpr = None if k_per_row is None else np.ascontiguousarray(k_per_row, np.int32)
    ua = np.zeros((B, K_max), np.float32) if ua is None else np.ascontiguousarray(ua, np.float32)
    ur = np.zeros(B, np.float32) if ur is None else np.ascontiguousarray(ur, np.float32)
    out = dict(
        tokens=np.empty((B, K_max + 1), np.int32), n_acc=np.empty(B, np.int32),
        p_draft=np.empty((B, K_max)), q_draft=np.empty((B, K_max)), accept_margin=np.empty((B, K_max)),
        sample_margin=np.empty(B), residual_mass=np.empty(B), row_lognorm=np.empty((B, 2 * K_max + 1)),
        nucleus_margin=np.empty((B, 2 * K_max + 1)), row_cut=np.empty((B, 2 * K_max + 1)),
        flags=np.empty(B, np.int32))
    tq = temperature if draft_temperature is None else draft_temperature
    cut_in = None if row_cut is None else np.ascontiguousarray(row_cut, np.float64).reshape(B, 2 * K_max + 1)
    rc = lib.oracle_verify_cuts(_ptr(p), _ptr(q), _ptr(draft), _ptr(kpr), _ptr(ua), _ptr(ur),
                                float(temperature), float(tq), int(top_k), float(top_p),
                                _ptr(out["tokens"]), _ptr(out["n_acc"]),
                                _ptr(out["p_draft"]), _ptr(out["q_draft"]), _ptr(out["accept_margin"]),
                                _ptr(out["sample_margin"]), _ptr(out["residual_mass"]), _ptr(out["row_lognorm"]),
                                _ptr(out["nucleus_margin"]), _ptr(cut_in), _ptr(out["row_cut"]),
                                _ptr(out["flags"]), B, K_max, V, dt, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_verify rejected its arguments")
    return out


def decide_multi(P: np.ndarray, Q: np.ndarray, x, ua, ur: float, lib=None):
    """The multi-draft decision of one request on fp64 distributions: P [N, K+1, V] (row 0 of chain
    0 is the shared first position), Q [N, K, V], x and ua [N, K] (ua as float64)."""
    lib = lib or load()
    P = np.ascontiguousarray(P, np.float64)
    N, K1, V = P.shape
    K = K1 - 1
    Q = np.ascontiguousarray(Q, np.float64).reshape(N, K, V) if K > 0 else np.zeros((N, 1, V))
    x = np.ascontiguousarray(x, np.int32).reshape(N, K) if K > 0 else np.zeros((N, 1), np.int32)
    ua = np.ascontiguousarray(ua, np.float64).reshape(N, K) if K > 0 else np.zeros((N, 1))
    tok = np.empty(K + 1, np.int32)
    n = np.empty(1, np.int32)
    ch = np.empty(1, np.int32)
    am = np.empty(max(N * K, 1))
    sm = np.empty(1)
    work = np.empty(2 * V)
    fl = lib.oracle_decide_multi(_ptr(P), _ptr(Q), V, N, K, _ptr(x), _ptr(ua), float(ur), _ptr(tok), _ptr(n),
                                 _ptr(ch), _ptr(am), _ptr(sm), _ptr(work))
    return dict(tokens=tok, n_acc=int(n[0]), chain=int(ch[0]), accept_margin=am[: N * K].reshape(N, K),
                sample_margin=float(sm[0]), flags=int(fl))


def verify_multi(p: np.ndarray, q: Optional[np.ndarray], draft: np.ndarray, ua: Optional[np.ndarray],
                 ur: Optional[np.ndarray], temperature: float, draft_temperature: Optional[float] = None,
                 nthreads: int = 1, lib=None) -> dict:
    """The multi-draft step on host arrays, same argument meaning as the CUDA ``spec_verify_multi``:
    p [B, N, K+1, V], q [B, N, K, V] (float32 or bf16 bits; None at temperature 0), draft and ua
    [B, N, K], ur [B].  Returns tokens [B, K+1], n_acc [B], chain [B], accept_margin [B, N, K],
    sample_margin [B], flags [B]."""
    lib = lib or load()
    p, dt = _logits(p)
    B, N, K1, V = p.shape
    K = K1 - 1
    if q is not None:
        q, dtq = _logits(q)
        assert dtq == dt and q.shape == (B, N, K, V)
    draft = np.ascontiguousarray(draft, np.int32).reshape(B, N, K)
    ua = np.zeros((B, N, K), np.float32) if ua is None else np.ascontiguousarray(ua, np.float32)
    ur = np.zeros(B, np.float32) if ur is None else np.ascontiguousarray(ur, np.float32)
    out = dict(tokens=np.empty((B, K + 1), np.int32), n_acc=np.empty(B, np.int32), chain=np.empty(B, np.int32),
               accept_margin=np.empty((B, N, K)), sample_margin=np.empty(B), flags=np.empty(B, np.int32))
    tq = temperature if draft_temperature is None else draft_temperature
    rc = lib.oracle_verify_multi(_ptr(p), _ptr(q), _ptr(draft), _ptr(ua), _ptr(ur), float(temperature), float(tq),
                                 _ptr(out["tokens"]), _ptr(out["n_acc"]), _ptr(out["chain"]),
                                 _ptr(out["accept_margin"]), _ptr(out["sample_margin"]), _ptr(out["flags"]),
                                 B, N, K, V, dt, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_verify_multi rejected its arguments")
    return out
