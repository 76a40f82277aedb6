"""Python binding of libspecverify.so — the speculative-sampling verify step on one GB300 GPU.

Argument marshalling only: every step of the verify computation runs in the library's CUDA
kernels (``csrc/spec_verify.cu``); PyTorch supplies device memory and the current stream.  There is
no CPU fallback: without the compiled library every call raises.

The C ABI is declared in ``include/spec_verify.h``; the names here mirror it:

* ``verify(p, q, draft, k_per_row, u_accept, u_resample, temperature, top_k, stats=False,
  draft_temperature=None, top_p=1.0)`` -> ``(tokens [B, K+1] int32, num_accepted [B] int32,
  stats dict | None)`` on device tensors, through ``spec_verify_ex``;
* ``verify_host(...)`` the same on host (numpy / CPU torch) arrays through ``spec_verify_host_ex``;
* ``verify_multi(p, q, draft, u_accept, u_resample, temperature, draft_temperature=None)`` ->
  ``(tokens, num_accepted, chain, flags)``: several draft chains per request through
  ``spec_verify_multi``;
* ``workspace_bytes(B, K, V, dtype, top_k)``;
* ``Controller(...)``: the host-side draft-length controller of ``include/spec_control.h``
  (2kiu.com/news/5895634 §4.4 and §7), fed with each batch's ``num_accepted``.

Logits are ``torch.float32`` or ``torch.bfloat16`` tensors ``p [B, K+1, V]`` and ``q [B, K, V]``
(q may be None at temperature 0).  The verify rule (cf-1.com/news/5155685 §2.2,
2kiu.com/news/5895634 §2.2 and §7, gsyq.cn/news/428210 §3.1-§3.3) is restated in the header.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Dict, Optional, Tuple

import numpy as np

from . import _build

SPEC_OK = 0
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA error", 4: "workspace", 5: "timeout"}
DTYPE_F32, DTYPE_BF16 = 0, 1

FLAG_RESIDUAL_ZERO = 1
FLAG_CDF_CLAMP = 2
FLAG_BAD_TOKEN = 4
FLAG_BAD_K = 8
FLAG_NONFINITE = 16
FLAG_TOPK_TIE = 32

MAX_K = 16
MAX_V = 2097152
MAX_TOPK = 256
MAX_DRAFTS = 4

EXPORTS = ("spec_verify_workspace_bytes", "spec_verify", "spec_verify_ex", "spec_verify_host_staging_bytes",
           "spec_verify_host", "spec_verify_host_ex", "spec_verify_static", "spec_verify_status_string",
           "spec_sample_workspace_bytes", "spec_sample", "spec_verify_set_test_hooks",
           "spec_verify_multi_workspace_bytes", "spec_verify_multi")
CONTROL_EXPORTS = ("spec_ctrl_default_config", "spec_ctrl_create", "spec_ctrl_destroy", "spec_ctrl_update",
                   "spec_ctrl_skip", "spec_ctrl_k", "spec_ctrl_window_mean", "spec_ctrl_window_fill",
                   "spec_ctrl_totals")
STATIC_SCRATCH_BYTES = 16 << 20


class SpecVerifyError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: status {code} ({STATUS.get(code, '?')})")
        self.code = code


class StatsStruct(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("p_draft", "q_draft", "accept_margin", "sample_margin", "residual_mass", "row_lognorm", "flags",
                 "pass1_done", "row_cut")]


class SamplingStruct(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("draft_temperature", ctypes.c_float),
                ("top_k", ctypes.c_int32), ("top_p", ctypes.c_float)]


def _sampling(temperature, draft_temperature, top_k, top_p) -> SamplingStruct:
    tq = temperature if draft_temperature is None else draft_temperature
    return SamplingStruct(float(temperature), float(tq), int(top_k), float(top_p))


class ControlConfig(ctypes.Structure):
    _fields_ = [("k_init", ctypes.c_int32), ("k_min", ctypes.c_int32), ("k_max", ctypes.c_int32),
                ("window", ctypes.c_int32), ("raise_above", ctypes.c_float), ("lower_below", ctypes.c_float),
                ("disable_below", ctypes.c_float), ("probe_after", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built (there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if build_if_missing and _build.stale():
                _build.build()
            if not os.path.exists(_build.LIB):
                raise RuntimeError(f"libspecverify.so is not built ({_build.LIB}); run "
                                   "`python -m speculative_decoding_rejection_verify_gb300._build`")
            lib = ctypes.CDLL(_build.LIB)
            P, I, F, Z = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
            lib.spec_verify_workspace_bytes.argtypes = [I, I, I, I, I]
            lib.spec_verify_workspace_bytes.restype = Z
            lib.spec_verify.argtypes = [P, P, P, P, P, P, F, I, P, P, ctypes.POINTER(StatsStruct),
                                        I, I, I, I, P, Z, P]
            lib.spec_verify.restype = I
            lib.spec_verify_ex.argtypes = [P, P, P, P, P, P, ctypes.POINTER(SamplingStruct), P, P,
                                           ctypes.POINTER(StatsStruct), I, I, I, I, P, Z, P]
            lib.spec_verify_ex.restype = I
            lib.spec_verify_host_staging_bytes.argtypes = [I, I, I, I, I, I]
            lib.spec_verify_host_staging_bytes.restype = Z
            lib.spec_verify_host.argtypes = [P, P, P, P, P, P, F, I, P, P, I, I, I, I, P, Z, P]
            lib.spec_verify_host.restype = I
            lib.spec_verify_host_ex.argtypes = [P, P, P, P, P, P, ctypes.POINTER(SamplingStruct), P, P, I, I, I, I,
                                                P, Z, P]
            lib.spec_verify_host_ex.restype = I
            lib.spec_verify_static.argtypes = [P, P, P, P, P, P, F, I, P, P, ctypes.POINTER(StatsStruct),
                                               I, I, I, I, P]
            lib.spec_verify_static.restype = I
            lib.spec_verify_status_string.argtypes = [I]
            lib.spec_verify_status_string.restype = ctypes.c_char_p
            lib.spec_sample_workspace_bytes.argtypes = [I, I, I, I]
            lib.spec_sample_workspace_bytes.restype = Z
            lib.spec_sample.argtypes = [P, P, ctypes.POINTER(SamplingStruct), P, P, I, I, I, P, Z, P]
            lib.spec_sample.restype = I
            lib.spec_verify_multi_workspace_bytes.argtypes = [I, I, I, I, I]
            lib.spec_verify_multi_workspace_bytes.restype = Z
            lib.spec_verify_multi.argtypes = [P, P, P, P, P, ctypes.POINTER(SamplingStruct), P, P, P, P, I, I, I, I,
                                              I, P, Z, P]
            lib.spec_verify_multi.restype = I
            lib.spec_verify_set_test_hooks.argtypes = [I]
            lib.spec_verify_set_test_hooks.restype = None
            CP = ctypes.POINTER(ControlConfig)
            lib.spec_ctrl_default_config.argtypes = [CP]
            lib.spec_ctrl_default_config.restype = None
            lib.spec_ctrl_create.argtypes = [CP]
            lib.spec_ctrl_create.restype = P
            lib.spec_ctrl_destroy.argtypes = [P]
            lib.spec_ctrl_destroy.restype = None
            lib.spec_ctrl_update.argtypes = [P, P, P, I, I]
            lib.spec_ctrl_update.restype = I
            lib.spec_ctrl_skip.argtypes = [P]
            lib.spec_ctrl_skip.restype = I
            lib.spec_ctrl_k.argtypes = [P]
            lib.spec_ctrl_k.restype = I
            lib.spec_ctrl_window_mean.argtypes = [P]
            lib.spec_ctrl_window_mean.restype = ctypes.c_double
            lib.spec_ctrl_window_fill.argtypes = [P]
            lib.spec_ctrl_window_fill.restype = I
            L = ctypes.POINTER(ctypes.c_int64)
            lib.spec_ctrl_totals.argtypes = [P, L, L, L]
            lib.spec_ctrl_totals.restype = None
            _lib = lib
    return _lib


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return DTYPE_F32
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def set_test_hooks(hooks: int) -> None:
    """spec_verify_set_test_hooks (test support: bit 0 makes the streaming pass treat every chunk
    as lost, so a batch comes out flagged non-finite)."""
    load().spec_verify_set_test_hooks(int(hooks))


def workspace_bytes(B: int, K: int, V: int, dtype: int, top_k: int = 0) -> int:
    n = load().spec_verify_workspace_bytes(B, K, V, dtype, top_k)
    if n == 0:
        raise SpecVerifyError(1, "spec_verify_workspace_bytes")
    return n


# Workspaces (per-call scratch) are cached per (device, stream) so repeated calls allocate nothing.
_ws_cache: Dict[Tuple[int, int], object] = {}


def workspace(nbytes: int, device, stream):
    """The cached scratch buffer of ``stream`` (a torch.cuda.Stream), grown to ``nbytes``.  It is
    allocated on that stream, so when a larger one replaces it the caching allocator hands the old
    memory out again only in that stream's order, after the calls that used it."""
    torch = _torch()
    key = (device.index if device.index is not None else torch.cuda.current_device(), stream.cuda_stream)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        with torch.cuda.stream(stream):
            ws = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check(t, name, shape, dtype, device):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)} != {tuple(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype} != {dtype}")
    if t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def verify(p, q, draft, k_per_row=None, u_accept=None, u_resample=None, temperature: float = 1.0,
           top_k: int = 0, stats: bool = False, workspace_tensor=None, stream=None, out=None,
           pass1_event=None, draft_temperature: Optional[float] = None, top_p: float = 1.0):
    """Run spec_verify_ex on device tensors; returns (tokens, num_accepted, stats | None).

    ``draft_temperature``: T_q of the q rows (None = ``temperature``); ``top_p``: nucleus mass
    (1 = off).  ``out``: optional (tokens, num_accepted) tensors to write into.  ``stream``: a
    torch.cuda.Stream (default: the current stream).  ``pass1_event``: a torch.cuda.Event
    recorded between the streaming pass and the per-request pass.  The call is asynchronous."""
    torch = _torch()
    lib = load()
    if p.dim() != 3:
        raise ValueError("p must be [B, K+1, V]")
    B, K1, V = p.shape
    K = K1 - 1
    dev = p.device
    if dev.type != "cuda":
        raise ValueError("verify() takes CUDA tensors; use verify_host() for host arrays")
    dt = _dtype_code(p)
    _check(p, "p", (B, K + 1, V), p.dtype, dev)
    if q is not None:
        _check(q, "q", (B, K, V), p.dtype, dev)
    if draft is not None:
        _check(draft, "draft", (B, K), torch.int32, dev)
    if k_per_row is not None:
        _check(k_per_row, "k_per_row", (B,), torch.int32, dev)
    if u_accept is not None:
        _check(u_accept, "u_accept", (B, K), torch.float32, dev)
    if u_resample is not None:
        _check(u_resample, "u_resample", (B,), torch.float32, dev)
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    handle = st.cuda_stream
    if out is None:
        tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
        nacc = torch.empty((B,), dtype=torch.int32, device=dev)
    else:
        tokens, nacc = out
    sd = None
    sp = None
    if stats:
        f32 = dict(dtype=torch.float32, device=dev)
        sd = dict(p_draft=torch.empty((B, K), **f32), q_draft=torch.empty((B, K), **f32),
                  accept_margin=torch.empty((B, K), **f32), sample_margin=torch.empty((B,), **f32),
                  residual_mass=torch.empty((B,), **f32), row_lognorm=torch.empty((B, 2 * K + 1), **f32),
                  flags=torch.empty((B,), dtype=torch.int32, device=dev),
                  row_cut=torch.empty((B, 2 * K + 1), **f32))
        sp = StatsStruct(**{k: v.data_ptr() for k, v in sd.items()})
    if pass1_event is not None:
        if pass1_event.cuda_event == 0:  # torch creates the event on its first record
            pass1_event.record(st)
        sp = sp if sp is not None else StatsStruct()
        sp.pass1_done = pass1_event.cuda_event
    nbytes = workspace_bytes(B, K, V, dt, top_k)
    ws = workspace_tensor if workspace_tensor is not None else workspace(nbytes, dev, st)
    smp = _sampling(temperature, draft_temperature, top_k, top_p)
    rc = lib.spec_verify_ex(_ptr(p), _ptr(q), _ptr(draft), _ptr(k_per_row), _ptr(u_accept), _ptr(u_resample),
                            ctypes.byref(smp), tokens.data_ptr(), nacc.data_ptr(),
                            ctypes.byref(sp) if sp is not None else None, B, K, V, dt, ws.data_ptr(),
                            ws.numel(), handle)
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_verify_ex")
    return tokens, nacc, sd


def sample(logits, u=None, temperature: float = 1.0, top_k: int = 0, top_p: float = 1.0, prob: bool = True,
           workspace_tensor=None, stream=None, out=None):
    """Draw one token per row of ``logits`` [rows, V] (device) with the uniforms ``u`` [rows]
    through ``spec_sample``; returns (tokens [rows] int32, q(x) [rows] float32 | None)."""
    torch = _torch()
    lib = load()
    if logits.dim() != 2:
        raise ValueError("logits must be [rows, V]")
    rows, V = logits.shape
    dev = logits.device
    dt = _dtype_code(logits)
    _check(logits, "logits", (rows, V), logits.dtype, dev)
    if u is not None:
        _check(u, "u", (rows,), torch.float32, dev)
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    if out is None:
        tokens = torch.empty((rows,), dtype=torch.int32, device=dev)
        pr = torch.empty((rows,), dtype=torch.float32, device=dev) if prob else None
    else:
        tokens, pr = out
    nbytes = lib.spec_sample_workspace_bytes(rows, V, dt, int(top_k))
    if nbytes == 0:
        raise SpecVerifyError(1, "spec_sample_workspace_bytes")
    ws = workspace_tensor if workspace_tensor is not None else workspace(nbytes, dev, st)
    smp = SamplingStruct(float(temperature), float(temperature), int(top_k), float(top_p))
    rc = lib.spec_sample(_ptr(logits), _ptr(u), ctypes.byref(smp), tokens.data_ptr(),
                         None if pr is None else pr.data_ptr(), rows, V, dt, ws.data_ptr(), ws.numel(),
                         st.cuda_stream)
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_sample")
    return tokens, pr


def verify_multi(p, q, draft, u_accept=None, u_resample=None, temperature: float = 1.0,
                 draft_temperature: Optional[float] = None, workspace_tensor=None, stream=None, out=None):
    """spec_verify_multi on device tensors: p [B, N, K+1, V], q [B, N, K, V] (None at temperature 0),
    draft and u_accept [B, N, K], u_resample [B].  Returns (tokens [B, K+1], num_accepted [B],
    chain [B], flags [B]) int32 tensors; the call is asynchronous."""
    torch = _torch()
    lib = load()
    if p.dim() != 4:
        raise ValueError("p must be [B, N, K+1, V]")
    B, N, K1, V = p.shape
    K = K1 - 1
    dev = p.device
    dt = _dtype_code(p)
    _check(p, "p", (B, N, K + 1, V), p.dtype, dev)
    if q is not None:
        _check(q, "q", (B, N, K, V), p.dtype, dev)
    if draft is not None:
        _check(draft, "draft", (B, N, K), torch.int32, dev)
    if u_accept is not None:
        _check(u_accept, "u_accept", (B, N, K), torch.float32, dev)
    if u_resample is not None:
        _check(u_resample, "u_resample", (B,), torch.float32, dev)
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    if out is None:
        i32 = dict(dtype=torch.int32, device=dev)
        out = (torch.empty((B, K + 1), **i32), torch.empty((B,), **i32), torch.empty((B,), **i32),
               torch.empty((B,), **i32))
    tokens, nacc, chain, flags = out
    nbytes = lib.spec_verify_multi_workspace_bytes(B, N, K, V, dt)
    if nbytes == 0:
        raise SpecVerifyError(1, "spec_verify_multi_workspace_bytes")
    ws = workspace_tensor if workspace_tensor is not None else workspace(nbytes, dev, st)
    smp = _sampling(temperature, draft_temperature, 0, 1.0)
    rc = lib.spec_verify_multi(_ptr(p), _ptr(q), _ptr(draft), _ptr(u_accept), _ptr(u_resample), ctypes.byref(smp),
                               tokens.data_ptr(), nacc.data_ptr(), _ptr(chain), _ptr(flags), B, N, K, V, dt,
                               ws.data_ptr(), ws.numel(), st.cuda_stream)
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_verify_multi")
    return tokens, nacc, chain, flags


_stage_cache: Dict[int, object] = {}


def staging_bytes(B: int, K: int, V: int, dtype: int, top_k: int, ragged: bool) -> int:
    n = load().spec_verify_host_staging_bytes(B, K, V, dtype, top_k, int(ragged))
    if n == 0:
        raise SpecVerifyError(1, "spec_verify_host_staging_bytes")
    return n


def verify_host(p, q, draft, k_per_row=None, u_accept=None, u_resample=None, temperature: float = 1.0,
                top_k: int = 0, staging=None, device=None, stream=None, out=None,
                draft_temperature: Optional[float] = None, top_p: float = 1.0):
    """spec_verify_host on host arrays (numpy, or CPU torch tensors; pinned memory recommended).

    ``p``/``q``: float32 arrays or bf16 bits as uint16 (numpy) / torch.bfloat16 (CPU tensors).
    Returns (tokens [B, K+1] int32, num_accepted [B] int32) as numpy arrays (or writes ``out``).
    The call blocks until the results are on the host."""
    torch = _torch()
    lib = load()

    def host(a, dtype=None):
        if a is None:
            return None, None
        if isinstance(a, np.ndarray):
            a = np.ascontiguousarray(a if dtype is None else a.astype(dtype, copy=False))
            return a, a.ctypes.data
        if a.device.type != "cpu" or not a.is_contiguous():
            raise ValueError("verify_host takes contiguous host arrays")
        return a, a.data_ptr()

    if isinstance(p, np.ndarray):
        dt = DTYPE_BF16 if p.dtype == np.uint16 else DTYPE_F32
        if p.dtype not in (np.uint16, np.float32):
            raise TypeError("p must be float32 or bf16 bits (uint16)")
    else:
        dt = _dtype_code(p)
    B, K1, V = p.shape
    K = K1 - 1
    p, pp = host(p)
    q, qp = host(q)
    draft, dp = host(draft, np.int32)
    k_per_row, kp = host(k_per_row, np.int32)
    u_accept, ap = host(u_accept, np.float32)
    u_resample, rp = host(u_resample, np.float32)
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    nbytes = staging_bytes(B, K, V, dt, top_k, k_per_row is not None)
    if staging is None:
        key = dev.index if dev.index is not None else torch.cuda.current_device()
        staging = _stage_cache.get(key)
        if staging is None or staging.numel() < nbytes:
            staging = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
            _stage_cache[key] = staging
    if out is None:
        tokens = np.empty((B, K + 1), np.int32)
        nacc = np.empty(B, np.int32)
        tp, npp = tokens.ctypes.data, nacc.ctypes.data
    else:
        tokens, nacc = out
        tp, npp = (tokens.ctypes.data, nacc.ctypes.data) if isinstance(tokens, np.ndarray) else \
            (tokens.data_ptr(), nacc.data_ptr())
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    smp = _sampling(temperature, draft_temperature, top_k, top_p)
    rc = lib.spec_verify_host_ex(pp, qp, dp, kp, ap, rp, ctypes.byref(smp), tp, npp, B, K, V, dt,
                                 staging.data_ptr(), staging.numel(), st.cuda_stream)
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_verify_host_ex")
    return tokens, nacc


class Controller:
    """The draft-length controller (``include/spec_control.h``): record each verified batch's
    ``num_accepted`` with :meth:`update` (or a batch decoded without drafts with :meth:`skip`);
    both return the K for the next batch, 0 meaning speculation is off.  Host-side; keyword
    arguments override the pages' defaults (k_init 4, k in [2, 10], window 100, raise above 0.8,
    lower below 0.6, switch off below 0.5, probe again after 100 batches)."""

    def __init__(self, **overrides):
        lib = load()
        cfg = ControlConfig()
        lib.spec_ctrl_default_config(ctypes.byref(cfg))
        for k, v in overrides.items():
            if not hasattr(cfg, k):
                raise TypeError(f"unknown controller setting {k}")
            setattr(cfg, k, v)
        self.config = cfg
        self._lib = lib
        self._h = lib.spec_ctrl_create(ctypes.byref(cfg))
        if not self._h:
            raise ValueError("controller settings out of range")

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            self._lib.spec_ctrl_destroy(h)

    def update(self, num_accepted, k_per_row=None, K_used: Optional[int] = None) -> int:
        """Record one verified batch (host arrays or tensors; copied to the host if needed)."""
        n = np.ascontiguousarray(_host_i32(num_accepted))
        kp = None if k_per_row is None else np.ascontiguousarray(_host_i32(k_per_row))
        K = self.k if K_used is None else int(K_used)
        r = self._lib.spec_ctrl_update(self._h, n.ctypes.data, None if kp is None else kp.ctypes.data,
                                       int(n.shape[0]), K)
        if r < 0:
            raise ValueError("spec_ctrl_update rejected its arguments")
        return r

    def skip(self) -> int:
        return self._lib.spec_ctrl_skip(self._h)

    @property
    def k(self) -> int:
        return self._lib.spec_ctrl_k(self._h)

    @property
    def window_mean(self) -> float:
        return self._lib.spec_ctrl_window_mean(self._h)

    @property
    def window_fill(self) -> int:
        return self._lib.spec_ctrl_window_fill(self._h)

    def totals(self) -> Tuple[int, int, int]:
        a, p, b = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        self._lib.spec_ctrl_totals(self._h, ctypes.byref(a), ctypes.byref(p), ctypes.byref(b))
        return a.value, p.value, b.value


def _host_i32(a) -> np.ndarray:
    if hasattr(a, "detach"):  # a torch tensor
        a = a.detach().cpu().numpy()
    return np.asarray(a, dtype=np.int32)
