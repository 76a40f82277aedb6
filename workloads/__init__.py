"""Seeded synthetic inputs for the speculative-sampling verify step.

This module serves the tests, the benchmark and the oracle alike, and holds none of the
verify step's arithmetic (no normaliser, no ratio test, no residual, no inverse CDF; the one
weighting in it is the draft sampler's own nucleus cut, made with numpy's cumulative sum).
It plays the part of the two models around the verify step:

* the draft model's logits: z_q = 3 * N(0, 1) - 1.1 * ln(rank_v), with rank a seeded
  permutation of 1..V shared by every row of a workload (a Zipf-like bias);
* the target model's logits: z_p = z_q + tau * N(0, 1) at the draft positions, and a fresh
  base row plus noise at the bonus position j = K_b;
* the draft model's own sampling of the draft tokens, by the Gumbel-max trick
  (argmax_v z_q[v] / T_q + G_v over the kept set; plain argmax when T == 0).  Gumbel-max
  draws exactly from softmax(z_q / T_q) on that set, the law the verify step assumes the draft
  used.  The kept set is the draft sampler's own truncation: top-k, then, when the workload sets
  top_p < 1, the most likely tokens up to mass top_p (the tied group at the cut whole);
* the uniforms the verify step consumes, on the grid k * 2^-24 so both sides see identical
  float32 values.

Logits are rounded to the workload's dtype (bf16 round-to-nearest-even, carried as uint16
bits) before anything else reads them.  Every request b draws from its own counter-keyed
streams ``(seed, stream, b)``, so any subset of requests of a full-size workload can be
regenerated on its own, bit for bit.

The target-noise scale tau of each workload is tuned so that the mean per-row acceptance
probability sum_v min(P, Q) hits the workload's alpha; the tuned values in ``tau.json`` are
written by ``oracle/tune_tau.py`` (which calls only the oracle and this module).
"""
from __future__ import annotations

import dataclasses
import json
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
TAU_FILE = os.path.join(_HERE, "tau.json")

SIGMA = 3.0          # spread of the base logits
ZIPF = 1.1           # bias_v = -ZIPF * ln(rank_v)
UGRID = 2.0 ** -24   # uniforms are k * UGRID, k in [0, 2^24)
BF16_NAN = 0x7FC0

# Streams of each request's counter-keyed generator (seed, stream, request).
_S_RANK, _S_ROWS, _S_KB, _S_DRAFT, _S_UNIF = 0, 1, 2, 3, 4


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic verify batch: sizes, sampling parameters and seeds."""
    name: str
    B: int
    K: int                       # K_max
    V: int
    dtype: str                   # "f32" or "bf16"
    temperature: float
    top_k: int
    seed: int
    alpha: Optional[float]       # target mean acceptance (None: tau given directly)
    tau: Optional[float] = None  # target-noise scale; None = look up tau.json
    ragged: Optional[tuple] = None  # (lo, hi) inclusive range of K_b, or None for K_b = K
    greedy: bool = False          # draft tokens by argmax, verified at T = 0
    draft_temperature: Optional[float] = None  # T_q of the draft; None = temperature
    top_p: float = 1.0            # nucleus mass of both sides; 1 = off

    @property
    def tq(self) -> float:
        return self.temperature if self.draft_temperature is None else self.draft_temperature

    @property
    def key(self) -> str:
        """Name of the tuned tau (a greedy batch shares the tau of its sampled twin)."""
        return self.name if self.alpha is None or self.name != "c5" else f"c5_a{self.alpha:g}"

    @property
    def label(self) -> str:
        return "c5_greedy" if self.greedy else self.key

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads (sizes, dtypes, temperatures, top-k and alpha targets as specified for this
# step; seeds 1001..1005, and 1051..1054 for the alpha sweep of the largest batch).
WORKLOADS: Dict[str, Workload] = {
    "c1": Workload("c1", B=1, K=4, V=1000, dtype="f32", temperature=1.0, top_k=0, seed=1001,
                   alpha=None, tau=0.5),
    "c2": Workload("c2", B=8, K=5, V=32000, dtype="bf16", temperature=0.8, top_k=0, seed=1002, alpha=0.8),
    "c3": Workload("c3", B=64, K=6, V=128256, dtype="bf16", temperature=1.0, top_k=0, seed=1003, alpha=0.6),
    "c4": Workload("c4", B=256, K=8, V=152064, dtype="f32", temperature=0.7, top_k=50, seed=1004,
                   alpha=0.75, ragged=(2, 8)),
}
for _a, _s in ((0.4, 1051), (0.6, 1052), (0.8, 1053), (0.9, 1054)):
    WORKLOADS[f"c5_a{_a:g}"] = Workload("c5", B=1024, K=4, V=128256, dtype="bf16", temperature=1.0,
                                        top_k=0, seed=_s, alpha=_a)
WORKLOADS["c5_greedy"] = WORKLOADS["c5_a0.8"].with_(temperature=0.0, greedy=True)
# Sampling-parameter variants of the largest batch: nucleus truncation on both sides, and a
# draft that samples at its own, lower temperature (T_q = 0.5 under a target at T = 1).
WORKLOADS["c5_topp0.9"] = Workload("c5_topp0.9", B=1024, K=4, V=128256, dtype="bf16", temperature=1.0,
                                   top_k=0, seed=1061, alpha=0.8, top_p=0.9)
WORKLOADS["c5_tq0.5"] = Workload("c5_tq0.5", B=1024, K=4, V=128256, dtype="bf16", temperature=1.0,
                                 top_k=0, seed=1062, alpha=0.45, draft_temperature=0.5)
# Multi-draft verify: 256 requests of 4 draft chains, 4 drafts each, over the largest batch's
# vocabulary (the target's noise scale 0.5 between each chain's first draft and the target).
WORKLOADS["multi_c5"] = Workload("multi_c5", B=256, K=4, V=128256, dtype="bf16", temperature=1.0, top_k=0,
                                 seed=1081, alpha=None, tau=0.5)
# Draft-token sampling (the step before verification): 1024 rows of 128256 bf16 logits, one draw
# each; a batch of requests with no drafts, whose one row is the row sampled from.
WORKLOADS["sample_c5"] = Workload("sample_c5", B=1024, K=0, V=128256, dtype="bf16", temperature=1.0,
                                  top_k=0, seed=1071, alpha=None, tau=0.5)


def get(name: str, **overrides) -> Workload:
    """A named workload, optionally with fields overridden (e.g. a smaller B for tests)."""
    return WORKLOADS[name].with_(**overrides) if overrides else WORKLOADS[name]


def load_tau() -> Dict[str, float]:
    if not os.path.exists(TAU_FILE):
        return {}
    with open(TAU_FILE) as f:
        return json.load(f)["tau"]


def tau_of(w: Workload) -> float:
    if w.tau is not None:
        return w.tau
    table = load_tau()
    if w.key not in table:
        raise KeyError(f"no tuned tau for {w.key}; run oracle/tune_tau.py")
    return table[w.key]


def _rng(seed: int, stream: int, b: int = 0) -> np.random.Generator:
    return np.random.default_rng([seed, stream, b])


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def as_f32(a: np.ndarray) -> np.ndarray:
    """Logits as float32 values (exact for both storage types)."""
    return bf16_bits_to_f32(a) if a.dtype == np.uint16 else a


def bias(w: Workload) -> np.ndarray:
    rank = _rng(w.seed, _S_RANK).permutation(w.V).astype(np.float64) + 1.0
    return (-ZIPF * np.log(rank)).astype(np.float32)


def k_per_row(w: Workload, requests: Optional[Sequence[int]] = None) -> np.ndarray:
    """K_b of each listed request (all of them by default); each from its own stream."""
    reqs = range(w.B) if requests is None else requests
    if w.ragged is None:
        return np.full(len(reqs), w.K, np.int32)
    lo, hi = w.ragged
    return np.array([_rng(w.seed, _S_KB, int(b)).integers(lo, hi + 1) for b in reqs], np.int32)


def _draft_token(zq: np.ndarray, T: float, top_k: int, greedy: bool, g: np.random.Generator,
                 top_p: float = 1.0) -> int:
    """The draft model's own sample from its row (Gumbel-max; argmax when greedy)."""
    z = zq.astype(np.float64)
    if greedy:
        return int(np.argmax(z))
    if 0 < top_k < z.shape[0]:
        kth = np.partition(z, z.shape[0] - top_k)[z.shape[0] - top_k]
        z = np.where(z >= kth, z, -np.inf)
    if top_p < 1.0:  # the draft sampler's nucleus: most likely tokens up to mass top_p
        w = np.exp((z - z.max()) / T)
        order = np.argsort(-z, kind="stable")
        cum = np.cumsum(w[order]) / w.sum()
        cut = z[order[min(int(np.searchsorted(cum, np.float32(top_p))), len(z) - 1)]]
        z = np.where(z >= cut, z, -np.inf)
    u = g.random(z.shape[0])
    gumbel = -np.log(-np.log(np.clip(u, 1e-300, None)))
    return int(np.argmax(z / T + gumbel))


def _request(w: Workload, tau: float, bias_v: np.ndarray, Kb: int, b: int, p_out, q_out, x_out):
    """Fill one request's rows (p_out [K+1, V], q_out [K, V]) and draft tokens in place."""
    r = _rng(w.seed, _S_ROWS, b)
    V = w.V
    bf = w.dtype == "bf16"
    for j in range(Kb + 1):
        zq = SIGMA * r.standard_normal(V, dtype=np.float32) + bias_v
        zp = zq + np.float32(tau) * r.standard_normal(V, dtype=np.float32)
        if bf:
            p_out[j] = to_bf16_bits(zp)
            if j < Kb:
                q_out[j] = to_bf16_bits(zq)
        else:
            p_out[j] = zp
            if j < Kb:
                q_out[j] = zq
    # padding rows are never read by the verify step: fill them with NaN so a stray read shows
    nan = BF16_NAN if bf else np.nan
    p_out[Kb + 1:] = nan
    q_out[Kb:] = nan
    g = _rng(w.seed, _S_DRAFT, b)
    x_out[:] = 0
    for j in range(Kb):
        zq = bf16_bits_to_f32(q_out[j]) if bf else q_out[j]
        x_out[j] = _draft_token(zq, w.tq, w.top_k, w.greedy, g, w.top_p)


def uniforms(w: Workload, requests: Sequence[int]):
    """(ua [n, K_max], ur [n]) on the 2^-24 grid for the given requests."""
    ua = np.empty((len(requests), w.K), np.float32)
    ur = np.empty(len(requests), np.float32)
    for i, b in enumerate(requests):
        k = _rng(w.seed, _S_UNIF, int(b)).integers(0, 1 << 24, size=w.K + 1)
        ua[i] = k[: w.K].astype(np.float32) * np.float32(UGRID)
        ur[i] = np.float32(k[w.K]) * np.float32(UGRID)
    return ua, ur


def generate(w: Workload, requests: Optional[Sequence[int]] = None, threads: int = 0,
             tau: Optional[float] = None) -> dict:
    """Materialise a workload (or the listed requests of it) as host arrays.

    Returns dict(p [n, K+1, V], q [n, K, V] (float32, or uint16 bf16 bits), draft [n, K] int32,
    k_per_row [n] int32, ua [n, K] f32, ur [n] f32, temperature, draft_temperature, top_k, top_p,
    workload)."""
    tau = tau_of(w) if tau is None else tau
    reqs = np.arange(w.B) if requests is None else np.asarray(requests, np.int64)
    n = len(reqs)
    st = np.uint16 if w.dtype == "bf16" else np.float32
    p = np.empty((n, w.K + 1, w.V), st)
    q = np.empty((n, w.K, w.V), st)
    x = np.zeros((n, w.K), np.int32)
    bias_v = bias(w)
    kb = k_per_row(w, reqs)

    def one(i):
        _request(w, tau, bias_v, int(kb[i]), int(reqs[i]), p[i], q[i], x[i])

    threads = threads or min(16, os.cpu_count() or 1)
    if n > 1 and threads > 1:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(one, range(n)))
    else:
        for i in range(n):
            one(i)
    ua, ur = uniforms(w, reqs)
    return dict(p=p, q=q, draft=x, k_per_row=kb.astype(np.int32), ua=ua, ur=ur,
                temperature=float(w.temperature), draft_temperature=float(w.tq), top_k=int(w.top_k),
                top_p=float(w.top_p), workload=w)


_S_MULTI = 10  # first stream of the multi-draft generator


def generate_multi(w: Workload, N: int, requests: Optional[Sequence[int]] = None, tau: Optional[float] = None) -> dict:
    """N draft chains per request (w.K drafts each), for the multi-draft verify step.

    At the shared first position the target's logits are a base row and each chain's draft logits
    that base plus tau * N(0, 1) of its own; along chain n (positions 1..K-1) the draft logits are
    fresh base rows and the target's the same plus noise, and row K is a fresh base row plus noise
    (the target after the chain's prefix).  Row 0 of chains n > 0 is NaN: the step never reads it.
    Draft tokens are the chains' own samples (Gumbel-max at T_q; argmax when greedy).
    Returns dict(p [n, N, K+1, V], q [n, N, K, V], draft [n, N, K], ua [n, N, K], ur [n], temperature,
    draft_temperature, N, workload)."""
    tau = (0.5 if w.tau is None else w.tau) if tau is None else tau
    reqs = np.arange(w.B) if requests is None else np.asarray(requests, np.int64)
    n_req, K, V = len(reqs), w.K, w.V
    bf = w.dtype == "bf16"
    st = np.uint16 if bf else np.float32
    p = np.empty((n_req, N, K + 1, V), st)
    q = np.empty((n_req, N, K, V), st)
    x = np.zeros((n_req, N, K), np.int32)
    ua = np.empty((n_req, N, K), np.float32)
    ur = np.empty(n_req, np.float32)
    bias_v = bias(w)
    cast = to_bf16_bits if bf else (lambda a: a)
    nan = BF16_NAN if bf else np.nan

    def one(i):
        b = int(reqs[i])
        r = _rng(w.seed, _S_MULTI, b)
        base0 = SIGMA * r.standard_normal(V, dtype=np.float32) + bias_v
        for n in range(N):
            p[i, n, 0] = cast(base0) if n == 0 else nan
            if K > 0:
                q[i, n, 0] = cast(base0 + np.float32(tau) * r.standard_normal(V, dtype=np.float32))
            for j in range(1, K + 1):
                base = SIGMA * r.standard_normal(V, dtype=np.float32) + bias_v
                p[i, n, j] = cast(base + np.float32(tau) * r.standard_normal(V, dtype=np.float32))
                if j < K:
                    q[i, n, j] = cast(base)
            g = _rng(w.seed, _S_MULTI + 1 + n, b)
            for j in range(K):
                x[i, n, j] = _draft_token(as_f32(q[i, n, j]), w.tq, 0, w.greedy, g)
        k = _rng(w.seed, _S_MULTI + 1 + N, b).integers(0, 1 << 24, size=N * K + 1)
        ua[i] = (k[: N * K].astype(np.float32) * np.float32(UGRID)).reshape(N, K)
        ur[i] = np.float32(k[N * K]) * np.float32(UGRID)

    threads = min(16, os.cpu_count() or 1)
    if n_req > 1 and threads > 1:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(one, range(n_req)))
    else:
        for i in range(n_req):
            one(i)
    return dict(p=p, q=q, draft=x, ua=ua, ur=ur, temperature=float(w.temperature),
                draft_temperature=float(w.tq), N=N, workload=w)


def multi_algorithmic_bytes(w: Workload, N: int, B: int) -> int:
    """Bytes one multi-draft pass must read at least: the shared first row, every chain's target
    rows 1..K and (unless greedy) its draft rows, once each, plus tokens, uniforms and outputs."""
    s = 2 if w.dtype == "bf16" else 4
    rows = 1 + N * w.K + (0 if w.temperature == 0.0 else N * w.K)
    per_req = 4 * N * w.K * 2 + 4 + 4 * (w.K + 1) + 4 * 3
    return B * (rows * w.V * s + per_req)


def algorithmic_bytes(w: Workload, kb: np.ndarray) -> int:
    """Bytes one verify pass must read at least: every valid logit row once (p rows 0..K_b and,
    unless greedy, q rows 0..K_b-1), plus the per-request draft tokens, uniforms and outputs."""
    s = 2 if w.dtype == "bf16" else 4
    kb = np.asarray(kb, np.int64)
    rows = (kb + 1).sum() if w.temperature == 0.0 else (2 * kb + 1).sum()
    per_req = 4 * w.K * 2 + 4 + 4 + 4 * (w.K + 1) + 4  # draft, ua, ur, k, tokens, n_acc
    return int(rows) * w.V * s + len(kb) * per_req
