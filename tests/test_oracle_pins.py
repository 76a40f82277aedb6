"""Pins of the fp64 oracle against what the pages and the mathematics fix (CPU only).

* Losslessness (cf-1.com §2.2, 2kiu.com §2.2: the accept/resample rule yields samples of p):
  exhaustive breakpoint enumeration at V = 4, K <= 3 — every decision is piecewise constant in
  each uniform, so splitting [0, 1) at every breakpoint and weighting each piece by its length
  gives the exact law of every emitted token; it must equal p at that position to 1e-12.
* The same in practice: chi-square over 1e6 seeded trials at V = 1000, K = 4.
* The acceptance count (gsyq.cn §3.2, 2kiu.com §3.1): the mean number of emitted tokens on inputs
  with exactly known alpha matches (1 - alpha^(K+1)) / (1 - alpha); the formula itself is pinned
  to the values the pages print (tests/golden/expected_accepted.txt).
* Normalisation with temperature and top-k (gsyq.cn §3.3) against a library softmax / top-k.
* Greedy limit against a library argmax (first index on ties).
* Planted mistakes: variants of oracle.c with a plausible error each must fail a pin.
"""
import os
import subprocess

import numpy as np
import pytest
import torch
from scipy import stats

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------------------------
def _pieces(weights):
    """Sub-intervals of [0, 1) on which an inverse-CDF draw over ``weights`` is constant.

    The edges are a superset of the draw's breakpoints; a wrong edge only makes the law check
    fail, never pass."""
    w = np.asarray(weights, np.float64)
    C = np.cumsum(w) / w.sum()
    edges = np.unique(np.clip(np.concatenate([[0.0], C, [1.0]]), 0.0, 1.0))
    return [(lo, hi) for lo, hi in zip(edges[:-1], edges[1:]) if hi > lo]


def enumerate_law(P, Q, lib=None):
    """Exact law of the emitted tokens under the oracle's decisions.

    Returns law [K+1, V]: law[i, v] = Pr(position i is emitted and equals v)."""
    K, V = P.shape[0] - 1, P.shape[1]
    law = np.zeros((K + 1, V))

    def call(xs, uas, ur, w):
        xs = list(xs) + [0] * (K - len(xs))
        uas = list(uas) + [0.5] * (K - len(uas))
        res = oracle.decide(P, Q, xs, uas, ur, lib=lib)
        for i in range(res["n_acc"] + 1):
            law[i, res["tokens"][i]] += w

    def dfs(j, xs, uas, w):
        if j == K:  # every draft accepted: the bonus draw from p at position K
            for lo, hi in _pieces(P[K]):
                call(xs, uas, 0.5 * (lo + hi), w * (hi - lo))
            return
        for x in range(V):
            if Q[j, x] <= 0.0:
                continue  # the draft never proposes it
            t = min(1.0, P[j, x] / Q[j, x])
            if t > 0.0:
                dfs(j + 1, xs + [x], uas + [0.5 * t], w * Q[j, x] * t)
            if t < 1.0:
                r = np.maximum(P[j] - Q[j], 0.0)
                for lo, hi in _pieces(r if r.sum() > 0 else P[j]):
                    call(xs + [x], uas + [0.5 * (1.0 + t)], 0.5 * (lo + hi), w * Q[j, x] * (1.0 - t) * (hi - lo))

    dfs(0, [], [], 1.0)
    return law


def check_lossless(P, Q, lib=None, tol=1e-12):
    """law[i] == Pr(n_acc >= i) * P[i] with Pr(n_acc >= i) = prod_{l<i} sum_v min(P_l, Q_l)."""
    law = enumerate_law(P, Q, lib)
    K = P.shape[0] - 1
    reach = 1.0
    for i in range(K + 1):
        np.testing.assert_allclose(law[i], reach * P[i], rtol=0, atol=tol)
        if i < K:
            reach *= np.minimum(P[i], Q[i]).sum()


def _dirichlet(rng, V, zeros=0):
    d = rng.dirichlet(np.ones(V))
    if zeros:
        d[rng.choice(V, zeros, replace=False)] = 0.0
        d /= d.sum()
    return d


# ----------------------------------------------------------------------------------------------
# losslessness by enumeration
# ----------------------------------------------------------------------------------------------
@pytest.mark.parametrize("K", [1, 2, 3])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_enumeration_random(K, seed):
    rng = np.random.default_rng(seed)
    V = 4
    P = np.stack([_dirichlet(rng, V, zeros=(seed + j) % 2) for j in range(K + 1)])
    Q = np.stack([_dirichlet(rng, V, zeros=(seed + j + 1) % 2) for j in range(K)])
    check_lossless(P, Q)


def test_enumeration_special_cases():
    V = 4
    e = np.eye(V)
    cases = [
        # p == q: every draft accepted
        (np.array([[.1, .2, .3, .4], [.4, .3, .2, .1], [.25, .25, .25, .25]]),
         np.array([[.1, .2, .3, .4], [.4, .3, .2, .1]])),
        # disjoint supports: always rejected, resample law is p
        (np.array([[.5, .5, 0, 0], [.3, .3, .2, .2]]), np.array([[0, 0, .5, .5]])),
        # q one-hot at x with p(x) = 0
        (np.array([[.2, .3, .5, 0], [.1, .1, .1, .7]]), np.array([e[3]])),
        # p one-hot at the draft token: accepted whenever q(x) > 0
        (np.array([e[2], e[1], [.1, .2, .3, .4]]), np.array([[.1, .1, .7, .1], e[1]])),
        # q wider than p, then p wider than q
        (np.array([[0, .5, .5, 0], [.25, .25, .25, .25], [.9, .1, 0, 0]]),
         np.array([[.25, .25, .25, .25], [0, 0, .5, .5]])),
    ]
    for P, Q in cases:
        check_lossless(np.asarray(P, float), np.asarray(Q, float))


def test_p_equals_q_always_accepts():
    rng = np.random.default_rng(5)
    P = np.stack([_dirichlet(rng, 50) for _ in range(4)])
    Q = P[:3].copy()
    N = 2000
    x = np.stack([rng.choice(50, N, p=Q[j]) for j in range(3)], 1)
    ua = rng.integers(0, 1 << 24, (N, 3)) * 2.0 ** -24
    ur = rng.integers(0, 1 << 24, N) * 2.0 ** -24
    tok, n, fl = oracle.decide_trials(P, Q, x, ua, ur)
    assert (n == 3).all() and (tok[:, :3] == x).all() and (fl == 0).all()


# ----------------------------------------------------------------------------------------------
# losslessness in practice: chi-square over 1e6 trials
# ----------------------------------------------------------------------------------------------
def _sample_from(rng, Prow, n):
    c = np.cumsum(Prow)
    return np.minimum(np.searchsorted(c, rng.random(n) * c[-1], side="right"), len(Prow) - 1)


def chisquare_pvalues(P, Q, N, seed, lib=None):
    rng = np.random.default_rng(seed)
    K, V = P.shape[0] - 1, P.shape[1]
    x = np.stack([_sample_from(rng, Q[j], N) for j in range(K)], 1).astype(np.int32)
    ua = (rng.integers(0, 1 << 24, (N, K)) * 2.0 ** -24).astype(np.float32)
    ur = (rng.integers(0, 1 << 24, N) * 2.0 ** -24).astype(np.float32)
    tok, n, fl = oracle.decide_trials(P, Q, x, ua, ur, lib=lib)
    pvals = []
    for i in range(K + 1):
        sel = n >= i
        obs = np.bincount(tok[sel, i], minlength=V).astype(float)
        exp = sel.sum() * P[i]
        small = exp < 5.0  # merge the bins expected below 5 into one
        o, e = obs[~small], exp[~small]
        if small.any():
            o, e = np.append(o, obs[small].sum()), np.append(e, exp[small].sum())
            if e[-1] < 5.0 and len(e) > 1:  # still too small: fold it into the smallest bin
                i0 = int(np.argmin(e[:-1]))
                o[i0] += o[-1]
                e[i0] += e[-1]
                o, e = o[:-1], e[:-1]
        e *= o.sum() / e.sum()
        pvals.append(stats.chisquare(o, e).pvalue)
    # the number of accepted drafts: Pr(n = m) = prod_{l<m} a_l * (1 - a_m), Pr(n = K) = prod a_l
    a = [np.minimum(P[l], Q[l]).sum() for l in range(K)]
    pm = [np.prod(a[:m]) * (1 - a[m]) for m in range(K)] + [np.prod(a)]
    obs = np.bincount(n, minlength=K + 1).astype(float)
    pvals.append(stats.chisquare(obs, np.asarray(pm) * N).pvalue)
    return pvals


def _c1_rows():
    w = W.get("c1")
    d = W.generate(w)
    K = int(d["k_per_row"][0])
    P = np.stack([oracle.row_dist(d["p"][0, j], w.temperature)[0] for j in range(K + 1)])
    Q = np.stack([oracle.row_dist(d["q"][0, j], w.temperature)[0] for j in range(K)])
    return P, Q


def test_chisquare_1e6_trials():
    P, Q = _c1_rows()
    pv = chisquare_pvalues(P, Q, N=1_000_000, seed=2024)
    assert min(pv) > 1e-3 / len(pv), pv


# ----------------------------------------------------------------------------------------------
# acceptance count: closed form and the pages' printed values
# ----------------------------------------------------------------------------------------------
def expected_emitted(alpha, K):
    """(1 - alpha^(K+1)) / (1 - alpha) = 1 + alpha + ... + alpha^K (gsyq.cn §3.2, 2kiu.com §3.1)."""
    return K + 1.0 if alpha == 1.0 else (1.0 - alpha ** (K + 1)) / (1.0 - alpha)


def _golden_rows():
    rows = []
    with open(os.path.join(GOLDEN, "expected_accepted.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                a, k, e, status = line.split()[:4]
                rows.append((float(a), int(k), float(e), status))
    return rows


def test_closed_form_matches_printed_values():
    rows = _golden_rows()
    assert sum(s == "pin" for *_, s in rows) >= 4
    for a, k, e, status in rows:
        got = expected_emitted(a, k)
        if status == "pin":
            assert abs(got - e) <= 0.005 + 1e-12, (a, k, e, got)
        else:  # values the pages print that the formula does not give (garbled arithmetic)
            assert abs(got - e) > 0.005, (a, k, e, got)


def known_alpha_rows(alpha, K, V, rng):
    """Rows with sum_v min(P, Q) == alpha exactly: q on A = {0..V-2}, p = alpha q + (1-alpha) e_{V-1}."""
    Q = np.zeros((K, V))
    P = np.zeros((K + 1, V))
    for j in range(K):
        Q[j, :-1] = _dirichlet(rng, V - 1)
        P[j] = alpha * Q[j]
        P[j, -1] = 1.0 - alpha
    P[K] = _dirichlet(rng, V)
    return P, Q


def mc_emitted_zscore(alpha, K, N, seed, lib=None):
    rng = np.random.default_rng(seed)
    V = 64
    P, Q = known_alpha_rows(alpha, K, V, rng)
    x = np.stack([_sample_from(rng, Q[j], N) for j in range(K)], 1).astype(np.int32)
    ua = (rng.integers(0, 1 << 24, (N, K)) * 2.0 ** -24).astype(np.float32)
    ur = (rng.integers(0, 1 << 24, N) * 2.0 ** -24).astype(np.float32)
    _, n, _ = oracle.decide_trials(P, Q, x, ua, ur, lib=lib)
    m = (n + 1).astype(float)
    return (m.mean() - expected_emitted(alpha, K)) / (m.std() / np.sqrt(N))


@pytest.mark.parametrize("alpha,K", [(0.4, 6), (0.6, 5), (0.75, 5), (0.8, 4), (0.9, 6)])
def test_mean_emitted_matches_closed_form(alpha, K):
    z = mc_emitted_zscore(alpha, K, N=1_000_000, seed=int(alpha * 100) + K)
    assert abs(z) < 4.0, z


# ----------------------------------------------------------------------------------------------
# normalisation: temperature, top-k, widening, non-finite rows
# ----------------------------------------------------------------------------------------------
@pytest.mark.parametrize("T", [1.0, 0.7, 1.3])
def test_softmax_against_library(T):
    rng = np.random.default_rng(11)
    z = (3 * rng.standard_normal(777)).astype(np.float32)
    P, info, fl = oracle.row_dist(z, T)
    ref = torch.softmax(torch.from_numpy(z.astype(np.float64)) / T, 0).numpy()
    assert fl == 0
    np.testing.assert_allclose(P, ref, rtol=1e-12, atol=1e-300)
    lse = torch.logsumexp(torch.from_numpy(z.astype(np.float64)) / T, 0).item()
    assert abs(info["lognorm"] - lse) < 1e-12
    assert info["m"] == z.max()


def test_constant_logits_are_uniform():
    P, _, fl = oracle.row_dist(np.full(1000, 2.5, np.float32), 0.8)
    assert fl == 0
    np.testing.assert_allclose(P, 1e-3, rtol=1e-14)


def test_bf16_widening_is_exact():
    bits = np.array([0x3F80, 0x0000, 0xBF80, 0x4000], np.uint16)  # 1, 0, -1, 2
    P, info, _ = oracle.row_dist(bits, 1.0)
    ref = torch.softmax(torch.tensor([1.0, 0.0, -1.0, 2.0], dtype=torch.float64), 0).numpy()
    np.testing.assert_allclose(P, ref, rtol=1e-14)
    assert info["m"] == 2.0
    # the generator's bf16 rounding is round-to-nearest-even
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -3.0 - 2 ** -9], np.float32)
    got = W.bf16_bits_to_f32(W.to_bf16_bits(x))
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("seed", range(6))
def test_topk_against_library(seed):
    rng = np.random.default_rng(100 + seed)
    V = int(rng.integers(5, 17))
    k = int(rng.integers(1, V))
    T = float(rng.choice([0.5, 1.0, 1.7]))
    z = rng.standard_normal(V).astype(np.float32)
    P, info, fl = oracle.row_dist(z, T, k)
    top = torch.topk(torch.from_numpy(z.astype(np.float64)), k)
    kept = np.zeros(V, bool)
    kept[top.indices.numpy()] = True
    assert fl == 0 and info["kept"] == k
    assert ((P > 0) == kept).all()
    ref = torch.softmax(top.values / T, 0).numpy()
    np.testing.assert_allclose(P[top.indices.numpy()], ref, rtol=1e-12)
    # top_k >= V and top_k == 0 are both "off"
    np.testing.assert_allclose(oracle.row_dist(z, T, V)[0], oracle.row_dist(z, T, 0)[0], rtol=0)


def test_topk_ties_kept_and_flagged():
    z = np.array([3.0, 1.0, 2.0, 2.0, 0.5, 2.0], np.float32)
    P, info, fl = oracle.row_dist(z, 1.0, 2)  # 2nd largest is 2.0, held three times
    assert fl & oracle.FLAG_TOPK_TIE
    assert info["kept"] == 4 and info["threshold"] == 2.0
    ref = np.exp(np.array([3.0, 2, 2, 2]) - 3.0)
    ref /= ref.sum()
    np.testing.assert_allclose(P[[0, 2, 3, 5]], ref, rtol=1e-14)
    assert P[1] == 0 and P[4] == 0


def test_nonfinite_rows_flagged():
    z = np.zeros(8, np.float32)
    for bad in (np.nan, np.inf):
        y = z.copy()
        y[3] = bad
        assert oracle.row_dist(y, 1.0)[2] & oracle.FLAG_NONFINITE
    assert oracle.row_dist(np.full(8, -np.inf, np.float32), 1.0)[2] & oracle.FLAG_NONFINITE
    y = z.copy()
    y[[1, 2]] = -np.inf  # -inf is allowed and means probability 0
    P, _, fl = oracle.row_dist(y, 1.0)
    assert fl == 0 and P[1] == 0 and P[2] == 0 and abs(P[0] - 1 / 6) < 1e-15


# ----------------------------------------------------------------------------------------------
# greedy limit
# ----------------------------------------------------------------------------------------------
def test_greedy_against_library_argmax():
    rng = np.random.default_rng(3)
    B, K, V = 40, 4, 300
    p = W.to_bf16_bits(np.round(rng.standard_normal((B, K + 1, V)) * 2) / 2)  # many exact ties
    pf = W.bf16_bits_to_f32(p)
    g = torch.argmax(torch.from_numpy(pf), dim=-1).numpy()  # first index among equal maxima
    assert (g == np.argmax(pf, -1)).all()
    draft = g[:, :K].copy()
    flip = rng.random((B, K)) < 0.3
    draft[flip] = (draft[flip] + 1) % V
    out = oracle.verify(p, None, draft, None, None, None, 0.0)
    for b in range(B):
        mism = np.nonzero(draft[b] != g[b, :K])[0]
        n = int(mism[0]) if len(mism) else K
        assert out["n_acc"][b] == n
        np.testing.assert_array_equal(out["tokens"][b, :n], draft[b, :n])
        assert out["tokens"][b, n] == g[b, n]
        assert (out["tokens"][b, n + 1:] == -1).all()
    # p == q in greedy mode with drafts = argmax q: everything accepted
    out = oracle.verify(p, p[:, :K].copy(), g[:, :K].copy(), None, None, None, 0.0)
    assert (out["n_acc"] == K).all()


def test_batch_entry_matches_per_request_decide():
    w = W.get("c4", B=3, V=4000, tau=0.6)
    d = W.generate(w)
    out = oracle.verify(d["p"], d["q"], d["draft"], d["k_per_row"], d["ua"], d["ur"], w.temperature, w.top_k)
    for b in range(3):
        K = int(d["k_per_row"][b])
        P = np.stack([oracle.row_dist(d["p"][b, j], w.temperature, w.top_k)[0] for j in range(K + 1)])
        Q = np.stack([oracle.row_dist(d["q"][b, j], w.temperature, w.top_k)[0] for j in range(K)])
        r = oracle.decide(P, Q, d["draft"][b, :K], d["ua"][b, :K].astype(np.float64), float(d["ur"][b]))
        assert r["n_acc"] == out["n_acc"][b]
        np.testing.assert_array_equal(r["tokens"], out["tokens"][b, :K + 1])
        assert (out["tokens"][b, K + 1:] == -1).all()


def test_bad_inputs_flagged():
    w = W.get("c1")
    d = W.generate(w)
    draft = d["draft"].copy()
    draft[0, 1] = 1000  # == V
    out = oracle.verify(d["p"], d["q"], draft, np.array([9], np.int32), d["ua"], d["ur"], 1.0)
    assert out["flags"][0] & oracle.FLAG_BAD_K
    out = oracle.verify(d["p"], d["q"], draft, None, np.zeros_like(d["ua"]), d["ur"], 1.0)
    assert out["n_acc"][0] <= 1 and (out["flags"][0] & oracle.FLAG_BAD_TOKEN or out["n_acc"][0] == 0)


# ----------------------------------------------------------------------------------------------
# the decision margins (a GPU result that differs from the oracle's is excused only where the
# margin of the decision that differs is below 1e-5, so the margins themselves are pinned)
# ----------------------------------------------------------------------------------------------
# Every probability and uniform below is a binary fraction, so each margin is exact in fp64:
#   accept margin = |u - p(x)/q(x)| (inf when q(x) = 0) at every examined position;
#   sample margin = min(u - C_{y-1}/R, C_y/R - u), C the cumulative weights of the draw in token
#   order and R their total.
HALF = [0.5, 0.25, 0.125, 0.125]
MARGIN_CASES = [
    # (P rows, Q rows, drafts, accept uniforms, resample uniform, expected result)
    # accepted (1/4 / 1/2 = 1/2 against u = 3/8), then the bonus draw from the uniform row at
    # u = 0.3: token 1, between the cumulative masses 1/4 and 1/2
    dict(P=[HALF, [0.25] * 4], Q=[[0.25, 0.5, 0.125, 0.125]], x=[1], ua=[0.375], ur=0.3,
         n_acc=1, tokens=[1, 1], accept_margin=[0.125], sample_margin=0.05, residual_mass=0.0),
    # rejected (1/8 / 1/2 = 1/4 against u = 5/8); residual (3/8, 1/8, 0, 0), R = 1/2, cumulative
    # C/R = (3/4, 1, 1, 1); u = 0.8 draws token 1, 0.05 above its lower edge
    dict(P=[HALF, [0.25] * 4], Q=[[0.125, 0.125, 0.5, 0.25]], x=[2], ua=[0.625], ur=0.8,
         n_acc=0, tokens=[1, -1], accept_margin=[0.375], sample_margin=0.05, residual_mass=0.5),
    # the same draw at u = 31/32: token 1, 1/32 below its upper edge
    dict(P=[HALF, [0.25] * 4], Q=[[0.125, 0.125, 0.5, 0.25]], x=[2], ua=[0.625], ur=31 / 32,
         n_acc=0, tokens=[1, -1], accept_margin=[0.375], sample_margin=1 / 32, residual_mass=0.5),
    # the same draw at u = 1/2: token 0, 1/4 below its upper edge (its lower edge is 0, 1/2 away)
    dict(P=[HALF, [0.25] * 4], Q=[[0.125, 0.125, 0.5, 0.25]], x=[2], ua=[0.625], ur=0.5,
         n_acc=0, tokens=[0, -1], accept_margin=[0.375], sample_margin=0.25, residual_mass=0.5),
    # two positions: the first accepted with q(x) = 0 (margin inf, accepted because p(x) > 0), the
    # second rejected (1/8 / 1/4 = 1/2 against u = 3/4, margin 1/4); the residual at position 1 is
    # (0, 0, 0, 1/8), so u = 1/4 draws token 3, 1/4 above its lower edge C_2 / R = 0
    dict(P=[[0.5, 0.5, 0, 0], [0.5, 0.25, 0.125, 0.125], [0.25] * 4], Q=[[1.0, 0, 0, 0], [0.5, 0.25, 0.25, 0]],
         x=[1, 2], ua=[0.875, 0.75], ur=0.25, n_acc=1, tokens=[1, 3, -1], accept_margin=[np.inf, 0.25],
         sample_margin=0.25, residual_mass=0.125),
]


def _margin_pin(lib=None):
    for c in MARGIN_CASES:
        r = oracle.decide(np.array(c["P"], float), np.array(c["Q"], float), c["x"], c["ua"], c["ur"], lib=lib)
        assert r["n_acc"] == c["n_acc"], (c, r)
        np.testing.assert_array_equal(r["tokens"], c["tokens"])
        np.testing.assert_array_equal(r["accept_margin"][: c["n_acc"] + 1], c["accept_margin"])
        assert abs(r["sample_margin"] - c["sample_margin"]) < 1e-15, (c, r)
        assert abs(r["residual_mass"] - c["residual_mass"]) < 1e-15, (c, r)


def test_margins_hand_computed():
    _margin_pin()


def test_margins_through_the_batch_entry():
    """The same cases as logits (ln of the probabilities, -inf for zeros) through oracle.verify:
    the margins come out as computed by hand, to the rounding of the float32 logits."""
    for c in MARGIN_CASES:
        K = len(c["x"])
        with np.errstate(divide="ignore"):
            p = np.log(np.array(c["P"], np.float64)).astype(np.float32)[None]
            q = np.log(np.array(c["Q"], np.float64)).astype(np.float32)[None]
        out = oracle.verify(p, q, np.array([c["x"]], np.int32), None, np.array([c["ua"]], np.float32),
                            np.array([c["ur"]], np.float32), 1.0)
        assert out["n_acc"][0] == c["n_acc"]
        np.testing.assert_array_equal(out["tokens"][0], c["tokens"])
        np.testing.assert_allclose(out["accept_margin"][0, : c["n_acc"] + 1], c["accept_margin"], rtol=0, atol=1e-6)
        assert abs(out["sample_margin"][0] - c["sample_margin"]) < 1e-6
        assert np.isnan(out["accept_margin"][0, c["n_acc"] + 1:]).all() and K >= c["n_acc"]


# ----------------------------------------------------------------------------------------------
# planted mistakes: every variant must fail at least one pin
# ----------------------------------------------------------------------------------------------
MUTANTS = {
    "resample_from_p": ("double d = Pj[v] - Qj[v];", "double d = Pj[v];"),
    "ratio_inverted": ("if (u * c < a) {", "if (u * a < c) {"),
    "bonus_wrong_row": ("const double* Pj = P + (size_t)jstar * V;",
                        "const double* Pj = P + (size_t)(jstar > 0 ? jstar - 1 : 0) * V;"),
    "no_temperature": ("exp((x - m) / T)", "exp(x - m)"),
    "topk_off_by_one": ("t = s[top_k - 1];", "t = s[top_k];"),
    "residual_sign": ("double d = Pj[v] - Qj[v];", "double d = Qj[v] - Pj[v];"),
    "cdf_from_top": ("for (int v = 0; v < V; ++v) {\n    double prev = C;",
                     "for (int v = V - 1; v >= 0; --v) {\n    double prev = C;"),
    # the margins the parity tests rely on
    "accept_margin_unnormalised": ("fabs(u - a / c)", "fabs(u * c - a)"),
    "accept_margin_swapped": ("fabs(u - a / c)", "fabs(u - c / a)"),
    "sample_margin_without_R": ("double lo = u - prev / R, hi = C / R - u;", "double lo = u - prev, hi = C - u;"),
    "sample_margin_lower_edge_off_by_one": ("double lo = u - prev / R, hi = C / R - u;",
                                            "double lo = u - (prev - (v > 0 ? r[v - 1] : 0.0)) / R, hi = C / R - u;"),
    "sample_margin_far_edge": ("*margin = lo < hi ? lo : hi;", "*margin = lo < hi ? hi : lo;"),
}


def _pins_fail(lib):
    """True if the variant fails any pin."""
    checks = []
    rng = np.random.default_rng(0)
    for K in (1, 2):
        P = np.stack([_dirichlet(rng, 4) for _ in range(K + 1)])
        Q = np.stack([_dirichlet(rng, 4) for _ in range(K)])
        checks.append(lambda P=P, Q=Q: check_lossless(P, Q, lib))
    checks.append(lambda: _softmax_pin(lib))
    checks.append(lambda: _topk_pin(lib))
    checks.append(lambda: _margin_pin(lib))
    for c in checks:
        try:
            c()
        except AssertionError:
            return True
    return False


def _softmax_pin(lib):
    rng = np.random.default_rng(1)
    z = rng.standard_normal(100).astype(np.float32)
    P, _, _ = oracle.row_dist(z, 0.7, lib=lib)
    ref = torch.softmax(torch.from_numpy(z.astype(np.float64)) / 0.7, 0).numpy()
    np.testing.assert_allclose(P, ref, rtol=1e-12)


def _topk_pin(lib):
    rng = np.random.default_rng(2)
    z = rng.standard_normal(12).astype(np.float32)
    P, _, _ = oracle.row_dist(z, 1.0, 5, lib=lib)
    assert (P > 0).sum() == 5
    top = torch.topk(torch.from_numpy(z.astype(np.float64)), 5).indices.numpy()
    assert (P[top] > 0).all()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new, 1)
    c = tmp_path / "oracle_mut.c"
    c.write_text(mutated)
    so = tmp_path / "liboracle_mut.so"
    subprocess.run(["gcc", *oracle.CFLAGS, str(c), "-o", str(so), "-lm"], check=True)
    lib = oracle.load(str(so))
    assert _pins_fail(lib), f"planted mistake {name} passed every pin"
    assert not _pins_fail(oracle.load())
