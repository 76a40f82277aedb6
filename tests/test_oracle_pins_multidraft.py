"""Pins of the oracle's multi-draft decision (CPU only).

2kiu.com §7 and cf-1.com §2.3 name ensembles of draft models whose best-accepted draft the target
keeps; the pages fix the property any verify rule must keep -- the emitted tokens are distributed as
p (cf-1.com §2.2, 2kiu.com §2.2) -- not a rule for several candidates.  The oracle tests the
candidates in turn, each against what the earlier rejections leave of p, and follows the first
accepted chain with the single-draft rule.  Pinned here by:

* one chain is exactly the single-draft rule (oracle_decide, itself pinned by enumeration);
* exhaustive breakpoint enumeration at V = 4 with 2 and 3 chains, K = 1 and 2, a target whose
  distribution at later positions depends on the emitted prefix and chains whose drafts depend on
  their own prefix: the law of the first emitted token is P_0, and the law of every later token
  given the prefix is the target's distribution after that prefix, to 1e-12;
* planted mistakes (every candidate tested against p, an unnormalised residual, the last draw from
  p, the wrong chain followed) each fail one of these.
"""
import itertools
import os
import subprocess

import numpy as np
import pytest

import oracle


def _pieces(weights):
    w = np.asarray(weights, np.float64)
    C = np.cumsum(w) / w.sum()
    edges = np.unique(np.clip(np.concatenate([[0.0], C, [1.0]]), 0.0, 1.0))
    return [(lo, hi) for lo, hi in zip(edges[:-1], edges[1:]) if hi > lo]


def _dirichlet(rng, V, zeros=0):
    d = rng.dirichlet(np.ones(V))
    if zeros:
        d[rng.choice(V, zeros, replace=False)] = 0.0
        d /= d.sum()
    return d


def make_case(rng, V, N, K, zeros=True):
    """A target P0 with prefix-dependent tables T1[t0], T2[t0, t1]; per chain a first-draft law Q0[n]
    and a prefix-dependent second-draft table Q1[n, t0]."""
    z = (lambda: int(rng.integers(0, 2))) if zeros else (lambda: 0)
    P0 = _dirichlet(rng, V, z())
    T1 = np.stack([_dirichlet(rng, V, z()) for _ in range(V)])
    T2 = np.stack([[_dirichlet(rng, V, z()) for _ in range(V)] for _ in range(V)])
    Q0 = np.stack([_dirichlet(rng, V, z()) for _ in range(N)])
    Q1 = np.stack([[_dirichlet(rng, V, z()) for _ in range(V)] for _ in range(N)])
    return dict(P0=P0, T1=T1, T2=T2, Q0=Q0, Q1=Q1, V=V, N=N, K=K)


def enumerate_multi(case, lib=None):
    """Exact law of the emitted tokens: {(t0, t1, ..., ) prefix: probability} for every emitted
    prefix, by enumerating each chain's drafts and every uniform's pieces."""
    V, N, K = case["V"], case["N"], case["K"]
    P0, T1, T2, Q0, Q1 = (case[k] for k in ("P0", "T1", "T2", "Q0", "Q1"))
    law = {}

    def call(xs, uas, ur, w):
        # the rows each chain presents: its target along its own prefix and its own draft law
        P = np.zeros((N, K + 1, V))
        Q = np.zeros((N, max(K, 1), V))
        x = np.zeros((N, max(K, 1)), np.int32)
        ua = np.full((N, max(K, 1)), 0.5)
        P[:, 0] = P0
        for n in range(N):
            x0 = xs[n][0]
            x[n, 0] = x0
            Q[n, 0] = Q0[n]
            ua[n, 0] = uas[n][0]
            if K >= 1:
                P[n, 1] = T1[x0]
            if K >= 2:
                x1 = xs[n][1]
                x[n, 1] = x1
                Q[n, 1] = Q1[n, x0]
                ua[n, 1] = uas[n][1]
                P[n, 2] = T2[x0, x1]
        res = oracle.decide_multi(P, Q[:, :K], x[:, :K], ua[:, :K], ur, lib=lib)
        t = tuple(int(v) for v in res["tokens"][: res["n_acc"] + 1])
        law[t] = law.get(t, 0.0) + w

    def chain(n, r, xs, uas, w):
        """Candidate n against what is left of P0 (r)."""
        if n == N:  # every candidate rejected: the last draw from r
            for lo, hi in _pieces(r):
                call(xs, uas, 0.5 * (lo + hi), w * (hi - lo))
            return
        for x0 in range(V):
            q = Q0[n][x0]
            if q <= 0.0:
                continue
            t = min(1.0, r[x0] / q)
            if t > 0.0:
                follow(n, x0, xs, uas, w * q * t, 0.5 * t)
            if t < 1.0:
                rest = np.maximum(r - Q0[n], 0.0)
                r2 = rest / rest.sum() if rest.sum() > 0 else r
                chain(n + 1, r2, xs + [[x0, 0]], uas + [[0.5 * (1.0 + t), 0.5]], w * q * (1.0 - t))

    def follow(n, x0, xs, uas, w, u0):
        """Chain n accepted at x0; the other chains' later entries are padding the rule never reads."""
        pad = [[0, 0]] * (N - n - 1)
        upad = [[0.5, 0.5]] * (N - n - 1)
        if K == 1:
            for lo, hi in _pieces(T1[x0]):
                call(xs + [[x0, 0]] + pad, uas + [[u0, 0.5]] + upad, 0.5 * (lo + hi), w * (hi - lo))
            return
        for x1 in range(V):  # K == 2: the chain's second draft, then the single-draft rule
            q = Q1[n, x0][x1]
            if q <= 0.0:
                continue
            t = min(1.0, T1[x0][x1] / q)
            if t > 0.0:
                for lo, hi in _pieces(T2[x0, x1]):
                    call(xs + [[x0, x1]] + pad, uas + [[u0, 0.5 * t]] + upad, 0.5 * (lo + hi),
                         w * q * t * (hi - lo))
            if t < 1.0:
                rest = np.maximum(T1[x0] - Q1[n, x0], 0.0)
                for lo, hi in _pieces(rest if rest.sum() > 0 else T1[x0]):
                    call(xs + [[x0, x1]] + pad, uas + [[u0, 0.5 * (1.0 + t)]] + upad, 0.5 * (lo + hi),
                         w * q * (1.0 - t) * (hi - lo))

    chain(0, P0.copy(), [], [], 1.0)
    return law


def check_lossless_multi(case, lib=None, tol=1e-12):
    law = enumerate_multi(case, lib)
    V, K = case["V"], case["K"]
    assert abs(sum(law.values()) - 1.0) < 1e-12
    first = np.zeros(V)
    for t, w in law.items():
        first[t[0]] += w
    np.testing.assert_allclose(first, case["P0"], rtol=0, atol=tol)
    # later positions: given the emitted prefix, the next token's law is the target's after it
    for depth in range(1, K + 1):
        table = case["T1"] if depth == 1 else None
        for prefix in itertools.product(range(V), repeat=depth):
            nxt = np.zeros(V)
            for t, w in law.items():
                if len(t) > depth and t[:depth] == prefix:
                    nxt[t[depth]] += w
            if nxt.sum() < 1e-14:
                continue
            ref = table[prefix[0]] if depth == 1 else case["T2"][prefix[0], prefix[1]]
            np.testing.assert_allclose(nxt / nxt.sum(), ref, rtol=0, atol=1e-10)


@pytest.mark.parametrize("N,K", [(2, 1), (3, 1), (2, 2)])
@pytest.mark.parametrize("seed", [0, 1])
def test_multi_draft_is_lossless(N, K, seed):
    check_lossless_multi(make_case(np.random.default_rng(100 + seed * 7 + N * 3 + K), 4, N, K))


def test_multi_draft_special_cases():
    rng = np.random.default_rng(9)
    # identical chains: a rejected first token is rejected again (nothing of p is left at it)
    c = make_case(rng, 4, 2, 1, zeros=False)
    c["Q0"][1] = c["Q0"][0]
    check_lossless_multi(c)
    # drafts that never cover p's support: every candidate rejected, the last draw is from p
    c = make_case(rng, 4, 3, 1, zeros=False)
    c["P0"] = np.array([0.5, 0.5, 0.0, 0.0])
    c["Q0"][:] = np.array([0.0, 0.0, 0.5, 0.5])
    check_lossless_multi(c)
    # a chain whose draft law is p itself is always accepted once reached
    c = make_case(rng, 4, 2, 1, zeros=False)
    c["Q0"][0] = c["P0"]
    law = enumerate_multi(c)
    assert all(len(t) == 2 for t in law)  # n_acc >= 1 on every path
    check_lossless_multi(c)


def test_one_chain_is_the_single_draft_rule():
    rng = np.random.default_rng(3)
    for trial in range(200):
        V, K = 6, int(rng.integers(1, 4))
        P = np.stack([_dirichlet(rng, V, int(rng.integers(0, 2))) for _ in range(K + 1)])
        Q = np.stack([_dirichlet(rng, V, int(rng.integers(0, 2))) for _ in range(K)])
        x = np.array([rng.choice(V, p=Q[j]) for j in range(K)], np.int32)
        ua = rng.integers(0, 1 << 24, K) * 2.0 ** -24
        ur = float(rng.integers(0, 1 << 24) * 2.0 ** -24)
        a = oracle.decide(P, Q, x, ua, ur)
        m = oracle.decide_multi(P[None], Q[None], x[None], ua[None], ur)
        np.testing.assert_array_equal(m["tokens"], a["tokens"])
        assert m["n_acc"] == a["n_acc"] and m["chain"] == (0 if a["n_acc"] >= 1 else -1) or \
            (m["n_acc"] == a["n_acc"] == 0 and m["chain"] in (-1, 0))
        np.testing.assert_array_equal(m["accept_margin"][0, : a["n_acc"] + 1], a["accept_margin"][: a["n_acc"] + 1])
        # the last draw runs over the renormalised residual here: the same token, the margin to rounding
        assert abs(m["sample_margin"] - a["sample_margin"]) <= 1e-12


def test_batch_entry_matches_the_decision():
    """oracle.verify_multi on logits = decide_multi on the distributions it normalises."""
    rng = np.random.default_rng(5)
    B, N, K, V = 3, 3, 2, 50
    p = rng.standard_normal((B, N, K + 1, V)).astype(np.float32)
    q = rng.standard_normal((B, N, K, V)).astype(np.float32)
    x = rng.integers(0, V, (B, N, K)).astype(np.int32)
    ua = (rng.integers(0, 1 << 24, (B, N, K)) * 2.0 ** -24).astype(np.float32)
    ur = (rng.integers(0, 1 << 24, B) * 2.0 ** -24).astype(np.float32)
    out = oracle.verify_multi(p, q, x, ua, ur, 0.9, draft_temperature=0.7)
    for b in range(B):
        P = np.stack([[oracle.row_dist(p[b, n, j], np.float32(0.9))[0] for j in range(K + 1)] for n in range(N)])
        P[1:, 0] = P[0, 0]  # row 0 of the other chains is not read: the shared first position
        Q = np.stack([[oracle.row_dist(q[b, n, j], np.float32(0.7))[0] for j in range(K)] for n in range(N)])
        r = oracle.decide_multi(P, Q, x[b], ua[b].astype(np.float64), float(ur[b]))
        np.testing.assert_array_equal(out["tokens"][b], r["tokens"])
        assert out["n_acc"][b] == r["n_acc"] and out["chain"][b] == r["chain"]


def test_greedy_multi():
    """T = 0: the first chain whose first draft is the argmax is followed with the greedy rule."""
    rng = np.random.default_rng(11)
    B, N, K, V = 20, 3, 3, 30
    p = np.round(rng.standard_normal((B, N, K + 1, V)) * 2).astype(np.float32) / 2  # ties
    g = np.argmax(p, -1)
    x = rng.integers(0, V, (B, N, K)).astype(np.int32)
    for b in range(B):
        n = int(rng.integers(0, N + 1))
        if n < N:
            x[b, n, 0] = g[b, 0, 0]
            x[b, n, 1:] = np.where(rng.random(K - 1) < 0.7, g[b, n, 1:K], x[b, n, 1:])
    out = oracle.verify_multi(p, None, x, None, None, 0.0)
    for b in range(B):
        hits = [n for n in range(N) if x[b, n, 0] == g[b, 0, 0]]
        assert out["tokens"][b, 0] == g[b, 0, 0]
        if not hits:
            assert out["chain"][b] == -1 and out["n_acc"][b] == 0
            continue
        c = hits[0]
        assert out["chain"][b] == c
        n = 1
        while n < K and x[b, c, n] == g[b, c, n]:
            n += 1
        assert out["n_acc"][b] == n
        np.testing.assert_array_equal(out["tokens"][b, 1: n + 1], list(x[b, c, 1:n]) + [g[b, c, n]])


def test_multi_margins_hand_computed(lib=None):
    """Margins of the multi-draft decision on binary-fraction rows (V = 4, N = 2, K = 1): each
    candidate's |u_n - r_n(x_n) / q_n(x_n)| and the draw's distance to the nearer CDF edge."""
    nan = np.nan
    # candidate 0 rejected (r_0(2) / q_0(2) = 0.5 < u_0 = 0.75), r_1 = norm(max(0, P_0 - Q_0)) =
    # [1, 0, 0, 0], candidate 1 accepted (r_1(0) / q_1(0) = 2), then chain 1's extra token from
    # its row 1 = [1/2, 1/2, 0, 0] at u = 0.3: token 0, margin min(0.3, 0.5 - 0.3) = 0.2
    P = np.array([[[0.5, 0.25, 0.125, 0.125], [0.25] * 4],
                  [[nan] * 4, [0.5, 0.5, 0.0, 0.0]]])
    Q = np.array([[[0.25] * 4], [[0.5, 0.5, 0.0, 0.0]]])
    o = oracle.decide_multi(P, Q, [[2], [0]], [[0.75], [0.9]], 0.3, lib=lib)
    assert o["chain"] == 1 and o["n_acc"] == 1 and list(o["tokens"]) == [0, 0]
    np.testing.assert_allclose(o["accept_margin"], [[0.25], [1.1]], rtol=0, atol=1e-12)
    assert abs(o["sample_margin"] - 0.2) < 1e-12
    # both candidates outside p's support: rejected with margins u_n, r_2 = P_0, the draw at
    # u = 0.7 over [1/2, 1/2, 0, 0]: token 1, margin min(0.7 - 0.5, 1 - 0.7) = 0.2
    P = np.array([[[0.5, 0.5, 0.0, 0.0], [0.25] * 4], [[nan] * 4, [0.25] * 4]])
    Q = np.array([[[0.0, 0.0, 0.5, 0.5]], [[0.0, 0.0, 0.5, 0.5]]])
    o = oracle.decide_multi(P, Q, [[2], [3]], [[0.3], [0.6]], 0.7, lib=lib)
    assert o["chain"] == -1 and o["n_acc"] == 0 and list(o["tokens"]) == [1, -1]
    np.testing.assert_allclose(o["accept_margin"], [[0.3], [0.6]], rtol=0, atol=1e-12)
    assert abs(o["sample_margin"] - 0.2) < 1e-12


MUTANTS = {
    "multi_accept_margin_unnormalised": ("accept_margin[(size_t)n * K] = (c > 0.0) ? fabs(u - a / c) : INFINITY;",
                                         "accept_margin[(size_t)n * K] = (c > 0.0) ? fabs(u * c - a) : INFINITY;"),
    "every_candidate_against_p": ("      a = r[xn];\n", "      a = P[xn];\n"),
    "residual_not_renormalised": ("      for (int v = 0; v < V; ++v) r[v] = rest[v] / R;", "      for (int v = 0; v < V; ++v) r[v] = rest[v];"),
    "last_draw_from_p": ("    return flags | inverse_cdf(r, V, R, ur, &out_tokens[0], sample_margin);",
                         "    return flags | inverse_cdf(P, V, 1.0, ur, &out_tokens[0], sample_margin);"),
    "follows_the_first_chain": ("flags |= oracle_decide(P + ((size_t)acc * (K + 1) + 1) * V, Q + ((size_t)acc * K + 1) * V,",
                                "flags |= oracle_decide(P + ((size_t)0 * (K + 1) + 1) * V, Q + ((size_t)acc * K + 1) * V,"),
}


def _pins_fail(lib):
    try:
        test_multi_margins_hand_computed(lib)
    except AssertionError:
        return True
    cases = [make_case(np.random.default_rng(100 + s), 4, N, K) for s, (N, K) in enumerate([(2, 1), (3, 1), (2, 2)])]
    for c in cases:
        try:
            check_lossless_multi(c, lib)
        except AssertionError:
            return True
    return False


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found"
    c = tmp_path / "oracle_mut.c"
    c.write_text(src.replace(old, new, 1))
    so = tmp_path / "liboracle_mut.so"
    subprocess.run(["gcc", *oracle.CFLAGS, str(c), "-o", str(so), "-lm"], check=True)
    assert _pins_fail(oracle.load(str(so))), f"planted mistake {name} passed every pin"
    assert not _pins_fail(oracle.load())
