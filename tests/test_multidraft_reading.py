"""Why the literal reading of multi-draft verify is not the one built (CPU only).

2kiu.com §7 suggests running several draft models at once and keeping the one that accepts the
most; the pages give no verify rule for it.  Read literally -- verify each draft independently
with the single-draft rule and keep the result with the most accepted drafts -- the selection
changes the output law: the first emitted token is no longer distributed as p.  The law is
computed exactly here, by breakpoint enumeration of each draft's verification through the
oracle's own decisions, then combined over the two independent verifications (the single-draft
law is checked beside it as the control).  The rule built instead tests the candidates in turn,
each against what the earlier rejections leave of p (oracle_decide_multi, pinned lossless in
test_oracle_pins_multidraft.py)."""
import numpy as np
import pytest

import oracle


def _pieces(weights):
    w = np.asarray(weights, np.float64)
    C = np.cumsum(w) / w.sum()
    edges = np.unique(np.clip(np.concatenate([[0.0], C, [1.0]]), 0.0, 1.0))
    return [(lo, hi) for lo, hi in zip(edges[:-1], edges[1:]) if hi > lo]


def outcomes(P, Q):
    """Every outcome of one request's verification with K = 1 as (n_acc, first token, weight),
    enumerated exactly over the draft token and both uniforms."""
    out = []

    def call(x, ua, ur, w):
        res = oracle.decide(P, Q, [x], [ua], ur)
        out.append((res["n_acc"], res["tokens"][0], w))

    V = P.shape[1]
    for x in range(V):
        if Q[0, x] <= 0.0:
            continue
        t = min(1.0, P[0, x] / Q[0, x])
        if t > 0.0:  # accepted: the bonus draw from p at position 1 follows
            for lo, hi in _pieces(P[1]):
                call(x, 0.5 * t, 0.5 * (lo + hi), Q[0, x] * t * (hi - lo))
        if t < 1.0:  # rejected: the residual draw
            r = np.maximum(P[0] - Q[0], 0.0)
            for lo, hi in _pieces(r if r.sum() > 0 else P[0]):
                call(x, 0.5 * (1.0 + t), 0.5 * (lo + hi), Q[0, x] * (1.0 - t) * (hi - lo))
    return out


def first_token_law(outs, V):
    law = np.zeros(V)
    for _, tok, w in outs:
        law[tok] += w
    return law


def best_of_two_law(P, Q1, Q2):
    """Law of the first emitted token when two drafts are verified independently and the result
    with more accepted drafts is kept (the first draft's on a tie)."""
    V = P.shape[1]
    o1, o2 = outcomes(P, Q1), outcomes(P, Q2)
    law = np.zeros(V)
    for n1, t1, w1 in o1:
        for n2, t2, w2 in o2:
            law[t1 if n1 >= n2 else t2] += w1 * w2
    return law


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_best_of_two_is_not_lossless(seed):
    rng = np.random.default_rng(seed)
    V = 4
    P = rng.dirichlet(np.ones(V), size=2)
    Q1 = rng.dirichlet(np.ones(V), size=1)
    Q2 = rng.dirichlet(np.ones(V), size=1)
    # the control: one draft, verified by the single-draft rule, emits exactly p
    np.testing.assert_allclose(first_token_law(outcomes(P, Q1), V), P[0], atol=1e-12)
    np.testing.assert_allclose(first_token_law(outcomes(P, Q2), V), P[0], atol=1e-12)
    law = best_of_two_law(P, Q1, Q2)
    assert abs(law.sum() - 1.0) < 1e-12
    # the selection biases the emitted token towards what the drafts propose
    assert np.abs(law - P[0]).max() > 1e-3, (law, P[0])


def test_best_of_two_closed_form():
    """The enumeration agrees with the closed form of the selection: with m_i = min(Q_i, P) and
    a_i = sum m_i, the first token's law is m_1 + (1 - a_1) m_2 + (1 - a_1)(1 - a_2) r_1, where
    r_1 = (P - m_1) / (1 - a_1) is the first draft's residual; it equals P only when
    m_2 = a_2 r_1."""
    rng = np.random.default_rng(5)
    V = 4
    P = rng.dirichlet(np.ones(V), size=2)
    Q1 = rng.dirichlet(np.ones(V), size=1)
    Q2 = rng.dirichlet(np.ones(V), size=1)
    m1, m2 = np.minimum(Q1[0], P[0]), np.minimum(Q2[0], P[0])
    a1, a2 = m1.sum(), m2.sum()
    r1 = (P[0] - m1) / (1.0 - a1)
    closed = m1 + (1.0 - a1) * m2 + (1.0 - a1) * (1.0 - a2) * r1
    np.testing.assert_allclose(best_of_two_law(P, Q1, Q2), closed, atol=1e-12)
