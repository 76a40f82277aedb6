"""Property-based pins of the oracle's accept / resample / bonus decisions (CPU only).

The verify rule is lossless (cf-1.com §2.2, 2kiu.com §2.2): whatever the draft proposes, the
emitted token at position i is distributed as p_i once the prefix is accepted.  The exact law of
every emitted token follows from the oracle's decisions by breakpoint enumeration (the helper of
the enumeration pins).  Here hypothesis draws the distributions from small integer weights, so
exact ties p(x) = q(x), zero mass on either side, one-hot rows and disjoint supports come up far
more often than with continuous draws; every case must be lossless to 1e-12, and the acceptance
probability at each position must equal sum_v min(p, q)."""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

from test_oracle_pins import check_lossless, enumerate_law  # noqa: E402


def _rows(draw, n, V):
    rows = []
    for _ in range(n):
        w = draw(st.lists(st.integers(0, 4), min_size=V, max_size=V).filter(lambda a: sum(a) > 0))
        rows.append(np.asarray(w, np.float64) / sum(w))
    return np.stack(rows)


@st.composite
def cases(draw):
    V = draw(st.integers(2, 5))
    K = draw(st.integers(1, 2))
    return _rows(draw, K + 1, V), _rows(draw, K, V)


@settings(max_examples=80, deadline=None, derandomize=True)
@given(cases())
def test_lossless_on_integer_weights(case):
    P, Q = case
    check_lossless(P, Q)


@settings(max_examples=40, deadline=None, derandomize=True)
@given(cases())
def test_acceptance_probability_is_the_overlap(case):
    P, Q = case
    law = enumerate_law(P, Q)
    K = Q.shape[0]
    reach = 1.0
    for i in range(K):
        # Pr(position i+1 is emitted) = Pr(drafts 0..i accepted)
        reach *= np.minimum(P[i], Q[i]).sum()
        assert abs(law[i + 1].sum() - reach) < 1e-12
