"""Property-based pins of the oracle's accept / resample / bonus decisions (CPU only).

The verify rule is lossless (cf-1.com §2.2, 2kiu.com §2.2): whatever the draft proposes, the
emitted token at position i is distributed as p_i once the prefix is accepted.  The exact law of
every emitted token follows from the oracle's decisions by breakpoint enumeration (the helper of
the enumeration pins).  Here hypothesis draws the distributions from small integer weights, so
exact ties p(x) = q(x), zero mass on either side, one-hot rows and disjoint supports come up far
more often than with continuous draws; every case must be lossless to 1e-12, and the acceptance
probability at each position must equal sum_v min(p, q).  The planted decision mistakes (resample
from p, inverted ratio, wrong bonus row, residual sign) each fail this enumeration on its own."""
import os
import subprocess

import numpy as np
import pytest

import oracle

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

from test_oracle_pins import MUTANTS, check_lossless, enumerate_law  # noqa: E402


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


# The decision mistakes among the planted ones must also fail this enumeration on its own, on a
# fixed set of integer-weight cases (so the property pin is not carried by the other pins).
DECISION_MUTANTS = ("resample_from_p", "ratio_inverted", "bonus_wrong_row", "residual_sign")


def _integer_cases(n=24, seed=7):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        V, K = int(rng.integers(2, 6)), int(rng.integers(1, 3))

        def rows(m):
            r = rng.integers(0, 5, size=(m, V)).astype(np.float64)
            r[r.sum(1) == 0, 0] = 1.0
            return r / r.sum(1, keepdims=True)

        out.append((rows(K + 1), rows(K)))
    return out


@pytest.mark.parametrize("name", DECISION_MUTANTS)
def test_integer_enumeration_catches_decision_mistakes(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    c = tmp_path / "oracle_mut.c"
    c.write_text(src.replace(old, new, 1))
    so = tmp_path / "liboracle_mut.so"
    subprocess.run(["gcc", *oracle.CFLAGS, str(c), "-o", str(so), "-lm"], check=True)
    lib = oracle.load(str(so))
    caught = False
    for P, Q in _integer_cases():
        try:
            check_lossless(P, Q, lib)
        except AssertionError:
            caught = True
            break
    assert caught, f"planted mistake {name} passed the integer-weight enumeration"
    for P, Q in _integer_cases():  # and the oracle as written passes every case
        check_lossless(P, Q)
