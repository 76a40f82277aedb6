"""Pins of the oracle's sampling-parameter variants (CPU only): a draft temperature of its own
(2kiu.com §7: the draft may sample cooler than the target) and top-p / nucleus truncation
(gsyq.cn §3.3 names top_p beside temperature and top-k as parameters both sides must share).

* top-p on a hand-built row whose probabilities are exact binary fractions, including a tie
  group that straddles the cut;
* top-p against a brute force over every candidate threshold (the largest logit t whose
  upper set {z >= t} holds mass >= top_p), on small random rows with ties, with and without
  top-k, at several temperatures;
* top_p = 1 is off; a vanishing top_p keeps exactly the maximal logits;
* the draft temperature reaches the q rows only: q logits built as T_q * ln(q_target) must
  come back as q_target, p rows follow the library softmax at T_p;
* losslessness with both variants on: exhaustive breakpoint enumeration at V = 4;
* planted mistakes in the new code each fail one of these pins.
"""
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from test_oracle_pins import check_lossless


# ----------------------------------------------------------------------------------------------
# top-p
# ----------------------------------------------------------------------------------------------
def _binary_row():
    # probabilities 1/2, 1/4, 1/8, 1/8 at T = 1: exact in fp32 logits up to ln rounding
    return np.log(np.array([0.5, 0.25, 0.125, 0.125])).astype(np.float32)


def test_topp_hand_example(lib=None):
    z = _binary_row()
    cases = {0.3: [1.0, 0, 0, 0], 0.6: [2 / 3, 1 / 3, 0, 0], 0.74: [2 / 3, 1 / 3, 0, 0],
             0.8: [0.5, 0.25, 0.125, 0.125], 0.95: [0.5, 0.25, 0.125, 0.125]}
    for top_p, ref in cases.items():
        P, info, fl = oracle.row_dist(z, 1.0, 0, top_p, lib=lib)
        assert fl == 0
        np.testing.assert_allclose(P, ref, rtol=1e-6, atol=1e-12, err_msg=f"top_p={top_p}")
        assert info["kept"] == int(np.count_nonzero(ref))
    # 0.8 needs the tied pair {2, 3}: the whole group is kept, not one of the two
    P, info, _ = oracle.row_dist(z, 1.0, 0, 0.8, lib=lib)
    assert info["threshold_p"] == z[2] and info["kept"] == 4
    # margin = distance of top_p to the cumulative masses around the cut (0.5 | 0.75 for 0.6)
    _, info, _ = oracle.row_dist(z, 1.0, 0, 0.6, lib=lib)
    assert abs(info["nucleus_margin"] - 0.1) < 1e-6
    # a cut at the first group: the mass before it is exactly 0, so only the far side counts
    _, info, _ = oracle.row_dist(z, 1.0, 0, 0.1, lib=lib)
    assert abs(info["nucleus_margin"] - 0.4) < 1e-6


def _brute_nucleus(z, T, top_k, top_p):
    """Kept mask and renormalised law by trying every threshold (library softmax / top-k)."""
    z64 = torch.from_numpy(z.astype(np.float64))
    V = z.shape[0]
    if 0 < top_k < V:
        kth = torch.topk(z64, top_k).values[-1]
        base = z64 >= kth
    else:
        base = torch.ones(V, dtype=torch.bool)
    P = torch.softmax(torch.where(base, z64 / T, torch.tensor(-np.inf, dtype=torch.float64)), 0).numpy()
    best, gap = None, np.inf
    for t in sorted(set(z[base.numpy()].tolist()), reverse=True):
        mass = P[z >= t].sum()
        gap = min(gap, abs(mass - top_p))
        if mass >= top_p:
            best = t
            break
    keep = base.numpy() & (z >= best)
    Pk = np.where(keep, P, 0.0)
    return keep, Pk / Pk.sum(), gap


@pytest.mark.parametrize("seed", range(12))
def test_topp_against_brute_force(seed, lib=None):
    rng = np.random.default_rng(500 + seed)
    checked = 0
    for _ in range(40):
        V = int(rng.integers(3, 11))
        z = (np.round(rng.standard_normal(V) * 2) / 2).astype(np.float32)  # many exact ties
        T = float(rng.choice([0.5, 1.0, 1.6]))
        top_k = int(rng.choice([0, 0, int(rng.integers(1, V))]))
        top_p = float(np.float32(rng.uniform(0.05, 0.999)))
        keep, ref, gap = _brute_nucleus(z, T, top_k, top_p)
        if gap < 1e-9:
            continue  # a cut within rounding of top_p: either side is correct
        P, info, _ = oracle.row_dist(z, T, top_k, top_p, lib=lib)
        assert ((P > 0) == keep).all(), (z, T, top_k, top_p)
        np.testing.assert_allclose(P, ref, rtol=1e-12, atol=1e-15)
        assert info["kept"] == keep.sum()
        checked += 1
    assert checked >= 30


def test_topp_limits(lib=None):
    rng = np.random.default_rng(7)
    z = rng.standard_normal(64).astype(np.float32)
    z[[5, 9]] = z.max() + 1.0  # two tied maxima
    off = oracle.row_dist(z, 0.8, 0, 1.0, lib=lib)[0]
    ref = torch.softmax(torch.from_numpy(z.astype(np.float64)) / 0.8, 0).numpy()
    np.testing.assert_allclose(off, ref, rtol=1e-12)
    np.testing.assert_allclose(oracle.row_dist(z, 0.8, 0, 1.5, lib=lib)[0], off, rtol=0)
    P = oracle.row_dist(z, 0.8, 0, 1e-6, lib=lib)[0]
    np.testing.assert_allclose(P[[5, 9]], [0.5, 0.5], rtol=1e-12)
    assert np.count_nonzero(P) == 2


# ----------------------------------------------------------------------------------------------
# draft temperature
# ----------------------------------------------------------------------------------------------
def test_draft_temperature_reaches_q_rows_only(lib=None):
    rng = np.random.default_rng(11)
    B, K, V = 6, 3, 50
    Tp, Tq = 1.3, 0.5
    q_target = rng.dirichlet(np.ones(V), size=(B, K))
    zq = (Tq * np.log(q_target)).astype(np.float32)
    zp = rng.standard_normal((B, K + 1, V)).astype(np.float32) * 2
    draft = np.stack([[rng.choice(V, p=q_target[b, j]) for j in range(K)] for b in range(B)]).astype(np.int32)
    ua = np.zeros((B, K), np.float32)  # u = 0 accepts every draft with p > 0: all positions examined
    ur = np.full(B, 0.5, np.float32)
    out = oracle.verify(zp, zq, draft, None, ua, ur, Tp, draft_temperature=Tq, lib=lib)
    Tp32 = float(np.float32(Tp))  # the batch entry takes temperatures as float32
    P = torch.softmax(torch.from_numpy(zp.astype(np.float64)) / Tp32, -1).numpy()
    for b in range(B):
        for j in range(K):
            np.testing.assert_allclose(out["q_draft"][b, j], q_target[b, j, draft[b, j]], rtol=1e-5)
            np.testing.assert_allclose(out["p_draft"][b, j], P[b, j, draft[b, j]], rtol=1e-12)
    # one temperature for both sides gives other q values: the parameter is not ignored
    same = oracle.verify(zp, zq, draft, None, ua, ur, Tp, lib=lib)
    assert not np.allclose(same["q_draft"], out["q_draft"], rtol=1e-3)


def test_lossless_with_draft_temperature_and_topp(lib=None):
    rng = np.random.default_rng(21)
    for K in (1, 2):
        zp = rng.standard_normal((K + 1, 4)).astype(np.float32)
        zq = rng.standard_normal((K, 4)).astype(np.float32)
        P = np.stack([oracle.row_dist(zp[j], 1.0, 0, 0.85, lib=lib)[0] for j in range(K + 1)])
        Q = np.stack([oracle.row_dist(zq[j], 0.6, 0, 0.85, lib=lib)[0] for j in range(K)])
        assert (P == 0).any() or (Q == 0).any()  # the truncation is active
        check_lossless(P, Q, lib)


# ----------------------------------------------------------------------------------------------
# planted mistakes
# ----------------------------------------------------------------------------------------------
MUTANTS = {
    "topp_drops_boundary_group": ("if (P_out[v] > 0.0 && logit_at(z, dtype, (size_t)v) >= tp) {",
                                  "if (P_out[v] > 0.0 && logit_at(z, dtype, (size_t)v) > tp) {"),
    "topp_no_renormalise": ("for (int v = 0; v < V; ++v) P_out[v] /= mass;", ""),
    "topp_walks_upwards": ("if (x->z != y->z) return (x->z < y->z) - (x->z > y->z);",
                           "if (x->z != y->z) return (x->z > y->z) - (x->z < y->z);"),
    "topp_stops_one_group_late": ("if (taken + g >= top_p) {", "if (taken >= top_p) {"),
    "draft_temperature_ignored": ("dtype, V, Tq, top_k, tp, cq, Qr", "dtype, V, T, top_k, tp, cq, Qr"),
}


def _pins_fail(lib):
    checks = [lambda: test_topp_hand_example(lib), lambda: test_topp_against_brute_force(0, lib),
              lambda: test_topp_limits(lib), lambda: test_draft_temperature_reaches_q_rows_only(lib)]
    for c in checks:
        try:
            c()
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
