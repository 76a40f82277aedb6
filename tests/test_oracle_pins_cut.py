"""Pins of the oracle's row cuts (CPU only).  The top-p parity tests lean on two oracle paths that
no other pin reaches: the cut each row reports (row_cut: the smallest logit the row keeps, the
larger of the top-k threshold and the nucleus cut, gsyq.cn §3.3) and the verify step rerun with
cuts given from outside (row_cut in, keep the logits >= cut inside the top-k set).

* a given cut on a hand-built row of binary-fraction probabilities, with and without top-k,
  including a tie group at the cut and a cut above every logit;
* the reported cut against a brute force over every candidate threshold (library top-k and
  softmax) on small random rows with ties, with and without top-k, at several temperatures;
* the verify step rerun with its own cuts gives the same tokens and margins;
* planted mistakes in these paths each fail one of the pins.
"""
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle

NONFINITE = 16


def _binary_row():
    # probabilities 1/2, 1/4, 1/8, 1/8 at T = 1, as float32 logits
    return np.log(np.array([0.5, 0.25, 0.125, 0.125])).astype(np.float32)


def test_given_cut_hand_row(lib=None):
    z = _binary_row()
    zc = z.astype(np.float64)  # cuts are compared with the logits as the step reads them
    cases = [  # (cut, top_k, expected law, expected kept count)
        (zc[0], 0, [1.0, 0, 0, 0], 1),
        (zc[1], 0, [2 / 3, 1 / 3, 0, 0], 2),
        (zc[2], 0, [0.5, 0.25, 0.125, 0.125], 4),  # the tie group at the cut is kept whole
        (zc[2] - 1.0, 0, [0.5, 0.25, 0.125, 0.125], 4),
        (zc[2], 2, [2 / 3, 1 / 3, 0, 0], 2),  # only logits inside the top-k set survive
        (zc[1], 3, [2 / 3, 1 / 3, 0, 0], 2),
    ]
    for cut, top_k, ref, kept in cases:
        P, info, fl = oracle.row_dist(z, 1.0, top_k, 1.0, lib=lib, cut=float(cut))
        assert fl & NONFINITE == 0
        np.testing.assert_allclose(P, ref, rtol=1e-6, atol=1e-12, err_msg=f"cut {cut} top_k {top_k}")
        assert info["kept"] == kept
        # the normaliser of the kept weights: m + log(sum of exp(z - m) over the kept logits)
        w = np.exp(zc - zc[0])[np.array(ref) > 0].sum()
        assert abs(info["lognorm"] - (zc[0] + np.log(w))) < 1e-12
    # a cut above every kept logit leaves nothing to sample from
    P, _, fl = oracle.row_dist(z, 1.0, 0, 1.0, lib=lib, cut=float(zc[0]) + 0.5)
    assert fl & NONFINITE and np.isnan(P).all()


def _brute_cut(z, T, top_k, top_p):
    """The smallest kept logit by trying every threshold: the top-k threshold (library topk), then
    the largest logit t of the top-k set whose upper set holds mass >= top_p (library softmax)."""
    z64 = torch.from_numpy(z.astype(np.float64))
    V = z.shape[0]
    if 0 < top_k < V:
        kth = float(torch.topk(z64, top_k).values[-1])
        base = z64 >= kth
    else:
        kth = -np.inf
        base = torch.ones(V, dtype=torch.bool)
    if top_p >= 1.0:
        return kth, np.inf
    P = torch.softmax(torch.where(base, z64 / T, torch.tensor(-np.inf, dtype=torch.float64)), 0).numpy()
    gap = np.inf
    for t in sorted(set(z[base.numpy()].astype(np.float64).tolist()), reverse=True):
        mass = P[z >= t].sum()
        gap = min(gap, abs(mass - top_p))
        if mass >= top_p:
            return max(t, kth), gap
    raise AssertionError("no threshold reaches top_p")


def _rows_verify(z, T, top_k, top_p, lib=None, row_cut=None):
    """The verify step on rows as requests without drafts (each row a bonus draw)."""
    B, V = z.shape
    p = z.reshape(B, 1, V)
    ur = ((np.arange(B) * 7919 % 4096) / 4096.0).astype(np.float32)
    return oracle.verify(p, None, np.zeros((B, 0), np.int32), None, None, ur, T, top_k, lib=lib, top_p=top_p,
                         row_cut=row_cut)


@pytest.mark.parametrize("seed", range(6))
def test_reported_cut_against_brute_force(seed, lib=None):
    rng = np.random.default_rng(900 + seed)
    checked = 0
    for _ in range(12):
        V = int(rng.integers(3, 12))
        B = 6
        z = (np.round(rng.standard_normal((B, V)) * 2) / 2).astype(np.float32)  # many exact ties
        T = float(rng.choice([0.6, 1.0, 1.5]))
        top_k = int(rng.choice([0, int(rng.integers(1, V))]))
        top_p = float(np.float32(rng.choice([1.0, rng.uniform(0.1, 0.99)])))
        o = _rows_verify(z, T, top_k, top_p, lib=lib)
        for b in range(B):
            ref, gap = _brute_cut(z[b], T, top_k, top_p)
            if gap < 1e-9:
                continue  # top_p within rounding of a cumulative mass: either side is correct
            got = o["row_cut"][b, 0]
            if ref == -np.inf:  # no truncation at all
                assert np.isnan(got) or got == -np.inf or got <= z[b].min(), (got, z[b])
            else:
                assert got == ref, (b, z[b], T, top_k, top_p, got, ref)
            checked += 1
    assert checked >= 40


def test_rerun_with_own_cuts_is_identical(lib=None):
    rng = np.random.default_rng(77)
    for top_k, top_p in [(0, 0.7), (5, 0.9), (8, 1.0)]:
        z = (rng.standard_normal((16, 40)) * 2).astype(np.float32)
        a = _rows_verify(z, 0.9, top_k, top_p, lib=lib)
        b = _rows_verify(z, 0.9, top_k, top_p, lib=lib, row_cut=a["row_cut"])
        np.testing.assert_array_equal(a["tokens"], b["tokens"])
        np.testing.assert_allclose(a["sample_margin"], b["sample_margin"], rtol=1e-12, atol=1e-15)
        np.testing.assert_array_equal(a["row_cut"], b["row_cut"])


# ----------------------------------------------------------------------------------------------
# planted mistakes
# ----------------------------------------------------------------------------------------------
MUTANTS = {
    "given_cut_drops_boundary": ("if (P_out[v] > 0.0 && logit_at(z, dtype, (size_t)v) >= cut) {",
                                 "if (P_out[v] > 0.0 && logit_at(z, dtype, (size_t)v) > cut) {"),
    "given_cut_ignores_topk": ("if (P_out[v] > 0.0 && logit_at(z, dtype, (size_t)v) >= cut) {",
                               "if (logit_at(z, dtype, (size_t)v) >= cut) {"),
    "reported_cut_nucleus_only": ("if (co) co[j] = info[4] > info[2] ? info[4] : info[2];",
                                  "if (co) co[j] = info[4];"),
}


def _pins_fail(lib):
    checks = [lambda: test_given_cut_hand_row(lib), lambda: test_reported_cut_against_brute_force(0, lib),
              lambda: test_rerun_with_own_cuts_is_identical(lib)]
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
