"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI and compare it with
the fp64 oracle element by element.

Acceptance criteria (the tolerances the verify step is held to):
* tokens and accepted counts identical, except where the decision that differs has an oracle
  margin below 1e-5 — |u - p/q| for an accept decision, the distance of u to the drawn token's
  CDF edge for a resample / bonus draw; such cases are counted and returned;
* p_j(x_j) and q_j(x_j) within 1e-5 relative; each row's log-normaliser within 1e-5 absolute
  (= 1e-5 relative on every probability of the row); the residual mass within 1e-5;
* the data flags (bad token, bad k, non-finite, top-k tie) identical; the rounding flags
  (zero residual, CDF clamp) are free to differ;
* each row's cut (the smallest kept logit, row_cut) identical: the top-k threshold is an exact
  order statistic;
* with top-p, the nucleus cut compares a float32 cumulative sum with top_p, so where the row's
  mass reaches top_p within rounding either neighbouring cut is right.  Every GPU cut that
  differs from the oracle's is first checked to be a correct one up to 1e-5 of mass (it is a
  logit of the row inside its top-k set; the mass strictly above it is below top_p + 1e-5 and
  the mass at or above it reaches top_p - 1e-5), and then the oracle is run again with the
  GPU's cuts and every request is compared element by element as above.
"""
from __future__ import annotations

import numpy as np

MARGIN = 1e-5
RTOL = 1e-5
DATA_FLAGS = 4 | 8 | 16 | 32


def to_dev(a, dev):
    import torch
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def run_gpu(d, dev="cuda:0", stats=True, k_per_row="auto", **kw):
    import torch
    import speculative_decoding_rejection_verify_gb300 as sv
    kpr = d["k_per_row"]
    w = d.get("workload")
    if isinstance(k_per_row, str):
        k_per_row = kpr if (w is None or w.ragged is not None) else None
    T = d["temperature"]
    greedy = T == 0.0
    kw.setdefault("draft_temperature", d.get("draft_temperature"))
    kw.setdefault("top_p", d.get("top_p", 1.0))
    tok, n, st = sv.verify(to_dev(d["p"], dev), None if greedy else to_dev(d["q"], dev),
                           to_dev(d["draft"], dev), to_dev(k_per_row, dev),
                           None if greedy else to_dev(d["ua"], dev), None if greedy else to_dev(d["ur"], dev),
                           T, d["top_k"], stats=stats, **kw)
    torch.cuda.synchronize()
    out = dict(tokens=tok.cpu().numpy(), n_acc=n.cpu().numpy())
    if st:
        out.update({k: v.cpu().numpy() for k, v in st.items()})
    return out


def run_oracle(d, nthreads=0, k_per_row="auto", row_cut=None):
    import os
    import oracle
    w = d.get("workload")
    kpr = d["k_per_row"]
    if isinstance(k_per_row, str):
        k_per_row = kpr if (w is None or w.ragged is not None) else None
    return oracle.verify(d["p"], d["q"], d["draft"], k_per_row, d["ua"], d["ur"], d["temperature"],
                         d["top_k"], nthreads=nthreads or (os.cpu_count() or 1),
                         draft_temperature=d.get("draft_temperature"), top_p=d.get("top_p", 1.0),
                         row_cut=row_cut)


def nucleus_cuts(d, g, o, kb=None, tol=MARGIN):
    """Checks that every valid row's nucleus cut on the GPU (g["row_cut"]) is a correct one up to
    rounding where it differs from the oracle's (o["row_cut"]), and returns the GPU's cuts for an
    oracle run that takes them (NaN where the oracle has none).  Returns (cuts, rows that differ)."""
    import oracle
    top_p = float(np.float32(d.get("top_p", 1.0)))
    gc, oc = g["row_cut"].astype(np.float64), o["row_cut"]
    B = gc.shape[0]
    Kmax = (gc.shape[1] - 1) // 2
    kb = d["k_per_row"] if kb is None else np.asarray(kb)
    T, Tq = d["temperature"], d.get("draft_temperature") or d["temperature"]
    differ = 0
    for b in range(B):
        if o["flags"][b] & 16:
            continue
        k = int(kb[b])
        rows = [(d["p"][b, j], T, j) for j in range(k + 1)] + [(d["q"][b, j], Tq, Kmax + 1 + j) for j in range(k)]
        for z, Tr, r in rows:
            if gc[b, r] == oc[b, r]:
                continue
            differ += 1
            c = gc[b, r]
            P, info, _ = oracle.row_dist(z, float(np.float32(Tr)), d["top_k"], 1.0)
            zf = z.astype(np.float64) if z.dtype == np.float32 else \
                (z.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            assert (zf == c).any() and c >= info["threshold"], f"b={b} row {r}: cut {c} is not a kept logit"
            above, incl = P[zf > c].sum(), P[zf >= c].sum()
            assert above < top_p + tol and incl >= top_p - tol, \
                f"b={b} row {r}: cut {c} keeps mass {incl} (above it {above}) for top_p {top_p}; oracle cut {oc[b, r]}"
    return np.where(np.isnan(oc), np.nan, gc), differ


def check(d, g, k_per_row="auto", check_stats=True):
    """The oracle on the same inputs (with top-p: again with the GPU's nucleus cuts, once they
    are checked to be correct) and the element-by-element comparison; returns the counts and
    the oracle's result."""
    o = run_oracle(d, k_per_row=k_per_row)
    kb = d["k_per_row"]
    if isinstance(k_per_row, np.ndarray):
        kb = np.clip(k_per_row, 0, d["workload"].K)
    differ = 0
    if d.get("top_p", 1.0) < 1.0 and d["temperature"] > 0:
        assert "row_cut" in g, "top-p parity needs the GPU's row cuts (stats=True)"
        cuts, differ = nucleus_cuts(d, g, o, kb)
        o = run_oracle(d, k_per_row=k_per_row, row_cut=cuts)
    res = compare(g, o, d["workload"].K, kb, check_stats=check_stats)
    res["cuts_differ"] = differ
    return res, o


def compare(g, o, K, kb=None, check_stats=True):
    """Element-by-element comparison; returns a dict of counts (raises AssertionError on failure)."""
    B = o["n_acc"].shape[0]
    kb = np.full(B, K) if kb is None else np.asarray(kb)
    low_margin = 0
    exact = 0
    for b in range(B):
        fo, fg = int(o["flags"][b]), int(g["flags"][b]) if "flags" in g else None
        if fg is not None:
            assert (fo & DATA_FLAGS) == (fg & DATA_FLAGS), f"b={b}: flags gpu {fg:#x} oracle {fo:#x}"
        if fo & 16:  # non-finite rows: the result is unspecified, only the flag is compared
            assert (g["tokens"][b] == -1).all() and g["n_acc"][b] == 0
            continue
        no, ng = int(o["n_acc"][b]), int(g["n_acc"][b])
        to, tg = o["tokens"][b], g["tokens"][b]
        assert 0 <= ng <= kb[b], f"b={b}: n_acc {ng} outside [0, {kb[b]}]"
        if no == ng and (to == tg).all():
            exact += 1
        else:
            j = min(no, ng)
            # the accepted prefix before the first decision that differs is the same draft tokens
            assert (to[:j] == tg[:j]).all(), f"b={b}: accepted prefix gpu {tg[:j]} oracle {to[:j]}"
            if no != ng:
                m = o["accept_margin"][b, j]
                assert m < MARGIN, f"b={b}: accept decision at {j} differs with margin {m} (gpu {ng}, oracle {no})"
            else:
                m = o["sample_margin"][b]
                assert m < MARGIN, f"b={b}: drawn token differs (gpu {tg[j]}, oracle {to[j]}) margin {m}"
                assert (to[:j] == tg[:j]).all()
            low_margin += 1
        assert (tg[ng + 1:] == -1).all(), f"b={b}: padding {tg}"
        assert 0 <= tg[ng] < 1 << 30
        if not check_stats or "p_draft" not in g:
            continue
        jj = min(min(no, ng) + 1, K)  # examined positions on both sides
        for key in ("p_draft", "q_draft"):
            a, r = g[key][b, :jj], o[key][b, :jj]
            sel = np.isfinite(r) & (np.arange(jj) < kb[b])
            np.testing.assert_allclose(a[sel], r[sel], rtol=RTOL, atol=1e-30, err_msg=f"b={b} {key}")
        ln_o, ln_g = o["row_lognorm"][b], g["row_lognorm"][b]
        fin = np.isfinite(ln_o)
        assert (np.isfinite(ln_g) == fin).all(), f"b={b}: lognorm validity {ln_g} vs {ln_o}"
        np.testing.assert_allclose(ln_g[fin], ln_o[fin], rtol=0, atol=RTOL, err_msg=f"b={b} lognorm")
        if "row_cut" in g and "row_cut" in o:
            np.testing.assert_array_equal(g["row_cut"][b][fin], o["row_cut"][b][fin].astype(np.float32),
                                          err_msg=f"b={b} row_cut")
        if no == ng:
            np.testing.assert_allclose(g["residual_mass"][b], o["residual_mass"][b], rtol=0, atol=RTOL)
    return dict(exact=exact, low_margin=low_margin, requests=B)
