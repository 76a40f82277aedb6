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
* with top-p, a request any of whose rows has its nucleus cut within 1e-5 of top_p (the
  oracle's nucleus margin) is counted as low-margin and only its output form is checked.
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


def run_oracle(d, nthreads=0, k_per_row="auto"):
    import os
    import oracle
    w = d.get("workload")
    kpr = d["k_per_row"]
    if isinstance(k_per_row, str):
        k_per_row = kpr if (w is None or w.ragged is not None) else None
    return oracle.verify(d["p"], d["q"], d["draft"], k_per_row, d["ua"], d["ur"], d["temperature"],
                         d["top_k"], nthreads=nthreads or (os.cpu_count() or 1),
                         draft_temperature=d.get("draft_temperature"), top_p=d.get("top_p", 1.0))


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
        nm = o.get("nucleus_margin")
        Kmax = (len(o["row_lognorm"][b]) - 1) // 2
        loose = np.zeros(2 * Kmax + 1, bool)  # rows whose top-p cut is within rounding of top_p
        if nm is not None:
            loose = nm[b] < MARGIN
            used = np.zeros_like(loose)
            used[: no + 1] = True                     # p rows 0..n_acc
            used[Kmax + 1: Kmax + 1 + min(no + 1, int(kb[b]))] = True  # q rows 0..n_acc (< K_b)
            if (loose & used).any():
                # a row the decision used has its cut within rounding of top_p: either kept set
                # is correct, so only the form of the result is checked
                low_margin += 1
                assert (tg[ng + 1:] == -1).all() and 0 <= tg[ng] < 1 << 30
                continue
        if no == ng and (to == tg).all():
            exact += 1
        else:
            j = min(no, ng)
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
        cmp = fin & ~loose
        np.testing.assert_allclose(ln_g[cmp], ln_o[cmp], rtol=0, atol=RTOL, err_msg=f"b={b} lognorm")
        if no == ng:
            np.testing.assert_allclose(g["residual_mass"][b], o["residual_mass"][b], rtol=0, atol=RTOL)
    return dict(exact=exact, low_margin=low_margin, requests=B)
