"""GPU parity of draft-token sampling (spec_sample, gsyq.cn §3.1 step 1) against the fp64 oracle:
the drawn token of every row must equal the oracle's inverse-CDF draw from the same row
(the verify step's bonus draw with no drafts), except where u lies within 1e-5 of a CDF edge,
and q(x) must match the oracle's probability of the drawn token within 1e-5 relative.
Covers the full 1024-row batch, temperature / top-k / top-p variants, greedy, small and odd
vocabularies, an empty batch and rows with NaN."""
import numpy as np
import pytest

import workloads as W
from _parity import MARGIN, RTOL, nucleus_cuts, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _run(d, top_p=1.0):
    import speculative_decoding_rejection_verify_gb300 as sv
    T = d["temperature"]
    logits = to_dev(d["p"][:, 0, :].copy(), "cuda:0")
    u = None if T == 0 else to_dev(d["ur"], "cuda:0")
    tok, pr = sv.sample(logits, u, T, d["top_k"], top_p)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), pr.cpu().numpy()


def _oracle(d, top_p=1.0, row_cut=None):
    import os
    import oracle
    B = d["p"].shape[0]
    o = oracle.verify(d["p"], None, np.zeros((B, 0), np.int32), None, None, d["ur"], d["temperature"],
                      d["top_k"], nthreads=os.cpu_count() or 1, top_p=top_p, row_cut=row_cut)
    return o


def _nucleus_cuts(d, tok, top_p):
    """The rows' nucleus cuts as the sampler's kernels find them (the verify step on the same rows
    as requests with no drafts, which reports them), each checked to be a correct cut up to 1e-5
    of mass where it differs from the oracle's."""
    import speculative_decoding_rejection_verify_gb300 as sv
    B = d["p"].shape[0]
    p = to_dev(d["p"], "cuda:0")
    t, _, st = sv.verify(p, None, torch.zeros((B, 0), dtype=torch.int32, device="cuda:0"), None, None,
                         to_dev(d["ur"], "cuda:0"), d["temperature"], d["top_k"], stats=True, top_p=top_p)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(t[:, 0].cpu().numpy(), tok)  # the same kernels, the same draws
    g = dict(row_cut=st["row_cut"].cpu().numpy())
    dd = dict(p=d["p"], q=None, temperature=d["temperature"], draft_temperature=None, top_k=d["top_k"],
              top_p=top_p)
    cuts, _ = nucleus_cuts(dd, g, _oracle(d, top_p), kb=np.zeros(B, np.int32))
    return cuts


def _check(d, top_p=1.0):
    import oracle
    tok, pr = _run(d, top_p)
    cuts = _nucleus_cuts(d, tok, top_p) if top_p < 1.0 and d["temperature"] > 0 else None
    o = _oracle(d, top_p, cuts)
    B = len(tok)
    exact = 0
    for b in range(B):
        if o["flags"][b] & 16:
            assert tok[b] == -1 and np.isnan(pr[b])
            continue
        if tok[b] == o["tokens"][b, 0]:
            exact += 1
        else:
            assert o["sample_margin"][b] < MARGIN, (b, tok[b], o["tokens"][b, 0], o["sample_margin"][b])
            continue
        if d["temperature"] == 0:
            assert pr[b] == 1.0
        else:
            cut = None if cuts is None else float(cuts[b, 0])
            P = oracle.row_dist(d["p"][b, 0], d["temperature"], d["top_k"], top_p, cut=cut)[0]
            np.testing.assert_allclose(pr[b], P[tok[b]], rtol=RTOL, err_msg=f"row {b}")
    assert exact >= B - max(2, B // 100), (exact, B)


@pytest.mark.parametrize("over", [dict(B=64), dict(B=32, temperature=0.7, top_k=50),
                                  dict(B=32, dtype="f32", V=50000, temperature=1.3)],
                         ids=["t1", "topk", "f32"])
def test_sample_variants(over):
    _check(W.generate(W.get("sample_c5", **over)))


@pytest.mark.parametrize("top_p", [0.5, 0.9])
def test_sample_topp(top_p):
    d = W.generate(W.get("sample_c5", B=32))
    _check(d, top_p)


def test_sample_greedy():
    d = W.generate(W.get("sample_c5", B=64, temperature=0.0))
    tok, pr = _run(d)
    ref = np.argmax(W.as_f32(d["p"][:, 0, :]), axis=-1)
    np.testing.assert_array_equal(tok, ref)
    assert (pr == 1.0).all()


def test_sample_full_batch():
    _check(W.generate(W.get("sample_c5")))


@pytest.mark.parametrize("V,dtype", [(1, "bf16"), (7, "f32"), (1001, "bf16"), (32003, "f32")])
def test_sample_odd_vocabularies(V, dtype):
    _check(W.generate(W.get("sample_c5", B=16, V=V, dtype=dtype)))


def test_sample_empty_and_nan_rows():
    import speculative_decoding_rejection_verify_gb300 as sv
    e = torch.empty((0, 100), dtype=torch.float32, device="cuda:0")
    tok, pr = sv.sample(e, torch.empty((0,), dtype=torch.float32, device="cuda:0"))
    assert tok.numel() == 0
    d = W.generate(W.get("sample_c5", B=8, V=3000, dtype="f32"))
    d["p"][3, 0, 17] = np.nan
    _check(d)
