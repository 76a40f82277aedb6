"""GPU parity of multi-draft verify (spec_verify_multi) against the fp64 oracle.

Several draft chains per request: their first drafts are tested in turn against what the earlier
rejections leave of p, and the first accepted chain is verified on with the single-draft rule (the
rule and its losslessness pins are in oracle.c and test_oracle_pins_multidraft.py).  The emitted
tokens, the accepted count and the chosen chain must equal the oracle's, except where a decision
that differs has an oracle margin below 1e-5 (at most max(2, B/100) requests).  One chain gives
spec_verify's tokens on the test's batch; greedy; bad tokens; a NaN in a row the step never reads (row 0 of
a later chain) changes nothing, a NaN in a row it reads flags the request; lost streaming items
flag every request; argument checks."""
import numpy as np
import pytest

import workloads as W
from _parity import MARGIN, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _gpu(d, dev="cuda:0"):
    import speculative_decoding_rejection_verify_gb300 as sv
    T = d["temperature"]
    greedy = T == 0.0
    tok, n, ch, fl = sv.verify_multi(to_dev(d["p"], dev), None if greedy else to_dev(d["q"], dev),
                                     to_dev(d["draft"], dev), None if greedy else to_dev(d["ua"], dev),
                                     None if greedy else to_dev(d["ur"], dev), T,
                                     draft_temperature=d["draft_temperature"])
    torch.cuda.synchronize()
    return dict(tokens=tok.cpu().numpy(), n_acc=n.cpu().numpy(), chain=ch.cpu().numpy(), flags=fl.cpu().numpy())


def _oracle(d):
    import os
    import oracle
    return oracle.verify_multi(d["p"], d["q"], d["draft"], d["ua"], d["ur"], d["temperature"],
                               draft_temperature=d["draft_temperature"], nthreads=os.cpu_count() or 1)


def compare_multi(g, o):
    B = len(o["n_acc"])
    low = 0
    for b in range(B):
        assert (int(g["flags"][b]) & (4 | 16)) == (int(o["flags"][b]) & (4 | 16)), (b, g["flags"][b], o["flags"][b])
        if o["flags"][b] & 16:
            assert (g["tokens"][b] == -1).all() and g["n_acc"][b] == 0 and g["chain"][b] == -1
            continue
        to, tg = o["tokens"][b], g["tokens"][b]
        no, ng, co, cg = int(o["n_acc"][b]), int(g["n_acc"][b]), int(o["chain"][b]), int(g["chain"][b])
        ng_valid = (tg[ng + 1:] == -1).all() and 0 <= tg[ng]
        assert ng_valid, (b, tg, ng)
        if no == ng and co == cg and (to == tg).all():
            continue
        am = o["accept_margin"][b]
        if co != cg:  # a first-position test came out differently: one of the tests taken was close
            tested = [n for n in range(am.shape[0]) if np.isfinite(am[n, 0]) or np.isinf(am[n, 0])]
            m = min(am[n, 0] for n in tested)
        elif no != ng:
            m = am[co, min(no, ng)]
            assert (to[: min(no, ng)] == tg[: min(no, ng)]).all()
        else:
            m = o["sample_margin"][b]
            assert (to[:no] == tg[:no]).all()
        assert m < MARGIN, f"b={b}: gpu {tg} n={ng} chain={cg} vs oracle {to} n={no} chain={co} (margin {m})"
        low += 1
    assert low <= max(2, B // 100), low
    return low


CASES = [
    dict(N=2, over=dict(B=64, K=3, V=32000, tau=1.5)),
    dict(N=4, over=dict(B=48, K=4, V=20000, dtype="f32", temperature=0.8, draft_temperature=0.6, tau=2.5)),
    dict(N=3, over=dict(B=40, K=1, V=3001, tau=3.0)),
    dict(N=4, over=dict(B=16, K=2, V=128256, tau=4.0)),
    dict(N=2, over=dict(B=200, K=4, V=40000, tau=0.8)),
    # rows of one or two 256-logit tiles: most blocks of a request's cluster hold no tile at all
    dict(N=3, over=dict(B=24, K=2, V=8, tau=3.0)),
    dict(N=4, over=dict(B=24, K=2, V=264, dtype="f32", tau=3.0)),
]


@pytest.mark.parametrize("case", CASES, ids=["n2", "n4_f32_tq", "n3_k1_odd_v", "n4_wide_low_alpha", "n2_many",
                                             "n3_one_tile", "n4_two_tiles_f32"])
def test_multi_parity(case):
    d = W.generate_multi(W.get("multi_c5", **case["over"]), case["N"])
    g, o = _gpu(d), _oracle(d)
    compare_multi(g, o)
    # the cases exercise every branch: chains after the first accepted, and every candidate rejected
    if case["over"].get("tau", 0) >= 2.5:
        assert (o["chain"] > 0).any() and (o["chain"] == -1).any(), (o["chain"])


def test_one_chain_is_spec_verify():
    import speculative_decoding_rejection_verify_gb300 as sv
    d = W.generate_multi(W.get("multi_c5", B=32, K=4, V=32000, tau=1.0), 1)
    g = _gpu(d)
    dev = "cuda:0"
    tok, n, _ = sv.verify(to_dev(d["p"][:, 0], dev), to_dev(d["q"][:, 0], dev), to_dev(d["draft"][:, 0], dev), None,
                          to_dev(d["ua"][:, 0], dev), to_dev(d["ur"], dev), d["temperature"], 0)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(g["tokens"], tok.cpu().numpy())
    np.testing.assert_array_equal(g["n_acc"], n.cpu().numpy())
    assert ((g["chain"] == 0) == (g["n_acc"] >= 1)).all()


def test_multi_greedy():
    w = W.get("multi_c5", B=40, K=3, V=5000, temperature=0.0, greedy=True)
    d = W.generate_multi(w, 3)
    # about half the requests: a chain whose first draft is the argmax, later drafts mostly too
    rng = np.random.default_rng(1)
    P = W.as_f32(d["p"])
    for b in range(0, 40, 2):
        n = int(rng.integers(0, 3))
        d["draft"][b, n, 0] = int(np.argmax(P[b, 0, 0]))
        for j in range(1, 3):
            if rng.random() < 0.7:
                d["draft"][b, n, j] = int(np.argmax(P[b, n, j]))
    g, o = _gpu(d), _oracle(d)
    np.testing.assert_array_equal(g["tokens"], o["tokens"])
    np.testing.assert_array_equal(g["n_acc"], o["n_acc"])
    np.testing.assert_array_equal(g["chain"], o["chain"])
    assert (o["chain"] >= 0).sum() >= 20


def test_multi_bad_tokens_and_nonfinite_rows():
    d = W.generate_multi(W.get("multi_c5", B=8, K=2, V=3000, dtype="f32", tau=2.0), 3)
    d["draft"][0, :, 0] = [-1, 3000, 7]          # the first two candidates cannot be accepted
    d["p"][1, 1, 0, 5] = np.inf                  # row 0 of a later chain: never read
    d["p"][2, 2, 1, 9] = np.nan                  # a row the step reads
    d["q"][3, 1, 0, :] = -np.inf                 # -inf is a legal logit, but a whole -inf row is not
    g, o = _gpu(d), _oracle(d)
    assert o["flags"][0] & 4 and not o["flags"][1] & 16 and o["flags"][2] & 16 and o["flags"][3] & 16
    compare_multi(g, o)


def test_multi_lost_items_flag_the_batch():
    import speculative_decoding_rejection_verify_gb300 as sv
    d = W.generate_multi(W.get("multi_c5", B=20, K=2, V=30000), 2)
    sv.set_test_hooks(1)
    try:
        g = _gpu(d)
    finally:
        sv.set_test_hooks(0)
    assert (g["flags"] & 16).all() and (g["n_acc"] == 0).all() and (g["tokens"] == -1).all()
    compare_multi(_gpu(d), _oracle(d))


def test_multi_argument_checks():
    import ctypes
    import speculative_decoding_rejection_verify_gb300 as sv
    lib = sv.load()
    dev = torch.device("cuda:0")
    one = torch.zeros(64, dtype=torch.int32, device=dev)
    p = one.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=dev)
    smp = sv.SamplingStruct(1.0, 1.0, 0, 1.0)
    call = lambda N, K=2, V=100, top_k=0, top_p=1.0: lib.spec_verify_multi(  # noqa: E731
        p, p, p, p, p, ctypes.byref(sv.SamplingStruct(1.0, 1.0, top_k, top_p)), p, p, p, p, 2, N, K, V, 0,
        ws.data_ptr(), ws.numel(), s)
    assert call(0) == 1 and call(sv.MAX_DRAFTS + 1) == 2 and call(2, K=sv.MAX_K + 1) == 2
    assert call(2, top_k=10) == 2 and call(2, top_p=0.9) == 2
    assert lib.spec_verify_multi(p, p, p, p, p, ctypes.byref(smp), p, p, p, p, 0, 2, 2, 100, 0, None, 0, s) == 0
    torch.cuda.synchronize()


def test_multi_full_size():
    """The benchmarked multi-draft batch (256 requests x 4 chains x 4 drafts over 128256 bf16
    logits), in the launch configuration bench.py times."""
    d = W.generate_multi(W.get("multi_c5"), 4)
    g, o = _gpu(d), _oracle(d)
    compare_multi(g, o)
    assert (o["chain"] == 0).any() and (o["chain"] > 0).any()
