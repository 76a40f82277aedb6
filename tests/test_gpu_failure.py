"""A lost streaming item is flagged, tested without any fault: under the test hook
(spec_verify_set_test_hooks, bit 0) every block of the streaming pass leaves the summaries of the
chunks it was to read NaN instead of reading them, and every request of the batch comes out
flagged non-finite with n_acc 0 and tokens -1.  With the hook cleared the next call on the same
context is exact again."""
import numpy as np
import pytest

import workloads as W
from _parity import compare, run_gpu, run_oracle, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

NONFINITE = 16


@pytest.mark.parametrize("name,over", [("c5_a0.8", dict(B=16)), ("c5_a0.8", dict(B=200)),
                                       ("c5_a0.8", dict(B=300, V=40000, ragged=(0, 4))),
                                       ("c5_greedy", dict(B=16)), ("c5_topp0.9", dict(B=8))],
                         ids=["cluster_tail", "block_tail", "block_tail_ragged", "greedy", "top_p"])
def test_lost_items_flag_the_batch(name, over):
    import speculative_decoding_rejection_verify_gb300 as sv
    d = W.generate(W.get(name, **over))
    sv.set_test_hooks(1)
    try:
        g = run_gpu(d)
    finally:
        sv.set_test_hooks(0)
    assert (g["flags"] & NONFINITE).all(), g["flags"]
    assert (g["n_acc"] == 0).all() and (g["tokens"] == -1).all()
    # the context is still usable and the next call exact
    g2 = run_gpu(d)
    o = run_oracle(d)
    res = compare(g2, o, d["workload"].K, d["k_per_row"])
    assert res["exact"] + res["low_margin"] == res["requests"]


@pytest.mark.parametrize("B", [32, 300])
def test_lost_items_in_the_sampler(B):
    import speculative_decoding_rejection_verify_gb300 as sv
    d = W.generate(W.get("sample_c5", B=B))
    logits = to_dev(d["p"][:, 0, :].copy(), "cuda:0")
    u = to_dev(d["ur"], "cuda:0")
    sv.set_test_hooks(1)
    try:
        tok, pr = sv.sample(logits, u, d["temperature"])
        torch.cuda.synchronize()
    finally:
        sv.set_test_hooks(0)
    assert (tok.cpu().numpy() == -1).all() and np.isnan(pr.cpu().numpy()).all()
    tok2, _ = sv.sample(logits, u, d["temperature"])
    torch.cuda.synchronize()
    assert (tok2.cpu().numpy() >= 0).all()
