"""GPU parity of the sampling-parameter variants against the fp64 oracle: a draft temperature of
its own (2kiu.com §7) and top-p / nucleus truncation (gsyq.cn §3.3), alone and with top-k, at
small sizes and at the full size of the largest batch (every request compared), plus the limits
(top_p = 1 and T_q = T reproduce spec_verify bit for bit; a vanishing top_p keeps the maximal
logits; greedy ignores both) and exact ties in bf16."""
import numpy as np
import pytest

import workloads as W
from _parity import check, run_gpu, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _check(d, **kw):
    """Element-by-element parity (with top-p, against the oracle run with the GPU's nucleus cuts
    once each cut that differs from the oracle's is checked to be a correct one up to 1e-5 of
    mass); at most max(2, B/100) requests may differ, each on a decision whose margin is below
    1e-5."""
    kw.setdefault("stats", True)
    g = run_gpu(d, **kw)
    res, o = check(d, g)
    assert res["low_margin"] <= max(2, res["requests"] // 100), res
    return res, g, o


@pytest.mark.parametrize("name,over", [("c5_topp0.9", dict(B=16)), ("c5_tq0.5", dict(B=16)),
                                       ("c5_topp0.9", dict(B=8, dtype="f32")),
                                       ("c5_tq0.5", dict(B=8, dtype="f32"))],
                         ids=["topp_bf16", "tq_bf16", "topp_f32", "tq_f32"])
def test_variant_small(name, over):
    _check(W.generate(W.get(name, **over)))


@pytest.mark.parametrize("top_p", [1e-6, 0.3, 0.7, 0.95, 0.999])
@pytest.mark.parametrize("tq", [None, 0.6])
def test_topp_sweep(top_p, tq):
    w = W.get("c2", B=8, top_p=top_p, draft_temperature=tq, tau=0.6)
    _check(W.generate(w))


def test_topp_with_topk_ragged():
    w = W.get("c4", B=8, top_p=0.8, draft_temperature=0.5, tau=0.6)
    _check(W.generate(w))


def test_topp_exact_ties_bf16():
    """Logits on a coarse grid: many equal values straddle every nucleus cut."""
    w = W.get("c2", B=8, top_p=0.6, tau=0.6)
    d = W.generate(w)
    for key in ("p", "q"):
        f = W.bf16_bits_to_f32(d[key])
        d[key] = W.to_bf16_bits(np.round(f * 2) / 2)
    _check(d)


def test_tiny_topp_keeps_the_maximum():
    w = W.get("c1", top_p=1e-6)
    d = W.generate(w)
    res, g, o = _check(d)
    # with only the argmax group kept, every draft that is not the argmax is rejected and the
    # resample / bonus draw returns the argmax of the row
    p = W.as_f32(d["p"])[0]
    n = int(g["n_acc"][0])
    assert g["tokens"][0, n] == int(np.argmax(p[n]))


def test_limits_match_spec_verify_bit_for_bit():
    import speculative_decoding_rejection_verify_gb300 as sv
    d = W.generate(W.get("c5_a0.8", B=16))
    a = run_gpu(d, top_p=1.0, draft_temperature=None)
    dev = "cuda:0"
    args = (to_dev(d["p"], dev), to_dev(d["q"], dev), to_dev(d["draft"], dev), None, to_dev(d["ua"], dev),
            to_dev(d["ur"], dev), 1.0, 0)
    b = sv.verify(*args, stats=True, top_p=1.5, draft_temperature=1.0)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(a["tokens"], b[0].cpu().numpy())
    np.testing.assert_array_equal(a["row_lognorm"], b[2]["row_lognorm"].cpu().numpy())


def test_greedy_ignores_sampling_parameters():
    d = W.generate(W.get("c5_greedy", B=16))
    a = run_gpu(d)
    b = run_gpu(d, top_p=0.5, draft_temperature=0.3)
    np.testing.assert_array_equal(a["tokens"], b["tokens"])
    np.testing.assert_array_equal(a["n_acc"], b["n_acc"])


@pytest.mark.parametrize("name", ["c5_topp0.9", "c5_tq0.5"])
def test_variant_full(name):
    """The full batch in the launch configuration the benchmark times; every request compared."""
    d = W.generate(W.get(name))
    res, _, _ = _check(d)
    print(name, res)
    assert res["requests"] == 1024, res


def test_host_entry_with_sampling():
    import speculative_decoding_rejection_verify_gb300 as sv
    d = W.generate(W.get("c5_topp0.9", B=8))
    g = run_gpu(d, stats=False)
    tok, n = sv.verify_host(d["p"], d["q"], d["draft"], None, d["ua"], d["ur"], d["temperature"], d["top_k"],
                            top_p=d["top_p"], draft_temperature=d["draft_temperature"])
    np.testing.assert_array_equal(tok, g["tokens"])
    np.testing.assert_array_equal(n, g["n_acc"])


# ---------------------------------------------------------------------------------------------
# the nucleus pass (top-p without top-k) on layouts and rows its common path does not settle
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_topp_both_dtypes(dtype):
    _check(W.generate(W.get("c5_topp0.9", B=12, dtype=dtype)))


def test_topp_ragged_sampling_mode():
    """Ragged K_b with top-p and no top-k: the nucleus pass takes its rows from the row table
    (rows past K_b are never read), with a draft temperature of its own."""
    w = W.get("c5_topp0.9", B=16, ragged=(0, 4), draft_temperature=0.7)
    _check(W.generate(w))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_topp_rows_off_the_common_path(dtype):
    """Rows the one-read common path cannot settle, mixed with ordinary ones in one batch:
    ascending rows (a crowded head), constant rows (every logit tied) and a row whose cut lies in
    the tail, below 2^-15 of the max's weight.  They take the multi-pass search and must come out
    exactly as the oracle has them."""
    w = W.get("c5_topp0.9", B=6, dtype=dtype)
    d = W.generate(w)
    V = w.V
    rng = np.random.default_rng(7)
    rows = {}
    ramp = np.linspace(-20.0, 10.0, V, dtype=np.float32)
    rows[(0, 0)] = ramp                                   # ascending p row
    rows[(1, 1)] = ramp + rng.normal(0, 0.05, V).astype(np.float32)
    rows[(2, 0)] = np.full(V, 1.5, np.float32)            # constant row
    # one spike over a low tail (each tail weight below 2^-15 of the spike's) that holds most of
    # the mass, so the cut lies in the tail
    tail = (-8.0 + rng.normal(0, 0.3, V)).astype(np.float32)
    tail[rng.integers(V)] = 3.0
    rows[(3, 2)] = tail
    for (b, j), z in rows.items():
        for key in ("p", "q"):
            if key == "q" and j >= w.K:
                continue
            d[key][b, j] = W.to_bf16_bits(z) if dtype == "bf16" else z
    _check(d)
