"""GPU parity: the CUDA verify step against the fp64 oracle on the same seeded inputs.

Each of the five workloads is checked at a size the oracle finishes in seconds (full vocabulary,
several chunks, ragged tails) and at its full size (the launch configuration the benchmark times),
where the oracle runs on every request with all host cores.  Edge cases: empty batch, bonus-only
requests, unaligned vocabularies and pointers, tiny vocabularies, NaN / -inf rows, bad tokens and
bad k_per_row, top-k ties and the exact top-k path, p == q, extreme uniforms, workspace reuse,
streams and the host-buffer entry point.
"""
import numpy as np
import pytest

import workloads as W
from _parity import check, compare, run_gpu, run_oracle, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _check(d, **kw):
    g = run_gpu(d, **kw)
    res, o = check(d, g)
    assert res["low_margin"] <= max(2, res["requests"] // 100), res
    return res, g, o


# ------------------------------------------------------------------------------------------------
# the five workloads, small
# ------------------------------------------------------------------------------------------------
SMALL = [("c1", {}), ("c2", {}), ("c3", dict(B=8)), ("c4", dict(B=8)), ("c5_a0.4", dict(B=16)),
         ("c5_a0.6", dict(B=16)), ("c5_a0.8", dict(B=16)), ("c5_a0.9", dict(B=16)), ("c5_greedy", dict(B=32))]


@pytest.mark.parametrize("name,over", SMALL, ids=[s[0] for s in SMALL])
def test_workload_small(name, over):
    d = W.generate(W.get(name, **over))
    _check(d)


# ------------------------------------------------------------------------------------------------
# full sizes (every request compared)
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["c3", "c4", "c5_a0.4", "c5_a0.8", "c5_a0.9", "c5_greedy"])
def test_workload_full(name):
    d = W.generate(W.get(name))
    res, g, o = _check(d)
    print(name, res)


def test_alpha_sweep_mean_emitted():
    """Mean emitted tokens per request near the closed form sum_n prod alpha (loose, statistical)."""
    for name in ("c5_a0.4", "c5_a0.9"):
        w = W.get(name, B=256)
        d = W.generate(w)
        g = run_gpu(d, stats=False)
        m = (g["n_acc"] + 1).mean()
        a = w.alpha
        e = (1 - a ** (w.K + 1)) / (1 - a)
        assert abs(m - e) < 0.25 * e, (name, m, e)


# ------------------------------------------------------------------------------------------------
# edge cases
# ------------------------------------------------------------------------------------------------
def _gen(name="c2", **over):
    return W.generate(W.get(name, **over))


def test_empty_batch():
    import speculative_decoding_rejection_verify_gb300 as sv
    dev = torch.device("cuda:0")
    p = torch.zeros((0, 5, 100), device=dev)
    tok, n, _ = sv.verify(p, torch.zeros((0, 4, 100), device=dev), torch.zeros((0, 4), dtype=torch.int32, device=dev),
                          None, torch.zeros((0, 4), device=dev), torch.zeros((0,), device=dev), 1.0, 0)
    assert tok.shape == (0, 5) and n.shape == (0,)


def test_ragged_with_bonus_only_requests():
    w = W.get("c3", B=12, V=50000, ragged=(0, 6), tau=1.0)
    d = W.generate(w)
    d["k_per_row"][:3] = 0
    d["k_per_row"][3] = 6
    _check(d, k_per_row=d["k_per_row"])


@pytest.mark.parametrize("V,dtype", [(1001, "bf16"), (1003, "f32"), (7, "f32"), (1, "bf16"), (8200, "bf16"),
                                     (8192 * 3 + 5, "f32")])
def test_odd_vocabularies(V, dtype):
    d = _gen("c2", B=5, V=V, dtype=dtype, tau=0.7)
    _check(d)


def test_unaligned_pointers():
    d = _gen("c2", B=3, V=4096, tau=0.7)
    dev = torch.device("cuda:0")
    import speculative_decoding_rejection_verify_gb300 as sv
    p = to_dev(d["p"], dev)
    q = to_dev(d["q"], dev)
    # shift both logit buffers by one element inside a larger allocation
    pbig = torch.empty(p.numel() + 1, dtype=p.dtype, device=dev)
    qbig = torch.empty(q.numel() + 1, dtype=q.dtype, device=dev)
    pbig[1:].copy_(p.flatten())
    qbig[1:].copy_(q.flatten())
    tok, n, st = sv.verify(pbig[1:].view(p.shape), qbig[1:].view(q.shape), to_dev(d["draft"], dev), None,
                           to_dev(d["ua"], dev), to_dev(d["ur"], dev), d["temperature"], 0, stats=True)
    torch.cuda.synchronize()
    g = dict(tokens=tok.cpu().numpy(), n_acc=n.cpu().numpy(), **{k: v.cpu().numpy() for k, v in st.items()})
    compare(g, run_oracle(d), d["workload"].K)


def test_nonfinite_rows_flagged():
    d = _gen("c2", B=6, V=3000, dtype="f32", tau=0.7)
    d["p"][0, 1, 17] = np.nan
    d["q"][1, 0, 5] = np.inf
    d["p"][2, :, :] = -np.inf
    d["q"][3, 2, :100] = -np.inf  # -inf entries are allowed
    d["p"][4, 0, :] = np.nan
    g, o = run_gpu(d), run_oracle(d)
    assert o["flags"][0] & 16 and o["flags"][1] & 16 and o["flags"][2] & 16 and o["flags"][4] & 16
    assert not o["flags"][3] & 16
    compare(g, o, d["workload"].K)


def test_bad_tokens_and_bad_k():
    w = W.get("c2", B=6, V=3000, tau=0.7, ragged=(1, 5))
    d = W.generate(w)
    d["draft"][0, 0] = -1
    d["draft"][1, 2] = 3000
    d["ua"][1, :2] = 0.0  # make sure the first two are accepted so position 2 is examined
    d["k_per_row"][2] = -3
    d["k_per_row"][3] = 9
    g, o = run_gpu(d, k_per_row=d["k_per_row"]), run_oracle(d, k_per_row=d["k_per_row"])
    assert o["flags"][0] & 4 and o["flags"][2] & 8 and o["flags"][3] & 8
    compare(g, o, w.K, np.clip(d["k_per_row"], 0, w.K))


def test_topk_variants():
    # k = 1, k >= V (off), bf16 logits with many ties, and a small vocabulary (exact top-k path)
    for over in (dict(top_k=1), dict(top_k=200000), dict(dtype="bf16", top_k=50), dict(V=900, top_k=50),
                 dict(top_k=256, B=4), dict(V=20000, top_k=7, temperature=1.3)):
        base = dict(B=6, V=40000, tau=0.6)
        base.update(over)
        d = W.generate(W.get("c4", **base))
        if over.get("dtype") == "bf16":
            for key in ("p", "q"):  # coarse logits: many exact ties around the k-th largest
                f = W.bf16_bits_to_f32(d[key])
                d[key] = W.to_bf16_bits(np.round(f * 2) / 2)
        _check(d)


@pytest.mark.parametrize("top_k", [32, 64, 65])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_topk_with_crowded_rows(top_k, dtype):
    """Rows that crowd the streaming pass's running candidate set, mixed with ordinary rows: a
    constant row (every logit tied, so the set overflows and the row takes the exact path) and an
    ascending row (every chunk raises the bound)."""
    w = W.get("c4", B=6, V=40000, tau=0.6, top_k=top_k, dtype=dtype)
    d = W.generate(w)
    V = w.V
    special = {(0, 0): np.full(V, 2.0, np.float32), (1, 1): np.linspace(-8.0, 8.0, V, dtype=np.float32)}
    for (b, j), z in special.items():
        if j > int(d["k_per_row"][b]):
            continue
        for key in ("p", "q"):
            if key == "q" and j >= int(d["k_per_row"][b]):
                continue
            d[key][b, j] = W.to_bf16_bits(z) if dtype == "bf16" else z
    _check(d)


def test_p_equals_q_accepts_everything():
    d = _gen("c2", B=8, V=5000, tau=0.0)
    d["p"][:, : d["q"].shape[1]] = d["q"]
    g = run_gpu(d)
    assert (g["n_acc"] == d["workload"].K).all()
    compare(g, run_oracle(d), d["workload"].K)


def test_extreme_uniforms():
    d = _gen("c2", B=8, V=5000, tau=0.7)
    d["ua"][:4] = 0.0
    d["ua"][4:] = np.float32(1 - 2 ** -24)
    d["ur"][::2] = 0.0
    d["ur"][1::2] = np.float32(1 - 2 ** -24)
    _check(d)


def test_workspace_reuse_and_determinism():
    d = _gen("c3", B=16, tau=1.0)
    a = run_gpu(d)
    b = run_gpu(d)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])


def test_side_stream():
    d = _gen("c2", B=8)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = run_gpu(d, stream=s)
    compare(g, run_oracle(d), d["workload"].K)


def test_greedy_without_q():
    d = _gen("c5_greedy", B=8, V=6000)
    g = run_gpu(d)  # run_gpu passes q=None at temperature 0
    compare(g, run_oracle(d), d["workload"].K)


def test_host_entry_point_matches_device():
    import speculative_decoding_rejection_verify_gb300 as sv
    for name, over in (("c2", {}), ("c4", dict(B=4)), ("c5_greedy", dict(B=8))):
        d = _gen(name, **over)
        w = d["workload"]
        kpr = d["k_per_row"] if w.ragged else None
        greedy = w.temperature == 0
        tok, n = sv.verify_host(d["p"], None if greedy else d["q"], d["draft"], kpr, None if greedy else d["ua"],
                                None if greedy else d["ur"], w.temperature, w.top_k)
        g = run_gpu(d, stats=False)
        np.testing.assert_array_equal(tok, g["tokens"])
        np.testing.assert_array_equal(n, g["n_acc"])


def test_errors_are_reported():
    import speculative_decoding_rejection_verify_gb300 as sv
    d = _gen("c2", B=2, V=1000)
    dev = torch.device("cuda:0")
    with pytest.raises(sv.SpecVerifyError):
        sv.verify(to_dev(d["p"], dev), to_dev(d["q"], dev), to_dev(d["draft"], dev), None, to_dev(d["ua"], dev),
                  to_dev(d["ur"], dev), -1.0, 0)
    with pytest.raises(sv.SpecVerifyError):
        sv.verify(to_dev(d["p"], dev), to_dev(d["q"], dev), to_dev(d["draft"], dev), None, to_dev(d["ua"], dev),
                  to_dev(d["ur"], dev), 1.0, 300)  # top-k above the supported bound


# ------------------------------------------------------------------------------------------------
# the small-batch tail (an 8-block cluster per request) and the one-block tail, at their switch
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("extra", [0, 1])
def test_cluster_tail_switch(extra):
    """B = the SM count takes the cluster tail, B = SMs + 1 the one-block tail; both must agree
    with the oracle (V = 16392 is just past the cluster tail's vocabulary threshold and leaves a
    ragged last tile in every cluster share)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    d = _gen("c2", B=sms + extra, V=16392, tau=0.9)
    res, _, _ = _check(d)
    assert res["requests"] == sms + extra


def test_cluster_tail_f32_and_zero_residual_fallback():
    # fp32 rows through the cluster tail, and p == q rows with u = 1 - 2^-24: the ratio test
    # accepts (u * q < p with p = q), and where rounding makes it reject, the residual is ~0 and
    # every block of the cluster must take the zero-residual fallback together
    d = _gen("c3", B=6, dtype="f32", V=40000)
    _check(d)
    d = _gen("c3", B=4, V=40000)
    d["p"][:, :6] = d["q"]
    d["ua"][:] = np.float32(1.0 - 2.0 ** -24)
    g = run_gpu(d)
    o = run_oracle(d)
    compare(g, o, d["workload"].K, d["k_per_row"])


@pytest.mark.parametrize("name,over", [("c2", {}), ("c5_a0.8", dict(B=200)), ("c5_topp0.9", dict(B=8))],
                         ids=["cluster_tail", "one_block_tail", "nucleus"])
def test_cuda_graph_replay_matches_direct_calls(name, over):
    """The step (dependent launches between its kernels, cluster tail, nucleus pass) captured in
    a CUDA graph replays to the results of direct calls."""
    import speculative_decoding_rejection_verify_gb300 as sv
    d = W.generate(W.get(name, **over))
    dev = "cuda:0"
    args = (to_dev(d["p"], dev), to_dev(d["q"], dev), to_dev(d["draft"], dev), None, to_dev(d["ua"], dev),
            to_dev(d["ur"], dev), d["temperature"], d["top_k"])
    kw = dict(top_p=d["top_p"], draft_temperature=d["draft_temperature"])
    ref_tok, ref_n, _ = sv.verify(*args, **kw)
    torch.cuda.synchronize()
    B, K1 = ref_tok.shape
    tok = torch.full((B, K1), -7, dtype=torch.int32, device=dev)
    n = torch.full((B,), -7, dtype=torch.int32, device=dev)
    ws = torch.zeros(sv.workspace_bytes(B, K1 - 1, d["p"].shape[-1], sv.DTYPE_BF16, d["top_k"]), dtype=torch.uint8,
                     device=dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # first call outside capture (kernel attributes)
        sv.verify(*args, **kw, workspace_tensor=ws, stream=s, out=(tok, n))
    torch.cuda.synchronize()
    tok.fill_(-7)
    n.fill_(-7)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sv.verify(*args, **kw, workspace_tensor=ws, stream=torch.cuda.current_stream(), out=(tok, n))
    for _ in range(2):
        tok.fill_(-7)
        n.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(tok, ref_tok) and torch.equal(n, ref_n)


# ------------------------------------------------------------------------------------------------
# more requests than SMs (the one-block-per-request tail): just above the SM count, ragged with
# bonus-only requests, one summary group per row block in fp32, and wide rows of 2^20 logits
# ------------------------------------------------------------------------------------------------
def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("over", [dict(B="sms+1"), dict(B=400, V=40000, ragged=(0, 4)),
                                  dict(B=300, V=3000, dtype="f32"), dict(B="sms+8", K=2, V=1 << 20)],
                         ids=["just_above_sms", "ragged_with_bonus_only", "small_rows_f32", "wide_rows"])
def test_many_requests(over):
    over = dict(over)
    if isinstance(over["B"], str):
        over["B"] = _sms() + int(over["B"].split("+")[1])
    d = W.generate(W.get("c5_a0.8", **over))
    if d["workload"].ragged:
        d["k_per_row"][:7] = 0  # bonus-only requests among the others
    res, _, _ = _check(d)
    assert res["requests"] == over["B"]


def test_pass_event_between_the_passes_matches():
    """An event recorded between the passes (the benchmark's pass split) turns the dependent
    launch into a plain one; the results are the same bit for bit."""
    d = W.generate(W.get("c5_a0.8", B=300, V=40000))
    a = run_gpu(d)
    b = run_gpu(d, pass1_event=torch.cuda.Event(enable_timing=True))
    for k in a:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_maximum_sizes(dtype):
    """K_max = 16 drafts over the largest supported vocabulary, 2^21 (SPEC_MAX_K, SPEC_MAX_V):
    rows of 4 (bf16) or 8 (f32) MB, 256 / 512 chunks each."""
    import speculative_decoding_rejection_verify_gb300 as sv
    d = W.generate(W.get("c5_a0.8", B=2, K=sv.MAX_K, V=sv.MAX_V, dtype=dtype))
    res, _, _ = _check(d)
    assert res["requests"] == 2


def test_maximum_k_with_topk_and_topp():
    import speculative_decoding_rejection_verify_gb300 as sv
    d = W.generate(W.get("c4", B=3, K=sv.MAX_K, ragged=None, V=60000, top_k=sv.MAX_TOPK, tau=0.6))
    _check(d)
    d = W.generate(W.get("c5_topp0.9", B=3, K=sv.MAX_K, V=60000, tau=0.6))
    res, _, _ = _check(d)
    assert res["requests"] == 3


# ------------------------------------------------------------------------------------------------
# the short-block streaming pass: each block takes two consecutive 16 KB items, so with an odd
# number of chunks per row blocks straddle rows (the second item in the next row, or the next
# request), and an odd number of items in all leaves the last block one item
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("V,dtype,B,K,greedy", [(16392, "bf16", 5, 3, False), (8196, "f32", 7, 2, False),
                                                 (16392, "bf16", 3, 4, True), (16392, "bf16", 200, 1, False)],
                         ids=["bf16_3chunks", "f32_3chunks", "greedy_odd_items", "many_requests"])
def test_streaming_blocks_straddle_rows(V, dtype, B, K, greedy):
    w = W.get("c5_greedy" if greedy else "c5_a0.8", B=B, K=K, V=V, dtype=dtype)
    per = 16384 // (2 if dtype == "bf16" else 4)
    nchunk = -(-V // per)
    rows = B * (K + 1 if greedy else 2 * K + 1)
    assert nchunk % 2 == 1 or (rows * nchunk) % 2 == 1  # the layouts this test is about
    d = W.generate(w)
    res, _, _ = _check(d)  # tokens, counts, flags and every row's normaliser against the oracle
    assert res["requests"] == B
