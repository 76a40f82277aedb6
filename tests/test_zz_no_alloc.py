"""spec_verify_static: the verify step for callers that cannot allocate device memory.

Some callers cannot give this library a workspace: an operator running inside a framework whose
memory pool owns all device memory, or a loop that must never block on cudaMalloc / cudaFree.
spec_verify_static keeps its scratch in one fixed device array instead.  This test calls it
through the C ABI and checks that two calls in a row give exactly what spec_verify gives with a
caller-provided workspace (same kernels, same inputs: every output and statistic agrees bit for
bit), with another batch run through the same array between the two calls so that nothing a
previous call left there can leak into the next; that the size limit follows the call's own mode
(a greedy fp32 batch of 1024 x 4 x 128256 fits, the sampled one does not); and that bad
arguments get the status codes spec_verify gives them.
"""
import ctypes

import numpy as np
import pytest

import workloads as W
from _parity import to_dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _run(lib, fn, d, ws=None):
    import speculative_decoding_rejection_verify_gb300 as sv
    dev = torch.device("cuda:0")
    w = d["workload"]
    B, K, V = w.B, w.K, w.V
    greedy = w.temperature == 0
    p, q = to_dev(d["p"], dev), None if greedy else to_dev(d["q"], dev)
    x = to_dev(d["draft"], dev)
    kpr = to_dev(d["k_per_row"], dev) if w.ragged else None
    ua = None if greedy else to_dev(d["ua"], dev)
    ur = None if greedy else to_dev(d["ur"], dev)
    tok = torch.full((B, K + 1), -7, dtype=torch.int32, device=dev)
    n = torch.full((B,), -7, dtype=torch.int32, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    st = dict(p_draft=torch.empty((B, K), **f32), q_draft=torch.empty((B, K), **f32),
              accept_margin=torch.empty((B, K), **f32), sample_margin=torch.empty(B, **f32),
              residual_mass=torch.empty(B, **f32), row_lognorm=torch.empty((B, 2 * K + 1), **f32),
              flags=torch.empty(B, dtype=torch.int32, device=dev), row_cut=torch.empty((B, 2 * K + 1), **f32))
    sp = sv.StatsStruct(**{k: v.data_ptr() for k, v in st.items()})
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    dt = sv.DTYPE_BF16 if w.dtype == "bf16" else sv.DTYPE_F32
    args = [ptr(p), ptr(q), ptr(x), ptr(kpr), ptr(ua), ptr(ur), float(w.temperature), int(w.top_k),
            tok.data_ptr(), n.data_ptr(), ctypes.byref(sp), B, K, V, dt]
    stream = torch.cuda.current_stream().cuda_stream
    if fn == "static":
        rc = lib.spec_verify_static(*args, stream)
    else:
        rc = lib.spec_verify(*args, ws.data_ptr(), ws.numel(), stream)
    torch.cuda.synchronize()
    out = dict(tokens=tok.cpu().numpy(), n_acc=n.cpu().numpy())
    out.update({k: v.cpu().numpy() for k, v in st.items()})
    return rc, out


STATS = ("p_draft", "q_draft", "accept_margin", "sample_margin", "residual_mass", "row_lognorm", "row_cut")


@pytest.mark.parametrize("name,over", [("c5_a0.8", dict(B=256)), ("c5_greedy", dict(B=128)), ("c2", {}),
                                       ("c4", dict(B=3, V=20000, tau=0.6))])
def test_static_scratch_matches_workspace_entry(name, over):
    import speculative_decoding_rejection_verify_gb300 as sv
    lib = sv.load()
    d = W.generate(W.get(name, **over))
    other = W.generate(W.get("c3", B=5, V=40000, tau=0.8))  # a different batch in between
    w = d["workload"]
    dt = sv.DTYPE_BF16 if w.dtype == "bf16" else sv.DTYPE_F32
    ws = torch.zeros(sv.workspace_bytes(w.B, w.K, w.V, dt, w.top_k), dtype=torch.uint8, device="cuda:0")
    rc, ref = _run(lib, "workspace", d, ws)
    assert rc == 0
    for _ in range(2):  # two calls in a row share the one array
        rc, got = _run(lib, "static", d)
        assert rc == 0, sv.STATUS.get(rc)
        for k in ("tokens", "n_acc", "flags") + STATS:
            np.testing.assert_array_equal(got[k], ref[k], err_msg=k)  # NaN where NaN, bit for bit
        rc, _ = _run(lib, "static", other)
        assert rc == 0


def _big_greedy(dtype):
    dev = torch.device("cuda:0")
    B, K, V = 1024, 4, 128256
    g = torch.Generator(device=dev).manual_seed(5)
    p = torch.randn((B, K + 1, V), generator=g, device=dev, dtype=dtype)
    x = torch.randint(0, V, (B, K), generator=g, device=dev, dtype=torch.int32)
    x[::2] = p[::2, :K].float().argmax(-1).int()  # half the requests match every draft
    return p, x


def test_static_scratch_sizes_follow_the_call_mode():
    """Greedy fp32 at 1024 x 4 x 128256 needs about 10.5 MB and fits the fixed array (matching the
    workspace entry bit for bit); the sampled fp32 batch of that size needs about 19 MB and is
    refused before anything is launched."""
    import speculative_decoding_rejection_verify_gb300 as sv
    lib = sv.load()
    p, x = _big_greedy(torch.float32)
    B, K1, V = p.shape
    K = K1 - 1
    dev = p.device
    stream = torch.cuda.current_stream().cuda_stream

    def call(fn, ws=None, T=0.0):
        tok = torch.full((B, K + 1), -7, dtype=torch.int32, device=dev)
        n = torch.full((B,), -7, dtype=torch.int32, device=dev)
        args = [p.data_ptr(), p.data_ptr() if T > 0 else None, x.data_ptr(), None,
                x.data_ptr() if T > 0 else None, x.data_ptr() if T > 0 else None, T, 0, tok.data_ptr(),
                n.data_ptr(), None, B, K, V, sv.DTYPE_F32]
        rc = lib.spec_verify_static(*args, stream) if fn == "static" else \
            lib.spec_verify(*args, ws.data_ptr(), ws.numel(), stream)
        torch.cuda.synchronize()
        return rc, tok.cpu().numpy(), n.cpu().numpy()

    ws = torch.zeros(sv.workspace_bytes(B, K, V, sv.DTYPE_F32, 0), dtype=torch.uint8, device=dev)
    rc, tok_ref, n_ref = call("workspace", ws)
    assert rc == 0
    rc, tok, n = call("static")
    assert rc == 0, sv.STATUS.get(rc)
    np.testing.assert_array_equal(tok, tok_ref)
    np.testing.assert_array_equal(n, n_ref)
    assert (n_ref[::2] == K).all()
    # sampled: the per-warp summaries of 9 rows x 32 chunks per request need about 19 MB
    rc, tok, _ = call("static", T=1.0)
    assert rc == 4 and (tok == -7).all()  # SPEC_ERR_WORKSPACE, nothing written


def test_static_scratch_refuses_oversized_batches():
    import speculative_decoding_rejection_verify_gb300 as sv
    lib = sv.load()
    B, K, V = 256, 8, 152064  # top-k candidates for this batch need far more than the fixed array
    need = sv.workspace_bytes(B, K, V, sv.DTYPE_F32, 50)
    assert need > sv.STATIC_SCRATCH_BYTES
    dev = torch.device("cuda:0")
    one = torch.zeros(16, dtype=torch.int32, device=dev)
    p = one.data_ptr()
    rc = lib.spec_verify_static(p, p, p, None, p, p, 0.7, 50, p, p, None, B, K, V, sv.DTYPE_F32,
                                torch.cuda.current_stream().cuda_stream)
    assert rc == 4  # SPEC_ERR_WORKSPACE, before anything is launched or read


def test_static_scratch_status_codes_match_spec_verify():
    """Host-checkable errors come back with spec_verify's codes (nothing is launched)."""
    import speculative_decoding_rejection_verify_gb300 as sv
    lib = sv.load()
    dev = torch.device("cuda:0")
    one = torch.zeros(16, dtype=torch.int32, device=dev)
    p = one.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=dev)
    cases = [dict(B=-1, K=4, V=100, dt=0, T=1.0), dict(B=2, K=sv.MAX_K + 1, V=100, dt=0, T=1.0),
             dict(B=2, K=4, V=sv.MAX_V + 1, dt=0, T=1.0), dict(B=2, K=4, V=100, dt=7, T=1.0),
             dict(B=2, K=4, V=100, dt=0, T=-1.0), dict(B=0, K=4, V=100, dt=0, T=1.0)]
    for c in cases:
        a = [p, p, p, None, p, p, c["T"], 0, p, p, None, c["B"], c["K"], c["V"], c["dt"]]
        want = lib.spec_verify(*a, ws.data_ptr(), ws.numel(), s)
        got = lib.spec_verify_static(*a, s)
        assert got == want, (c, got, want)
    # a missing required pointer
    a = [None, p, p, None, p, p, 1.0, 0, p, p, None, 2, 4, 100, 0]
    assert lib.spec_verify_static(*a, s) == lib.spec_verify(*a, ws.data_ptr(), ws.numel(), s) == 1
    torch.cuda.synchronize()
