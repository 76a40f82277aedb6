"""spec_verify_static: the verify step for callers that cannot allocate device memory.

Some callers cannot give this library a workspace: an operator running inside a framework whose
memory pool owns all device memory, or a loop that must never block on cudaMalloc / cudaFree.
spec_verify_static keeps its scratch in one fixed device array instead.  This test calls it
through the C ABI and checks that two calls in a row give exactly what spec_verify gives with a
caller-provided workspace (same kernels, same inputs: the results agree bit for bit), and that
sizes beyond the fixed array are refused.
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
              flags=torch.empty(B, dtype=torch.int32, device=dev))
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


@pytest.mark.parametrize("name,over", [("c5_a0.8", dict(B=256)), ("c5_greedy", dict(B=128)), ("c2", {}),
                                       ("c4", dict(B=3, V=20000, tau=0.6))])
def test_static_scratch_matches_workspace_entry(name, over):
    import speculative_decoding_rejection_verify_gb300 as sv
    lib = sv.load()
    d = W.generate(W.get(name, **over))
    w = d["workload"]
    dt = sv.DTYPE_BF16 if w.dtype == "bf16" else sv.DTYPE_F32
    ws = torch.zeros(sv.workspace_bytes(w.B, w.K, w.V, dt, w.top_k), dtype=torch.uint8, device="cuda:0")
    rc, ref = _run(lib, "workspace", d, ws)
    assert rc == 0
    for _ in range(2):  # two calls in a row share the one array
        rc, got = _run(lib, "static", d)
        assert rc == 0, sv.STATUS.get(rc)
        for k in ("tokens", "n_acc", "flags"):
            np.testing.assert_array_equal(got[k], ref[k], err_msg=k)
        for k in ("p_draft", "q_draft", "accept_margin", "sample_margin", "residual_mass", "row_lognorm"):
            np.testing.assert_allclose(got[k], ref[k], rtol=1e-5, atol=0, equal_nan=True, err_msg=k)


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
