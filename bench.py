"""Benchmark of the speculative-sampling verify step (one JSON line on rank 0).

A step is one spec_verify call over one batch of synthetic requests whose logits are already
resident in HBM.  The default workload is the largest batch, B=1024 requests x K=4 drafts over a
128256-token vocabulary in bf16 (alpha ~ 0.8, T = 1): 2.36 GB of logits per step, well above the
129 MB L2, and two copies of the inputs alternate between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c5_a0.8] [--graph] [--impl reference]

--graph replays each step from a CUDA graph captured once per input copy (the launch-bound small
workloads); the per-pass split is then unavailable and the roofline covers the whole step.

value     = verified draft positions per second over all ranks (sum_b K_b / step time)
roofline  = logits bytes per launch / mean kernel time, against the measured HBM copy peak
            (and against the nominal 8 TB/s); median_step_ms = median of per-step event times
e2e       = the same metric through spec_verify_host (pinned host buffers, copies included)
cpu_baseline = the fp64 oracle on the host cores, on a bounded sample of the same workload
Multi-GPU (torchrun): every rank verifies its own batch of distinct requests (weak scaling, no
collective on the data path); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "verified draft positions/s and logits GB/s (fraction of GB300 HBM peak)"
NOMINAL_HBM_GBS = 8000.0  # the nominal GB300 HBM3e bandwidth the fraction is also quoted against
UNIT = "positions/s"
KERNEL_SRC = os.path.join(ROOT, "speculative_decoding_rejection_verify_gb300", "csrc", "spec_verify.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


# ------------------------------------------------------------------------------------------------
# distributed plumbing (host logic; tested with gloo on CPU)
# ------------------------------------------------------------------------------------------------
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def shard_requests(B: int, rank: int) -> range:
    """The requests rank `rank` verifies: its own B distinct requests (weak scaling)."""
    return range(rank * B, (rank + 1) * B)


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for _, _, fl in rows for n, v in zip(names, fl) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------------------------------------
# helpers
# ------------------------------------------------------------------------------------------------
def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_hash() -> str:
    with open(KERNEL_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def traffic_for(workload_key: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken on this kernel."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        t = json.load(f)
    if t.get("kernel_sha256_16") != kernel_hash():
        return None
    e = t.get("workloads", {}).get(workload_key)
    return None if e is None else e.get("dram_bytes_per_launch")


def describe(w: W.Workload) -> str:
    kk = f"K_b~U{{{w.ragged[0]}..{w.ragged[1]}}}" if w.ragged else f"K={w.K}"
    extra = " greedy" if w.temperature == 0 else f" T={w.temperature:g}" + (f" top_k={w.top_k}" if w.top_k else "")
    if w.temperature and w.tq != w.temperature:
        extra += f" T_q={w.tq:g}"
    if w.temperature and w.top_p < 1.0:
        extra += f" top_p={w.top_p:g}"
    return f"{w.label}: B={w.B} {kk} V={w.V} {w.dtype}{extra}" + \
        (f" alpha~{w.alpha:g}" if w.alpha is not None and not w.greedy else "")


def stream_kernel(w: W.Workload) -> str:
    """The streaming pass's kernel for rows of whole 16-byte vectors (every workload here):
    short-lived blocks in sampling and greedy modes, the persistent candidate-set grid for top-k."""
    return "stats_kernel" if 0 < w.top_k < w.V and w.temperature > 0 else "stats_item_kernel"


def launches_per_step(w: W.Workload) -> int:
    """Kernels of one step: the streaming pass and the per-request pass, plus the ragged row
    table and the nucleus pass (top-p without top-k).  The sampler's q(x) comes from the
    per-request pass."""
    n = 2 + (w.ragged is not None)
    if w.temperature > 0 and w.top_p < 1.0 and not (0 < w.top_k < w.V):
        n += 1
    return n


def _time_oracle(w: W.Workload, d, nthreads: int, seconds: float):
    """Repeated oracle calls on the sample `d` for about `seconds`: (positions/s, calls, seconds)."""
    import oracle
    kpr = d["k_per_row"] if w.ragged else None
    calls = 0
    t0 = time.perf_counter()
    while True:
        oracle.verify(d["p"], None if w.temperature == 0 else d["q"], d["draft"], kpr, d["ua"], d["ur"],
                      w.temperature, w.top_k, nthreads=nthreads, draft_temperature=w.tq, top_p=w.top_p)
        calls += 1
        dt = time.perf_counter() - t0
        if dt >= seconds:
            break
    return int(d["k_per_row"].sum()) * calls / dt, calls, dt


def cpu_baseline(w: W.Workload, budget_requests: int, seconds: float = 10.0, single_requests: int = 16,
                 single_seconds: float = 5.0):
    """The oracle, as it stands, on the host cores over a bounded sample of the workload: the
    first `budget_requests` requests with OpenMP over requests on every core, verified repeatedly
    until about `seconds` have passed; then the first `single_requests` requests on one thread."""
    n = min(budget_requests, w.B)
    d = W.generate(w, requests=range(n))
    cores = os.cpu_count() or 1
    v, calls, dt = _time_oracle(w, d, cores, seconds)
    n1 = min(single_requests, n)
    d1 = {k: (a[:n1] if isinstance(a, np.ndarray) and a.ndim >= 1 and a.shape[0] == n else a) for k, a in d.items()}
    v1, calls1, dt1 = _time_oracle(w, d1, 1, single_seconds)
    return {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"first {n} of the {w.B} requests, {calls} oracle calls, OpenMP over requests "
                      f"({dt:.1f} s)",
            "single_thread": {"value": v1, "unit": UNIT, "cores": 1,
                              "sample": f"first {n1} of the {w.B} requests, {calls1} oracle calls on one "
                                        f"thread ({dt1:.1f} s)"}}, None, dt


# ------------------------------------------------------------------------------------------------
# arms
# ------------------------------------------------------------------------------------------------
def run_reference(args, w: W.Workload):
    """The oracle timed on the host cores: --warmup + --steps oracle calls, each over a sample of
    the workload's requests sized so the whole run stays within about two minutes."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    cores = os.cpu_count() or 1
    q_of = lambda d: None if w.temperature == 0 else d["q"]  # noqa: E731
    kpr_of = lambda d: d["k_per_row"] if w.ragged else None  # noqa: E731
    multi = MULTI_CHAINS.get(w.label)

    def gen(reqs):
        return W.generate_multi(w, multi, requests=reqs) if multi else W.generate(w, requests=reqs)

    def run(d):
        if multi:
            oracle.verify_multi(d["p"], q_of(d), d["draft"], d["ua"], d["ur"], w.temperature,
                                draft_temperature=w.tq, nthreads=cores)
        else:
            oracle.verify(d["p"], q_of(d), d["draft"], kpr_of(d), d["ua"], d["ur"], w.temperature, w.top_k,
                          nthreads=cores, draft_temperature=w.tq, top_p=w.top_p)

    probe = gen(range(min(8, w.B)))
    t0 = time.perf_counter()
    run(probe)
    per_req = (time.perf_counter() - t0) / probe["p"].shape[0]
    budget = args.ref_seconds / max(1, args.steps + args.warmup)
    n = int(max(1, min(args.ref_requests, w.B, budget / max(per_req, 1e-9))))
    d = gen(range(n))

    def one():
        run(d)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    dt = (time.perf_counter() - t0) / args.steps
    pos = n * w.K if multi else int(d["k_per_row"].sum())
    v = pos / dt
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded generator; no dataset)",
            "config": {"workload": describe(w), "sample_requests": n},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"first {n} of the {w.B} requests per step, OpenMP over requests"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


MULTI_CHAINS = {"multi_c5": 4}  # draft chains per request of the multi-draft workloads


def run_gpu_multi(args, w: W.Workload):
    """Multi-draft verify (spec_verify_multi): N chains of K drafts per request; a step is one call
    over the batch.  value = B K / step time (the positions a request can advance by)."""
    import torch
    import speculative_decoding_rejection_verify_gb300 as sv
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sv.load()
    N = MULTI_CHAINS[w.label]
    d = W.generate_multi(w, N, requests=shard_requests(w.B, rank))
    B, K, V = w.B, w.K, w.V

    def up(a):
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 else torch.from_numpy(a)
        return t.to(dev)

    copies = [dict(p=up(d["p"]), q=up(d["q"]), x=up(d["draft"]), ua=up(d["ua"]), ur=up(d["ur"])) for _ in range(2)]
    dt_code = sv.DTYPE_BF16 if w.dtype == "bf16" else sv.DTYPE_F32
    lib = sv.load()
    ws = torch.zeros(lib.spec_verify_multi_workspace_bytes(B, N, K, V, dt_code), dtype=torch.uint8, device=dev)
    i32 = dict(dtype=torch.int32, device=dev)
    out = (torch.empty((B, K + 1), **i32), torch.empty((B,), **i32), torch.empty((B,), **i32), torch.empty((B,), **i32))
    stream = torch.cuda.current_stream(dev)

    def step(i):
        c = copies[i & 1]
        sv.verify_multi(c["p"], c["q"], c["x"], c["ua"], c["ur"], w.temperature, draft_temperature=w.tq,
                        workspace_tensor=ws, stream=stream, out=out)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(min(args.steps, 200))]
    with ClockSampler(str(local)) as clk:
        barrier(world)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(args.steps):
            step(i)
        t1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        for i, (a, z) in enumerate(ev):
            a.record(stream)
            step(i)
            z.record(stream)
        torch.cuda.synchronize()
    step_ms = max_over_ranks(t0.elapsed_time(t1) / args.steps, world, dev)
    per_step = [a.elapsed_time(z) for a, z in ev]
    value = sum_over_ranks(B * K, world, dev) / (step_ms * 1e-3)
    if rank != 0:
        return 0
    nbytes = W.multi_algorithmic_bytes(w, N, B)
    peak, peak_kind = measured_peak()
    achieved = nbytes / (step_ms * 1e-3) / 1e9
    line = {"metric": "verified draft positions/s (multi-draft) and logits GB/s", "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic (seeded generator; no dataset)",
            "config": {"workload": f"{w.label}: B={B} N={N} chains K={K} V={V} {w.dtype} T={w.temperature:g}",
                       "logits_bytes_per_step": nbytes, "launch": "direct launches",
                       "parallelism": f"{world} independent batches (no collective)"},
            "median_step_ms": statistics.median(per_step),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                         "frac_vs_nominal": achieved / NOMINAL_HBM_GBS, "traffic": None,
                         "kernel": "whole step (row table, streaming pass, per-request pass)"},
            "gpu_launches": args.steps * 3, "clocks": clk.summary()}
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args, w: W.Workload):
    import torch
    import speculative_decoding_rejection_verify_gb300 as sv
    rank, world, local = dist_env()
    if w.label in MULTI_CHAINS:
        return run_gpu_multi(args, w)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sv.load()

    reqs = shard_requests(w.B, rank)
    d = W.generate(w, requests=reqs)
    ragged = w.ragged is not None
    greedy = w.temperature == 0
    kb = d["k_per_row"]
    positions = int(kb.sum())
    logits_bytes = W.algorithmic_bytes(w, kb)

    def up(a):
        if a is None:
            return None
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 else torch.from_numpy(a)
        return t.to(dev)

    # two copies of the inputs alternate, so no step finds the previous step's logits in L2
    copies = []
    for _ in range(2):
        copies.append(dict(p=up(d["p"]), q=None if greedy else up(d["q"]), x=up(d["draft"]),
                           k=up(kb) if ragged else None, ua=None if greedy else up(d["ua"]),
                           ur=None if greedy else up(d["ur"])))
    B, K, V = len(reqs), w.K, w.V
    dt_code = sv.DTYPE_BF16 if w.dtype == "bf16" else sv.DTYPE_F32
    ws = torch.zeros(sv.workspace_bytes(B, K, V, dt_code, w.top_k), dtype=torch.uint8, device=dev)
    tok = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    nacc = torch.empty((B,), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    sampling = K == 0  # draft-token sampling: one draw per row through spec_sample
    if sampling:
        for c in copies:
            c["rows"] = c["p"][:, 0, :].contiguous()
        sws = torch.zeros(sv.load().spec_sample_workspace_bytes(B, V, dt_code, w.top_k), dtype=torch.uint8,
                          device=dev)
        sprob = torch.empty((B,), dtype=torch.float32, device=dev)

    def launch(i, st, mid=None):
        c = copies[i & 1]
        if sampling:
            sv.sample(c["rows"], c["ur"], w.temperature, w.top_k, w.top_p, workspace_tensor=sws, stream=st,
                      out=(nacc, sprob))
            return
        sv.verify(c["p"], c["q"], c["x"], c["k"], c["ua"], c["ur"], w.temperature, w.top_k,
                  workspace_tensor=ws, stream=st, out=(tok, nacc), pass1_event=mid,
                  draft_temperature=w.tq, top_p=w.top_p)

    graphs = None
    if args.graph:
        launch(0, stream)  # first call outside capture: sets the kernels' attributes
        torch.cuda.synchronize()
        graphs = []
        for i in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                launch(i, torch.cuda.current_stream(dev))
            graphs.append(g)
        torch.cuda.synchronize()

    def step(i, mid=None):
        if graphs is not None:
            graphs[i & 1].replay()
        else:
            launch(i, stream, mid)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    # per step: start -> (streaming pass) -> mid -> (per-request pass) -> end, all on the launch stream
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(args.steps)]
    for e in ev:  # create the events before the timed region
        for x in e:
            x.record(stream)
    torch.cuda.synchronize()
    gpu_id = "0"
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    with ClockSampler(gpu_id) as clk:
        barrier(world)
        torch.cuda.synchronize()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(args.steps):
            step(i)
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        # per-step times (events around each step, nothing between its kernels)
        nsplit = min(args.steps, 200)
        for i in range(nsplit):
            ev[i][0].record(stream)
            step(i)
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        per_step = [a.elapsed_time(z) for a, _, z in ev[:nsplit]]
        # the pass split, on separate steps: an event between the passes serialises them fully
        for i in range(nsplit):
            ev[i][0].record(stream)
            step(i, None if (graphs or sampling) else ev[i][1])
            ev[i][2].record(stream)
        torch.cuda.synchronize()
    total_ms = t_start.elapsed_time(t_end)
    ev = ev[:nsplit]
    if graphs is None and not sampling:
        pass1_ms = statistics.mean(a.elapsed_time(m) for a, m, _ in ev)
        pass2_ms = statistics.mean(m.elapsed_time(z) for _, m, z in ev)
    else:  # no event between the passes inside a graph: the whole step stands for the pass
        pass1_ms = statistics.mean(a.elapsed_time(z) for a, _, z in ev)
        pass2_ms = None
    step_ms = max_over_ranks(total_ms / args.steps, world, dev)
    all_positions = sum_over_ranks(B if sampling else positions, world, dev)
    value = all_positions / (step_ms * 1e-3)

    # end to end: host buffers through spec_verify_host (H2D + verify + D2H, synchronous)
    e2e = None
    if args.e2e_steps > 0 and not sampling:
        pin = lambda a: None if a is None else torch.from_numpy(a).pin_memory().numpy()  # noqa: E731
        hp = dict(p=pin(d["p"]), q=None if greedy else pin(d["q"]), x=pin(d["draft"]), k=pin(kb) if ragged else None,
                  ua=None if greedy else pin(d["ua"]), ur=None if greedy else pin(d["ur"]))
        htok = torch.empty((B, K + 1), dtype=torch.int32).pin_memory().numpy()
        hn = torch.empty((B,), dtype=torch.int32).pin_memory().numpy()

        def hstep():
            sv.verify_host(hp["p"], hp["q"], hp["x"], hp["k"], hp["ua"], hp["ur"], w.temperature, w.top_k,
                           device=dev, stream=stream, out=(htok, hn), draft_temperature=w.tq, top_p=w.top_p)

        for _ in range(2):
            hstep()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            hstep()
        e2e_s = max_over_ranks((time.perf_counter() - t0) / args.e2e_steps, world, dev)
        h2d = sum(a.nbytes for a in hp.values() if a is not None)
        e2e = {"value": all_positions / e2e_s, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(htok.nbytes + hn.nbytes), "ms_per_step": e2e_s * 1e3,
               "steps": args.e2e_steps}

    if rank != 0:
        return 0
    peak, peak_kind = measured_peak()
    achieved = logits_bytes / (pass1_ms * 1e-3) / 1e9  # the streaming pass reads every logit once
    in_bytes = sum(t.numel() * t.element_size() for t in copies[0].values() if t is not None)
    l2_bytes = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129 << 20
    if 2 * in_bytes > l2_bytes:
        l2_note = f"inputs larger than L2 ({l2_bytes / 1e6:.0f} MB); two input copies alternate between steps"
    else:
        l2_note = f"hot L2: both input copies ({2 * in_bytes / 1e6:.2f} MB) fit in L2 ({l2_bytes / 1e6:.0f} MB)"
    line = {
        "metric": "sampled tokens/s and logits GB/s" if sampling else METRIC, "value": value,
        "unit": "tokens/s" if sampling else UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded generator; no dataset)",
        "config": {"workload": describe(w), "B_per_gpu": B, "K": K, "V": V, "temperature": w.temperature,
                   "draft_temperature": w.tq, "top_k": w.top_k, "top_p": w.top_p,
                   "logits_bytes_per_step": logits_bytes,
                   "l2": l2_note, "launch": "CUDA graph replay" if graphs else "direct launches",
                   "parallelism": f"{world} independent batches (no collective)"},
        "logits_gbs": logits_bytes / (step_ms * 1e-3) / 1e9,
        "median_step_ms": statistics.median(per_step), "step_ms_p10_p90": [float(np.percentile(per_step, 10)),
                                                                        float(np.percentile(per_step, 90))],
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "frac_vs_nominal": achieved / NOMINAL_HBM_GBS,
                     "step_frac_vs_nominal": logits_bytes / (step_ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS,
                     "traffic": traffic_for(w.label),
                     "kernel": (stream_kernel(w) + " (streaming pass)" if graphs is None and not sampling else
                                "whole step" + (" (graph replay)" if graphs else "")),
                     "per_launch_ms": pass1_ms,
                     "step_frac": logits_bytes / (step_ms * 1e-3) / 1e9 / peak,
                     "pass2_ms": pass2_ms},
        "gpu_launches": args.steps * launches_per_step(w),
        "clocks": clk.summary(),
    }
    if e2e is not None:
        line["e2e"] = e2e
    if not args.no_cpu_baseline:
        cb, _, _ = cpu_baseline(w, args.cpu_requests, args.cpu_seconds)
        line["cpu_baseline"] = cb
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="c5_a0.8", choices=sorted(W.WORKLOADS))
    ap.add_argument("--batch", type=int, default=0, help="override B (profiling a smaller case)")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--graph", action="store_true", help="replay each step from a captured CUDA graph")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-requests", type=int, default=1024)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle baseline: time budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-requests", type=int, default=64, help="reference arm: max requests per step")
    ap.add_argument("--ref-seconds", type=float, default=120.0, help="reference arm: time budget")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = W.get(args.workload)
    if args.batch:
        w = w.with_(B=args.batch)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_gpu(args, w)


if __name__ == "__main__":
    sys.exit(main())
