"""bench.py's reference arm (the fp64 oracle timed on the host cores) and its argument checks,
run here without a GPU: the JSON line keeps the contract the GPU arm's line keeps."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=e,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_contract_line():
    r = _bench("--impl", "reference", "--steps", "1", "--warmup", "3", "--workload", "c2")
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "positions/s"
    assert d["higher_is_better"] is True and d["vs_baseline"] is None and d["steps"] == 1
    assert d["config"]["workload"].startswith("c2:")
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_do_no_work():
    r = _bench("--impl", "reference", "--steps", "1", "--warmup", "3", "--workload", "c2",
               env=dict(RANK="1", LOCAL_RANK="1", WORLD_SIZE="2"))
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_fewer_than_three_warmup_steps_refused():
    r = _bench("--impl", "reference", "--steps", "1", "--warmup", "2")
    assert r.returncode != 0 and "warmup" in r.stderr


def test_cpu_baseline_reports_all_cores_and_one_thread():
    """The GPU arm's cpu_baseline: the oracle with OpenMP over requests on every core, and on one
    thread over a smaller sample, each a positions/s figure with its sample stated."""
    import bench
    import workloads as W
    cb, _, _ = bench.cpu_baseline(W.get("c2", V=2000), 4, seconds=0.2, single_requests=2, single_seconds=0.2)
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["unit"] == "positions/s"
    st = cb["single_thread"]
    assert st["cores"] == 1 and st["value"] > 0 and "first 2 of the 8 requests" in st["sample"]
