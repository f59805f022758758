"""bench.py's reference arm on the host (no GPU needed): the oracle timed on
the tiny workload prints exactly one JSON line with the benchmark's keys, and
a rank other than 0 of a multi-rank launch prints nothing and exits 0."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CMD = [sys.executable, "bench.py", "--impl", "reference", "--config", "1", "--steps", "3", "--warmup", "3"]


def _run(env_extra):
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "LOCAL_RANK", "WORLD_SIZE")}
    env.update(env_extra)
    return subprocess.run(CMD, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_one_line_with_the_benchmark_keys():
    r = _run({})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.lstrip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["metric"] == "sparse-decode tokens/s" and d["unit"] == "tokens/s"
    assert d["value"] > 0 and d["steps"] == 3 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny-bf16-L1024"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert isinstance(cb["cpu_model"], str) and cb["cpu_model"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_print_nothing():
    r = _run({"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [ln for ln in r.stdout.splitlines() if ln.lstrip().startswith("{")]


def test_oracle_timed_on_one_core_then_restored():
    sys.path.insert(0, ROOT)
    import bench
    import oracle as O
    from block_sparse_paged_score_gb300 import workloads as W
    before = O.num_threads()
    rate, cores, desc = bench.cpu_oracle_rate(W.workload(1), seconds=0.05, threads=1)
    assert rate > 0 and cores == 1 and desc
    assert O.num_threads() == before
