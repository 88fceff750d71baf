"""The JSON line of bench.py's reference arm (the CPU oracle timed on the host cores), on one
token of the decode workload: the keys the line carries, a cpu_baseline and an e2e that
describe this same run, and a config equal to the GPU arm's on every key both describe.
Under torch.distributed.run with two ranks, rank 0 alone prints it."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARGS = ["--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-tokens", "1", "--cpu-budget", "2"]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _json_lines(stdout: str):
    return [json.loads(l) for l in stdout.splitlines() if l.startswith("{")]


def _check_line(o: dict, n_gpus: int):
    import bench

    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in o, key
    assert o["impl"] == "reference"
    assert o["metric"] == bench.METRIC and o["unit"] == "tok/s" and o["higher_is_better"] is True
    assert o["n_gpus"] == n_gpus and o["steps"] == 1 and o["warmup"] >= 3
    assert o["value"] > 0 and o["ms_per_step"] > 0
    assert o["dtype"] == "f64" and o["vs_baseline"] is None
    cb = o["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == o["value"] and cb["unit"] == o["unit"]
    assert cb["cores"] >= 1 and "1 tokens" in cb["sample"]
    e = o["e2e"]
    assert e["value"] == o["value"] and e["unit"] == o["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
    # the GPU arm describes the same workload; it adds only what has no meaning for the oracle
    ours = bench._config_desc(bench._workload(), None, 512)
    shared = set(ours) & set(o["config"])
    assert {"workload", "n_layers", "hidden", "n_experts", "top_k", "cache_slots", "bp_bh_gbps"} <= shared
    for key in shared - {"parallelism"}:
        assert o["config"][key] == ours[key], key
    assert set(ours) - set(o["config"]) <= {"cache_warm_prefix_tokens"}


def test_reference_arm_line_single_process():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *ARGS], capture_output=True, text=True,
                       cwd=ROOT, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_line(lines[0], 1)


def test_reference_arm_two_ranks_rank0_prints_once():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"), "--gpus", "2", *ARGS]
    r = subprocess.run(cmd, capture_output=True, text=True, cwd=ROOT, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_line(lines[0], 2)
