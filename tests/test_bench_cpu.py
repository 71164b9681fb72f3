"""bench.py's reference arm (the float64 oracle on host cores) needs no GPU: it
prints one JSON line with the contract's keys, and under torchrun with two ranks
rank 0 alone prints it while the other rank exits 0 without work."""

import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
        "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"}


def _lines(out):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def _check(line, n_gpus):
    assert KEYS <= set(line), KEYS - set(line)
    assert line["impl"] == "reference" and line["n_gpus"] == n_gpus
    assert line["unit"] == "tokens/s" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["steps"] == 2 and line["warmup"] == 3
    assert line["config"]["workload"] == "llama3_8b_packed_outliers"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == line["value"] and cb["sample"]
    assert cb["rows"] == 512 and cb["passes"] == 2 and cb["cpu_model"] and cb["host_logical_cores"] >= 1
    assert cb["tokens_per_s_label"] == "extrapolated" and "extrapolated" in cb["sample"]
    assert set(cb["per_operator"]) == {"positions", "rmsnorm_fwd", "rope_fwd", "swiglu_fwd", "swiglu_bwd",
                                       "rope_bwd", "rmsnorm_bwd"}
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_one_process():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3",
                        "--oracle-rows", "512"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = _lines(r.stdout)
    assert len(lines) == 1
    _check(lines[0], 1)


def test_reference_arm_under_torchrun_prints_once():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3",
           "--oracle-rows", "512"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _lines(r.stdout)
    assert len(lines) == 1, r.stdout
    _check(lines[0], 2)


def test_gpu_arm_refuses_to_run_without_a_gpu():
    # The measured path has no CPU fallback: on a machine without a CUDA device the
    # bench's own arm exits non-zero instead of timing something else.
    import pytest
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    r = subprocess.run([sys.executable, "bench.py", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0
    assert "no CUDA device" in r.stderr and not _lines(r.stdout)
