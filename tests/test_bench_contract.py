"""bench.py's command-line contract on a machine without a GPU.

The reference arm times the CPU oracle on the host cores (here on a cut of
the workload, every tensor at most 65,536 elements, so that it is quick): one JSON line with the keys the contract fixes, and under a
two-rank launch only rank 0 prints.  The CUDA arm must refuse to run without
a device rather than fall back to anything.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout=300, env=None):
    return subprocess.run([sys.executable] + args, cwd=ROOT, capture_output=True, text=True,
                          timeout=timeout, env=env)


def _json_lines(out):
    return [json.loads(line) for line in out.splitlines() if line.startswith("{")]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _check_reference_line(d, n_gpus, steps, warmup):
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["n_gpus"] == n_gpus and d["steps"] == steps and d["warmup"] == warmup
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["vs_baseline"] is None and d["data"] == "synthetic"
    assert "workload" in d["config"] and d["config"]["n_params"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == d["value"] and cb["unit"] == d["unit"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_prints_one_contract_line():
    r = _run(["bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3",
              "--max-elems", "65536"])
    assert r.returncode == 0, r.stderr
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_reference_line(lines[0], 1, 2, 3)


def test_reference_arm_under_two_ranks_prints_once():
    port = _free_port()
    env = dict(os.environ, MASTER_ADDR="127.0.0.1")
    r = _run(["-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
              "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
              "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
              "--max-elems", "65536"], env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_reference_line(lines[0], 2, 1, 3)


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="needs a machine without a GPU")
def test_cuda_arm_refuses_to_run_without_a_device():
    r = _run(["bench.py", "--steps", "3", "--warmup", "3"], timeout=120)
    assert r.returncode != 0
    assert "CUDA device" in (r.stderr + r.stdout)
    assert not _json_lines(r.stdout)
