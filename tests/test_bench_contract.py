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


def test_algorithmic_byte_accounting():
    """42 B/param for the three passes (2 + 22 + 18), 30 for tensors finished
    in one pass (2 + 28 + 0); speculative mode 40 for a step that stands and
    22 + 40 (28 for one-pass tensors) for one that is clipped and redone."""
    n, p = 1_000_000, 12_345
    assert sum(bench.kernel_bytes(n, 0).values()) == 42 * n
    assert sum(bench.kernel_bytes(n, n).values()) == 30 * n
    kb = bench.kernel_bytes(n, p)
    assert kb == {"grad_norm": 2 * n, "moments": 22 * (n - p) + 28 * p, "apply": 18 * (n - p)}
    assert sum(bench.spec_kernel_bytes(n, p, False).values()) == 40 * n
    assert bench.spec_kernel_bytes(n, p, True) == {"spec_step": 22 * n,
                                                   "redo": 40 * (n - p) + 28 * p}
    assert bench.FLOOR_BYTES_PER_PARAM == 28


def test_recorded_traffic_applies_only_to_the_source_it_was_taken_on(tmp_path, monkeypatch):
    """The committed DRAM-byte record scales with the params while the kernel
    code is unchanged (comments and blank lines do not count), and is dropped
    as soon as the code changes."""
    rec = json.load(open(bench.TRAFFIC_FILE))
    per = rec["dram_bytes_per_param"]["moments"]
    src = open(bench.KERNEL_SOURCE).read()
    assert bench.kernel_source_hash() == rec["kernel_source_sha256"]
    assert bench.traffic_per_launch("moments", 1000) == pytest.approx(per * 1000)
    commented = tmp_path / "commented.cu"
    commented.write_text("// a new comment\n\n" + src.replace("\n", "  // note\n", 3))
    monkeypatch.setattr(bench, "KERNEL_SOURCE", str(commented))
    assert bench.traffic_per_launch("moments", 1000) == pytest.approx(per * 1000)
    changed = tmp_path / "changed.cu"
    changed.write_text(src + "\nint one_more_line;\n")
    monkeypatch.setattr(bench, "KERNEL_SOURCE", str(changed))
    assert bench.traffic_per_launch("moments", 1000) is None
