"""The benchmark's command-line contract, checked on the CPU.

- The reference arm (the CPU oracle timed on the host) prints exactly one
  JSON line with impl "reference" and the native arm's metric, unit and
  workload. Its e2e object moves no host-device bytes, and its cpu_baseline
  says what was timed.
- Under a two-rank launch, rank 0 alone prints it.
- Without a GPU the native arm stops with an error: there is no CPU fallback.
"""
import json
import os
import socket
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
REF_ARGS = ["--impl", "reference", "--steps", "1", "--warmup", "0", "--cpu-budget", "1"]


def _run(cmd, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=e)


def _json_lines(stdout):
    return [json.loads(l) for l in stdout.splitlines() if l.strip().startswith("{")]


def _check_reference_line(d, n_gpus):
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["higher_is_better"] is True and d["value"] > 0
    assert d["n_gpus"] == n_gpus and d["steps"] == 1 and d["warmup"] == 0
    assert d["config"]["workload"] == "quest_8k"
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]


def test_reference_arm_prints_one_contract_line():
    r = _run([sys.executable, "bench.py", *REF_ARGS])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_reference_line(lines[0], 1)


def test_reference_arm_two_ranks_prints_once():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = _run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
              "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--gpus", "2", *REF_ARGS],
             env={"OMP_NUM_THREADS": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_reference_line(lines[0], 2)


def test_native_arm_without_gpu_fails_loudly():
    r = _run([sys.executable, "bench.py", "--steps", "1", "--warmup", "3"], env={"CUDA_VISIBLE_DEVICES": ""})
    assert r.returncode != 0
    assert "needs a CUDA GPU" in r.stderr
    assert _json_lines(r.stdout) == []


def test_recorded_traffic_holds_only_for_the_captured_sources(tmp_path, monkeypatch):
    """The DRAM traffic bench.py reports comes from the record only while the
    hash of every source file of the kernel matches the capture's."""
    rec = json.load(open(os.path.join(bench.HERE, "profiles", "dram_traffic.json")))
    ent = rec["pa_decode"]["quest_8k"]
    assert ent["source"] == "decode.cu+common.cuh+kernels.h"
    # the committed record was taken on the committed sources
    assert bench.recorded_traffic("pa_decode", "quest_8k") == ent["dram_bytes_per_launch"]
    assert ent["dram_bytes_per_launch"] == ent["dram_bytes_read"] + ent["dram_bytes_write"]
    # a copy of the tree with one source byte changed: no traffic
    csrc = tmp_path / "paged_gqa_decode_reshape_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(rec))
    for name in ent["source"].split("+"):
        src = os.path.join(bench.HERE, "paged_gqa_decode_reshape_gb300", "csrc", name)
        (csrc / name).write_bytes(open(src, "rb").read())
    monkeypatch.setattr(bench, "HERE", str(tmp_path))
    assert bench.recorded_traffic("pa_decode", "quest_8k") == ent["dram_bytes_per_launch"]
    with open(csrc / "common.cuh", "ab") as f:
        f.write(b"\n")
    assert bench.recorded_traffic("pa_decode", "quest_8k") is None
    assert bench.recorded_traffic("pa_decode", "no_such_workload") is None
