"""The host side of bench.py, on the CPU: the traffic table goes stale when
a kernel's sources change, the L2 rule and workload description, and the
reference arm's JSON line (the float64 oracle timed on a small sample)."""

import json
import os
import subprocess
import sys

import pytest

import bench
from linear_cross_entropy_lce_gb300.workloads import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_traffic_entries_name_known_kernels_and_workloads():
    for (workload, kernel), (nbytes, commit, src) in bench.MEASURED_TRAFFIC.items():
        assert workload in WORKLOADS
        assert kernel in bench.KERNEL_SOURCES
        assert nbytes > 0 and len(commit) >= 7 and len(src) == 16


def test_traffic_is_reported_only_while_the_sources_hash_the_same(monkeypatch):
    (workload, kernel), (nbytes, commit, src) = next(iter(bench.MEASURED_TRAFFIC.items()))
    monkeypatch.setattr(bench, "kernel_sources_hash", lambda k: src)
    got, note = bench.measured_traffic(workload, kernel)
    assert got == nbytes and commit in note
    monkeypatch.setattr(bench, "kernel_sources_hash", lambda k: "0" * 16)
    got, note = bench.measured_traffic(workload, kernel)
    assert got is None and note.startswith("stale")
    # a variant of a workload (another dtype, class weights, the autograd
    # API) has no capture of its own
    got, note = bench.measured_traffic(workload + "+f16", kernel)
    assert got is None and "no ncu capture" in note


def test_source_hash_covers_the_kernel_files(tmp_path, monkeypatch):
    files = bench.KERNEL_SOURCES["gemm_logits_tc"]
    for fn in files:
        (tmp_path / fn).write_text("a")
    monkeypatch.setattr(bench, "CSRC", str(tmp_path))
    h0 = bench.kernel_sources_hash("gemm_logits_tc")
    (tmp_path / files[0]).write_text("b")
    assert bench.kernel_sources_hash("gemm_logits_tc") != h0


@pytest.mark.parametrize("name,flushed", [("tiny_fp32", True), ("fp32_mid", True), ("bf16_llm_head", False),
                                          ("bf16_large_head", False), ("ce_logits_fp32", False)])
def test_l2_rule_and_config(name, flushed):
    w = WORKLOADS[name]
    assert bench.flushes_l2(w) == flushed
    cfg = bench._config(w, 1)
    assert cfg["workload"] == name and cfg["N"] == w.N and cfg["C"] == w.C
    assert cfg["l2"].startswith("L2 flushed") == flushed
    assert cfg["parallelism"] == "single" and bench._config(w, 4)["parallelism"] == "replicas"


def test_reference_arm_prints_one_json_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_fp32",
                          "--steps", "2", "--warmup", "1", "--ref-rows", "16"],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["dtype"] == "f64" and d["value"] > 0
    assert d["config"]["workload"] == "tiny_fp32"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_committed_traffic_was_captured_from_the_committed_kernels():
    """Every entry's source hash is the current one: the table in the tree
    describes the kernels in the tree (a change to a kernel's sources needs
    a new capture, or the entry removed)."""
    stale = [(w, k) for (w, k), (_, _, src) in bench.MEASURED_TRAFFIC.items() if src != bench.kernel_sources_hash(k)]
    assert not stale, stale
