"""bench.py without a GPU: its helpers and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.argv = ["bench.py"]
import bench  # noqa: E402


def test_kernel_names_and_bytes():
    assert bench.kernel_of(synth.WORKLOADS[2], "encode") == "encode_k2_tc"
    assert bench.kernel_of(synth.WORKLOADS[3], "encode") == "encode_k4_grid"
    assert bench.kernel_of(synth.WORKLOADS[4], "encode") == "encode_kq_tc"
    assert bench.kernel_of(synth.WORKLOADS[5], "encode") == "encode_full_tc"
    assert bench.kernel_of(synth.WORKLOADS[4], "decode") == "decode_ws"
    assert bench.kernel_of(synth.WORKLOADS[2], "decode") == "decode_tc"
    enc, gat = bench.workload_bytes(synth.WORKLOADS[2], 256)
    assert enc == 2 * 64 + 4 + 32 and gat == 8 + 4 + 32 + 128


def test_committed_traffic_requires_matching_sources(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (tmp_path / "random_access_kv_gb300").symlink_to(os.path.join(ROOT, "random_access_kv_gb300"))
    h = bench.source_hash("decode_tc")
    (prof / "decode_tc_w2.md").write_text(
        f"# x\n\n- source_hash: `{h}`\n- rows_per_launch: 1000\n- dram_bytes_per_launch: 5000\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.committed_traffic("decode_tc", 2, 4000) == pytest.approx(20000.0)
    (prof / "decode_tc_w2.md").write_text("- source_hash: `stale`\n- rows_per_launch: 1\n- dram_bytes_per_launch: 5\n")
    assert bench.committed_traffic("decode_tc", 2, 4000) is None
    assert bench.committed_traffic("encode_k2_tc", 2, 1) is None


def test_committed_traffic_of_a_named_archive_workload(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (tmp_path / "random_access_kv_gb300").symlink_to(os.path.join(ROOT, "random_access_kv_gb300"))
    h = bench.source_hash("archive_access")
    (prof / "archive_access_kv-streams.md").write_text(
        f"- source_hash: `{h}`\n- rows_per_launch: 1048576\n- dram_bytes_per_launch: 19202560\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.committed_traffic("archive_access", "kv-streams", 1 << 19) == pytest.approx(9601280.0)
    assert bench.committed_traffic("archive_access", "document", 1 << 20) is None


def test_archive_params_are_the_librarys_bound():
    from oracle import fractal as ofa
    from random_access_kv_gb300 import build as fbuild
    fbuild.build()
    r, L = bench.archive_params(256)
    assert r == pytest.approx(0.75 * ofa.ratio_limit(256), rel=1e-15) and L == ofa.max_segment(256, r) == 7


def test_reference_arm_prints_one_contract_line():
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "1",
                        "--steps", "1", "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert p.returncode == 0, p.stderr
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_archive_reference_arm_prints_one_contract_line():
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--archive",
                        "--steps", "1", "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert p.returncode == 0, p.stderr
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "symbols/s" and d["value"] > 0
    assert d["cpu_baseline"]["cores"] == 1 and "document" in d["config"]["workload"]
