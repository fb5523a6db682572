"""Host-side pieces of bench.py that need no GPU: the algorithmic work and byte counts
behind the roofline, the DRAM-traffic table lookup (valid only while the kernel sources
it was captured from are unchanged), and the pipe peaks."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_layer1_work_and_bytes():
    s = bench.LAYERS["layer1"]
    # 2 * B * P * OC * IC * K * K with P = 3 * 4
    assert bench.flops(B=1024, **s) == 2 * 1024 * 12 * 128 * 59 * 25
    x, w, y = 1024 * 59 * 11 * 15, 128 * 59 * 25, 1024 * 128 * 12
    assert bench.alg_bytes("fwd", B=1024, esize=4, **s) == (x + w + y) * 4
    # with the mask the backward reads y as well
    assert bench.alg_bytes("dgrad", B=1024, esize=4, **s) == (y + w + x + y) * 4
    assert bench.alg_bytes("wgrad", B=1024, esize=2, **s) == (x + y + w + y) * 2


def test_traffic_lookup_follows_the_source_hash(tmp_path, monkeypatch):
    csrc = tmp_path / "implicit_gemm_conv2d_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "a.cu").write_text("kernel a\n")
    (csrc / "b.cuh").write_text("header b\n")
    sha = bench.source_sha([str(csrc / "a.cu"), str(csrc / "b.cuh")])
    (tmp_path / "profiles" / "dram_traffic.txt").write_text(
        "# comment\n"
        f"fwd:layer1:f32:B1024 1234 5.0 a.cu+b.cuh:{sha}\n"
        "dgrad:layer1:f32:B1024 99 5.0 a.cu+b.cuh:0000000000000000\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.read_traffic("fwd:layer1:f32:B1024") == 1234.0
    assert bench.read_traffic("dgrad:layer1:f32:B1024") is None      # stale hash
    assert bench.read_traffic("wgrad:layer1:f32:B1024") is None      # no entry
    (csrc / "b.cuh").write_text("header b, edited\n")                # a source changed
    assert bench.read_traffic("fwd:layer1:f32:B1024") is None


def test_committed_traffic_table_names_existing_sources():
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    keys = 0
    for line in open(path):
        line = line.split("#", 1)[0].split()
        if not line:
            continue
        assert len(line) == 4
        names, sha = line[3].split(":")
        assert len(sha) == 16
        for n in names.split("+"):
            assert os.path.exists(os.path.join(ROOT, "implicit_gemm_conv2d_gb300", "csrc", n)), n
        keys += 1
    assert keys == 6


def test_pipe_peaks():
    peaks = {"hbm_gbs": 6777.0, "bf16_tflops": 1920.6}
    pk, _ = bench.pipe_peak("tc", "bf16", 152, 2070.0, peaks)
    assert pk == pytest.approx(1920.6)
    pk, _ = bench.pipe_peak("tc", "f32", 152, 2070.0, peaks)
    assert pk == pytest.approx(1920.6 * 1.1 / 2.25 / 3)
    pk, _ = bench.pipe_peak("ffma", "f32", 152, 2070.0, peaks)
    assert pk == pytest.approx(152 * 128 * 2 * 2070e6 / 1e12)


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` times the oracle on the host cores and prints one JSON
    line with the contract's keys (no GPU needed)."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"]
