"""Host-side pieces of bench.py that need no GPU: the algorithmic work and byte counts
behind the roofline, the DRAM-traffic table lookup (valid only while the kernel sources
it was captured from are unchanged), and the pipe peaks."""
import os
import types
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
    keys = set()
    for line in open(path):
        line = line.split("#", 1)[0].split()
        if not line:
            continue
        assert len(line) == 4
        names, sha = line[3].split(":")
        assert len(sha) == 16
        for n in names.split("+"):
            assert os.path.exists(os.path.join(ROOT, "implicit_gemm_conv2d_gb300", "csrc", n)), n
        keys.add(line[0])
    # the fused step's two operations for both encoder layers and both dtypes at the bench batch
    for layer in ("layer1", "layer2"):
        for dt in ("f32", "bf16"):
            for op in ("fwd", "bwd"):
                assert f"{op}:{layer}:{dt}:B1024" in keys


def _ncu_csv(path, launches):
    """An ncu --csv log of the three metrics for [(kernel name, us, read bytes, write bytes)]."""
    rows = ['==PROF== Connected to process 1',
            '"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size",'
            '"Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"']
    for i, (name, us, rd, wr) in enumerate(launches):
        for metric, unit, v in (("dram__bytes_read.sum", "byte", rd), ("dram__bytes_write.sum", "Kbyte", wr / 1e3),
                                ("gpu__time_duration.sum", "us", us)):
            rows.append(f'"{i}","1","python3","h","{name}","1","7","(256, 1, 1)","(1, 1, 1)","0","10.3",'
                        f'"Command line profiler metrics","{metric}","{unit}","{v:,}"')
    path.write_text("\n".join(rows) + "\n")


def test_write_traffic_groups_calls_between_flushes(tmp_path, monkeypatch):
    # two operations, warmup 1 + steps 2 each: flush-separated calls; warm-up calls dropped
    flush = ("igc::<unnamed>::l2_flush_kernel(float4 *, unsigned long, float)", 70.0, 0, 5e8)
    pack = "void igc::<unnamed>::pack_fwd_w_kernel<float>(ConvParams, const T1 *, unsigned char *, int, int)"
    fwd = "void igc::<unnamed>::fwd_tc_kernel<float, 1>(ConvParams, const T1 *)"
    bwd = "void igc::<unnamed>::bwd_tc_kernel<float, 1>(ConvParams, const T1 *)"
    seq = [("void at::vectorized_elementwise_kernel<4, at::copy>(int)", 3.0, 1e6, 0)]
    for rd in (9e6, 1e6, 3e6):                  # fwd: warm-up, then 1 and 3 MB in its main kernel
        seq += [flush, (pack, 4.0, 1e5, 0), (fwd, 40.0, rd, 2e3)]
    for rd in (9e6, 5e6, 7e6):                  # bwd
        seq += [flush, (pack, 4.0, 0, 0), (bwd, 90.0, rd, 0)]
    csv = tmp_path / "t.csv"
    _ncu_csv(csv, seq)
    (tmp_path / "profiles").mkdir()
    csrc = tmp_path / "implicit_gemm_conv2d_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for n in bench.TRAFFIC_SOURCES:
        (csrc / n).write_text(n)
    (tmp_path / "profiles" / "dram_traffic.txt").write_text("# header\nfwd:layer1:f32:B1024 1 1.0 a.cu:0000000000000000\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    args = types.SimpleNamespace(write_traffic=str(csv), profile_ops="fwd,bwd", warmup=1, steps=2, layer="layer1",
                                 dtype="f32", batch=1024)
    assert bench.write_traffic(args) == 0
    assert bench.read_traffic("fwd:layer1:f32:B1024") == pytest.approx(1e5 + 2e6 + 2e3, abs=1)
    assert bench.read_traffic("bwd:layer1:f32:B1024") == pytest.approx(6e6, abs=1)
    lines = [l for l in (tmp_path / "profiles" / "dram_traffic.txt").read_text().splitlines() if l.startswith("fwd:")]
    assert len(lines) == 1  # the stale line was replaced
    # a capture with the wrong number of calls is refused
    args.steps = 3
    with pytest.raises(SystemExit):
        bench.write_traffic(args)


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
    # the same config object our arm reports for the default workload
    args = types.SimpleNamespace(layer="layer1", dtype="f32", batch=1024, step="fused", no_graphs=False, algo="auto")
    assert d["config"] == bench.arm_config(args)
    assert "B=1024" in d["config"]["workload"] and "8 of the workload's 1024 samples" in d["sample"]
