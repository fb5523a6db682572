#!/usr/bin/env python3
"""Benchmark of the implicit-GEMM conv2d layer on one or more GPUs.

A step is one pass of the whole hot path -- forward (+ fused ReLU), d_input and
wgrad (split-K partials + reduction) -- over one batch of seeded synthetic input
of layer 1 of PufferLib PR #522's encoder in fp32: B=1024, IC=59, OC=128, 11x15
input, K=5, S=3 -> 3x4, ReLU.  The value is whole-job GFLOP/s (algorithmic
FLOPs 2*B*P*OC*IC*K*K per operation) with inputs resident in HBM; L2 is flushed
(a 512 MiB write) between timed steps, outside the timed region.  The JSON line
also carries per-operation us/iter for both layers in both dtypes, the roofline
of the dominant kernel, the fp64 oracle's CPU throughput on a bounded sample,
an end-to-end number through host buffers, and SM clocks sampled during the
timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU (torchrun): every rank runs the same per-GPU workload (weak scaling,
independent replicas; the layer needs no exchange for this measurement) and the
slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs/iter and GFLOP/s for conv fwd/dgrad/wgrad at B=1024; % of roofline"
LAYERS = {
    "layer1": dict(IC=59, OC=128, H=11, W=15, K=5, S=3, relu=1),
    "layer2": dict(IC=128, OC=128, H=3, W=4, K=3, S=1, relu=0),
}
# PufferLib PR #522 bench output at B=1024 on a GPU the page does not name:
# (forward us/iter, backward = wgrad + d_input us/iter) of its gemm_fast kernels.
PR522_US = {("layer1", "f32"): (192.4102, 541.7361), ("layer2", "f32"): (56.8698, 100.2875),
            ("layer1", "bf16"): (106.4277, 403.5356), ("layer2", "bf16"): (18.4427, 49.1440)}
# The same PR's "n3_conv_bias_grad" blocks: bias-gradient us/iter of its fast kernel at
# B=32768, OC=128 (conv1: 12 positions, 50.3 M gradient elements; conv2: 2 positions).
PR522_BIAS_GRAD_US = {"layer1": 136.5968, "layer2": 40.9008}
BIAS_GRAD_BATCH = 32768
FLUSH_BYTES = 512 << 20
OPS = ("fwd", "dgrad", "wgrad")
STEP_OPS = ("fwd", "bwd")  # the timed step: the forward, then the whole backward in one call


def flops(B, IC, OC, H, W, K, S, **_):
    OH, OW = (H - K) // S + 1, (W - K) // S + 1
    return 2.0 * B * OH * OW * OC * IC * K * K


def alg_bytes(op, B, IC, OC, H, W, K, S, relu, esize):
    """Algorithmic HBM bytes of one operation: each tensor read or written once ("bwd": d_input and
    wgrad in one call read x, dy, w and y once and write dx and dw)."""
    OH, OW = (H - K) // S + 1, (W - K) // S + 1
    nx, ny, nw = B * IC * H * W, B * OC * OH * OW, OC * IC * K * K
    if op == "fwd":
        n = nx + nw + ny
    elif op == "dgrad":
        n = ny + nw + nx + (ny if relu else 0)
    elif op == "bwd":
        n = nx + ny + nw + nx + nw + (ny if relu else 0)
    else:
        n = nx + ny + nw + (ny if relu else 0)
    return n * esize


def op_flops(op, flops_per_op):
    """The fused backward does d_input's and wgrad's FLOPs."""
    return 2 * flops_per_op if op == "bwd" else flops_per_op


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--batch", type=int, default=1024)
    ap.add_argument("--layer", choices=tuple(LAYERS), default="layer1",
                    help="workload of the timed step (default: layer 1, the headline)")
    ap.add_argument("--dtype", choices=("f32", "bf16"), default="f32")
    ap.add_argument("--algo", choices=("auto", "direct", "ffma", "tc"), default="auto",
                    help="force one kernel family for all three operations")
    ap.add_argument("--no-graphs", action="store_true",
                    help="launch each operation eagerly instead of replaying a captured CUDA graph")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other-config table, e2e and CPU baseline")
    ap.add_argument("--step", choices=("fused", "split"), default="fused",
                    help="fused: conv_fwd_ws then conv_bwd; split: the three operations one call each")
    ap.add_argument("--chain-only", action="store_true",
                    help="time only the fused two-layer forward chain against the two forward calls")
    ap.add_argument("--profile-ops", default=None, metavar="OPS",
                    help="comma-separated operations (" + ", ".join(PROFILE_OPS) + "): run each --warmup + "
                    "--steps times, eagerly, each call after an L2 flush, and exit -- the launch sequence an ncu "
                    "capture of the whole run reads (see --write-traffic)")
    ap.add_argument("--write-traffic", default=None, metavar="CSV",
                    help="host only: from `ncu --csv --metrics gpu__time_duration.sum,dram__bytes_read.sum,"
                    "dram__bytes_write.sum` of a --profile-ops run (same --profile-ops, --steps, --warmup, --layer, "
                    "--dtype, --batch), write each operation's DRAM bytes per call into profiles/dram_traffic.txt")
    return ap.parse_args()


def combine_ranks(ms_step, world, device):
    """The slowest rank's step time (every rank gets it): replicas finish together only as
    fast as the slowest one."""
    if world == 1:
        return ms_step
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms_step)], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(ms_step_max, world, flops_per_op):
    """Whole-job GFLOP/s: every rank runs the full three-operation step on its own batch."""
    return world * 3 * flops_per_op / (ms_step_max * 1e-3) / 1e9


def workload_config(layer, dtype, batch):
    shp = LAYERS[layer]
    OH, OW = (shp["H"] - shp["K"]) // shp["S"] + 1, (shp["W"] - shp["K"]) // shp["S"] + 1
    return {"workload": (f"{layer} conv {dtype} fwd+dgrad+wgrad"
                         f"{', fused ReLU' if shp['relu'] else ''}, B={batch} IC={shp['IC']} "
                         f"OC={shp['OC']} {shp['H']}x{shp['W']} K={shp['K']} S={shp['S']} -> {OH}x{OW} "
                         "(PufferLib PR #522 encoder conv" + ("1)" if layer == "layer1" else "2)")),
            "inputs": "x~N(0,1), w~U(+-1/sqrt(IC*K*K)), dy~N(0,1), SplitMix64 seed 0x5EED2026"}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ----------------------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 100 ms; only the samples that
    arrive between mark_start() and mark_end() (the timed region) are summarised."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.oneshot = []
        self.t = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            deadline = time.monotonic() + 5.0  # wait until the sampler is live
            while not self.lines and time.monotonic() < deadline and self.proc.poll() is None:
                time.sleep(0.01)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def query_once(self):
        """One nvidia-smi query now (the timed region of a short run can fall between two
        100 ms samples; a query right before and right after it always lands)."""
        try:
            r = subprocess.run(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=10)
            if r.returncode == 0 and r.stdout.strip():
                self.oneshot.append((time.monotonic(), r.stdout.strip().splitlines()[0]))
        except (OSError, subprocess.TimeoutExpired):
            pass

    def mark_start(self):
        self.query_once()
        self.t0 = time.monotonic()

    def mark_end(self):
        self.t1 = time.monotonic()
        self.query_once()

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.t:
                self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        inside = [(ts, ln) for ts, ln in self.lines
                  if not (self.t0 is not None and ts < self.t0) and not (self.t1 is not None and ts > self.t1 + 0.1)]
        n_inside = len(inside)
        for ts, ln in inside + self.oneshot:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        how = ("nvidia-smi: one query right before and one right after the timed region, plus "
               "100 ms samples inside it")
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "samples_inside": 0,
                    "how": how}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "samples_inside": n_inside, "how": how}


# ----------------------------------------------------------------------------------------
# reference arm: the fp64 CPU oracle (the only other implementation of this layer)
# ----------------------------------------------------------------------------------------
def oracle_step(inp, shape):
    import oracle
    y, _ = oracle.conv_fwd(inp["x"], inp["w"], shape["S"], shape["relu"])
    oracle.conv_bwd_data(inp["dy"], inp["w"], y, shape["H"], shape["W"], shape["S"], shape["relu"])
    oracle.conv_bwd_filter(inp["x"], inp["dy"], y, shape["K"], shape["S"], shape["relu"])


def cpu_baseline(shape, b_sample, min_seconds):
    import oracle
    from implicit_gemm_conv2d_gb300 import synth
    oracle.build()
    inp = synth.conv_inputs(b_sample, shape["IC"], shape["OC"], shape["H"], shape["W"], shape["K"],
                            shape["S"], dtype="f32")
    oracle_step(inp, shape)  # warm-up (page-in, thread start)
    n, t0 = 0, time.perf_counter()
    while True:
        oracle_step(inp, shape)
        n += 1
        el = time.perf_counter() - t0
        if el >= min_seconds:
            break
    gflop = 3 * flops(B=b_sample, **shape) * n / 1e9
    return {"value": gflop / el, "unit": "GFLOP/s", "cores": oracle.default_threads(), "kind": "oracle",
            "sample": f"{n} step(s) of fwd+dgrad+wgrad on {b_sample} of the 1024 samples "
                      f"(same shapes and seeded inputs), fp64 direct loops, {el:.1f} s"}


def arm_config(args):
    """The `config` both arms report: the workload of the timed step and how it is run."""
    return dict(workload_config(args.layer, args.dtype, args.batch),
                l2="flushed (512 MiB write) between timed steps, outside the timed region",
                calls=("step: conv_fwd_ws, then conv_bwd (d_input + wgrad in one launch), caller-owned "
                       "workspaces, captured together as one CUDA graph" if args.step == "fused" else
                       "step: conv_fwd_ws, conv_bwd_data_ws, conv_bwd_filter (caller-owned workspaces)"),
                launch=("each operation replayed from a captured CUDA graph" if not args.no_graphs
                        else "eager launches"),
                algo=args.algo)


def run_reference(args):
    """The oracle on the host cores, on our arm's config (the same `config` object), each step a
    bounded sample of its workload: B_SAMPLE of its samples, the same shapes, dtype and seeded
    inputs; the value counts the sample's FLOPs (the `sample` fields say so)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    shape = LAYERS[args.layer]
    b_sample = min(8, args.batch)
    from implicit_gemm_conv2d_gb300 import synth
    import oracle
    oracle.build()
    inp = synth.conv_inputs(b_sample, shape["IC"], shape["OC"], shape["H"], shape["W"], shape["K"],
                            shape["S"], dtype=args.dtype)
    for _ in range(args.warmup):
        oracle_step(inp, shape)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(inp, shape)
    el = time.perf_counter() - t0
    value = 3 * flops(B=b_sample, **shape) * args.steps / 1e9 / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": arm_config(args),
        "sample": (f"each step runs the fp64 oracle on {b_sample} of the workload's {args.batch} samples (same "
                   "shapes, dtype and seeded inputs); the value counts those samples' FLOPs"),
        "cpu_baseline": {"value": value, "unit": "GFLOP/s", "cores": oracle.default_threads(),
                         "kind": "oracle",
                         "sample": f"each step the fp64 oracle on {b_sample} of the {args.batch} samples (the same "
                                   "shapes, dtype and seeded inputs); GFLOP/s counts the sample's FLOPs"},
        "e2e": {"value": value, "unit": "GFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------------------
def source_sha(paths):
    """First 16 hex digits of the SHA-256 of the concatenated files."""
    h = hashlib.sha256()
    for path in paths:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


TRAFFIC_SOURCES = ("kernels_tc.cu", "tc_ptx.cuh", "common.cuh", "kernels_ffma.cu")
PROFILE_OPS = ("fwd", "dgrad", "wgrad", "bwd", "fwd_plain", "dgrad_plain", "bias_grad", "chain")
FLUSH_KERNEL = "l2_flush_kernel"


def ncu_launches(csv_path):
    """[(kernel name, us, DRAM bytes read + written)] in launch order from an ncu --csv log."""
    import csv
    with open(csv_path) as f:
        rows = list(csv.reader(line for line in f if not line.startswith("==")))
    hdr = rows[0]
    col = {k: hdr.index(k) for k in ("ID", "Kernel Name", "Metric Name", "Metric Value", "Metric Unit")}
    scale = {"nsecond": 1e-3, "ns": 1e-3, "usecond": 1.0, "us": 1.0, "msecond": 1e3, "ms": 1e3, "byte": 1.0,
             "Kbyte": 1e3, "KB": 1e3, "Mbyte": 1e6, "MB": 1e6, "Gbyte": 1e9, "GB": 1e9}
    per = {}
    for r in rows[1:]:
        if len(r) <= col["Metric Value"]:
            continue
        lid = int(r[col["ID"]])
        name = r[col["Kernel Name"]].replace("<unnamed>", "").replace("(anonymous namespace)", "")
        name = name.split("(")[0].split("<")[0].split("::")[-1].replace("void ", "").strip()
        v = float(r[col["Metric Value"]].replace(",", "")) * scale.get(r[col["Metric Unit"]], 1.0)
        e = per.setdefault(lid, [name, 0.0, 0.0])
        if r[col["Metric Name"]] == "gpu__time_duration.sum":
            e[1] += v
        elif r[col["Metric Name"]].startswith("dram__bytes_"):
            e[2] += v
    return [tuple(per[k]) for k in sorted(per)]


def write_traffic(args):
    """Per-call DRAM bytes of each --profile-ops operation, from the ncu capture of that run:
    the launches between two L2 flushes are one call; an operation's --warmup first calls are
    dropped and the rest averaged.  Replaces the table's lines for the same keys and stamps
    them with the hash of the kernel sources they were taken from."""
    ops = args.profile_ops.split(",")
    launches = ncu_launches(args.write_traffic)
    first = next(i for i, l in enumerate(launches) if l[0] == FLUSH_KERNEL)
    calls, cur = [], None
    for name, us, nbytes in launches[first:]:
        if name == FLUSH_KERNEL:
            cur = [0.0, 0.0, []]
            calls.append(cur)
        else:
            cur[0] += us
            cur[1] += nbytes
            cur[2].append(name)
    per_op = args.warmup + args.steps
    if len(calls) != len(ops) * per_op:
        raise SystemExit(f"{len(calls)} flush-separated calls in the capture, expected {len(ops)} x {per_op}")
    srcs = [os.path.join(ROOT, "implicit_gemm_conv2d_gb300", "csrc", n) for n in TRAFFIC_SOURCES]
    stamp = "+".join(TRAFFIC_SOURCES) + ":" + source_sha(srcs)
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    lines = open(path).read().splitlines() if os.path.exists(path) else []
    new = {}
    for i, op in enumerate(ops):
        timed = calls[i * per_op + args.warmup:(i + 1) * per_op]
        key = f"{op}:{args.layer}:{args.dtype}:B{args.batch}"
        nbytes = statistics.mean(c[1] for c in timed)
        us = statistics.mean(c[0] for c in timed)
        new[key] = f"{key} {int(round(nbytes))} {us:.1f} {stamp}"
        print(f"{key}: {nbytes / 1e6:.2f} MB, {us:.1f} us under ncu, kernels {' + '.join(timed[0][2])}")
    out = [l for l in lines if not (l.split() and l.split()[0] in new)]
    if not any(l.startswith("#") for l in out):
        out = ["# DRAM bytes per operation call: the sum over the call's launches of dram__bytes_read.sum +",
               "# dram__bytes_write.sum, L2 flushed before the call.  Columns: key  bytes  us_under_ncu",
               "# sources:sha16 (the kernel sources the capture was taken from, '+'-joined, and the first 16",
               "# hex digits of the SHA-256 of their concatenation).  Written by bench.py --write-traffic;",
               "# the commands are in profiles/traffic_b1024.md."] + out
    out += [new[k] for k in new]
    with open(path, "w") as f:
        f.write("\n".join(out) + "\n")
    return 0


def run_profile_ops(args, wl, flush_buf):
    """The launch sequence --write-traffic reads: each operation --warmup + --steps times,
    eagerly, an L2 flush before each call."""
    import torch
    from implicit_gemm_conv2d_gb300 import binding
    ops = args.profile_ops.split(",")
    for op in ops:
        if op not in PROFILE_OPS:
            raise SystemExit(f"unknown operation {op!r}")
    for op in ops:
        for _ in range(args.warmup + args.steps):
            binding.conv_l2_flush(flush_buf)
            wl.op(op)
    torch.cuda.synchronize()
    assert binding.conv_device_status(reset=True) == 0
    print(json.dumps({"profile_ops": ops, "calls_each": args.warmup + args.steps,
                      "launches": {o: wl.plans[o]["launches"] for o in ops}}))
    return 0


def read_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if the kernel sources it was
    taken from are unchanged (their '+'-joined names and sha in the table); else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        line = line.split("#", 1)[0].split()
        if len(line) == 4 and line[0] == kernel_key:
            names, sha = line[3].split(":")
            srcs = [os.path.join(ROOT, "implicit_gemm_conv2d_gb300", "csrc", n) for n in names.split("+")]
            if all(os.path.exists(x) for x in srcs) and source_sha(srcs) == sha:
                return float(line[1])
    return None


class Workload:
    def __init__(self, layer, dtype, B, device, on_device=False):
        """on_device: draw the inputs with a seeded torch generator on the GPU (same
        distributions as synth.conv_inputs, other values) instead of the host generator;
        for timing-only sweeps at large B, where host generation would take minutes."""
        import torch
        from implicit_gemm_conv2d_gb300 import binding, synth
        self.layer, self.dtype, self.B = layer, dtype, B
        self.shape = dict(LAYERS[layer])
        self.tdt = torch.float32 if dtype == "f32" else torch.bfloat16
        s = self.shape
        OH, OW = (s["H"] - s["K"]) // s["S"] + 1, (s["W"] - s["K"]) // s["S"] + 1
        if on_device:
            g = torch.Generator(device=device)
            g.manual_seed(synth.SEED)
            a = 1.0 / math.sqrt(s["IC"] * s["K"] * s["K"])
            self.inp = None
            self.x = torch.randn((B, s["IC"], s["H"], s["W"]), generator=g, device=device).to(self.tdt)
            self.w = ((torch.rand((s["OC"], s["IC"], s["K"], s["K"]), generator=g, device=device) * 2 - 1) * a).to(
                self.tdt)
            self.dy = torch.randn((B, s["OC"], OH, OW), generator=g, device=device).to(self.tdt)
        else:
            inp = synth.conv_inputs(B, s["IC"], s["OC"], s["H"], s["W"], s["K"], s["S"], dtype=dtype)
            self.inp = inp
            self.x = torch.from_numpy(inp["x"]).to(device).to(self.tdt).contiguous()
            self.w = torch.from_numpy(inp["w"]).to(device).to(self.tdt).contiguous()
            self.dy = torch.from_numpy(inp["dy"]).to(device).to(self.tdt).contiguous()
        self.desc = binding.make_desc(B, s["IC"], s["OC"], s["H"], s["W"], s["K"], s["S"], s["relu"], self.tdt)
        OH, OW = binding.out_dims(self.desc)
        self.y = torch.empty((B, s["OC"], OH, OW), dtype=self.tdt, device=device)
        self.dx = torch.empty_like(self.x)
        self.dw = torch.empty_like(self.w)
        self.ws = torch.empty(max(16, binding.conv_bwd_filter_workspace_size(self.desc)), dtype=torch.uint8,
                              device=device)
        # The step runs the workspace-taking forward and d_input (weights packed once per call into
        # these caller-owned buffers); "fwd_plain" / "dgrad_plain" are the no-workspace entry points.
        self.ws_fwd = torch.empty(max(16, binding.conv_fwd_workspace_size(self.desc)), dtype=torch.uint8, device=device)
        self.ws_dgrad = torch.empty(max(16, binding.conv_bwd_data_workspace_size(self.desc)), dtype=torch.uint8,
                                    device=device)
        self.flops = flops(B=B, **s)
        step_ops = (binding.OP_FWD_WS, binding.OP_BWD_DATA_WS, binding.OP_BWD_FILTER)
        self.launches = sum(binding.conv_query(op, self.desc)["launches"] for op in step_ops)
        self.plans = {name: binding.conv_query(op, self.desc) for op, name in zip(step_ops, OPS)}
        self.plans["fwd_plain"] = binding.conv_query(binding.OP_FWD, self.desc)
        self.plans["dgrad_plain"] = binding.conv_query(binding.OP_BWD_DATA, self.desc)
        self.plans["bwd"] = binding.conv_query(binding.OP_BWD, self.desc)
        self.ws_bwd = torch.empty(max(16, binding.conv_bwd_workspace_size(self.desc)), dtype=torch.uint8, device=device)
        self.step_launches = self.plans["fwd"]["launches"] + self.plans["bwd"]["launches"]
        self.plans["bias_grad"] = binding.conv_query(binding.OP_BWD_BIAS, self.desc)
        self.db = torch.empty((s["OC"],), dtype=self.tdt, device=device)
        self.chain = None  # the layer-2 half of the encoder chain, made on first use (layer 1 only)

    def _chain(self):
        """Layer 2's weights, descriptor, output and the chain's workspace (for "chain")."""
        import torch
        from implicit_gemm_conv2d_gb300 import binding
        if self.chain is None:
            if self.layer != "layer1":
                raise SystemExit("the chain op takes the layer-1 workload (its output feeds layer 2)")
            s2 = LAYERS["layer2"]
            g = torch.Generator(device=self.x.device)
            g.manual_seed(7)
            w2 = ((torch.rand((s2["OC"], s2["IC"], s2["K"], s2["K"]), generator=g, device=self.x.device) * 2 - 1)
                  / math.sqrt(s2["IC"] * s2["K"] ** 2)).to(self.tdt)
            d2 = binding.make_desc(self.B, *(s2[k] for k in ("IC", "OC", "H", "W", "K", "S", "relu")), self.tdt)
            OH2, OW2 = binding.out_dims(d2)
            y2 = torch.empty((self.B, s2["OC"], OH2, OW2), dtype=self.tdt, device=self.x.device)
            ws = torch.empty(max(16, binding.conv_fwd_chain2_workspace_size(self.desc, d2)), dtype=torch.uint8,
                             device=self.x.device)
            self.chain = (d2, w2, y2, ws)
            q = binding.conv_query_chain2(self.desc, d2)
            self.plans["chain"] = q
        return self.chain

    def capture(self):
        """One CUDA graph per operation (captured after a warm-up call), so that
        replays carry no host launch overhead into the timed region; and the training step's
        calls (conv_fwd_ws, then conv_bwd) as one graph, "step", the way a caller captures a
        step (one graph launch per step instead of one per call)."""
        import torch
        self.graphs = {}
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for o in OPS + ("fwd_plain", "dgrad_plain", "bwd"):
                self.op(o)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        for o in OPS + ("fwd_plain", "dgrad_plain", "bwd"):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                self.op(o)
            self.graphs[o] = g
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for o in STEP_OPS:
                self.op(o)
        self.graphs["step"] = g
        torch.cuda.synchronize()

    def run(self, name):
        g = getattr(self, "graphs", None)
        if g:
            g[name].replay()
        else:
            self.op(name)

    def op(self, name, stream=None):
        from implicit_gemm_conv2d_gb300 import binding
        relu_y = self.y if self.shape["relu"] else None
        if name == "fwd":
            binding.conv_fwd_ws(self.desc, self.x, self.w, None, self.y, self.ws_fwd, stream)
        elif name == "dgrad":
            binding.conv_bwd_data_ws(self.desc, self.dy, self.w, relu_y, self.dx, self.ws_dgrad, stream)
        elif name == "fwd_plain":
            binding.conv_fwd(self.desc, self.x, self.w, self.y, stream)
        elif name == "dgrad_plain":
            binding.conv_bwd_data(self.desc, self.dy, self.w, relu_y, self.dx, stream)
        elif name == "bwd":
            binding.conv_bwd(self.desc, self.x, self.dy, self.w, relu_y, self.dx, self.dw, None, self.ws_bwd, stream)
        elif name == "bias_grad":
            binding.conv_bwd_bias(self.desc, self.dy, relu_y, self.db, stream)
        elif name == "chain":
            d2, w2, y2, ws = self._chain()
            binding.conv_fwd_chain2(self.desc, d2, self.x, self.w, None, w2, None, self.y, y2, ws, stream)
        else:
            binding.conv_bwd_filter(self.desc, self.x, self.dy, relu_y, self.dw, self.ws, stream)


def time_step(wl, flush_buf, steps, warmup, flush=True):
    """Per-op device times (ms) for `steps` steps, L2 flushed before each step."""
    import torch
    from implicit_gemm_conv2d_gb300 import binding
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        for o in OPS:
            wl.run(o)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for i in range(steps):
        if flush:
            binding.conv_l2_flush(flush_buf)
        e = ev[i]
        e[0].record(stream)
        wl.run("fwd")
        e[1].record(stream)
        wl.run("dgrad")
        e[2].record(stream)
        wl.run("wgrad")
        e[3].record(stream)
    torch.cuda.synchronize()
    per = {o: [] for o in OPS}
    total = []
    for e in ev:
        for j, o in enumerate(OPS):
            per[o].append(e[j].elapsed_time(e[j + 1]))
        total.append(e[0].elapsed_time(e[3]))
    return per, total


def time_fused_step(wl, flush_buf, steps, warmup):
    """Device times (ms) of the step the bench reports: the forward, then conv_bwd (d_input and
    wgrad in one call), replayed as the one "step" graph (eagerly without graphs); L2 flushed
    before each step, outside the timed region.  `per` times the two calls the same way, each
    from its own graph, in a second pass."""
    import torch
    from implicit_gemm_conv2d_gb300 import binding
    stream = torch.cuda.current_stream()
    graphs = getattr(wl, "graphs", None)

    def step():
        if graphs:
            graphs["step"].replay()
        else:
            for o in STEP_OPS:
                wl.op(o)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for i in range(steps):
        binding.conv_l2_flush(flush_buf)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    total = [e[0].elapsed_time(e[1]) for e in ev]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(steps):
        binding.conv_l2_flush(flush_buf)
        e = ev[i]
        e[0].record(stream)
        wl.run("fwd")
        e[1].record(stream)
        wl.run("bwd")
        e[2].record(stream)
    torch.cuda.synchronize()
    per = {o: [e[j].elapsed_time(e[j + 1]) for e in ev] for j, o in enumerate(STEP_OPS)}
    return per, total


def warm_us(wl, iters=200, warmup=50):
    """PR-style warm timing: back-to-back iterations of one op between two events."""
    import torch
    out = {}
    for o in OPS:
        for _ in range(warmup):
            wl.run(o)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(iters):
            wl.run(o)
        b.record()
        torch.cuda.synchronize()
        out[o] = a.elapsed_time(b) / iters * 1e3
    return out


def e2e(wl, flush_buf, steps, chunks=4):
    """Same step through the public API with host buffers: every step copies the pinned host
    inputs in and the three results out.  The batch is cut into `chunks` sample ranges so
    that copies overlap compute: per range, x and dy go in on a copy-in stream, the forward and
    d_input of that range run on the compute stream, and y and dx come out on a copy-out
    stream; wgrad runs once on the whole batch when every range is in, then dw comes out.
    Events order the three streams.  The step -- copies included -- is captured as one CUDA
    graph (as a caller would capture it) and replayed; the timed region of a step runs from
    before its first copy to after its last, on the device, L2 flushed between steps."""
    import torch
    from implicit_gemm_conv2d_gb300 import binding
    B = wl.B
    chunks = max(1, min(chunks, B))
    bounds = [B * i // chunks for i in range(chunks + 1)]
    s = wl.shape
    relu = s["relu"]
    descs = [binding.make_desc(bounds[i + 1] - bounds[i], s["IC"], s["OC"], s["H"], s["W"], s["K"], s["S"],
                               relu, wl.tdt) for i in range(chunks)]
    ws_f = [torch.empty(max(16, binding.conv_fwd_workspace_size(d)), dtype=torch.uint8, device=wl.x.device)
            for d in descs]
    ws_d = [torch.empty(max(16, binding.conv_bwd_data_workspace_size(d)), dtype=torch.uint8, device=wl.x.device)
            for d in descs]
    xh = wl.x.cpu().pin_memory()
    wh = wl.w.cpu().pin_memory()
    dyh = wl.dy.cpu().pin_memory()
    yh = torch.empty(wl.y.shape, dtype=wl.tdt).pin_memory()
    dxh = torch.empty(wl.dx.shape, dtype=wl.tdt).pin_memory()
    dwh = torch.empty(wl.dw.shape, dtype=wl.tdt).pin_memory()
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def step():
        main = torch.cuda.current_stream()
        s_in.wait_stream(main)
        s_cmp.wait_stream(main)
        s_out.wait_stream(main)
        with torch.cuda.stream(s_in):
            wl.w.copy_(wh, non_blocking=True)
        ins = []
        for i in range(chunks):
            a, b = bounds[i], bounds[i + 1]
            with torch.cuda.stream(s_in):
                wl.x[a:b].copy_(xh[a:b], non_blocking=True)
                wl.dy[a:b].copy_(dyh[a:b], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(s_in)
                ins.append(ev)
        for i in range(chunks):
            a, b = bounds[i], bounds[i + 1]
            s_cmp.wait_event(ins[i])
            binding.conv_fwd_ws(descs[i], wl.x[a:b], wl.w, None, wl.y[a:b], ws_f[i], s_cmp)
            binding.conv_bwd_data_ws(descs[i], wl.dy[a:b], wl.w, wl.y[a:b] if relu else None, wl.dx[a:b], ws_d[i],
                                     s_cmp)
            done = torch.cuda.Event()
            done.record(s_cmp)
            s_out.wait_event(done)
            with torch.cuda.stream(s_out):
                yh[a:b].copy_(wl.y[a:b], non_blocking=True)
                dxh[a:b].copy_(wl.dx[a:b], non_blocking=True)
        binding.conv_bwd_filter(wl.desc, wl.x, wl.dy, wl.y if relu else None, wl.dw, wl.ws, s_cmp)
        done = torch.cuda.Event()
        done.record(s_cmp)
        s_out.wait_event(done)
        with torch.cuda.stream(s_out):
            dwh.copy_(wl.dw, non_blocking=True)
        main.wait_stream(s_out)
        main.wait_stream(s_in)
        main.wait_stream(s_cmp)

    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        for _ in range(2):  # warm-up calls outside the capture
            step()
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        step()
    torch.cuda.synchronize()
    main = torch.cuda.current_stream()
    evs = []
    for i in range(steps + 3):
        binding.conv_l2_flush(flush_buf)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(main)
        g.replay()
        b.record(main)
        if i >= 3:
            evs.append((a, b))
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    esz = wl.x.element_size()
    return {"value": 3 * wl.flops / (ms * 1e-3) / 1e9, "unit": "GFLOP/s", "ms_per_step": ms,
            "h2d_bytes_per_step": (wl.x.numel() + wl.w.numel() + wl.dy.numel()) * esz,
            "d2h_bytes_per_step": (wl.y.numel() + wl.dx.numel() + wl.dw.numel()) * esz,
            "overlap": f"{chunks} sample ranges; copy-in, compute and copy-out on three streams, "
                       "the step captured as one CUDA graph (copies from / to pinned host memory included)"}


_SIDE = []


def graphed(fn):
    """Capture fn (a sequence of library calls) into a CUDA graph on a side stream, after
    a warm-up call there (kernel attributes and lazy module loading happen outside capture)."""
    import torch
    if not _SIDE:
        _SIDE.append(torch.cuda.Stream())
    s = _SIDE[0]
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    torch.cuda.synchronize()
    return g


def time_graph(g, flush_buf=None, iters=50, warmup=5):
    """Mean device ms of one replay: cold (L2 flushed before each, one event pair per
    replay) when flush_buf is given, else warm (iters back-to-back replays)."""
    import torch
    from implicit_gemm_conv2d_gb300 import binding
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    if flush_buf is None:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(iters):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / iters
    evs = []
    for _ in range(iters):
        binding.conv_l2_flush(flush_buf)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        evs.append((a, b))
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in evs)


def bias_extras(wls, flush_buf, peaks, device):
    """The per-channel bias: forward with the bias against the plain forward, and the bias
    gradient, for each layer / dtype workload at the bench batch; then the bias gradient at
    the PR's bias-grad batch (B=32768, no mask, as its blocks time it), warm and cold L2."""
    import torch
    from implicit_gemm_conv2d_gb300 import binding, synth
    hbm = peaks["hbm_gbs"]
    out = {}
    for key, wl in wls.items():
        s = wl.shape
        b_np = synth.conv_inputs(wl.B, s["IC"], s["OC"], s["H"], s["W"], s["K"], s["S"], dtype=wl.dtype,
                                 need=("bias",))["bias"]
        bias = torch.from_numpy(b_np).to(device).to(wl.tdt)
        db = torch.empty_like(bias)
        relu_y = wl.y if s["relu"] else None
        g_fb = graphed(lambda: binding.conv_fwd_bias(wl.desc, wl.x, wl.w, bias, wl.y))
        g_f = graphed(lambda: binding.conv_fwd(wl.desc, wl.x, wl.w, wl.y))
        g_db = graphed(lambda: binding.conv_bwd_bias(wl.desc, wl.dy, relu_y, db))
        esz = wl.x.element_size()
        nbytes = (wl.dy.numel() * (2 if s["relu"] else 1) + db.numel()) * esz
        t_db = time_graph(g_db, flush_buf)
        plan = binding.conv_query(binding.OP_BWD_BIAS, wl.desc)
        out[key] = {"fwd_us_cold_l2": time_graph(g_f, flush_buf) * 1e3,
                    "fwd_bias_us_cold_l2": time_graph(g_fb, flush_buf) * 1e3,
                    "bias_grad_us_cold_l2": t_db * 1e3, "bias_grad_us_warm": time_graph(g_db, None, 200, 50) * 1e3,
                    "bias_grad_bytes": nbytes, "bias_grad_gbs": nbytes / (t_db * 1e-3) / 1e9,
                    "bias_grad_frac_hbm": nbytes / (t_db * 1e-3) / 1e9 / hbm,
                    "bias_grad_plan": {k: plan[k] for k in ("algo_name", "launches", "grid", "block", "splits")}}
    big = {}
    for layer in ("layer1", "layer2"):
        s = LAYERS[layer]
        for dt in ("f32", "bf16"):
            tdt = torch.float32 if dt == "f32" else torch.bfloat16
            dy_np = synth.conv_inputs(BIAS_GRAD_BATCH, s["IC"], s["OC"], s["H"], s["W"], s["K"], s["S"], dtype=dt,
                                      need=("dy",))["dy"]
            dy = torch.from_numpy(dy_np).to(device).to(tdt)
            del dy_np
            db = torch.empty((s["OC"],), dtype=tdt, device=device)
            desc = binding.bias_desc(tuple(dy.shape), False, tdt)
            g = graphed(lambda: binding.conv_bwd_bias(desc, dy, None, db))
            nbytes = (dy.numel() + db.numel()) * dy.element_size()
            warm = time_graph(g, None, 200, 50)
            cold = time_graph(g, flush_buf, 50, 5)
            big[f"{layer}_{dt}"] = {"grad_elems": dy.numel(), "us_warm": warm * 1e3, "us_cold_l2": cold * 1e3,
                                    "gbs_cold_l2": nbytes / (cold * 1e-3) / 1e9,
                                    "frac_hbm_cold_l2": nbytes / (cold * 1e-3) / 1e9 / hbm,
                                    "pr522_fast_us": PR522_BIAS_GRAD_US[layer]}
            del dy, g
    out[f"bias_grad_b{BIAS_GRAD_BATCH}_norelu"] = big
    return out


def chain_extras(flush_buf, device, batches=(256, 1024, 4096, 16384)):
    """The encoder's two-layer forward fused (conv_fwd_chain2: layer 1's output tile stays in
    shared memory as layer 2's input) against the two layers' forward calls one after the other
    (conv_fwd_ws each), cold L2; layer 2's share of the chain = chain - layer 1 alone."""
    import torch
    from implicit_gemm_conv2d_gb300 import binding
    out = {}
    s1, s2 = LAYERS["layer1"], LAYERS["layer2"]
    for dt in ("bf16", "f32"):
        tdt = torch.float32 if dt == "f32" else torch.bfloat16
        for B in batches:
            g = torch.Generator(device=device)
            g.manual_seed(7)
            x = torch.randn((B, s1["IC"], s1["H"], s1["W"]), generator=g, device=device).to(tdt)
            w1 = ((torch.rand((s1["OC"], s1["IC"], s1["K"], s1["K"]), generator=g, device=device) * 2 - 1)
                  / math.sqrt(s1["IC"] * s1["K"] ** 2)).to(tdt)
            w2 = ((torch.rand((s2["OC"], s2["IC"], s2["K"], s2["K"]), generator=g, device=device) * 2 - 1)
                  / math.sqrt(s2["IC"] * s2["K"] ** 2)).to(tdt)
            d1 = binding.make_desc(B, *(s1[k] for k in ("IC", "OC", "H", "W", "K", "S", "relu")), tdt)
            d2 = binding.make_desc(B, *(s2[k] for k in ("IC", "OC", "H", "W", "K", "S", "relu")), tdt)
            y1 = torch.empty((B, 128, 3, 4), dtype=tdt, device=device)
            y2 = torch.empty((B, 128, 1, 2), dtype=tdt, device=device)
            wsc = torch.empty(max(16, binding.conv_fwd_chain2_workspace_size(d1, d2)), dtype=torch.uint8, device=device)
            ws1 = torch.empty(max(16, binding.conv_fwd_workspace_size(d1)), dtype=torch.uint8, device=device)
            ws2 = torch.empty(max(16, binding.conv_fwd_workspace_size(d2)), dtype=torch.uint8, device=device)
            gc = graphed(lambda: binding.conv_fwd_chain2(d1, d2, x, w1, None, w2, None, y1, y2, wsc))
            g1 = graphed(lambda: binding.conv_fwd_ws(d1, x, w1, None, y1, ws1))
            g2 = graphed(lambda: binding.conv_fwd_ws(d2, y1, w2, None, y2, ws2))
            tc, t1, t2 = (time_graph(gg, flush_buf, 30, 3) * 1e3 for gg in (gc, g1, g2))
            q = binding.conv_query_chain2(d1, d2)
            out[f"{dt}_B{B}"] = {"chain_us_cold_l2": tc, "layer1_fwd_us_cold_l2": t1, "layer2_fwd_us_cold_l2": t2,
                                 "unfused_us": t1 + t2, "layer2_share_of_chain_us": tc - t1,
                                 "chain_plan": {k: q[k] for k in ("algo_name", "launches", "grid", "block")}}
            # fp32 runs unfused by default; the fused kernel, forced, for the record
            binding.conv_set_algo(binding.OP_FWD, binding.ALGO_TC)
            try:
                if q["algo"] == binding.ALGO_AUTO and binding.conv_query_chain2(d1, d2)["algo"] == binding.ALGO_TC:
                    wsf = torch.empty(max(16, binding.conv_fwd_chain2_workspace_size(d1, d2)), dtype=torch.uint8,
                                      device=device)
                    gf = graphed(lambda: binding.conv_fwd_chain2(d1, d2, x, w1, None, w2, None, y1, y2, wsf))
                    out[f"{dt}_B{B}"]["fused_forced_us_cold_l2"] = time_graph(gf, flush_buf, 30, 3) * 1e3
                    del gf
            finally:
                binding.conv_set_algo(binding.OP_FWD, binding.ALGO_AUTO)
            del gc, g1, g2, x, y1, y2
            torch.cuda.empty_cache()
    return out


def chain_bwd_extras(flush_buf, device, batches=(256, 1024, 4096)):
    """The encoder's two-layer backward (conv_bwd_chain2: layer 2's dx kept in the workspace and
    fed to layer 1's backward) with and without layer 1's input gradient, against the two
    layers' conv_bwd calls one after the other, cold L2."""
    import torch
    from implicit_gemm_conv2d_gb300 import binding
    out = {}
    s1, s2 = LAYERS["layer1"], LAYERS["layer2"]
    for dt in ("f32", "bf16"):
        tdt = torch.float32 if dt == "f32" else torch.bfloat16
        for B in batches:
            g = torch.Generator(device=device)
            g.manual_seed(11)
            x = torch.randn((B, s1["IC"], s1["H"], s1["W"]), generator=g, device=device).to(tdt)
            w1 = ((torch.rand((s1["OC"], s1["IC"], s1["K"], s1["K"]), generator=g, device=device) * 2 - 1)
                  / math.sqrt(s1["IC"] * s1["K"] ** 2)).to(tdt)
            w2 = ((torch.rand((s2["OC"], s2["IC"], s2["K"], s2["K"]), generator=g, device=device) * 2 - 1)
                  / math.sqrt(s2["IC"] * s2["K"] ** 2)).to(tdt)
            dy2 = torch.randn((B, 128, 1, 2), generator=g, device=device).to(tdt)
            d1 = binding.make_desc(B, *(s1[k] for k in ("IC", "OC", "H", "W", "K", "S", "relu")), tdt)
            d2 = binding.make_desc(B, *(s2[k] for k in ("IC", "OC", "H", "W", "K", "S", "relu")), tdt)
            y1 = torch.empty((B, 128, 3, 4), dtype=tdt, device=device)
            y2 = torch.empty((B, 128, 1, 2), dtype=tdt, device=device)
            binding.conv_fwd(d1, x, w1, y1)
            binding.conv_fwd(d2, y1, w2, y2)
            dx1, dx2 = torch.empty_like(x), torch.empty_like(y1)
            dw1, dw2 = torch.empty_like(w1), torch.empty_like(w2)
            wsc = torch.empty(max(16, binding.conv_bwd_chain2_workspace_size(d1, d2)), dtype=torch.uint8,
                              device=device)
            ws1 = torch.empty(max(16, binding.conv_bwd_workspace_size(d1)), dtype=torch.uint8, device=device)
            ws2 = torch.empty(max(16, binding.conv_bwd_workspace_size(d2)), dtype=torch.uint8, device=device)
            gc = graphed(lambda: binding.conv_bwd_chain2(d1, d2, x, w1, y1, w2, y2, dy2, dx1, dw1, None, dw2, None, wsc))
            gn = graphed(lambda: binding.conv_bwd_chain2(d1, d2, x, w1, y1, w2, y2, dy2, None, dw1, None, dw2, None,
                                                         wsc))

            def two_calls():
                binding.conv_bwd(d2, y1, dy2, w2, y2, dx2, dw2, None, ws2)
                binding.conv_bwd(d1, x, dx2, w1, y1, dx1, dw1, None, ws1)
            gu = graphed(two_calls)
            tc, tn, tu = (time_graph(gg, flush_buf, 30, 3) * 1e3 for gg in (gc, gn, gu))
            out[f"{dt}_B{B}"] = {"chain_us_cold_l2": tc, "chain_no_dx1_us_cold_l2": tn, "two_conv_bwd_us_cold_l2": tu}
            del gc, gn, gu, x, y1, y2, dx1, dx2
            torch.cuda.empty_cache()
    return out


SWEEP_BATCHES = (256, 1024, 4096, 16384)


def batch_sweep(flush_buf, sms, sm_mhz, peaks, device):
    """Per-operation cold-L2 time, throughput and roofline fraction of both layers in both
    dtypes over a range of batch sizes (the plans the library picks for each), inputs drawn
    on the device."""
    import torch
    out = {}
    for layer in ("layer1", "layer2"):
        for dt in ("f32", "bf16"):
            for B in SWEEP_BATCHES:
                wl = Workload(layer, dt, B, device, on_device=True)
                wl.capture()
                per, _ = time_step(wl, flush_buf, 30, 3)
                entry = {}
                for o in OPS:
                    t_ms = statistics.mean(per[o])
                    r = roofline_of(wl, o, t_ms, sms, sm_mhz, peaks)
                    pl = wl.plans[o]
                    entry[o] = {"us_cold_l2": t_ms * 1e3, "tflops": wl.flops / (t_ms * 1e-3) / 1e12,
                                "bound": r["bound"], "frac": r["frac"], "algo": pl["algo_name"],
                                "grid": pl["grid"], "splits": pl["splits"], "launches": pl["launches"]}
                out[f"{layer}_{dt}_B{B}"] = entry
                del wl
                torch.cuda.empty_cache()
    return out


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}, \
        "fallback"


def pipe_peak(algo, dtype, sms, sm_mhz, peaks):
    """Peak of the pipe an algorithm family runs on, in TFLOP/s of the layer's own
    (algorithmic) FLOPs, and a description of where it comes from."""
    if algo == "tc" and dtype == "bf16":
        return peaks["bf16_tflops"], f"measured dense bf16 tensor peak ({peaks['bf16_tflops']:.0f} TF/s, burst)"
    if algo == "tc":
        tf32 = peaks["bf16_tflops"] * (1.1 / 2.25)
        return tf32 / 3.0, (f"measured bf16 peak x nominal tf32/bf16 ratio (1.1/2.25) = {tf32:.0f} TF/s, "
                            "/3 for the three tf32 MMAs per fp32 product (3xTF32)")
    return sms * 128 * 2 * sm_mhz * 1e6 / 1e12, f"{sms} SMs x 128 FP32 lanes x 2 FLOP x {sm_mhz:.0f} MHz (FFMA)"


def roofline_of(wl, op, t_ms, sms, sm_mhz, peaks):
    plan = wl.plans[op]
    esz = 4 if wl.dtype == "f32" else 2
    ab = alg_bytes(op, B=wl.B, esize=esz, **wl.shape)
    fl = op_flops(op, wl.flops)
    pk, src = pipe_peak(plan["algo_name"], wl.dtype, sms, sm_mhz, peaks)
    t_flop = fl / (pk * 1e12)
    t_mem = ab / (peaks["hbm_gbs"] * 1e9)
    t = t_ms * 1e-3
    if t_flop >= t_mem:
        bound = "alu" if plan["algo_name"] != "tc" else "tensor"
        r = {"bound": bound, "achieved": fl / t / 1e12, "peak": pk, "unit": "TFLOP/s"}
        src_s = src
    else:
        r = {"bound": "hbm", "achieved": ab / t / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
        src_s = f"measured HBM copy bandwidth ({peaks['hbm_gbs']:.0f} GB/s)"
    r["frac"] = r["achieved"] / r["peak"]
    r["roofline_us"] = max(t_flop, t_mem) * 1e6
    r["algorithmic_bytes"] = ab
    r["flops"] = fl
    r["peak_source"] = src_s
    return r


def run_ours(args):
    import torch
    import torch.distributed as dist
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
    from implicit_gemm_conv2d_gb300 import binding, build as libbuild
    if rank == 0 and not libbuild.up_to_date():
        libbuild.build()
    if world > 1:
        dist.barrier()
    binding.lib()
    algo = {"auto": 0, "direct": 1, "ffma": 2, "tc": 3}[args.algo]
    for op in range(3):
        binding.conv_set_algo(op, algo)
    props = torch.cuda.get_device_properties(device)
    sms = props.multi_processor_count
    peaks, peaks_kind = load_peaks()

    flush_buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    if args.chain_only:
        print(json.dumps({"chain_fwd": chain_extras(flush_buf, device), "chain_bwd": chain_bwd_extras(flush_buf, device)}))
        return 0
    # Above 4096 samples the inputs are drawn on the device (host generation would take minutes).
    wl = Workload(args.layer, args.dtype, args.batch, device, on_device=args.batch > 4096)
    if args.profile_ops:
        return run_profile_ops(args, wl, flush_buf)
    if not args.no_graphs:
        wl.capture()

    # ---- the timed region ----
    step = STEP_OPS if args.step == "fused" else OPS
    for _ in range(args.warmup):
        for o in step:
            wl.run(o)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        clk.mark_start()
        if args.step == "fused":
            per, total = time_fused_step(wl, flush_buf, args.steps, 0)
        else:
            per, total = time_step(wl, flush_buf, args.steps, 0)
        torch.cuda.synchronize()
        clk.mark_end()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ms_step = combine_ranks(sum(total) / len(total), world, device)
    value = job_value(ms_step, world, wl.flops)

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return 0

    # ---- per-op summary and roofline of the dominant kernel ----
    clocks = clk.summary()
    sm_mhz = clocks["sm_max_mhz"] or peaks.get("sm_max_mhz", 2070.0)
    step_ms = {o: statistics.mean(per[o]) for o in step}
    dom = max(step, key=lambda o: step_ms[o])
    # the three operations one call each (cold L2), for the per-operation table
    if args.step == "fused":
        per3, _ = time_step(wl, flush_buf, 50, 3)
        op_ms = {o: statistics.mean(per3[o]) for o in OPS}
        op_ms["bwd"] = step_ms["bwd"]
    else:
        op_ms = dict(step_ms)
    plan = wl.plans[dom]
    roofline = roofline_of(wl, dom, step_ms[dom], sms, sm_mhz, peaks)
    roofline["kernel"] = f"{dom} ({plan['algo_name']}, {plan['launches']} launch(es))"
    roofline["traffic"] = read_traffic(f"{dom}:{args.layer}:{args.dtype}:B{args.batch}")
    roofline["traffic_note"] = ("dram__bytes_read.sum + dram__bytes_write.sum per call (sum over its launches) from "
                                "one ncu capture of the same kernel source, L2 flushed before the step; output "
                                "lines still dirty in L2 when the kernel ends are not in dram__bytes_write, so "
                                "the figure is mostly reads; null when the kernel source changed since")
    ops = {}
    for o in op_ms:
        r = roofline_of(wl, o, op_ms[o], sms, sm_mhz, peaks)
        ops[o] = {"us": op_ms[o] * 1e3, "gflops": op_flops(o, wl.flops) / (op_ms[o] * 1e-3) / 1e9,
                  "algo": wl.plans[o]["algo_name"], "launches": wl.plans[o]["launches"],
                  "bound": r["bound"], "frac": r["frac"], "roofline_us": r["roofline_us"]}
    # The no-workspace entry points (weights formatted inside the kernels), same workload, cold L2.
    plain = {}
    if getattr(wl, "graphs", None):
        for o, name in (("fwd", "fwd_plain"), ("dgrad", "dgrad_plain")):
            t_ms = time_graph(wl.graphs[name], flush_buf, 50, 5)
            plain[o] = {"us": t_ms * 1e3, "gflops": wl.flops / (t_ms * 1e-3) / 1e9,
                        "launches": wl.plans[name]["launches"]}
    pr = PR522_US.get((args.layer, args.dtype))
    pr_gflops = 3 * wl.flops / ((pr[0] + pr[1]) * 1e-6) / 1e9 if (pr and args.batch == 1024) else None
    line = {
        "metric": METRIC, "value": value, "unit": "GFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": (value / world / pr_gflops) if pr_gflops else None,
        "dtype": args.dtype, "data": "synthetic",
        "config": arm_config(args),
        "ops": ops,
        "ops_no_workspace": plain,
        "roofline": roofline,
        "gpu_launches": (wl.step_launches if args.step == "fused" else wl.launches) * args.steps,
        "clocks": clocks,
        "peaks": {"source": peaks_kind, "hbm_gbs": peaks["hbm_gbs"], "bf16_tflops": peaks.get("bf16_tflops")},
    }
    if not args.no_extras:
        line["e2e"] = e2e(wl, flush_buf, min(args.steps, 50))
        others = {}
        wls = {}
        for layer in ("layer1", "layer2"):
            for dt in ("f32", "bf16"):
                w2 = wl if (layer, dt) == (args.layer, args.dtype) else Workload(layer, dt, args.batch, device)
                wls[f"{layer}_{dt}"] = w2
                if not args.no_graphs and not getattr(w2, "graphs", None):
                    w2.capture()
                p2, _ = time_step(w2, flush_buf, 50, 5)
                warm = warm_us(w2)
                entry = {}
                for o in OPS:
                    t_ms = statistics.mean(p2[o])
                    r = roofline_of(w2, o, t_ms, sms, sm_mhz, peaks)
                    entry[o] = {"us_cold_l2": t_ms * 1e3, "us_warm": warm[o],
                                "gflops": w2.flops / (t_ms * 1e-3) / 1e9, "algo": w2.plans[o]["algo_name"],
                                "bound": r["bound"], "frac": r["frac"], "roofline_us": r["roofline_us"]}
                if getattr(w2, "graphs", None):
                    t_ms = time_graph(w2.graphs["bwd"], flush_buf, 50, 5)
                    r = roofline_of(w2, "bwd", t_ms, sms, sm_mhz, peaks)
                    entry["bwd"] = {"us_cold_l2": t_ms * 1e3, "gflops": 2 * w2.flops / (t_ms * 1e-3) / 1e9,
                                    "algo": w2.plans["bwd"]["algo_name"], "bound": r["bound"], "frac": r["frac"],
                                    "roofline_us": r["roofline_us"]}
                if args.batch == 1024:
                    f, b = PR522_US[(layer, dt)]
                    entry["pr522_us"] = {"fwd": f, "bwd": b}
                others[f"{layer}_{dt}"] = entry
        line["configs_b%d" % args.batch] = others
        line["bias"] = bias_extras(wls, flush_buf, peaks, device)
        line["chain_fwd"] = chain_extras(flush_buf, device)
        line["chain_bwd"] = chain_bwd_extras(flush_buf, device)
        line["batch_sweep"] = batch_sweep(flush_buf, sms, sm_mhz, peaks, device)
        if world == 1:
            line["cpu_baseline"] = cpu_baseline(LAYERS[args.layer], 128, 10.0)
    print(json.dumps(line))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.write_traffic:
        return write_traffic(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
