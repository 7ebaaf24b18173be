"""Benchmark of the scaled FP8 / BF16 GEMM hot path on GB300.

One step = one launch of every workload in the suite below, each on its own
synthetic inputs already resident in HBM: the M x 7168 x K ptpc shapes (tail-only
K=256, K=512, K=1792), blockscale 16384x7168x2048, mxfp8 32768x7168x1792, the
unpadded-N ptpc shapes at K=7168 (N = 6288, 3648, 6400) and the BF16
[4096,1024]x[1024,896] GEMM.  `value` is the suite's total FLOPs (2MNK per GEMM)
divided by its device time, in TFLOP/s; per-workload times, TFLOP/s and
fractions of peak are in `per_config`.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) every rank runs the same suite on its own GPU (replicas:
the GEMM needs no exchange); the step time is the max over ranks and `value`
counts the work of all ranks.  `--impl reference` times the CPU oracle on a
bounded row sample of the same workloads instead (rank 0 only).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "scaled-FP8 GEMM TFLOPS & % FP8 peak at M×7168×K; bad launches per 20 (must be 0)"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Control:
    """Host-side control plane across replicas (gloo): barrier and reductions."""

    def __init__(self, world):
        self.world = world
        self.dist = None
        if world > 1:
            import torch.distributed as dist

            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("gloo")
            self.dist = dist

    def barrier(self):
        if self.dist:
            self.dist.barrier()

    def max(self, x):
        if not self.dist:
            return float(x)
        t = torch.tensor([float(x)], dtype=torch.float64)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x):
        if not self.dist:
            return float(x)
        t = torch.tensor([float(x)], dtype=torch.float64)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.dist:
            self.dist.destroy_process_group()


def aggregate(control, local_flops, local_seconds):
    """Whole-job throughput: work of all ranks over the slowest rank's time."""
    total = control.sum(local_flops)
    t = control.max(local_seconds)
    return total, t, (total / t / 1e12 if t > 0 else 0.0)


def make_suite(only=None, rows=None):
    """The suite's cases; `only` keeps one workload and `rows` shrinks its M (profiling runs)."""
    cases, cache = [], {}
    for name in synth.SUITE if only is None else [only]:
        mode, M, N, K, seed, a_std, b_std = synth.CONFIGS[name]
        if rows:
            M = rows
        cases.append((name, synth.make_case(mode, M, N, K, seed=seed, a_std=a_std, b_std=b_std, cache=cache)))
    return cases


# --------------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while a region runs."""

    QUERY = (
        "index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
        "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
        "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap"
    )

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL,
            )
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), float(f[3]), f[4], f[5], f[6], f[7], f[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        loaded = [r for r in rows if r[2] > 300.0] or rows  # samples under load (power)
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for nm, v in zip(names, r[4:]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {
            "sm_mhz": statistics.median(r[0] for r in loaded),
            "sm_max_mhz": max(r[1] for r in rows),
            "power_w_max": max(r[2] for r in rows),
            "reasons": sorted(reasons),
            "samples": len(rows),
            "samples_under_load": len(loaded),
        }


# --------------------------------------------------------------------------- oracle baseline


def cpu_baseline(cases, rows, seconds_cap=None):
    """The CPU oracle on rows [0, rows) of every workload: (TFLOP/s, seconds, threads, flops)."""
    import oracle

    flops = 0.0
    t0 = time.perf_counter()
    for name, c in cases:
        r = min(rows, c.M)
        oracle.gemm(c.mode, *c.numpy(), rows=(0, r), want_r=False)
        flops += 2.0 * r * c.N * c.K
        if seconds_cap and time.perf_counter() - t0 > seconds_cap:
            break
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, dt, oracle.num_threads(), flops


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    import platform

    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


C0_ONE_CORE = r"""
import json, sys, time
sys.path.insert(0, %r)
import oracle, synth
mode, M, N, K, seed, a, b = synth.CONFIGS["c0_ptpc_256x512x256"]
c = synth.make_case(mode, M, N, K, seed=seed, a_std=a, b_std=b)
args = c.numpy()
oracle.gemm(mode, *args, want_r=False)
t0 = time.perf_counter()
oracle.gemm(mode, *args, want_r=False)
dt = time.perf_counter() - t0
print(json.dumps({"seconds": dt, "gflops": c.flops / dt / 1e9, "threads": oracle.num_threads()}))
"""


def c0_one_core():
    """The oracle on the whole 256 x 512 x 256 ptpc workload with one OpenMP thread
    (a child process started with OMP_NUM_THREADS=1)."""
    env = dict(os.environ, OMP_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, "-c", C0_ONE_CORE % ROOT], capture_output=True, text=True, env=env,
                           timeout=300)
        d = json.loads(r.stdout.strip().splitlines()[-1])
        return {"workload": "c0_ptpc_256x512x256", "seconds": round(d["seconds"], 4),
                "gflops": round(d["gflops"], 3), "threads": d["threads"]}
    except (OSError, subprocess.SubprocessError, ValueError, IndexError, KeyError) as e:
        return {"workload": "c0_ptpc_256x512x256", "error": str(e)[:200]}


def choose_peak(clk):
    """Burst or sustained FP8 / BF16 peak for this run, from its clock record: the
    burst figure (a short cuBLAS burst at full clock) when the SM clock held within
    3% of its maximum with no power cap active during the timed region, else the
    sustained one (a seconds-long loop under the power cap).  Returns (kind, why)."""
    sm, smax, reasons = clk.get("sm_mhz"), clk.get("sm_max_mhz"), clk.get("reasons") or []
    if sm is None or not smax:
        return "sustained", "no clock record"
    if "sw_power_cap" in reasons:
        return "sustained", "sw_power_cap was active (median SM clock %.0f of %.0f MHz)" % (sm, smax)
    if sm < 0.97 * smax:
        return "sustained", "median SM clock %.0f MHz < 0.97 x max %.0f" % (sm, smax)
    return "burst", "median SM clock %.0f of %.0f MHz, no power cap" % (sm, smax)


# Workloads shorter than this are also timed per call in a CUDA graph.
GRAPH_MAX_US = 100.0


def graph_per_call(launch_fn, stream, calls=200, batches=9, gpu_index=None):
    """Median device time per call over `batches` replays of a CUDA graph of
    `calls` back-to-back launches on the same operands (deepseek-ai/DeepGEMM PR
    453, Performance Overhead: CUDA-graph median per call over 9 x 200 calls).
    The operands stay in L2 between calls where they fit.  With `gpu_index`, the
    SM clock and throttle reasons sampled during the replays come back too (the
    replays follow the timed steps, so the clocks there may have dropped)."""
    clocks = None
    try:
        with torch.cuda.stream(stream):
            launch_fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(calls):
                launch_fn()
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        per = []
        if gpu_index is not None:
            clocks = ClockSampler(gpu_index)
            clocks.start()
        for _ in range(batches):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            per.append(1e3 * e0.elapsed_time(e1) / calls)
        del g
        out = {"us_median": round(statistics.median(per), 2), "us_min": round(min(per), 2),
               "calls": calls, "batches": batches}
        if clocks is not None:
            clk = clocks.stop()
            clocks = None
            out["clocks"] = {"sm_mhz": clk["sm_mhz"], "reasons": clk["reasons"]}
        return out
    except RuntimeError as e:
        return {"error": str(e)[:200]}
    finally:
        if clocks is not None:
            clocks.stop()


# --------------------------------------------------------------------------- GPU arm


def run_gpu(args, control, rank, local):
    from fp8_scaled_gemm_sm_gb300 import binding, build

    build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_kind = load_peaks()
    fp8_peak_sustained = 2.0 * peaks["bf16_tflops_sustained"]
    fp8_peak_burst = 2.0 * peaks["bf16_tflops"]
    hbm = peaks["hbm_gbs"]

    cases = make_suite(args.only, args.rows)
    stream = torch.cuda.Stream(dev)
    sraw = stream.cuda_stream
    work = []
    for name, c in cases:
        d = {
            "name": name,
            "case": c,
            "A": c.A.to(dev),
            "B": c.B.to(dev),
            "sa": None if c.sa is None else c.sa.to(dev),
            "sb": None if c.sb is None else c.sb.to(dev),
            "C": torch.empty((c.M, c.N), dtype=torch.bfloat16, device=dev),
            "h": binding.scaled_gemm_create(c.mode, c.N, c.K, c.M, local),
        }
        d["cfg"] = binding.scaled_gemm_get_config(d["h"])
        work.append(d)
    torch.cuda.synchronize()

    def launch(d, C=None):
        binding.scaled_gemm_launch(
            d["h"], d["A"].data_ptr(), d["B"].data_ptr(),
            0 if d["sa"] is None else d["sa"].data_ptr(),
            0 if d["sb"] is None else d["sb"].data_ptr(),
            (d["C"] if C is None else C).data_ptr(), d["case"].M, sraw,
        )

    # warm-up
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            for d in work:
                launch(d)
    torch.cuda.synchronize()

    # timed steps: one event pair around the step plus one per GEMM
    n = len(work)
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)] for _ in range(args.steps)]
    e_all0, e_all1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    control.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        e_all0.record(stream)
        for s in range(args.steps):
            for i, d in enumerate(work):
                ev[s][i][0].record(stream)
                launch(d)
                ev[s][i][1].record(stream)
        e_all1.record(stream)
    torch.cuda.synchronize()
    control.barrier()
    wall1 = time.perf_counter()
    clk = clocks.stop()
    local_s = e_all0.elapsed_time(e_all1) / 1e3
    peak_kind_run, peak_why = choose_peak(clk)
    fp8_peak = fp8_peak_burst if peak_kind_run == "burst" else fp8_peak_sustained
    bf16_peak = peaks["bf16_tflops"] if peak_kind_run == "burst" else peaks["bf16_tflops_sustained"]
    flops_step = sum(d["case"].flops for d in work)
    total_flops, t_max, value = aggregate(control, flops_step * args.steps, local_s)

    per = {}
    for i, d in enumerate(work):
        c = d["case"]
        ms = [ev[s][i][0].elapsed_time(ev[s][i][1]) for s in range(args.steps)]
        us = 1e3 * sum(ms) / len(ms)
        tf = c.flops / (us * 1e-6) / 1e12
        byts = synth.gemm_bytes(c.mode, c.M, c.N, c.K)
        peak = bf16_peak if c.mode == "bf16" else fp8_peak
        per[d["name"]] = {
            "mode": c.mode, "M": c.M, "N": c.N, "K": c.K,
            "us": round(us, 2), "us_min": round(1e3 * min(ms), 2),
            "tflops": round(tf, 1),
            "frac_peak": round(tf / peak, 3),
            "frac_peak_burst": round(tf / (peaks["bf16_tflops"] if c.mode == "bf16" else fp8_peak_burst), 3),
            "frac_peak_sustained": round(tf / (peaks["bf16_tflops_sustained"] if c.mode == "bf16" else fp8_peak_sustained), 3),
            "gbs": round(byts / (us * 1e-6) / 1e9, 1),
            "frac_hbm": round(byts / (us * 1e-6) / 1e9 / hbm, 3),
            "tile": "%dx%d" % (d["cfg"]["bm"], d["cfg"]["bn"]), "grid": d["cfg"]["grid"],
        }

    # dominant kernel: the one with the largest share of the step's device time
    # (the ptpc pair kernel); its launch with the most work is reported
    share = {}
    for k, v in per.items():
        share[v["mode"]] = share.get(v["mode"], 0.0) + v["us"]
    dom_mode = max(share, key=share.get)
    dom = max((k for k in per if per[k]["mode"] == dom_mode), key=lambda k: per[k]["M"] * per[k]["N"] * per[k]["K"])
    pc = per[dom]
    dom_flops = 2.0 * pc["M"] * pc["N"] * pc["K"]
    achieved = dom_flops / (pc["us"] * 1e-6) / 1e12
    dom_peak = bf16_peak if pc["mode"] == "bf16" else fp8_peak
    # the same kernel over all of its launches in the step (every workload it runs)
    dom_all = [k for k in per if per[k]["mode"] == dom_mode]
    all_flops = sum(2.0 * per[k]["M"] * per[k]["N"] * per[k]["K"] for k in dom_all)
    all_us = sum(per[k]["us"] for k in dom_all)
    achieved_all = all_flops / (all_us * 1e-6) / 1e12
    traffic = stored_traffic(dom)
    roofline = {
        "bound": "tensor", "achieved": round(achieved, 1), "peak": round(dom_peak, 1), "unit": "TFLOP/s",
        "frac": round(achieved / dom_peak, 3), "traffic": traffic,
        "kernel": kernel_name(pc["mode"], pc["K"]),
        "workload": dom,
        "achieved_all_launches": round(achieved_all, 1),
        "frac_all_launches": round(achieved_all / dom_peak, 3),
        "launches_per_step": len(dom_all),
        "peak_source": "%s: 2 x bf16_tflops%s (fp8 = 2 x bf16 nominal ratio); %s peak because %s" % (
            peak_kind, "" if peak_kind_run == "burst" else "_sustained", peak_kind_run, peak_why),
    }

    # bad launches: 20 launches per workload into NaN-poisoned outputs followed by
    # a guard tail, each bit-identical to the first, NaN-free and leaving the tail
    # untouched (parity against the oracle is in tests/)
    bad = 0
    with torch.cuda.stream(stream):
        for d in ([] if args.no_bad_check else work):
            c = d["case"]
            buf = torch.empty(c.M * c.N + 4096, dtype=torch.int16, device=dev)
            Cg, tail = buf[: c.M * c.N].view(c.M, c.N), buf[c.M * c.N:]
            tail.fill_(0x5A5A)
            first = None
            for _ in range(20):
                Cg.fill_(0x7FC0)
                launch(d, Cg.view(torch.bfloat16))
                isnan = torch.isnan(Cg.view(torch.bfloat16)).any()
                ok = (not bool(isnan)) and bool((tail == 0x5A5A).all())
                if first is None:
                    first = Cg.clone()
                else:
                    ok = ok and torch.equal(Cg, first)
                bad += 0 if ok else 1
            del first, buf
    torch.cuda.synchronize()
    status_bad = 0
    for d in work:
        code, _ = binding.scaled_gemm_debug_status(d["h"], sraw)
        status_bad += code != 0

    if not args.no_graph:
        for d in work:
            if per[d["name"]]["us"] < GRAPH_MAX_US:
                per[d["name"]]["graph"] = graph_per_call(lambda d=d: launch(d), stream, gpu_index=local)

    quant = None if args.no_quant else run_quantize(binding, dev, stream, hbm)
    extra = None if (args.no_quant or args.only) else run_extra(binding, dev, stream, local, fp8_peak_burst)

    # end to end through the C ABI with host buffers: H2D inputs, GEMM, D2H C
    e2e = None if args.no_e2e else run_e2e(work, launch, stream, args, control, dev)

    cpu = None
    if rank == 0 and control.world == 1 and not args.no_cpu_baseline:
        v, dt, cores, fl = cpu_baseline(cases, args.cpu_rows)
        cpu = {
            "value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
            "sample": "rows [0,%d) of every suite workload (%.1f GFLOP, %.1f s)" % (args.cpu_rows, fl / 1e9, dt),
            "c0_one_core": c0_one_core(),
        }

    for d in work:
        binding.scaled_gemm_destroy(d["h"])

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": control.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * t_max / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 x e4m3 (bf16 x bf16 for the BF16 GEMM), fp32 accumulate, bf16 out",
        "data": "synthetic (seeded normals quantised per the workload's scale mode)",
        "config": {
            "workload": "suite: " + ", ".join(name for name, _ in cases) + (" (M=%d)" % args.rows if args.rows else ""),
            "parallelism": "replicas" if control.world > 1 else "single GPU",
            "l2": "inputs larger than L2 (suite operands %.2f GB; each GEMM's operands last touched one full step earlier)"
            % (sum(d["A"].numel() * d["A"].element_size() + d["B"].numel() * d["B"].element_size() for d in work) / 1e9),
        },
        "roofline": roofline,
        "quantize": quant,
        "extra": extra,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": clk,
        "gpu_launches": args.steps * sum(KERNELS_PER_LAUNCH.get(d["case"].mode, 1) for d in work),
        "bad_launches": {"per_workload": 0 if args.no_bad_check else 20, "workloads": n, "bad": bad,
                         "checks": "NaN-free, bit-identical to the first launch, 4096-element guard tail untouched",
                         "watchdog_timeouts": status_bad},
        "per_config": per,
        "wall_s_timed": round(wall1 - wall0, 4),
        "peaks": {"source": peak_kind, "used": peak_kind_run, "fp8_tflops_sustained": fp8_peak_sustained,
                  "fp8_tflops_burst": fp8_peak_burst, "bf16_tflops_sustained": peaks["bf16_tflops_sustained"],
                  "bf16_tflops_burst": peaks["bf16_tflops"], "hbm_gbs": hbm},
    }
    return line


# Kernels one scaled_gemm_launch enqueues: mxfp8 rearranges its scales first.
KERNELS_PER_LAUNCH = {"mxfp8": 2}


def kernel_name(mode, K):
    """The kernel that runs a (mode, K) launch."""
    if mode == "mxfp8":
        return "mxfp8_pair_kernel"
    if mode == "blockscale":
        return "blockscale_pair_kernel"
    return "dense_pair_kernel<%s>" % mode


def run_extra(binding, dev, stream, local, fp8_peak_burst, iters=20):
    """Shapes outside the suite (not part of `value`), each timed on its own:
    3 warm-up launches, then `iters` launches between CUDA events; inputs plus
    output are larger than L2.  Includes the gather-GEMM workload (16384 rows
    gathered from a 65536-row paged cache, N = 8192, K = 512) through
    scaled_gemm_launch_gather."""
    out = {}
    sraw = stream.cuda_stream
    for name in synth.EXTRA:
        mode, M, N, K, seed, a_std, b_std = synth.CONFIGS[name]
        c = synth.make_case(mode, M, N, K, seed=seed, a_std=a_std, b_std=b_std)
        A, B = c.A.to(dev), c.B.to(dev)
        sa, sb = c.sa.to(dev), c.sb.to(dev)
        C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        h = binding.scaled_gemm_create(mode, N, K, M, local)
        f = lambda: binding.scaled_gemm_launch(h, A.data_ptr(), B.data_ptr(), sa.data_ptr(), sb.data_ptr(),  # noqa: E731
                                               C.data_ptr(), M, sraw)
        with torch.cuda.stream(stream):
            for _ in range(3):
                f()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(iters):
                f()
            e1.record(stream)
        torch.cuda.synchronize()
        us = 1e3 * e0.elapsed_time(e1) / iters
        tf = c.flops / (us * 1e-6) / 1e12
        out[name] = {"mode": mode, "M": M, "N": N, "K": K, "us": round(us, 2), "tflops": round(tf, 1),
                     "frac_peak_burst": round(tf / fp8_peak_burst, 3), "kernel": kernel_name(mode, K)}
        binding.scaled_gemm_destroy(h)
        del A, B, sa, sb, C
    for name, (M, R, N, K, seed) in synth.GATHER_CONFIGS.items():
        c = synth.make_gather_case(M, R, N, K, seed=seed)
        A, sa, idx = c.A_src.to(dev), c.sa_src.to(dev), c.idx.to(dev)
        B, sb = c.B.to(dev), c.sb.to(dev)
        C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        h = binding.scaled_gemm_create("ptpc", N, K, M, local)
        f = lambda: binding.scaled_gemm_launch_gather(h, A.data_ptr(), R, idx.data_ptr(), B.data_ptr(),  # noqa: E731
                                                      sa.data_ptr(), sb.data_ptr(), C.data_ptr(), M, sraw)
        with torch.cuda.stream(stream):
            for _ in range(3):
                f()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(iters):
                f()
            e1.record(stream)
        torch.cuda.synchronize()
        us = 1e3 * e0.elapsed_time(e1) / iters
        tf = c.flops / (us * 1e-6) / 1e12
        byts = M * K + N * K + 2.0 * M * N + 4.0 * (2 * M + N)  # gathered A, B, C, a/b scales, idx
        out[name] = {"mode": "ptpc gather", "M": M, "N": N, "K": K, "R": R, "us": round(us, 2),
                     "tflops": round(tf, 1), "frac_peak_burst": round(tf / fp8_peak_burst, 3),
                     "gbs": round(byts / (us * 1e-6) / 1e9, 1), "kernel": "gather_gemm_kernel"}
        binding.scaled_gemm_destroy(h)
        del A, sa, idx, B, sb, C
    return out


def run_quantize(binding, dev, stream, hbm, R=32768, C=7168, iters=20):
    """The quantisation step before the GEMM, timed on its own (not part of the
    suite value): the largest activation of the workloads, R x C bf16, in every
    mode.  HBM-bound: algorithmic bytes = 2RC read + RC written + the scales."""
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    x = torch.randn(R, C, generator=g, device=dev, dtype=torch.float32).bfloat16()
    out = {}
    sraw = stream.cuda_stream
    for mode in ("ptpc", "blockscale", "mxfp8"):
        q = torch.empty((R, C), dtype=torch.uint8, device=dev)
        if mode == "ptpc":
            sc = torch.empty(R, dtype=torch.float32, device=dev)
        elif mode == "blockscale":
            sc = torch.empty((C // 128, R), dtype=torch.float32, device=dev)
        else:
            sc = torch.empty((C // 32, R), dtype=torch.uint8, device=dev)
        f = lambda: binding.scaled_gemm_quantize(mode, "bf16", x.data_ptr(), R, C, q.data_ptr(), sc.data_ptr(), sraw)  # noqa: E731
        with torch.cuda.stream(stream):
            for _ in range(3):
                f()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(iters):
                f()
            e1.record(stream)
        torch.cuda.synchronize()
        us = 1e3 * e0.elapsed_time(e1) / iters
        byts = 3.0 * R * C + sc.numel() * sc.element_size()
        gbs = byts / (us * 1e-6) / 1e9
        out[mode] = {"us": round(us, 2), "gbs": round(gbs, 1), "frac_hbm": round(gbs / hbm, 3)}
    out["workload"] = "%dx%d bf16 -> e4m3 + scales, %d launches per mode, inputs larger than L2" % (R, C, iters)
    return out


def run_e2e(work, launch, stream, args, control, dev):
    """The suite end to end through the C ABI with pinned host buffers.

    Per step and workload: H2D copy of its inputs, the GEMM, D2H copy of its C.
    Copy streams (each copy split over `--e2e-split` of them, so several copy
    engines work at once) overlap the copies of one workload with the GEMMs of
    its neighbours; events keep each workload's device buffers from being
    refilled (or its C overwritten) before the previous use has finished.
    """
    steps = max(1, args.e2e_steps)
    host_in, host_out = [], []
    h2d = d2h = 0
    for d in work:
        ins = []
        for key in ("A", "B", "sa", "sb"):
            t = d[key]
            if t is None:
                ins.append(None)
                continue
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            ins.append(h)
            h2d += t.numel() * t.element_size()
        host_in.append(ins)
        host_out.append(torch.empty(d["C"].shape, dtype=d["C"].dtype, pin_memory=True))
        d2h += d["C"].numel() * d["C"].element_size()
    torch.cuda.synchronize()
    nsplit = max(1, args.e2e_split)
    s_in = [torch.cuda.Stream(dev) for _ in range(nsplit)]
    s_out = [torch.cuda.Stream(dev) for _ in range(nsplit)]
    n = len(work)
    in_done, gemm_done, out_done = [None] * n, [None] * n, [None] * n

    def chunks(t):
        flat = t.view(-1)
        step_ = (flat.numel() + nsplit - 1) // nsplit
        return [flat[j * step_:(j + 1) * step_] for j in range(nsplit)]

    def step():
        for i, (d, ins, out) in enumerate(zip(work, host_in, host_out)):
            # inputs: every tensor split over the copy streams
            done = []
            for j, q in enumerate(s_in):
                with torch.cuda.stream(q):
                    if gemm_done[i] is not None:
                        q.wait_event(gemm_done[i])  # previous GEMM i has read its inputs
                    for key, h in zip(("A", "B", "sa", "sb"), ins):
                        if h is not None:
                            chunks(d[key])[j].copy_(chunks(h)[j], non_blocking=True)
                    e = torch.cuda.Event()
                    e.record(q)
                    done.append(e)
            in_done[i] = done
            with torch.cuda.stream(stream):
                for e in in_done[i]:
                    stream.wait_event(e)
                for e in out_done[i] or []:
                    stream.wait_event(e)  # previous C i has been copied out
                launch(d)
                gemm_done[i] = torch.cuda.Event()
                gemm_done[i].record(stream)
            done = []
            for j, q in enumerate(s_out):
                with torch.cuda.stream(q):
                    q.wait_event(gemm_done[i])
                    chunks(out)[j].copy_(chunks(d["C"])[j], non_blocking=True)
                    e = torch.cuda.Event()
                    e.record(q)
                    done.append(e)
            out_done[i] = done

    step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    control.barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for q in s_in + s_out:
        q.wait_event(e0)
    for _ in range(steps):
        step()
    for q in s_in + s_out:
        j = torch.cuda.Event()
        j.record(q)
        stream.wait_event(j)
    e1.record(stream)
    torch.cuda.synchronize()
    control.barrier()
    secs = e0.elapsed_time(e1) / 1e3
    flops = steps * sum(d["case"].flops for d in work)
    _, _, v = aggregate(control, flops, secs)
    return {"value": round(v, 1), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "ms_per_step": round(1e3 * secs / steps, 3),
            "pipeline": "H2D / GEMM / D2H overlapped across workloads; each copy split over %d streams" % nsplit}


def stored_traffic(workload):
    """DRAM bytes per launch of `workload` from profiles/traffic.txt, if they were
    measured on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    rev = kernel_revision(synth.CONFIGS[workload][0])
    for line in open(path):
        f = line.split()
        if len(f) >= 3 and not line.startswith("#") and f[0] == workload and f[1] == rev:
            return float(f[2])
    return None


KERNEL_FILES = {
    "ptpc": ["sg_dense.cu", "sg_common.cuh", "sg_ptx.cuh"],
    "bf16": ["sg_dense.cu", "sg_common.cuh", "sg_ptx.cuh"],
    "mxfp8": ["sg_mxfp8.cu", "sg_common.cuh", "sg_ptx.cuh"],
    "blockscale": ["sg_blockscale.cu", "sg_common.cuh", "sg_ptx.cuh"],
}


def kernel_revision(mode="ptpc"):
    """Hash of the CUDA sources of one kernel family, to tell whether stored
    counters still apply to the code that runs."""
    import hashlib

    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "fp8_scaled_gemm_sm_gb300", "csrc")
    for f in KERNEL_FILES[mode]:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:12]


# --------------------------------------------------------------------------- reference arm


def run_reference(args, control, rank):
    if rank != 0:
        return None
    cases = make_suite()
    rows = args.ref_rows
    times, flops = [], 0.0
    for s in range(args.warmup + args.steps):
        v, dt, cores, fl = cpu_baseline(cases, rows)
        if s >= args.warmup:
            times.append(dt)
            flops = fl
    t = sum(times)
    value = flops * len(times) / t / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": control.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * t / len(times), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 (CPU oracle: exact e4m3/e8m0 decode, binary64 accumulation)",
        "data": "synthetic (seeded normals quantised per the workload's scale mode)",
        "config": {"workload": "suite: " + ", ".join(synth.SUITE), "sample": "rows [0,%d) of every workload per step" % rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "rows [0,%d) of every suite workload per step" % rows},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-split", type=int, default=1, help="copy streams per direction in the e2e leg")
    ap.add_argument("--cpu-rows", type=int, default=1536)
    ap.add_argument("--ref-rows", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (profiling runs)")
    ap.add_argument("--no-quant", action="store_true", help="skip the quantisation measurement (profiling runs)")
    ap.add_argument("--no-bad-check", action="store_true", help="skip the 20-launch check (profiling runs)")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph per-call timing (profiling runs)")
    ap.add_argument("--only", default=None, choices=synth.SUITE + synth.EXTRA, help="one workload (profiling runs)")
    ap.add_argument("--rows", type=int, default=None, help="override M of the workload(s) (profiling runs)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3  # timing rule: at least 3 warm-up steps
    world, rank, local = dist_env()
    control = Control(world)
    try:
        if args.impl == "reference":
            line = run_reference(args, control, rank)
        else:
            line = run_gpu(args, control, rank, local)
    finally:
        control.close()
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
