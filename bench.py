"""Benchmark: training steps/s and achieved TFLOP/s per step on one GB300.

A step is one full training step of the workload (forward, loss, backward,
optimizer) through the C ABI (libmg.so).  Default workload: the large GELU MLP
(4096-4096-4096-4096-1000, batch 8192, bf16, Adam) -- the configuration the
throughput target is quoted on.  ``--config`` selects another workload.

Prints one JSON line (rank 0).  Under torchrun each rank runs an independent
replica on its own GPU (the step has no exchange: replicas only), timing is the
max over ranks, and ``value`` is the total steps/s of all ranks.

``--impl reference`` times the CPU oracle (float64 numpy) on a bounded row
sample of the same workload instead: the reference arm.
"""
from __future__ import annotations

import argparse
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

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of a
# kernel family, averaged over the launches of one training step, from one ncu
# capture of the current code (summary and command under profiles/); keyed by
# (workload, family); absent when not captured for that pair, or when the
# kernel has changed since its capture.
TRAFFIC = {
    # profiles/gemm_pair_c3_step_dram_traffic.md: eleven launches of one step
    ("c3_mlp4096_gelu", "gemm_pair_kernel (tcgen05 cta_group::2)"): 246.9e6,
}

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


class NvmlSampler:
    """SM clock and clock-event reasons read through NVML (read-only queries)
    every ~2 ms from a background thread while the timed region runs."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_index):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        bus = None
        try:   # NVML numbers GPUs on its own; match the CUDA device by PCI address
            import torch
            pr = torch.cuda.get_device_properties(gpu_index)
            bus = b"%08x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
        except Exception:
            bus = None
        if bus is None or self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(self.h)) != 0:
            if self.lib.nvmlDeviceGetHandleByIndex_v2(int(gpu_index), ctypes.byref(self.h)) != 0:
                raise RuntimeError("no NVML handle")
        self.samples, self.reasons = [], set()
        self.stop_flag = False
        self.thread = None

    def _one(self):
        ct = self.ct
        clk, mx, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(clk))          # NVML_CLOCK_SM
        self.max = self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ct.byref(mx)) == 0 and mx.value
        f = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        if f(self.h, ct.byref(rs)) == 0:
            for bit, name in self.REASONS.items():
                if rs.value & bit:
                    self.reasons.add(name)
        self.samples.append(clk.value)

    def _run(self):
        while not self.stop_flag:
            self._one()
            time.sleep(0.002)

    def start(self):
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def stop(self):
        self.stop_flag = True
        self.thread.join(timeout=2)
        self._one()
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max or None, "reasons": sorted(self.reasons),
                "samples": len(self.samples), "source": "nvml"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm = [float(r[1]) for r in self.rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in self.rows:
            if len(r) < 9:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(self.rows)}


def kernel_family(site_name: str) -> str:
    """The CUDA kernel a schedule entry launches, from its name."""
    n = site_name
    if n.startswith(("fwd[", "dX[", "dW[")):
        if "tcgen05x2" in n:
            return "gemm_pair_kernel (tcgen05 cta_group::2)"
        if "tcgen05" in n:
            return "gemm_tc_kernel (tcgen05)"
        if "f32-ffma" in n:
            return "gemm_simt (fp32 FFMA)"
        if "skinny" in n:
            return "gemm_skinny (bf16, narrow side in shared memory)"
        return "gemm_simt (bf16)"
    if n.startswith("attn_fwd"):
        return "attn_fwd" + (" (tcgen05)" if "tcgen05" in n else " (simt)")
    if n.startswith("attn_bwd"):
        return "attn_bwd dq+dkdv" + (" (tcgen05)" if "tcgen05" in n else " (simt)")
    return n.split("[")[0].split(" ")[0]


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def workload_for(key, precision):
    from static_graph_nn_gb300 import workloads as W
    w = W.workload(key)
    if precision is None:
        precision = "bf16" if "bf16" in w.precisions else w.precisions[0]
    return w, precision


def _oracle_inputs(w):
    import numpy as np

    from static_graph_nn_gb300 import workloads as W
    p0 = W.init_params(w)
    return p0, W.make_x(w), W.make_labels(w), [np.zeros_like(a) for a in p0]


def _oracle_rows(w, rows, precision, inputs):
    import oracle
    p0, x, y, z = inputs
    t0 = time.perf_counter()
    oracle.train_step(w.layers, p0, x[:rows], y[:rows], w.loss, precision, w.optimizer, w.lr, 1,
                      z, z, w.beta1, w.beta2, w.adam_eps)
    return time.perf_counter() - t0


def calibrate_rows(w, precision, inputs, target_s):
    """Largest row sample (doubling, a multiple of the attention sequence) whose
    oracle step stays near target_s seconds."""
    unit = 1
    for l in w.layers:
        if l["op"] == "causal_attention":
            unit = l["seq_len"]
    rows = max(unit, min(w.batch, 32))
    while rows < w.batch:
        dt = _oracle_rows(w, rows, precision, inputs)
        if dt * 2.2 > target_s:
            break
        rows = min(w.batch, rows * 2)
    return rows


def cpu_oracle_sample(w, precision, target_s=12.0):
    """Times the oracle as it stands on a row sample of the workload.  Returns
    (seconds per full step extrapolated by rows, rows sampled, threads)."""
    inputs = _oracle_inputs(w)
    rows = calibrate_rows(w, precision, inputs, target_s)
    dt = _oracle_rows(w, rows, precision, inputs)
    return dt * w.batch / rows, rows, os.cpu_count()


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w, prec = workload_for(args.config, args.precision)
    inputs = _oracle_inputs(w)
    per_step = min(10.0, 150.0 / max(1, args.steps + args.warmup))
    rows = calibrate_rows(w, prec, inputs, per_step)
    times = [_oracle_rows(w, rows, prec, inputs) * w.batch / rows
             for _ in range(args.warmup + args.steps)]
    sec = statistics.mean(times[args.warmup:] or times)
    value = 1.0 / sec
    flops = w.flops_per_step()
    line = {
        "impl": "reference", "metric": "training steps/s (achieved TFLOP/s per step)",
        "value": value, "unit": "steps/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "precision": prec,
                   "optimizer": w.optimizer},
        "tflops": flops / sec / 1e12,
        "cpu_baseline": {"value": value, "unit": "steps/s", "cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": f"each step: the oracle on {rows} of {w.batch} rows, "
                                   f"time scaled by rows"},
        "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def make_plan(w, prec, graph=True):
    """A plan for the workload; graph=False creates it with the step's graph
    replay turned off (MG_GRAPH=0, read at plan creation)."""
    from static_graph_nn_gb300 import Plan
    if graph:
        return Plan.for_workload(w, prec)
    old = os.environ.get("MG_GRAPH")
    os.environ["MG_GRAPH"] = "0"
    try:
        return Plan.for_workload(w, prec)
    finally:
        if old is None:
            del os.environ["MG_GRAPH"]
        else:
            os.environ["MG_GRAPH"] = old


class Session:
    """One workload's plan and its device and pinned host buffers."""

    def __init__(self, w, prec):
        import torch

        from static_graph_nn_gb300 import workloads as W
        self.w, self.prec = w, prec
        t0 = time.perf_counter()
        self.plan = make_plan(w, prec)
        self.create_ms = (time.perf_counter() - t0) * 1e3
        p0 = W.init_params(w)
        flat = torch.zeros(self.plan.param_count, dtype=torch.float32)
        for (off, r, c), t in zip(self.plan.param_info(), p0):
            flat[off:off + r * c] = torch.from_numpy(t.reshape(-1))
        self.params = flat.cuda()
        self.grads = torch.zeros_like(self.params)
        self.m = torch.zeros_like(self.params) if w.optimizer in ("adam", "laprop", "sgd_momentum") else None
        self.v = torch.zeros_like(self.params) if w.optimizer in ("adam", "laprop") else None
        xt = torch.from_numpy(W.make_x(w))
        if prec == "bf16":
            xt = xt.to(torch.bfloat16)
        yt = torch.from_numpy(W.make_labels(w))
        if w.loss == "mse" and prec == "bf16":
            yt = yt.to(torch.bfloat16)
        self.x_host = xt.contiguous().pin_memory()
        self.y_host = yt.contiguous().pin_memory()
        self.x_dev = self.x_host.cuda()
        self.y_dev = self.y_host.cuda()
        self.stream = torch.cuda.current_stream()
        self.step = 0

    def one_step(self, plan=None, x=None, y=None):
        self.step += 1
        (plan or self.plan).train_step(self.params, self.grads, self.m, self.v,
                                       self.x_dev if x is None else x,
                                       self.y_dev if y is None else y, self.w.lr, self.step,
                                       self.stream)

    def close(self):
        self.plan.close()


def time_reps(sess, plan, steps, reps, dist):
    """reps timed regions of `steps` steps each (device-resident inputs, CUDA
    events on the launching stream, a barrier and a synchronize on both
    sides); milliseconds per region."""
    import torch
    out = []
    for _ in range(reps):
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(sess.stream)
        for _ in range(steps):
            sess.one_step(plan)
        ev1.record(sess.stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        out.append(ev0.elapsed_time(ev1))
    return out


def time_e2e(sess, steps, warmup, dist):
    """Seconds per step end to end: a training loop as a user pipelines it.
    Every step's inputs are copied from pinned host memory on a copy stream
    into one of two device buffers while the previous step computes, and every
    step's loss (with the pipeline's error flag) is copied back and read on the
    host one step later, so the copies overlap the compute and the host
    enqueues the next step while the GPU runs this one."""
    import torch
    plan, stream = sess.plan, sess.stream
    e2e_steps = max(10, steps)
    e2e_warm = max(4, warmup)
    total = e2e_warm + e2e_steps
    copy_stream = torch.cuda.Stream()
    xb = [sess.x_dev, torch.empty_like(sess.x_dev)]
    yb = [sess.y_dev, torch.empty_like(sess.y_dev)]
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(total)]
    loss_host = torch.zeros(total, 2, dtype=torch.float32).pin_memory()
    losses = []
    x_host, y_host = sess.x_host, sess.y_host
    # inputs under 1 MiB are copied on the compute stream itself: their copy is
    # shorter than the cross-stream synchronisation it would overlap with
    overlap = (x_host.numel() * x_host.element_size() + y_host.numel() * y_host.element_size()
               >= 1 << 20)

    def enqueue_copy(t):
        b = t & 1
        if not overlap:
            return
        with torch.cuda.stream(copy_stream):
            if t >= 2:
                copy_stream.wait_event(consumed[b])   # step t-2 is done reading buffer b
            xb[b].copy_(x_host, non_blocking=True)
            yb[b].copy_(y_host, non_blocking=True)
            copied[b].record(copy_stream)

    # the loop's first e2e_warm steps are untimed warm-up (each buffer's step
    # graph is captured on its second use); the clock starts at the step after
    t0 = None
    enqueue_copy(0)
    for t in range(total):
        if t == e2e_warm:
            torch.cuda.synchronize()
            if dist:
                dist.barrier()
            t0 = time.perf_counter()
            enqueue_copy(t)
        if t + 1 < total and t + 1 != e2e_warm:
            enqueue_copy(t + 1)
        b = t & 1
        if overlap:
            stream.wait_event(copied[b])
        else:
            xb[b].copy_(x_host, non_blocking=True)    # on the compute stream
            yb[b].copy_(y_host, non_blocking=True)
        sess.one_step(plan, xb[b], yb[b])
        if overlap:
            consumed[b].record(stream)
        plan.loss_async(loss_host[t].data_ptr(), stream)
        done[t].record(stream)
        if t > e2e_warm:
            done[t - 1].synchronize()
            losses.append(float(loss_host[t - 1, 0]))
    done[total - 1].synchronize()
    losses.append(float(loss_host[total - 1, 0]))
    sec = (time.perf_counter() - t0) / e2e_steps
    if any(loss_host.view(torch.int32)[:, 1].tolist()) or not all(map(math.isfinite, losses)):
        raise RuntimeError("end-to-end steps reported a timed-out pipeline or a non-finite loss")
    h2d = x_host.numel() * x_host.element_size() + y_host.numel() * y_host.element_size()
    return sec, h2d


def pick_peak(prec, peaks, peak_src, clk, ffma):
    """The roofline denominator: the strict path's measured FFMA rate; for bf16
    the measured burst peak when the timed region ran at full clock with no
    power cap (short steps between idle gaps), the sustained peak otherwise."""
    if prec != "bf16":
        return "alu", "TFLOP/s", ffma, "FP32 FFMA peak measured by mg_ffma_peak in this run"
    capped = "sw_power_cap" in (clk.get("reasons") or []) or (
        clk.get("sm_mhz") and clk.get("sm_max_mhz") and clk["sm_mhz"] < 0.95 * clk["sm_max_mhz"])
    if capped:
        return ("tensor", "TFLOP/s", peaks.get("bf16_tflops_sustained", 1700.0),
                f"sustained bf16 peak ({peak_src}): the timed region ran power-capped or below "
                f"95% of the maximum SM clock")
    return ("tensor", "TFLOP/s", peaks.get("bf16_tflops", 1900.0),
            f"burst bf16 peak ({peak_src}): the timed region ran at full clock with no power cap")


def measure(w, prec, args, dist, world, rank, local, peaks, peak_src, ffma, reps=5):
    """Everything the JSON line reports for one workload."""
    import torch

    from static_graph_nn_gb300.replicas import job_throughput, max_over_ranks
    sess = Session(w, prec)
    for _ in range(args.warmup):
        sess.one_step()
    torch.cuda.synchronize()

    # ---- timed region: device-resident inputs, the steps as a user runs
    # them (from the second call on, each step is a CUDA-graph replay);
    # `reps` repetitions, the median reported ----
    try:
        clocks = NvmlSampler(local)
    except Exception:
        clocks = ClockSampler(local)
    clocks.start()
    replays0 = sess.plan.graph_replays()
    first = time_reps(sess, sess.plan, args.steps, 1, dist)
    replays = sess.plan.graph_replays() - replays0
    launches = sess.plan.last_launch_count() * args.steps
    clk = clocks.stop()
    # the measurement protocol's repetitions: the first region and `reps` - 1
    # more, with graph replay, then `reps` with every kernel launched directly
    reps_graph = first + time_reps(sess, sess.plan, args.steps, reps - 1, dist)

    # the same repetitions with every kernel launched directly (a second plan
    # created with graph replay off, on the same buffers)
    plan_ng = make_plan(w, prec, graph=False)
    for _ in range(2):
        sess.one_step(plan_ng)
    reps_direct = time_reps(sess, plan_ng, args.steps, reps, dist)
    plan_ng.close()

    # ---- kernel timing: the same K steps again, launched directly with a
    # CUDA event pair around every kernel on the stream it runs on ----
    sess.plan.profile_begin(args.steps)
    ev2 = torch.cuda.Event(enable_timing=True)
    ev3 = torch.cuda.Event(enable_timing=True)
    ev2.record(sess.stream)
    for _ in range(args.steps):
        sess.one_step()
    ev3.record(sess.stream)
    torch.cuda.synchronize()
    ms_prof = ev2.elapsed_time(ev3)
    prof = sess.plan.profile_end()
    loss = sess.plan.loss(sess.stream)

    e2e_s, h2d = time_e2e(sess, args.steps, args.warmup, dist)

    ms = first[0]
    ms_med = statistics.median(reps_graph)
    ms_direct = statistics.median(reps_direct)
    ms, ms_med, ms_direct, e2e_s = max_over_ranks([ms, ms_med, ms_direct, e2e_s], device="cuda")
    ms_step = ms / args.steps
    flops = w.flops_per_step()
    bound, unit, peak, peak_note = pick_peak(prec, peaks, peak_src, clk, ffma)
    hbm_peak = peaks.get("hbm_gbs", 6800.0)

    # dominant kernel: schedule entries grouped by the kernel they launch (the
    # view of the ncu launch list); achieved = algorithmic work per launch /
    # average launch duration, i.e. the group's work / its time
    fam = {}
    for e in prof:
        k = kernel_family(e["name"])
        f = fam.setdefault(k, {"name": k, "launches": 0, "total_ms": 0.0, "flops": 0.0, "bytes": 0.0})
        f["launches"] += e["launches"]
        f["total_ms"] += e["total_ms"]
        f["flops"] += e["flops"] * e["launches"]
        f["bytes"] += e["bytes"] * e["launches"]
    top = max(fam.values(), key=lambda f: f["total_ms"])
    if top["flops"] > 0:
        achieved = top["flops"] / (top["total_ms"] * 1e-3) / 1e12
    else:
        bound, unit, peak, peak_note = "hbm", "GB/s", hbm_peak, f"HBM copy bandwidth ({peak_src})"
        achieved = top["bytes"] / (top["total_ms"] * 1e-3) / 1e9
    total_prof = sum(e["total_ms"] for e in prof)
    kernels = [{"name": e["name"], "share": e["total_ms"] / total_prof if total_prof else None,
                "avg_ms": e["total_ms"] / max(1, e["launches"]),
                "tflops": (e["flops"] / (e["total_ms"] / max(1, e["launches"]) * 1e-3) / 1e12)
                if e["flops"] and e["total_ms"] else None,
                "gbs": (e["bytes"] / (e["total_ms"] / max(1, e["launches"]) * 1e-3) / 1e9)
                if e["total_ms"] else None}
               for e in sorted(prof, key=lambda e: -e["total_ms"])[:8]]
    out = {
        "value": job_throughput(world, args.steps, ms * 1e-3),
        "ms_per_step": ms_step,
        "dtype": prec if prec == "bf16" else "f32",
        "config": {"workload": w.name, "batch": w.batch, "precision": prec,
                   "optimizer": w.optimizer, "flops_per_step": flops,
                   "parallelism": f"replicas x{world}",
                   "l2": "working set per step >> 129 MB L2 (weights, activations, optimizer "
                         "state); no flush between steps"},
        "tflops": flops / (ms_step * 1e-3) / 1e12,
        "pct_of_peak": flops / (ms_step * 1e-3) / 1e12 / peak if bound != "hbm" else None,
        "roofline": {"kernel": top["name"], "launches_timed": top["launches"],
                     "share": top["total_ms"] / total_prof if total_prof else None,
                     "bound": bound, "achieved": achieved, "peak": peak,
                     "unit": unit, "frac": achieved / peak,
                     "traffic": TRAFFIC.get((w.name, top["name"])),
                     "peak_note": peak_note},
        "repetitions": {"how": f"{reps} timed regions of {args.steps} steps each, back to back, "
                               f"with graph replay (the first is the headline region) and "
                               f"with every kernel launched directly; medians",
                        "graph_ms_per_step": [r / args.steps for r in reps_graph],
                        "direct_ms_per_step": [r / args.steps for r in reps_direct],
                        "graph_median_value": job_throughput(world, args.steps, ms_med * 1e-3),
                        "direct_median_value": job_throughput(world, args.steps, ms_direct * 1e-3)},
        "kernels": kernels,
        "kernel_families": [{"kernel": f["name"], "launches": f["launches"],
                             "share": f["total_ms"] / total_prof if total_prof else None,
                             "tflops": f["flops"] / (f["total_ms"] * 1e-3) / 1e12 if f["flops"] and f["total_ms"] else None,
                             "gbs": f["bytes"] / (f["total_ms"] * 1e-3) / 1e9 if f["total_ms"] else None}
                            for f in sorted(fam.values(), key=lambda f: -f["total_ms"])],
        "gpu_launches": launches,
        "graph_replays_timed": replays,
        "kernel_timing": {"steps": args.steps, "ms_per_step": ms_prof / args.steps,
                          "how": "the K steps after the timed region, launched directly with a "
                                 "CUDA event pair around every kernel (roofline and kernels)"},
        "loss": loss,
        "clocks": clk,
        "e2e": {"value": job_throughput(world, 1, e2e_s), "unit": "steps/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 8},
        "plan_workspace_bytes": sess.plan.workspace_bytes,
        "plan_create_ms": sess.create_ms,
    }
    sess.close()
    return out


def plan_create_times(reps=3):
    """Wall time of mg_step_plan_create (validation, layout, schedule, the
    workspace allocation) for every workload, the median of `reps`; the
    pages' counterpart is the session's compile time."""
    from static_graph_nn_gb300 import Plan
    from static_graph_nn_gb300 import workloads as W
    out = {}
    for key in ("c1", "c2", "c3", "c4", "c5"):
        w = W.workload(key)
        for prec in w.precisions:
            ts = []
            for _ in range(reps):
                t0 = time.perf_counter()
                p = Plan.for_workload(w, prec)
                ts.append((time.perf_counter() - t0) * 1e3)
                p.close()
            out[f"{w.name}/{prec}"] = statistics.median(ts)
    return out


EXTRA = {"c3": ("c5", "c4")}   # the default run also times these after the headline


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="c3", choices=["c1", "c2", "c3", "c4", "c5"])
    ap.add_argument("--precision", default=None, choices=[None, "strict", "bf16"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="time only --config (the default run adds the attention and "
                         "residual-network workloads after the large MLP)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)

    import torch

    import __graft_entry__

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if dist:
        dist.barrier()
    from static_graph_nn_gb300 import binding
    binding.load()

    peaks, peak_src = load_peaks()
    w, prec = workload_for(args.config, args.precision)
    ffma = binding.ffma_peak()[0] if prec != "bf16" else None
    head = measure(w, prec, args, dist, world, rank, local, peaks, peak_src, ffma)
    extras = {}
    if not args.no_extra and args.precision in (None, "bf16"):
        for key in EXTRA.get(args.config, ()):
            we, pe = workload_for(key, None)
            extras[we.name] = measure(we, pe, args, dist, world, rank, local, peaks, peak_src, None)
    creates = plan_create_times()
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    line = {
        "metric": "training steps/s (achieved TFLOP/s per step)",
        "value": head["value"], "unit": "steps/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"], "data": "synthetic",
        "config": head["config"], "roofline": head["roofline"], "clocks": head["clocks"],
        "e2e": head["e2e"], "gpu_launches": head["gpu_launches"], "peak_source": peak_src,
    }
    for k, v in head.items():
        line.setdefault(k, v)
    if ffma is not None:
        line["ffma_peak_tflops"] = ffma
    line["plan_create_ms"] = {"this_workload": head["plan_create_ms"], "all": creates,
                              "pages_compile_s": "0.1-2.4 (consumer GPUs, Vulkan/Metal)"}
    if extras:
        line["configs"] = extras
    if not args.no_cpu_baseline and world == 1:
        sec, rows, threads = cpu_oracle_sample(w, prec)
        line["cpu_baseline"] = {"value": 1.0 / sec, "unit": "steps/s", "cores": threads,
                                "kind": "oracle",
                                "sample": f"one oracle step on {rows} of {w.batch} rows, "
                                          f"time scaled by rows"}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
