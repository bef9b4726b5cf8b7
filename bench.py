"""Benchmark of the fused ZeRO update step on one GB300 (or N independent replicas).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload flat1b_n8] [--api plan|step] [--in-place]
                [--staging tma|registers] [--pingpong auto|on|off] [--sequence|--no-sequence]

One step is one pass of the whole hot path over one batch of synthetic
gradients, resident in device memory when the timed region starts:
  - reduce-scatter of the N ranks' gradients with 1/N batch-mean scaling and
    loss-scale removal;
  - the overflow check and the global norm;
  - owner-local Adam on the FP32 master/m/v;
  - the BF16 cast and all-gather into the full working-weight view;
  - the host bookkeeping (step counter, dynamic loss scale).
The default workload is flat1b_n8: 1,000,000,000 parameters, N=8 BF16 ranks,
25,000,000-element buckets, dynamic loss scale from 65536, skip on overflow.
It runs out of place (the plan entry points, as zero_step_into), so the skip
decision needs no second pass, with ping-pong state sets: the device keeps
which of the two sets is current, so a skipped step copies nothing.  The
one-pass kernel stages every 2048-element tile in shared memory with TMA bulk
copies (ZERO_STAGING_TMA); --staging registers times the kernel that loads
straight into registers instead.

The steady-state steps all reuse step 1's gradients.  For a workload with an
injected overflow (flat1b_n8) the line also carries `sequence`: the workload's
own steps as its configuration lists them, fresh gradients each step and the
+inf on step 3, each step timed on its own.

The printed JSON line carries:
  - value: params/s over all GPUs;
  - the dominant kernel's roofline: algorithmic bytes per launch over its
    CUDA-event duration, against the measured HBM copy peak (and, beside it,
    the nominal HBM3e bandwidth);
  - the oracle timed on host cores (cpu_baseline);
  - an end-to-end figure: gradients streamed from pinned host memory through
    two device slots, and the result read back to the host;
  - the SM clocks sampled during the timed region, and the count of this
    library's kernel launches.
Under torchrun each rank runs an independent replica on its own GPU ("replicas
only": the in-device step has no cross-GPU exchange); a gloo group carries
only the barrier and the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "params/sec and achieved HBM GB/s (fraction of GB300 peak) per fused ZeRO step"
UNIT = "params/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e, nominal
# the step kernels' code: the profile summaries are tied to a hash of these
KERNEL_SOURCES = [os.path.join(ROOT, "zero_sharded_mixed_04_gb300", "csrc", f)
                  for f in ("zero_kernels.cuh", "zero_elem.cuh", "zero_common.cuh")]
# the committed ncu summary of each one-pass kernel on the full flat1b_n8 workload
PROFILE_SUMMARY = {
    "zero_fused_kernel": os.path.join(ROOT, "profiles", "zero_fused_kernel_flat1b_n8.md"),
    "zero_fused_staged_kernel": os.path.join(ROOT, "profiles",
                                             "zero_fused_staged_kernel_flat1b_n8.md"),
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="flat1b_n8")
    ap.add_argument("--api", choices=["plan", "step"], default="plan")
    ap.add_argument("--in-place", action="store_true",
                    help="zero_step in place (two passes when skipping) instead of zero_step_into")
    ap.add_argument("--e2e-steps", type=int, default=0, help="0 = min(steps, 10)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--policy", choices=["auto", "host", "device"], default="auto",
                    help="where t and the loss scale are kept: 'device' runs steps back to "
                         "back with no host read in between; 'auto' picks the device when the "
                         "workload skips on overflow or has a dynamic loss scale (otherwise "
                         "no step outcome is needed on the host anyway)")
    ap.add_argument("--host-grad-accum", action="store_true",
                    help="keep the owner's FP32 gradient shard in pinned host memory "
                         "(reached over the host link); forces the two-pass form")
    ap.add_argument("--staging", choices=["registers", "tma"], default="tma",
                    help="how the one-pass kernel reads its inputs: straight into registers, or "
                         "tile by tile into shared-memory stages by TMA bulk copies")
    ap.add_argument("--micro-batches", type=int, default=0,
                    help="accumulate each step's gradient over this many micro-batches "
                         "(reduce-scattered bucket by bucket); 0 = one batch")
    ap.add_argument("--zero3-gather", action="store_true",
                    help="time the ZeRO-3 per-layer gather (two views, one-ahead prefetch) "
                         "over the workload's layers instead of the step")
    ap.add_argument("--zero3-layer-elems", type=int, default=50_000_000,
                    help="layer size for flat workloads in --zero3-gather")
    ap.add_argument("--zero3-side-streams", type=int, choices=[1, 2], default=2,
                    help="--zero3-gather: gather on one side stream (each gather chained to the "
                         "previous) or on one per view (neighbouring layers concurrent)")
    ap.add_argument("--bucket-elems", type=int, default=-1,
                    help="override the workload's bucket size (0: one bucket, the whole vector)")
    ap.add_argument("--ranks", type=int, default=0,
                    help="override the workload's rank count N (for instance k*N, to time one "
                         "pass over every micro-batch's gradients held at once)")
    ap.add_argument("--psi", type=int, default=0,
                    help="reduced parameter count of the same workload (profiling captures "
                         "only; the benchmark line is the full size)")
    ap.add_argument("--pingpong", choices=["auto", "on", "off"], default="auto",
                    help="ping-pong state sets (the device keeps which out-of-place set is "
                         "current, so a skipped step copies nothing and no restore kernel is "
                         "launched); 'auto' uses them for every out-of-place step")
    ap.add_argument("--profile-graph", action="store_true",
                    help="before the timed steps, capture one step as a CUDA graph and replay "
                         "it between cudaProfilerStart/Stop, so that an ncu range capture holds "
                         "one graph launch instead of the step's host calls (needs the device "
                         "policy and ping-pong sets, which keep the step's host state on the "
                         "device)")
    ap.add_argument("--profile-step", type=int, default=-1,
                    help="bracket timed step K (0-based) with cudaProfilerStart/Stop, so that "
                         "ncu --replay-mode app-range measures that "
                         "step's launches as one range, overlapping as they run")
    seq = ap.add_mutually_exclusive_group()
    seq.add_argument("--sequence", dest="sequence", action="store_true", default=None,
                     help="also time the workload's own step sequence (fresh gradients each "
                          "step, the injected overflow included)")
    seq.add_argument("--no-sequence", dest="sequence", action="store_false")
    return ap.parse_args(argv)


def select_workload(args):
    import dataclasses
    from zero_sharded_mixed_04_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    if args.psi:
        wl = dataclasses.replace(wl, name=f"{wl.name}[psi={args.psi}]", psi_flat=args.psi,
                                 tensor_sizes=())
    if args.bucket_elems >= 0:
        wl = dataclasses.replace(wl, name=f"{wl.name}[bucket={args.bucket_elems}]",
                                 bucket_elems=args.bucket_elems)
    if args.ranks:
        wl = dataclasses.replace(wl, name=f"{wl.name}[N={args.ranks}]", N=args.ranks)
    return wl


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class Group:
    """Barrier and max over ranks on a gloo group (control plane only)."""

    def __init__(self, world: int):
        self.world = world
        if world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("gloo")
            self.dist = dist

    def barrier(self):
        if self.world > 1:
            self.dist.barrier()

    def max(self, x: float) -> float:
        if self.world == 1:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t[0])

    def sum(self, x: float) -> float:
        if self.world == 1:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.SUM)
        return float(t[0])

    def close(self):
        if self.world > 1:
            self.dist.destroy_process_group()


# ------------------------------------------------------------------ clocks

CLOCK_FIELDS = ["uuid", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
                "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons every 100 ms."""

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={','.join(CLOCK_FIELDS)}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = []
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(CLOCK_FIELDS):
                continue
            if self.uuid and parts[0] != self.uuid:
                continue
            rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        sm = [num(r[1]) for r in rows]
        mx = [num(r[2]) for r in rows]
        reasons = sorted({REASONS[k] for r in rows for k in range(4) if r[5 + k] == "Active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(num(r[3]) for r in rows)}


# ------------------------------------------------------------------ helpers

def read_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    """sha256 (first 16 hex digits) of the step kernels' code (the kernel file
    and the headers it includes, in that order): comments, trailing spaces and
    blank lines removed, so that a comment edit does not void the profiles
    taken on the same code."""
    text = ""
    for path in KERNEL_SOURCES:
        with open(path) as f:
            text += f.read() + "\n"
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = [re.sub(r"//.*$", "", line).rstrip() for line in text.splitlines()]
    code = "\n".join(line for line in lines if line)
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def profiled_figures(kernel: str) -> dict | None:
    """From a one-pass kernel's committed ncu summary, if it was taken on the
    kernel source as it is now: DRAM bytes per parameter and, when given, the
    serialised duration of one full-size launch under ncu."""
    try:
        text = open(PROFILE_SUMMARY[kernel]).read()
    except OSError:
        return None
    h = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    b = re.search(r"traffic_bytes_per_param:\s*([0-9.]+)", text)
    d = re.search(r"ncu_launch_us:\s*([0-9.]+)", text)
    if not h or not b or h.group(1) != kernel_source_hash():
        return None
    return {"traffic_bytes_per_param": float(b.group(1)),
            "ncu_launch_us": float(d.group(1)) if d else None}


def cpu_model() -> str:
    """The host CPU's model name, as lscpu or /proc/cpuinfo gives it."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine() or "unknown"


def alg_bytes_per_param(wl) -> int:
    """N*g grad reads + 12 state reads + 12 state writes + 2 weight writes."""
    return wl.N * wl.grad_bytes + 26


def cpu_baseline(oracle, wl, grads, master, budget_s: float, max_elems: int) -> dict:
    """The oracle on the first elements of the same gradients and master
    weights (copied from the device), stepped until ``budget_s`` of wall time
    is used: single-threaded, as it stands (the reported value), and then its
    OpenMP build on every host core (``all_cores``)."""
    import numpy as np
    from zero_sharded_mixed_04_gb300 import synth
    n = min(max_elems, wl.psi_pad) // (wl.N * 128) * (wl.N * 128)
    g = [synth.to_numpy_grad(x[:n]) for x in grads]
    p0 = master[:n].cpu().numpy().copy()
    hp = oracle.Hparams(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps,
                        weight_decay=wl.weight_decay, max_grad_norm=wl.max_grad_norm)

    def timed(parallel: bool, budget: float):
        p = p0.copy()
        m, v, w = np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)
        oracle.zero_step(g, p, m, v, w, hp, 1, wl.loss_scale, wl.skip_on_overflow,
                         parallel=parallel)   # loads the library, faults the pages in
        steps, w0 = 0, time.perf_counter()
        while True:
            oracle.zero_step(g, p, m, v, w, hp, steps + 2, wl.loss_scale, wl.skip_on_overflow,
                             parallel=parallel)
            steps += 1
            if time.perf_counter() - w0 >= budget:
                break
        return steps, time.perf_counter() - w0

    steps, wall = timed(False, budget_s)
    out = {"value": steps * n / wall, "unit": UNIT, "cores": 1, "kind": "oracle",
           "ns_per_param": round(wall / (steps * n) * 1e9, 3), "cpu_model": cpu_model(),
           "nproc": os.cpu_count() or 1,
           "sample": f"{steps} oracle step(s) of {wl.name} on its first {n} parameters "
                     f"(all {wl.N} ranks), single-threaded C, {wall:.1f} s wall"}
    try:
        cores = os.cpu_count() or 1
        steps_p, wall_p = timed(True, budget_s / 2)
        out["all_cores"] = {
            "value": steps_p * n / wall_p, "unit": UNIT, "cores": cores, "kind": "oracle (OpenMP build)",
            "ns_per_param": round(wall_p / (steps_p * n) * 1e9, 4),
            "sample": f"{steps_p} step(s) of the same sample, the oracle's elementwise loops on "
                      f"{cores} threads, {wall_p:.1f} s wall"}
    except Exception as exc:  # no OpenMP runtime on this host
        out["all_cores"] = {"unavailable": str(exc).splitlines()[0]}
    return out


# ------------------------------------------------------------------ our arm

def run_ours(args, world, rank, local):
    import torch
    from zero_sharded_mixed_04_gb300 import build
    build.build_library()
    from zero_sharded_mixed_04_gb300 import synth
    from zero_sharded_mixed_04_gb300 import zero as Z
    from zero_sharded_mixed_04_gb300.optim import ZeroAdam

    group = Group(world)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = select_workload(args)
    out_of_place = not args.in_place
    device_policy = args.policy == "device" or (
        args.policy == "auto" and (wl.skip_on_overflow or wl.dynamic_loss_scale))
    pingpong = out_of_place and args.pingpong in ("on", "auto")
    grads = synth.make_grads(wl, 1, dev)  # step-1 gradients: no injected inf
    # the end-to-end leg's pinned host copy of the gradients, made before the
    # large device allocations as an application would hold it from the start
    host_grads, e2e_unavailable = None, None
    if not args.no_e2e:
        try:
            host_grads = pin_host_grads(grads)
        except RuntimeError as exc:  # not enough host memory to pin, say
            e2e_unavailable = f"pinned host copy of the gradients failed: {exc}".splitlines()[0]
        # every rank takes the same branch, since run_e2e holds barriers
        if group.max(1.0 if e2e_unavailable else 0.0) > 0.0 and e2e_unavailable is None:
            e2e_unavailable = "another rank could not pin its host copy of the gradients"
            host_grads = None
    master = synth.make_master(wl, dev)
    opt = ZeroAdam(wl.psi_pad, wl.N, wl.grad_dtype, lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2,
                   eps=wl.eps, weight_decay=wl.weight_decay, max_grad_norm=wl.max_grad_norm,
                   skip_on_overflow=wl.skip_on_overflow, bucket_elems=wl.bucket_elems,
                   loss_scale=wl.loss_scale, dynamic_loss_scale=wl.dynamic_loss_scale,
                   out_of_place=out_of_place, device=dev, master=master,
                   micro_batches=args.micro_batches, host_grad_accum=args.host_grad_accum,
                   device_policy=device_policy, pingpong=pingpong,
                   smem_staging=Z.ZERO_STAGING_TMA if args.staging == "tma" else 0,
                   # a captured step reads its bias corrections from a table
                   policy_table_steps=(args.warmup + args.steps + 64
                                       if args.profile_graph and device_policy else 0))
    buckets = opt.bucket_bounds()
    k_micro = max(1, args.micro_batches)
    # One event pair per step around its sequence of first-pass launches.
    # Nothing is recorded between the launches, so they overlap as in zero_step.
    # When the host bookkeeping needs no step outcome (no skip, static loss
    # scale) the host runs ahead of the device and the spans are read at the
    # end.
    stream = torch.cuda.current_stream(dev)
    # A step whose bytes could stay in L2 until the next one (the small parity
    # configs) gets L2 flushed before every timed step, by a write larger than
    # L2, and each step is timed on its own events so the flush stays out.
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129 << 20)
    step_bytes = alg_bytes_per_param(wl) * wl.psi_pad * max(1, args.micro_batches)
    flush_l2 = step_bytes < 2 * l2_bytes
    flush_buf = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev) if flush_l2 else None
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)] if flush_l2 else None
    # with micro-batches a third event, recorded before the last micro-batch,
    # splits the accumulate passes from the last one
    n_ev = 3 if k_micro > 1 else 2
    spans = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(n_ev))
             for _ in range(max(args.steps, args.warmup))]

    def one_step(k: int):
        ev = spans[k] if args.api == "plan" else None
        if k_micro > 1:
            # every micro-batch reads the same synthetic gradients
            res = opt.step_accumulated_async([grads] * k_micro, stream, span_events=ev)
        else:
            res = opt.step_async(grads, stream, api=args.api, span_events=ev)
        if res is not None and not res["applied"]:
            raise RuntimeError("benchmark step was skipped: the synthetic gradients overflowed")

    for k in range(args.warmup):
        one_step(k)
    torch.cuda.synchronize(dev)
    if args.profile_graph:
        # One more step, captured as a graph (ZeroAdam.capture_step) and
        # replayed once inside the profiler range.  Capturing runs nothing:
        # with the device policy, its table and ping-pong sets, t, the loss
        # scale, the bias corrections and the current set all live on the
        # device.
        if not (device_policy and pingpong and k_micro == 1):
            raise SystemExit("--profile-graph needs the device policy and ping-pong sets")
        graph = opt.capture_step(grads)
        torch.cuda.synchronize(dev)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.profiler.start()
        g0.record(stream)
        graph.replay()
        g1.record(stream)
        torch.cuda.profiler.stop()
        torch.cuda.synchronize(dev)
        if not opt.last_result(stream)["applied"]:
            raise RuntimeError("the profiled graph step was skipped")
        print(f"graph step: {g0.elapsed_time(g1):.4f} ms", file=sys.stderr)
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    clocks.start()
    launch_ms: list[float] = []
    last_ms: list[float] = []
    group.barrier()
    torch.cuda.synchronize(dev)
    launches0 = Z.zero_launch_count()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(args.steps):
        if flush_l2:
            flush_buf.zero_()
            step_ev[k][0].record(stream)
        if k == args.profile_step:
            torch.cuda.profiler.start()
        one_step(k)
        if k == args.profile_step:
            torch.cuda.profiler.stop()
        if flush_l2:
            step_ev[k][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    if not opt.last_result(stream)["applied"]:
        raise RuntimeError("benchmark step was skipped: the synthetic gradients overflowed")
    if args.api == "plan":
        launch_ms = [ev[0].elapsed_time(ev[1]) for ev in spans[:args.steps]]
        last_ms = ([ev[1].elapsed_time(ev[2]) for ev in spans[:args.steps]]
                   if k_micro > 1 else [])
    group.barrier()
    launches = Z.zero_launch_count() - launches0
    clock_info = clocks.stop()
    ms = (sum(a.elapsed_time(b) for a, b in step_ev) if flush_l2
          else t_start.elapsed_time(t_end)) / args.steps
    ms_max = group.max(ms)
    params_total = group.sum(float(wl.psi))
    value = params_total / (ms_max / 1e3)

    peak, peak_kind = read_peaks()
    b_alg = alg_bytes_per_param(wl)
    roofline = None
    two_pass = (opt.hp.max_grad_norm > 0 or (not out_of_place and opt.hp.skip_on_overflow)
                or args.host_grad_accum)
    if launch_ms:
        # the bucket launches of a step: their total span over the launch count
        # is the average launch duration
        per_step_kernel_ms = sum(launch_ms) / args.steps
        # algorithmic bytes of the timed kernel: the whole step's for the fused
        # kernel, the gradient reads for the first pass of the two-pass form
        b_kernel = wl.N * wl.grad_bytes if two_pass else b_alg
        n_launch = opt.first_pass_launches
        if k_micro > 1:
            # the accumulate passes: every micro-batch but the last, whose pass
            # the third event times apart (it is a pass of the accumulate
            # kernel too when the step has a second pass)
            b_kernel = (k_micro - 1) * wl.N * wl.grad_bytes   # their gradient reads
            n_launch = sum(opt.pass_launches[:-1])
        achieved = b_kernel * wl.psi_pad / (per_step_kernel_ms / 1e3) / 1e9
        # the committed ncu summary covers the fused kernel on the full flat1b_n8
        # workload only
        staged = args.staging == "tma" and not two_pass and k_micro == 1
        prof = (profiled_figures("zero_fused_staged_kernel" if staged else "zero_fused_kernel")
                if wl.name == "flat1b_n8" and not two_pass and k_micro == 1 else None)
        traffic = (None if prof is None
                   else round(prof["traffic_bytes_per_param"] * wl.psi_pad / n_launch))
        ncu_gbs = (None if prof is None or not prof["ncu_launch_us"]
                   else round(traffic / (prof["ncu_launch_us"] * 1e-6) / 1e9, 1))
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                    "frac": round(achieved / peak, 4),
                    "traffic": traffic,
                    "peak_kind": peak_kind,
                    "peak_label": "measured HBM copy" if peak_kind == "measured"
                                  else "fallback HBM copy",
                    "nominal_peak": NOMINAL_HBM_GBS,
                    "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                    # DRAM bytes of one launch over its serialised, cold-cache
                    # duration under ncu (the committed summary's figures)
                    "ncu_gbs": ncu_gbs,
                    "ncu_frac": None if ncu_gbs is None else round(ncu_gbs / peak, 4),
                    "kernel": ("zero_reduce_kernel" if two_pass else
                               "zero_fused_staged_kernel" if staged else "zero_fused_kernel"),
                    "buckets_per_step": len(buckets),
                    "launches_per_step": n_launch,
                    "avg_launch_ms": round(per_step_kernel_ms / n_launch, 5),
                    "alg_bytes_per_param": b_kernel}
    if k_micro > 1:
        # a step reads k micro-batches of gradients; the accumulator's round
        # trips are an implementation cost, not algorithmic bytes
        b_alg = k_micro * wl.N * wl.grad_bytes + 26
        ng = wl.N * wl.grad_bytes
        if roofline:
            roofline["kernel"] = "zero_accum_kernel"
            # k - 1 accumulate passes: the first writes the accumulator, the
            # others read and write it
            roofline["moved_bytes_per_param"] = (k_micro - 1) * ng + 8 * (k_micro - 1) - 4
            last_step_ms = sum(last_ms) / args.steps
            # the last micro-batch: fused with the update (reads the
            # accumulator, 26 B of state), or one more accumulate pass
            last_moved = ng + 4 + 26 if not two_pass else ng + 8
            roofline["last_micro_batch"] = {
                "kernel": "zero_accum_kernel" if two_pass else "zero_fused_kernel (accumulator in)",
                "ms": round(last_step_ms, 4), "moved_bytes_per_param": last_moved,
                "moved_gbs": round(last_moved * wl.psi_pad / (last_step_ms / 1e3) / 1e9, 1)}
            roofline["step_moved_bytes_per_param"] = (
                k_micro * ng + 8 * (k_micro - 1) + 26 if not two_pass
                else k_micro * ng + 8 * k_micro - 4 + 30)
    step_gbs = b_alg * wl.psi_pad / (ms / 1e3) / 1e9

    sequence = None
    run_seq = args.sequence if args.sequence is not None else bool(wl.inject_inf_step)
    if run_seq and k_micro == 1 and not args.host_grad_accum:
        sequence = run_sequence(opt, wl, grads, stream, dev, group, b_alg, flush_buf)

    e2e = None
    if e2e_unavailable is not None:
        e2e = {"unavailable": e2e_unavailable}
    elif not args.no_e2e:
        e2e = run_e2e(args, opt, grads, host_grads, wl, stream, dev, group)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        cpu = cpu_baseline(oracle, wl, grads, opt.state()["master"], budget_s=10.0,
                           max_elems=1 << 24)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": wl.name, "psi": wl.psi, "psi_pad": wl.psi_pad, "N": wl.N,
                   "grad_dtype": wl.grad_dtype, "bucket_elems": wl.bucket_elems,
                   "loss_scale": wl.loss_scale, "dynamic_loss_scale": wl.dynamic_loss_scale,
                   "skip_on_overflow": wl.skip_on_overflow, "max_grad_norm": wl.max_grad_norm,
                   "micro_batches": k_micro, "staging": args.staging,
                   "grad_shard": "pinned host memory" if args.host_grad_accum else "HBM",
                   "step_policy": "device" if device_policy else "host",
                   "state_sets": ("ping-pong (device keeps the current set)" if pingpong else
                                  "swapped by the host" if out_of_place else "one, in place"),
                   "entry": ("zero_plan_* (= zero_step_into)" if args.api == "plan"
                             else "zero_step_into") if out_of_place else
                   ("zero_plan_* (= zero_step)" if args.api == "plan" else "zero_step"),
                   "l2": ("L2 flushed before every timed step (a %d MB write outside the "
                          "step's own events): %.1f MB moved per step" %
                          (2 * l2_bytes >> 20, step_bytes / 1e6) if flush_l2 else
                          "inputs larger than L2: %.1f GB moved per step" %
                          (b_alg * wl.psi_pad / 1e9)),
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU, N ranks in HBM"},
        "achieved_hbm_gbs": round(step_gbs, 1),
        "hbm_frac": round(step_gbs / peak, 4),
        "hbm_frac_of_nominal": round(step_gbs / NOMINAL_HBM_GBS, 4),
        "roofline": roofline,
        "sequence": sequence,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clock_info,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    group.close()


def run_sequence(opt, wl, grads, stream, dev, group, b_alg, flush_buf=None) -> dict:
    """The workload's own steps as its configuration lists them: fresh seeded
    gradients every step, drawn at the loss scale that step uses, and the
    injected +inf on its step, which must be skipped.  Each step is timed on
    its own by CUDA events around its launches; the gradients are drawn
    between the timed regions.  Steps are enqueued as the timed steps are
    (with a device policy, back to back with no host read); the outcome is
    checked against the workload's script at the end.  With ``flush_buf`` (a
    workload whose step fits in L2) it is written before every step, outside
    the step's events."""
    import torch
    from zero_sharded_mixed_04_gb300 import synth
    opt.finish_pending()
    t0, scale = opt.t, opt.scaler.scale
    evs = []
    for step in range(1, wl.steps + 1):
        synth.make_grads(wl, step, dev, loss_scale=scale, out=grads)
        e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        if flush_buf is not None:
            flush_buf.zero_()
        e[0].record(stream)
        res = opt.step_async(grads, stream)
        e[1].record(stream)
        evs.append(e)
        overflow = step == wl.inject_inf_step
        if res is not None and res["applied"] == overflow:
            raise RuntimeError(f"sequence step {step}: expected it {'skipped' if overflow else 'applied'}")
        if overflow and wl.dynamic_loss_scale:
            scale *= 0.5   # the scale the next step's gradients carry
    opt.finish_pending()
    skipped = [s for s in range(1, wl.steps + 1) if s == wl.inject_inf_step]
    if opt.t != t0 + wl.steps - len(skipped) or (wl.dynamic_loss_scale and opt.scaler.scale != scale):
        raise RuntimeError("the step sequence did not skip exactly its injected step")
    ms = [group.max(a.elapsed_time(b)) for a, b in evs]
    applied_ms = [m for s, m in enumerate(ms, 1) if s not in skipped]
    mean = sum(ms) / len(ms)
    return {"steps": wl.steps, "skipped_steps": skipped, "ms": [round(m, 4) for m in ms],
            "applied_ms_mean": round(sum(applied_ms) / len(applied_ms), 4),
            "skipped_ms": round(ms[skipped[0] - 1], 4) if skipped else None,
            "mean_ms": round(mean, 4),
            "value": round(group.sum(float(wl.psi)) / (mean / 1e3), 1), "unit": UNIT,
            "achieved_hbm_gbs": round(b_alg * wl.psi_pad / (mean / 1e3) / 1e9, 1),
            "gradients": "fresh seeded draws per step, at the step's loss scale; "
                         "the injected +inf on its step"}


def pin_host_grads(grads):
    """The gradients in one page-locked host buffer backed by huge pages
    (hostmem.HostBuffer), every rank's a slice of it, placed on the host
    memory node next to the GPU."""
    from zero_sharded_mixed_04_gb300.hostmem import HostBuffer, gpu_numa_node
    n = grads[0].numel()
    # every rank on this node allocates one such buffer at about the same time
    ranks_here = int(os.environ.get("LOCAL_WORLD_SIZE", os.environ.get("WORLD_SIZE", "1")))
    buf = HostBuffer(n * len(grads), grads[0].dtype, share=ranks_here,
                     numa_node=gpu_numa_node(grads[0].device))
    host = [buf.tensor[i * n:(i + 1) * n] for i in range(len(grads))]
    for h, g in zip(host, grads):
        h.copy_(g)
    return buf, host


def run_e2e(args, opt, grads, host_grads, wl, stream, dev, group) -> dict:
    """The same step through the public API with the gradients in pinned host
    memory: every step copies them host-to-device through two bucket slots
    (overlapped with the reduction of the previous bucket) and reads the
    step result back to the host."""
    import torch
    buf, host = host_grads
    slots = opt.make_slots()
    copy_stream = torch.cuda.Stream(dev)
    steps = args.e2e_steps or max(1, min(args.steps, 10))
    opt.enqueue_from_host(host, slots, copy_stream, stream)  # one untimed warm-up step
    opt.finish(stream)
    h2d = sum(g.numel() * g.element_size() for g in grads)

    def copies_only() -> float:
        # the host link on its own: the step's own host-to-device copies
        # (bucket by bucket, rank by rank, into the two slots on the copy
        # stream) with no kernel in between
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        b = slots[0][0].numel()
        with torch.cuda.stream(copy_stream):
            for k, b0 in enumerate(range(0, wl.psi_pad, b)):
                b1 = min(wl.psi_pad, b0 + b)
                for i in range(wl.N):
                    slots[k % 2][i][:b1 - b0].copy_(host[i][b0:b1], non_blocking=True)
        copy_stream.synchronize()
        return time.perf_counter() - t0

    link = [copies_only() for _ in range(2)]
    group.barrier()
    torch.cuda.synchronize(dev)
    # each step timed on its own (it ends with the host reading its result):
    # the median is robust to a transient slowdown of the shared host link,
    # and the mean and the slowest step are reported beside it
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        opt.enqueue_from_host(host, slots, copy_stream, stream)
        res = opt.finish(stream)  # the step result, read on the host
        times.append(time.perf_counter() - t0)
        if not res["applied"]:
            raise RuntimeError("e2e step was skipped")
    link.append(copies_only())
    link_s = min(link)
    link_gbs = h2d / link_s / 1e9
    dt = group.max(statistics.median(times))
    mean = group.max(sum(times) / len(times))
    from zero_sharded_mixed_04_gb300.hostmem import cpu_nodes
    kind, numa_node, numa_placed = buf.kind, buf.numa_node, buf.numa_placed
    del host, slots, host_grads
    torch.cuda.synchronize(dev)
    buf.close()
    return {"value": round(group.sum(float(wl.psi)) / dt, 1), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 16, "ms_per_step": round(dt * 1e3, 3),
            "steps": steps, "statistic": "median step",
            "mean_ms_per_step": round(mean * 1e3, 3),
            "max_ms_per_step": round(group.max(max(times)) * 1e3, 3),
            "h2d_link_gbs": round(link_gbs, 1),
            "h2d_copies_only_ms": round(link_s * 1e3, 3),
            "host_buffer": kind,
            "host_numa_node": numa_node,
            "host_pages_on_node": numa_placed,
            "host_cpu_nodes": len(cpu_nodes()),
            "weights_d2h": "none: the BF16 working weights stay on the device for the next "
                           "forward pass; the host reads the 16-byte step result",
            "path": "pinned host grads -> two device bucket slots -> zero_plan_bucket; "
                    "result read by the host"}


# ------------------------------------------------------------------ reference arm (the oracle)

def run_reference(args, world, rank):
    if rank != 0:
        return
    import numpy as np
    import torch
    import oracle
    from zero_sharded_mixed_04_gb300 import synth
    wl = select_workload(args)
    oracle.build()
    unit = wl.N * 128
    # size each step's sample so the whole run takes about a minute
    calib_n = 1 << 18
    hp = oracle.Hparams(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps,
                        weight_decay=wl.weight_decay, max_grad_norm=wl.max_grad_norm)

    def sample(n):
        grads = synth.make_grads(wl, 1, "cpu", psi=n, psi_pad=n)
        g = [synth.to_numpy_grad(x) for x in grads]
        p = synth.make_master(wl, "cpu", psi_pad=n, psi=n).numpy()
        return g, p, np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)

    g, p, m, v, w = sample(calib_n)
    t0 = time.perf_counter()
    oracle.zero_step(g, p, m, v, w, hp, 1, wl.loss_scale, wl.skip_on_overflow)
    ns = (time.perf_counter() - t0) / calib_n * 1e9
    n = int(60.0 / (args.steps + args.warmup) / (ns * 1e-9))
    n = max(unit, min(1 << 25, n // unit * unit))
    g, p, m, v, w = sample(n)
    for k in range(args.warmup):
        oracle.zero_step(g, p, m, v, w, hp, k + 1, wl.loss_scale, wl.skip_on_overflow)
    t0 = time.perf_counter()
    for k in range(args.steps):
        oracle.zero_step(g, p, m, v, w, hp, args.warmup + k + 1, wl.loss_scale,
                         wl.skip_on_overflow)
    dt = (time.perf_counter() - t0) / args.steps
    value = n / dt
    desc = (f"each step: one oracle step of {wl.name} on a {n}-parameter sample (all {wl.N} "
            f"ranks), single-threaded C on the host")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "psi": wl.psi, "N": wl.N, "grad_dtype": wl.grad_dtype,
                   "sample_params": n},
        "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "ns_per_param": round(dt / n * 1e9, 3), "cpu_model": cpu_model(),
                         "nproc": os.cpu_count() or 1, "sample": desc},
        "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def zero3_layers(wl, layout_offsets, sizes, layer_elems):
    """Flat [begin, end) ranges of the workload's layers: GPT-2-small's
    embedding, twelve blocks and final norm; equal layers for flat vectors."""
    if wl.name.startswith("gpt2small"):
        bounds = [0, 1] + [1 + 10 * (i + 1) for i in range(12)] + [len(sizes)]
        return [(layout_offsets[bounds[i]],
                 layout_offsets[bounds[i + 1] - 1] + sizes[bounds[i + 1] - 1])
                for i in range(len(bounds) - 1)]
    return [(b, min(wl.psi, b + layer_elems)) for b in range(0, wl.psi, layer_elems)]


def run_zero3_gather(args, world, rank, local):
    """Times passes of the ZeRO-3 per-layer gather over the workload's layers,
    after one step has written the owners' BF16 shards."""
    import torch
    from zero_sharded_mixed_04_gb300 import build
    build.build_library()
    from zero_sharded_mixed_04_gb300 import synth
    from zero_sharded_mixed_04_gb300 import zero as Z
    from zero_sharded_mixed_04_gb300.optim import ZeroAdam, Zero3Views
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = select_workload(args)
    sizes = wl.sizes
    rc, lay, offs = Z.zero_init_layout(sizes, wl.N)
    Z.check(rc, "zero_init_layout")
    layers = zero3_layers(wl, offs, sizes, args.zero3_layer_elems)
    grads = synth.make_grads(wl, 1, dev)
    opt = ZeroAdam(wl.psi_pad, wl.N, wl.grad_dtype, lr=wl.lr, weight_decay=wl.weight_decay,
                   loss_scale=wl.loss_scale, device=dev, master=synth.make_master(wl, dev))
    opt.step(grads)
    del grads
    torch.cuda.empty_cache()
    w = opt.state()["w"]
    S = lay.shard
    views = Zero3Views([w[r * S:(r + 1) * S] for r in range(wl.N)], S, layers, device=dev,
                       side_streams=args.zero3_side_streams)
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(one_pass) -> float:
        for _ in range(args.warmup):
            one_pass()
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.steps):
            one_pass()                 # the stream waits for every layer's gather
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / args.steps

    # issued from Python layer by layer, then as one captured CUDA graph
    ms_eager = timed(lambda: views.run(lambda i, v: None))
    graph = views.capture()
    ms = timed(graph.replay)
    peak, peak_kind = read_peaks()
    gbs = 4 * wl.psi / (ms / 1e3) / 1e9   # 2 B read from a shard + 2 B written to a view
    numel = [e - b for b, e in layers]
    if rank == 0:
        print(json.dumps({
            "metric": "ZeRO-3 per-layer gather: gathered params/s (two views, one-ahead prefetch, "
                      "CUDA graph of the pass)",
            "value": round(wl.psi / (ms / 1e3), 1), "unit": "params/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_pass": round(ms, 4),
            "higher_is_better": True,
            "config": {"workload": wl.name, "N": wl.N, "layers": len(layers),
                       "largest_layer": max(numel), "side_streams": args.zero3_side_streams},
            "achieved_gbs": round(gbs, 1), "peak": peak, "peak_kind": peak_kind,
            "frac": round(gbs / peak, 4),
            "eager": {"ms_per_pass": round(ms_eager, 4),
                      "achieved_gbs": round(4 * wl.psi / (ms_eager / 1e3) / 1e9, 1)},
            "ledger_bytes_per_rank": {"zero3_persistent": Z.zero_ledger(wl.psi, wl.N, 3),
                                      "zero3_peak_two_views": Z.zero3_peak_bytes(numel, wl.N)},
        }), flush=True)


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_env()
    if args.zero3_gather and args.impl == "ours":
        run_zero3_gather(args, world, rank, local)
        return
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
