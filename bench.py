"""Benchmark of the layout-aware reduce-scatter + placement hot path.

One step = one reduce-scatter (N simulated ranks' per-parameter bf16
gradients -> every rank's fp32 dim-0 shards) plus one all-gather placement
(rank-major bf16 buffer -> per-parameter storage) over one synthetic
workload, through the C ABI.  Default workload: the Llama-3.1-70B-shaped
decoder layer, N = 8.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                  [--impl tide|reference]

Prints ONE JSON line on rank 0.  Under torchrun (--gpus > 1) every rank runs
an independent replica on its own GPU (the path has no cross-GPU step on one
box); value = all ranks' bytes / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "RS / AG-placement HBM GB/s and % of GB300 peak; concurrent GEMM slowdown %"
L2_BYTES = 129 * 1024 * 1024  # GB300; used when the device does not report its L2 size
FALLBACK_HBM_GBS = 6800.0
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.txt")
KERNEL_SRC = os.path.join(ROOT, "layout_aware_collectives_gb300", "csrc", "kernels.cu")
HBM_LIB = os.path.join(ROOT, "libbench_hbm.so")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="llama70b")
    ap.add_argument("--impl", default="tide", choices=["tide", "reference"])
    ap.add_argument("--no-interference", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-stock", action="store_true")
    ap.add_argument("--no-hbm-mix", action="store_true")
    ap.add_argument("--no-sustained", action="store_true",
                    help="skip the ~2 s back-to-back run with its clock record")
    ap.add_argument("--no-next-ops", action="store_true",
                    help="skip the single-rank RS, pack and Slot-Reuse figures")
    ap.add_argument("--hbm-mix-only", action="store_true",
                    help="only measure the HBM read/write-mix streams and print them as one JSON line")
    ap.add_argument("--no-second", action="store_true",
                    help="skip the second throughput workload (MoE layer after the 70B layer)")
    ap.add_argument("--mode", default="uncapped", choices=["uncapped", "capped", "bulk"],
                    help="kernel mode of the timed step")
    ap.add_argument("--cap", type=int, default=0, help="CTA cap for --mode capped / bulk")
    ap.add_argument("--out", default=None, help="also append the JSON line to this file")
    ap.add_argument("--collective", default="replicas", choices=["replicas", "ipc"],
                    help="replicas: every process runs all N simulated ranks on its own GPU; "
                         "ipc: one process per rank (N = world size), peers' buffers mapped over CUDA IPC")
    return ap.parse_args()


# ---------------------------------------------------------------- distributed
def dist_setup(n):
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def reduce_max(x: float, world: int) -> float:
    """Maximum of x over all ranks (the slowest replica's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(step_ms_local: float, bytes_per_step: int, world: int):
    """Whole-job figures of N independent replicas: every rank moves
    bytes_per_step per step; the job's step time is the slowest rank's."""
    step_ms = reduce_max(step_ms_local, world)
    return step_ms, world * bytes_per_step / (step_ms * 1e-3) / 1e9


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: str):
        self.dev = device
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.dev)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.time(), ln.strip()))

    def stop(self, t0=None, t1=None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        return self.summary(t0, t1)

    def summary(self, t0=None, t1=None):
        """Median SM clock and the throttle reasons seen in [t0, t1] (host time)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        lines = list(self.lines)
        sel = [ln for ts, ln in lines if t0 is None or (t0 - 0.06 <= ts <= t1 + 0.06)]
        if not sel and t0 is None:
            sel = [ln for _, ln in lines]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in sel:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(workload: str):
    """Per-launch DRAM bytes of the reduce-scatter kernel from the committed
    ncu summary, or None when absent or taken on another kernel source."""
    try:
        src_hash = hashlib.sha256(open(KERNEL_SRC, "rb").read()).hexdigest()[:16]
        with open(PROFILE_TRAFFIC) as f:
            for ln in f:
                parts = ln.split()
                if len(parts) == 4 and parts[0] == workload and parts[1] == "rs":
                    if parts[2] == src_hash:
                        return int(parts[3])
    except OSError:
        pass
    return None


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def oracle_sample(wl, budget_s, max_elems=48 * 2**20):
    """A bounded sample of the workload for the CPU oracle: every parameter
    with its rows capped at R (at least N, so every rank owns rows), R chosen
    so one oracle pass takes about budget_s seconds and the sample holds at
    most max_elems elements per rank."""
    import synth

    n = wl.num_ranks

    def shapes_for(R):
        return [s if not s else (min(int(s[0]), R),) + tuple(int(d) for d in s[1:])
                for s in wl.shapes]

    def elems(shapes):
        return sum(synth.numel(s) for s in shapes)

    cal = shapes_for(n)
    rate = max(1, elems(cal)) / max(time_oracle_pass(wl, cal), 1e-6)
    R = n
    while True:
        nxt = shapes_for(R * 2)
        if nxt == shapes_for(R) or elems(nxt) / rate > budget_s or elems(nxt) > max_elems:
            break
        R *= 2
    return shapes_for(R)


def _sample_inputs(wl, shapes):
    import numpy as np

    import synth
    import oracle

    sub = synth.Workload(wl.name + "_sample", wl.num_ranks, shapes, wl.names, wl.sigma, wl.seed,
                         wl.outlier_every, wl.outlier_mult, wl.zero_groups, wl.zero_pct)
    grads = [[sub.host_grad_at(k, p, np.arange(synth.numel(s))) for p, s in enumerate(shapes)]
             for k in range(wl.num_ranks)]
    offs, S = oracle.layout(shapes, wl.num_ranks, 8)
    buf = np.full(wl.num_ranks * S, synth.SENTINEL_BF16, dtype=np.uint16)
    for p, s in enumerate(shapes):
        d0, inner = synth.dim0_inner(s)
        c = -(-d0 // wl.num_ranks)
        full = sub.host_param_value(p)
        for r in range(wl.num_ranks):
            v = max(0, min(c, d0 - r * c)) * inner
            buf[r * S + offs[p]: r * S + offs[p] + v] = full[r * c * inner: r * c * inner + v]
    return grads, buf, offs, S


def time_oracle_pass(wl, shapes, inputs=None):
    import oracle

    grads, buf, offs, S = inputs if inputs is not None else _sample_inputs(wl, shapes)
    t0 = time.perf_counter()
    oracle.rs(shapes, wl.num_ranks, grads, wl.scale)
    oracle.ag_place(shapes, wl.num_ranks, buf, offs, S)
    return time.perf_counter() - t0


def sample_bytes(wl, shapes):
    import synth

    psi = sum(synth.numel(s) for s in shapes)
    return 2 * wl.num_ranks * psi + 4 * psi + 4 * psi


def describe_sample(wl, shapes):
    import synth

    cap = max((s[0] for s in shapes if s), default=1)
    return (f"{wl.name} (N={wl.num_ranks}): all {len(shapes)} parameters with dim 0 capped at "
            f"{cap} rows, {sum(synth.numel(s) for s in shapes)} elements per rank; one "
            "reduce-scatter + one placement pass of the single-threaded C oracle")


def cpu_baseline(wl, budget_s):
    """The oracle, as it stands, on a bounded sample: passes repeated until
    about budget_s seconds of single-thread CPU work."""
    shapes = oracle_sample(wl, budget_s)
    inputs = _sample_inputs(wl, shapes)
    total, passes = 0.0, 0
    while total < budget_s or passes == 0:
        total += time_oracle_pass(wl, shapes, inputs)
        passes += 1
    return {"value": round(sample_bytes(wl, shapes) * passes / total / 1e9, 4), "unit": "GB/s",
            "cores": 1, "kind": "oracle",
            "sample": describe_sample(wl, shapes) + f"; {passes} passes",
            "seconds": round(total, 2), "host_cores": cpu_cores()}


# ---------------------------------------------------------------- reference arm
def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import synth

    wl = synth.WORKLOADS[args.config]()
    per_step = max(0.05, min(5.0, 150.0 / max(1, args.steps + args.warmup)))
    shapes = oracle_sample(wl, per_step)
    inputs = _sample_inputs(wl, shapes)
    for _ in range(args.warmup):
        time_oracle_pass(wl, shapes, inputs)
    times = [time_oracle_pass(wl, shapes, inputs) for _ in range(args.steps)]
    total = sum(times)
    nbytes = sample_bytes(wl, shapes)
    value = nbytes * args.steps / total / 1e9
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "num_ranks": wl.num_ranks, "num_params": wl.num_params,
                   "psi": wl.psi, "sample": "bounded CPU sample, see cpu_baseline"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": describe_sample(wl, shapes),
                         "host_cores": cpu_cores()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    emit(out, args)
    return 0


def emit(out, args):
    """The one JSON line on stdout, optionally appended to --out."""
    line = json.dumps(out)
    print(line)
    if args.out:
        with open(args.out, "a") as f:
            f.write(line + "\n")


# ---------------------------------------------------------------- GPU arm
def smi_device(dev: int) -> str:
    """nvidia-smi -i takes an index, a UUID or a PCI id: pass the visible entry as is."""
    visible = [v.strip() for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    return visible[dev] if dev < len(visible) else str(dev)


def timed_steps(layout, job, wl, stream, K, warmup, world, smi_dev, l2_bytes):
    """W untimed steps, then K timed steps (one reduce-scatter + one
    placement each) bracketed by a barrier and a device synchronise, with CUDA
    events on the launching stream around every launch and nvidia-smi clock
    samples over the timed region."""
    import torch

    import layout_aware_collectives_gb300 as tide

    gptr = tide.PointerTable(job.grad_ptrs())
    sptr = tide.PointerTable(job.shard_ptrs())
    pptr = tide.PointerTable(job.param_ptrs())
    scale = wl.scale
    rs_bytes, ag_bytes = wl.rs_bytes(), wl.ag_bytes()
    small = (rs_bytes + ag_bytes) < 2 * l2_bytes
    flush = torch.empty(2 * l2_bytes // 4, dtype=torch.float32, device="cuda") if small else None
    with torch.cuda.stream(stream):
        for _ in range(max(3, warmup)):
            layout.reduce_scatter(gptr, sptr, scale, stream)
            layout.place(job.gathered, pptr, stream)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    clocks = ClockSampler(smi_dev)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    with torch.cuda.stream(stream):
        for i in range(K):
            if flush is not None:
                flush.fill_(float(i))
            ev[i][0].record(stream)
            layout.reduce_scatter(gptr, sptr, scale, stream)
            ev[i][1].record(stream)
            layout.place(job.gathered, pptr, stream)
            ev[i][2].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    clk = clocks.stop(t0, t1)
    rs_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    ag_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    if flush is None:
        step_ms_local = ev[0][0].elapsed_time(ev[K - 1][2]) / K
    else:
        step_ms_local = sum(r + a for r, a in zip(rs_ms, ag_ms)) / K
    del flush
    return {"step_ms_local": step_ms_local, "rs_ms": rs_ms, "ag_ms": ag_ms, "clocks": clk,
            "l2": "flushed between steps" if small else
            f"inputs larger than L2 ({(rs_bytes + ag_bytes) / 1e9:.1f} GB per step)"}


def run_sustained(layout, job, wl, stream, smi_dev, world, seconds=2.0):
    """The same step back to back for about `seconds` (after the timed
    region, same mode): GB/s over the whole run by CUDA events and the SM
    clocks sampled throughout (tens of samples, where the short timed region
    gets a few)."""
    import torch

    import layout_aware_collectives_gb300 as tide

    gptr = tide.PointerTable(job.grad_ptrs())
    sptr = tide.PointerTable(job.shard_ptrs())
    pptr = tide.PointerTable(job.param_ptrs())
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):  # one step to size the run
        e0.record(stream)
        layout.reduce_scatter(gptr, sptr, wl.scale, stream)
        layout.place(job.gathered, pptr, stream)
        e1.record(stream)
    torch.cuda.synchronize()
    steps = max(10, int(seconds * 1e3 / max(e0.elapsed_time(e1), 1e-3)))
    clocks = ClockSampler(smi_dev)
    clocks.start()
    time.sleep(0.1)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            layout.reduce_scatter(gptr, sptr, wl.scale, stream)
            layout.place(job.gathered, pptr, stream)
        e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    clk = clocks.stop(t0, t1)
    ms = e0.elapsed_time(e1)
    return {"steps": steps, "seconds": round(ms * 1e-3, 3),
            "GB/s": round(steps * (wl.rs_bytes() + wl.ag_bytes()) / (ms * 1e-3) / 1e9, 1), "clocks": clk}


def mix_ratio(num_ranks: int) -> int:
    """Reads per write of the reduce-scatter (2N bytes read per 4 written),
    rounded to a ratio the HBM-mix probe has."""
    want = max(1, num_ranks // 2)
    return min((1, 2, 4, 8, 16), key=lambda r: abs(r - want))


def run_tide(args):
    import torch

    world, rank, local = dist_setup(args.gpus)
    import layout_aware_collectives_gb300 as tide
    import synth
    from synth.device import DeviceJob

    dev = torch.cuda.current_device()
    props = torch.cuda.get_device_properties(dev)
    smi_dev = smi_device(dev)
    l2_bytes = getattr(props, "L2_cache_size", 0) or L2_BYTES  # queried; the constant if unknown
    wl = synth.WORKLOADS[args.config]()
    layout = tide.Layout(wl.shapes, wl.num_ranks)
    job = DeviceJob(wl, layout, guard=False)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    rs_bytes, ag_bytes = wl.rs_bytes(), wl.ag_bytes()

    step_mode = {"uncapped": tide.TIDE_MODE_UNCAPPED, "capped": tide.TIDE_MODE_CAPPED,
                 "bulk": tide.TIDE_MODE_BULK}[args.mode]
    if args.mode == "capped" and args.cap < 1:
        raise SystemExit("--mode capped needs --cap >= 1")
    layout.set_mode(step_mode, args.cap)

    K = args.steps
    run = timed_steps(layout, job, wl, stream, K, args.warmup, world, smi_dev, l2_bytes)
    rs_ms, ag_ms = run["rs_ms"], run["ag_ms"]
    step_ms, value = aggregate(run["step_ms_local"], rs_bytes + ag_bytes, world)
    rs_avg = statistics.mean(rs_ms)
    ag_avg = statistics.mean(ag_ms)

    peak, peak_src = measured_peaks()
    rs_gbs = rs_bytes / (rs_avg * 1e-3) / 1e9
    ag_gbs = ag_bytes / (ag_avg * 1e-3) / 1e9
    grid_rs, block_rs = layout.launch_shape(tide.TIDE_OP_RS)
    grid_ag, block_ag = layout.launch_shape(tide.TIDE_OP_AG)
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": round(step_ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "num_ranks": wl.num_ranks, "num_params": wl.num_params,
                   "psi": wl.psi, "rs_bytes": rs_bytes, "ag_bytes": ag_bytes,
                   "io": "bf16 gradients -> fp32 shards (fp32 sums); bf16 placement (bit copy)",
                   "l2": run["l2"],
                   "mode": args.mode + (f" cap {args.cap}" if args.cap else ""),
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm",
                     "kernel": "tide rs_bulk_kernel" if args.mode == "bulk" else "tide rs_kernel",
                     "achieved": round(rs_gbs, 1),
                     "peak": peak, "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "unit": "GB/s", "frac": round(rs_gbs / peak, 4),
                     "traffic": recorded_traffic(wl.name) if args.mode == "uncapped" else None},
        "clocks": run["clocks"],
        "gpu_launches": 2 * K,
        "device": props.name,
        "kernels": {
            "rs": {"ms": round(rs_avg, 4), "GB/s": round(rs_gbs, 1), "frac": round(rs_gbs / peak, 4),
                   "ms_median": round(statistics.median(rs_ms), 4), "grid": grid_rs, "block": block_rs},
            "ag": {"ms": round(ag_avg, 4), "GB/s": round(ag_gbs, 1), "frac": round(ag_gbs / peak, 4),
                   "ms_median": round(statistics.median(ag_ms), 4), "grid": grid_ag, "block": block_ag},
        },
    }

    layout.check_device()  # raises if a bounded device wait ran out during the timed steps
    if not args.no_sustained and rs_bytes + ag_bytes >= 2 * l2_bytes:  # no L2 flush between its steps
        out["sustained"] = run_sustained(layout, job, wl, stream, smi_dev, world)
    layout.set_mode(tide.TIDE_MODE_UNCAPPED)
    if not args.no_next_ops:
        out["next_ops"] = run_next_ops(tide, layout, job, wl, stream)
    if not args.no_stock:
        out["stock_fsdp2"] = run_stock(job, wl, stream, rs_avg, ag_avg)
    if not args.no_e2e:
        try:
            out["e2e"] = run_e2e(tide, layout, job, wl, stream, K, world)
        except (RuntimeError, torch.OutOfMemoryError) as e:  # pinned host memory can run out
            torch.cuda.synchronize()
            out["e2e"] = {"value": None, "unit": "GB/s", "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0, "unavailable": f"{type(e).__name__}: {e}"[:300]}
    if not args.no_interference:
        out["interference"] = run_interference(tide, layout, job, wl, props, smi_dev)
    layout.set_mode(tide.TIDE_MODE_UNCAPPED)
    layout.close()
    del job
    torch.cuda.empty_cache()

    # HBM streams of the reduce-scatter's own read:write mix (the copy peak is 1:1)
    second = "moe" if args.config != "moe" else "llama70b"
    ratios = sorted({mix_ratio(wl.num_ranks), mix_ratio(synth.WORKLOADS[second]().num_ranks)})
    if not args.no_hbm_mix:
        mix = run_hbm_mix(ratios, smi_dev)
        out["hbm_mix"] = mix
        ceiling = mix.get(f"read{mix_ratio(wl.num_ranks)}_write1")
        if ceiling:
            out["roofline"]["mix_peak"] = ceiling
            out["roofline"]["frac_vs_mix"] = round(rs_gbs / ceiling, 4)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(wl, 10.0)
    if not args.no_second:
        out[second] = run_second(second, args, world, smi_dev, l2_bytes, peak, out.get("hbm_mix"))
    if "interference" in out:
        out["interference_summary"] = interference_summary(out["interference"])
    if rank == 0:
        emit(out, args)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def run_second(name, args, world, smi_dev, l2_bytes, peak, mix):
    """The step on the other throughput workload (MoE layer after the 70B
    layer, or the reverse), timed the same way, reported compactly."""
    import torch

    import layout_aware_collectives_gb300 as tide
    import synth
    from synth.device import DeviceJob

    wl = synth.WORKLOADS[name]()
    layout = tide.Layout(wl.shapes, wl.num_ranks)
    job = DeviceJob(wl, layout, guard=False)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    run = timed_steps(layout, job, wl, stream, args.steps, args.warmup, world, smi_dev, l2_bytes)
    step_ms, value = aggregate(run["step_ms_local"], wl.rs_bytes() + wl.ag_bytes(), world)
    rs_gbs = wl.rs_bytes() / (statistics.mean(run["rs_ms"]) * 1e-3) / 1e9
    ag_gbs = wl.ag_bytes() / (statistics.mean(run["ag_ms"]) * 1e-3) / 1e9
    res = {"workload": wl.name, "N": wl.num_ranks, "P": wl.num_params, "value_GB/s": round(value, 1),
           "ms_per_step": round(step_ms, 4), "rs_GB/s": round(rs_gbs, 1), "rs_frac": round(rs_gbs / peak, 4),
           "ag_GB/s": round(ag_gbs, 1), "ag_frac": round(ag_gbs / peak, 4)}
    ceiling = (mix or {}).get(f"read{mix_ratio(wl.num_ranks)}_write1")
    if ceiling:
        res["rs_frac_vs_mix"] = round(rs_gbs / ceiling, 4)
    c = run["clocks"]
    res["clocks"] = {"sm_mhz": c.get("sm_mhz"), "reasons": c.get("reasons"), "samples": c.get("samples")}
    layout.check_device()
    layout.close()
    del job
    torch.cuda.empty_cache()
    return res


def run_hbm_mix(ratios, smi_dev, out_bytes=1 << 30, reps=10):
    """HBM rates of streams with a fixed read:write mix (bench_hbm.cu):
    read-only, write-only, and R reads per write for each R in `ratios`
    (plus R = 1, a copy); median of `reps` launches by CUDA events, 1 GiB
    written per launch (R GiB read)."""
    import ctypes

    import torch

    lib = ctypes.CDLL(HBM_LIB)
    for f in (lib.hbm_read, lib.hbm_write, lib.hbm_mix):
        f.restype = ctypes.c_int
    lib.hbm_read.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    lib.hbm_write.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint32, ctypes.c_void_p]
    lib.hbm_mix.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
    lib.hbm_sm_stream.restype = ctypes.c_int
    lib.hbm_sm_stream.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_void_p, ctypes.c_void_p]
    rmax = max([1] + list(ratios))
    src = torch.empty(max(rmax, 4) * out_bytes, dtype=torch.uint8, device="cuda")
    dst = torch.empty(out_bytes, dtype=torch.uint8, device="cuda")
    sink = torch.zeros(16, dtype=torch.uint8, device="cuda")
    src.fill_(0x5A)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    sh = stream.cuda_stream

    def rate(launch, nbytes):
        with torch.cuda.stream(stream):
            for _ in range(3):
                assert launch() == 0
            ms = []
            for _ in range(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                assert launch() == 0
                e1.record(stream)
                ms.append((e0, e1))
        torch.cuda.synchronize()
        t = statistics.median(a.elapsed_time(b) for a, b in ms)
        return round(nbytes / (t * 1e-3) / 1e9, 1)

    clocks = ClockSampler(smi_dev)
    clocks.start()
    time.sleep(0.2)
    t0 = time.time()
    rd_bytes = src.numel()
    wr_bytes = 4 * out_bytes
    res = {"kernel": "bench_hbm.cu: one 512-thread CTA per tile, 16-byte ld.global.nc / st.global.cs",
           "read_only": rate(lambda: lib.hbm_read(src.data_ptr(), rd_bytes, sink.data_ptr(), sh), rd_bytes),
           "write_only": rate(lambda: lib.hbm_write(src.data_ptr(), wr_bytes, 7, sh), wr_bytes)}
    for r in sorted({1} | set(ratios)):
        res[f"read{r}_write1"] = rate(lambda r=r: lib.hbm_mix(src.data_ptr(), dst.data_ptr(), out_bytes, r, sh),
                                      (r + 1) * out_bytes)
    # what one SM moves: 8 persistent 1024-thread CTAs (the CTA-capped kernels' shape), per CTA
    half = out_bytes // 2
    per_cta = {}
    for name, mode, nbytes in (("read", 0, half), ("write", 1, half), ("copy_read_plus_write", 2, 2 * half)):
        gbs = rate(lambda mode=mode: lib.hbm_sm_stream(src.data_ptr(), dst.data_ptr(), half, mode, 8,
                                                       sink.data_ptr(), sh), nbytes)
        per_cta[name] = round(gbs / 8, 1)
    res["per_sm_8_ctas"] = {"kernel": "bench_hbm.cu hbm_sm_stream: 8 CTAs x 1024 threads, 8 accesses in "
                                      "flight per thread; GB/s per CTA (each CTA holds one SM)", **per_cta}
    t1 = time.time()
    rd, wr = res["read_only"], res["write_only"]
    # the rate a stream with read fraction f would reach if reads ran at the
    # read-only rate and writes at the write-only rate, one after the other
    res["bound_from_read_and_write_rates"] = {
        f"read{r}_write1": round(1.0 / ((r / (r + 1)) / rd + (1 / (r + 1)) / wr), 1) for r in sorted({1} | set(ratios))}
    res["clocks"] = clocks.stop(t0, t1)
    del src, dst, sink
    torch.cuda.empty_cache()
    return res


def run_next_ops(tide, layout, job, wl, stream, reps=20):
    """Device time of the per-GPU operations next to the step: the
    single-rank reduce-scatter (rank 0: what one GPU of the job computes) and
    the all-gather input pack of every rank (fp32 shard -> bf16 slot)."""
    import torch

    N = wl.num_ranks
    valid0 = sum(max(0, min(c, d0 - 0 * c)) * inner
                 for c, (d0, inner) in zip(job.chunk, job.dims))
    padded = sum(job.shard_numel)
    outs = [torch.empty(n, dtype=torch.float32, device="cuda") for n in job.shard_numel]
    job.make_pack_inputs()
    torch.cuda.synchronize()  # the generator fills run on the default stream
    gptr = tide.PointerTable(job.grad_ptrs())
    optr = tide.PointerTable(outs)
    pptr = tide.PointerTable(job.pack_src_ptrs())
    res = {}
    for name, op, nbytes in (
            ("rs_rank0", lambda: layout.reduce_scatter_rank(0, gptr, optr, wl.scale, stream),
             2 * N * valid0 + 4 * valid0),
            ("ag_pack_all_ranks", lambda: layout.pack(-1, pptr, job.packed, stream),
             6 * N * padded)):
        with torch.cuda.stream(stream):
            for _ in range(3):
                op()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                op()
            e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        res[name] = {"ms": round(ms, 4), "bytes": nbytes,
                     "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1)}
    del outs, job.pack_src, job.packed
    # Slot-Reuse two-stage path: stage every rank's gradients into its slot,
    # then reduce-scatter from the slots
    job.make_slots()
    torch.cuda.synchronize()
    sptr = tide.PointerTable(job.shard_ptrs())
    slot_tab = tide.PointerTable(job.slots)
    gtabs = [tide.PointerTable([job.grads[k][p] for p in range(job.P)]) for k in range(N)]

    def stage_all():
        for k in range(N):
            layout.stage(gtabs[k], job.slots[k], stream)

    for name, op, nbytes in (
            ("stage_all_ranks", stage_all, 4 * N * wl.psi),
            ("rs_from_staged_slots", lambda: layout.reduce_scatter_staged(slot_tab, sptr, wl.scale, stream),
             wl.rs_bytes())):
        with torch.cuda.stream(stream):
            for _ in range(3):
                op()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                op()
            e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        res[name] = {"ms": round(ms, 4), "bytes": nbytes,
                     "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1)}
    del job.slots
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------- stock FSDP2 emulation
class StockFSDP2:
    """What stock FSDP2 does around its collectives, in the PyTorch ops it
    uses, on the same N simulated ranks: the reduce-scatter input is built by
    copying every rank's per-parameter bf16 gradients into one flat fp32
    rank-major buffer (torch._chunk_cat with a cast, dense dim-0 chunks, zero
    padding); the reduction then runs on the flat buffers (here a rank-order
    fp32 sum, on the wire in a real job); the all-gather output, a flat bf16
    rank-major buffer, is copied out into padded per-parameter storage
    (torch.split_with_sizes_copy).  The copy-in and copy-out are the layout
    conversion ("FSDP通信终局：TIDE零拷贝集合通信优化" §FSDP2通信开销的根源) that
    TIDE's fused reduce-scatter and direct placement avoid."""

    def __init__(self, job):
        import torch

        self.job = job
        N = job.N
        self.sizes = list(job.shard_numel)            # c_p * inner_p
        self.S1 = sum(self.sizes)                      # dense rank block
        self.offs1 = [sum(self.sizes[:p]) for p in range(job.P)]
        dev = job.device
        self.flat = [torch.empty(N, self.S1, dtype=torch.float32, device=dev) for _ in range(N)]
        self.out = torch.empty(N * self.S1, dtype=torch.float32, device=dev)
        self.gathered = torch.zeros(N, self.S1, dtype=torch.bfloat16, device=dev)
        self.padded = [torch.empty(N * n, dtype=torch.bfloat16, device=dev) for n in self.sizes]
        # the stock all-gather output holds the same chunks as TIDE's buffer
        for p in range(job.P):
            o, o1, n = job.layout.param_offset(p), self.offs1[p], self.sizes[p]
            for r in range(N):
                self.gathered[r, o1:o1 + n] = job.gathered[r * job.S + o: r * job.S + o + n].view(torch.bfloat16)
        self.grad_views = [[self._view(job.grads[k][p], job.wl.shapes[p]) for p in range(job.P)]
                           for k in range(N)]

    @staticmethod
    def _view(t, shape):
        import torch

        shp = tuple(shape) if len(shape) else (1,)
        return t.view(torch.bfloat16).view(shp)

    def copy_in(self):
        import torch

        for k in range(self.job.N):
            torch._chunk_cat(self.grad_views[k], dim=0, num_chunks=self.job.N, out=self.flat[k])

    def flat_reduce(self, scale):
        self.out.zero_()
        for k in range(self.job.N):
            self.out.add_(self.flat[k].view(-1))
        self.out.mul_(scale)

    def copy_out(self):
        import torch

        torch.split_with_sizes_copy(self.gathered, self.sizes, dim=1,
                                    out=[b.view(self.job.N, n) for b, n in zip(self.padded, self.sizes)])

    def shard(self, r, p):
        o1 = r * self.S1 + self.offs1[p]
        return self.out[o1: o1 + self.sizes[p]]

    def param(self, p):
        d0, inner = self.job.dims[p]
        return self.padded[p][: d0 * inner]


def run_stock(job, wl, stream, tide_rs_ms, tide_ag_ms, reps=10):
    """Times of the stock emulation's three parts next to TIDE's kernels."""
    import torch

    st = StockFSDP2(job)
    torch.cuda.synchronize()  # set-up work ran on the default stream
    flat_bytes = sum(t.numel() * t.element_size() for t in st.flat)
    N, psi, padded = wl.num_ranks, wl.psi, sum(job.shard_numel)
    flat = N * padded  # elements of one rank's flat buffer (every destination block)
    parts = {"rs_copy_in": (st.copy_in, N * (2 * psi + 4 * flat)),
             # zero_, N rank-order add_ passes (read out + read flat_k + write out), mul_
             "flat_reduce": (lambda: st.flat_reduce(wl.scale), 4 * flat + N * 12 * flat + 8 * flat),
             "ag_copy_out": (st.copy_out, 4 * flat)}
    res = {}
    with torch.cuda.stream(stream):
        for name, (fn, nbytes) in parts.items():
            fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / reps
            res[name] = {"ms": round(ms, 4), "bytes": nbytes, "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1)}
    conv = res["rs_copy_in"]["ms"] + res["ag_copy_out"]["ms"]
    total = conv + res["flat_reduce"]["ms"]
    res["layout_conversion_ms"] = round(conv, 4)
    res["stock_step_ms"] = round(total, 4)
    res["tide_step_ms"] = round(tide_rs_ms + tide_ag_ms, 4)
    res["tide_speedup_vs_stock"] = round(total / (tide_rs_ms + tide_ag_ms), 2)
    res["note"] = ("stock = chunk_cat copy-in (bf16->fp32) + torch rank-order fp32 sum of flat "
                   "buffers + split_with_sizes_copy copy-out; TIDE = fused RS + placement")
    # Device memory beyond what both paths hold (gradients, shards, the
    # rank-major all-gather buffer, parameters), per rank.  Stock: the fp32
    # flat reduce-scatter input.  TIDE: the reduce-scatter reads the gradients in
    # place and Slot-Reuse stages them into the vacated all-gather slot, so
    # neither needs a buffer; the library's own device state is its tile
    # lists and cached pointer tables.  (Stock: the flat tensors' sizes over
    # the N simulated ranks, divided by N.)
    import layout_aware_collectives_gb300 as tide

    lay = job.layout
    tile_bytes = 32 * sum(len(lay.tiles(op)) for op in (tide.TIDE_OP_RS, tide.TIDE_OP_AG, tide.TIDE_OP_PACK,
                                                          tide.TIDE_OP_STAGED_RS))
    # SM time (kernel time x SMs occupied; every launch here spans the GPU),
    # the analog of the pages' reduce-scatter SM-time comparison
    # ("FSDP通信终局：TIDE零拷贝集合通信优化" §性能表现)
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    stock_rs = res["rs_copy_in"]["ms"] + res["flat_reduce"]["ms"]
    res["sm_ms"] = {"stock_rs_copy_in_plus_flat_reduce": round(stock_rs * sms, 1),
                    "stock_flat_reduce": round(res["flat_reduce"]["ms"] * sms, 1),
                    "tide_rs": round(tide_rs_ms * sms, 1),
                    "stock_rs_over_tide_rs": round(stock_rs / tide_rs_ms, 2),
                    "note": "kernel ms x SMs occupied (all of them for these launches); the CTA-capped "
                            "reduce-scatter's SM.ms is in the interference table"}
    res["memory_per_rank"] = {
        "stock_rs_input_bytes": flat_bytes // N,
        "tide_rs_extra_bytes": 0,
        "slot_reuse_extra_bytes": 0,
        "tide_library_device_bytes": {"tile_lists": tile_bytes,
                                      "per_cached_pointer_table": 16 * N * job.P, "max_cached_tables": 8}}
    del st
    torch.cuda.empty_cache()
    return res


def _host_mapped(tensors) -> bool:
    """True when every pinned host tensor is mapped into the device address
    space at its own address (UVA), so kernels may read and write it."""
    import ctypes

    lib = None
    for name in ("libcudart.so", "/usr/local/cuda/lib64/libcudart.so"):
        try:
            lib = ctypes.CDLL(name)
            break
        except OSError:
            continue
    if lib is None:
        return False
    for t in tensors:
        if t.numel() == 0:
            continue
        dp = ctypes.c_void_p(0)
        rc = lib.cudaHostGetDevicePointer(ctypes.byref(dp), ctypes.c_void_p(t.data_ptr()), 0)
        if rc != 0 or dp.value != t.data_ptr():
            return False
    return True


def run_e2e(tide, layout, job, wl, stream, K, world):
    """Same metric through the public API with the step's inputs and results
    in pinned HOST memory, every step:
      zero_copy    the kernels read the gradients and the gathered buffer from
                   host memory and write shards and parameters to host memory
                   over NVLink-C2C (pinned memory is device-mapped on Grace);
      copy_engine  cudaMemcpyAsync of the inputs in, both kernels on device
                   buffers, cudaMemcpyAsync of the results out.
    `value` is the zero-copy figure when every buffer is mapped (checked with
    cudaHostGetDevicePointer), else the copy-engine one."""
    import torch

    flat_g = [g for row in job.grads for g in row]
    flat_s = [s for row in job.shards for s in row]
    h_g = [torch.empty(g.shape, dtype=g.dtype, pin_memory=True) for g in flat_g]
    h_s = [torch.empty(s.shape, dtype=s.dtype, pin_memory=True) for s in flat_s]
    h_buf = torch.empty(job.gathered.shape, dtype=job.gathered.dtype, pin_memory=True)
    h_p = [torch.empty(p.shape, dtype=p.dtype, pin_memory=True) for p in job.params]
    for h, d in zip(h_g, flat_g):
        h.copy_(d)
    h_buf.copy_(job.gathered)
    torch.cuda.synchronize()
    steps = max(3, min(K, 20))
    nbytes = wl.rs_bytes() + wl.ag_bytes()

    def timed(one):
        with torch.cuda.stream(stream):
            one()
            torch.cuda.synchronize()
            barrier(world)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                one()
            e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return aggregate(e0.elapsed_time(e1) / steps, nbytes, world)

    # copy-engine staging
    gptr = tide.PointerTable(job.grad_ptrs())
    sptr = tide.PointerTable(job.shard_ptrs())
    pptr = tide.PointerTable(job.param_ptrs())

    def one_ce():
        for d, h in zip(flat_g, h_g):
            d.copy_(h, non_blocking=True)
        job.gathered.copy_(h_buf, non_blocking=True)
        layout.reduce_scatter(gptr, sptr, wl.scale, stream)
        layout.place(job.gathered, pptr, stream)
        for h, d in zip(h_s, flat_s):
            h.copy_(d, non_blocking=True)
        for h, d in zip(h_p, job.params):
            h.copy_(d, non_blocking=True)

    ms_ce, val_ce = timed(one_ce)
    ce = {"value": round(val_ce, 2), "ms_per_step": round(ms_ce, 3),
          "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in h_g) + h_buf.numel() * 2,
          "d2h_bytes_per_step": sum(h.numel() * 4 for h in h_s) + sum(h.numel() * 2 for h in h_p)}
    out = {"unit": "GB/s", "steps": steps, "copy_engine": ce}

    if _host_mapped(h_g + h_s + h_p + [h_buf]):
        hg = tide.PointerTable(h_g)
        hs = tide.PointerTable(h_s)
        hp = tide.PointerTable(h_p)

        def one_zc():
            layout.reduce_scatter(hg, hs, wl.scale, stream)
            layout.place(h_buf, hp, stream)

        ms_zc, val_zc = timed(one_zc)
        same = all(torch.equal(h.view(torch.int32), d.view(torch.int32).cpu())
                   for h, d in zip(h_s[:2] + h_s[-2:], flat_s[:2] + flat_s[-2:]))
        out.update({"value": round(val_zc, 2), "ms_per_step": round(ms_zc, 3),
                    "mode": "zero_copy: kernels read inputs from / write results to pinned host memory",
                    "h2d_bytes_per_step": 2 * wl.num_ranks * wl.psi + 2 * wl.psi,
                    "d2h_bytes_per_step": 4 * sum(job.shard_numel) * wl.num_ranks + 2 * wl.psi,
                    "results_match_device_run": bool(same)})
    else:
        out.update({"value": ce["value"], "ms_per_step": ce["ms_per_step"], "mode": "copy_engine",
                    "h2d_bytes_per_step": ce["h2d_bytes_per_step"],
                    "d2h_bytes_per_step": ce["d2h_bytes_per_step"]})
    del h_g, h_s, h_buf, h_p
    return out


def run_interference(tide, layout, job, wl, props, smi_dev, repeats=3, window_s=0.3):
    """Slowdown of a bf16 8192^3 GEMM on one stream while the reduce-scatter
    (or placement) loops on another, per mode; the op's bandwidth during the
    GEMM window and its SM.time.  Modes marked `_lowprio` put the GEMM on a
    high-priority stream and the op on a low-priority one: the block
    scheduler then dispatches pending GEMM CTAs first, and the op's
    one-CTA-per-tile launches fill whatever the GEMM leaves.

    Per mode, `repeats` pairs of windows of at least `window_s` seconds each
    (several nvidia-smi samples per window): the GEMMs alone, then the same
    number of GEMMs beside the op.  Reported: the median slowdown and its
    range over the repeats, and the slowdown in GEMM clock cycles (window
    time x median SM clock of the window), which takes out the part a lower
    clock under the shared power cap explains."""
    import math

    import torch

    n = 8192
    a = torch.randn(n, n, dtype=torch.bfloat16, device="cuda")
    b = torch.randn(n, n, dtype=torch.bfloat16, device="cuda")
    c = torch.empty(n, n, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()  # the operands are written on the default stream
    least, greatest = torch.cuda.Stream.priority_range()
    streams = {False: (torch.cuda.Stream(), torch.cuda.Stream()),
               True: (torch.cuda.Stream(priority=greatest), torch.cuda.Stream(priority=least))}
    gptr = tide.PointerTable(job.grad_ptrs())
    sptr = tide.PointerTable(job.shard_ptrs())
    pptr = tide.PointerTable(job.param_ptrs())

    def gemm_window(sg, count):
        """Events around `count` back-to-back GEMMs on sg (not synchronised)."""
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(sg):
            e0.record(sg)
            for _ in range(count):
                torch.matmul(a, b, out=c)
            e1.record(sg)
        return e0, e1

    def gemm_alone(sg, count):
        e0, e1 = gemm_window(sg, count)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / count

    def concurrent(sg, sr, op, count, launches, nbytes):
        """`launches` op launches on sr (an event pair each), enqueued by a
        second host thread, and `count` GEMMs on sg enqueued by this one once
        the op loop has started: GEMM ms, bytes the op moved inside the GEMM
        window, mean op launch ms.  Enqueuing both at once keeps an op whose
        calls cost more host time than device time (the copy-engine
        placement of many tensors) running beside the GEMMs."""
        evs = []

        def enqueue_ops():
            with torch.cuda.stream(sr):
                for _ in range(launches):
                    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    x0.record(sr)
                    op()
                    x1.record(sr)
                    evs.append((x0, x1))

        th = threading.Thread(target=enqueue_ops)
        th.start()
        time.sleep(0.002)
        e0, e1 = gemm_window(sg, count)
        th.join()
        torch.cuda.synchronize()
        window = e0.elapsed_time(e1)
        moved = 0.0
        for x0, x1 in evs:
            st, en = e0.elapsed_time(x0), e0.elapsed_time(x1)
            if en > st:
                moved += nbytes * max(0.0, min(en, window) - max(st, 0.0)) / (en - st)
        return window / count, moved / (window * 1e-3) / 1e9, evs[0][0].elapsed_time(evs[-1][1]) / launches

    for prio in (False, True):
        for _ in range(3):
            gemm_window(streams[prio][0], 8)
    torch.cuda.synchronize()
    t0 = statistics.median(gemm_alone(streams[False][0], 8) for _ in range(5))
    t0_hi = statistics.median(gemm_alone(streams[True][0], 8) for _ in range(5))
    count = max(8, math.ceil(window_s * 1e3 / t0))
    flops = 2 * n ** 3
    res = {"gemm": f"bf16 {n}x{n}x{n} torch.matmul", "gemm_ms_alone": round(t0, 4),
           "gemm_tflops_alone": round(flops / (t0 * 1e-3) / 1e12, 1),
           "gemm_ms_alone_high_priority": round(t0_hi, 4),
           "stream_priorities": {"least": least, "greatest": greatest},
           "windows": f"{repeats} repeats per mode of {count} GEMMs alone, then {count} GEMMs beside the op",
           "op_GB/s_during_gemm": "bytes the op moved inside the GEMM window (each launch weighted by "
                                  "its overlap with the window) / window length",
           "slowdown_cycles": "slowdown of GEMM time x median SM MHz of its window (clock-normalised)",
           "modes": []}
    U, C, B, CE = (tide.TIDE_MODE_UNCAPPED, tide.TIDE_MODE_CAPPED, tide.TIDE_MODE_BULK,
                   tide.TIDE_MODE_COPY_ENGINE)
    modes = [("rs", "uncapped", U, 0, False), ("rs", "uncapped_lowprio", U, 0, True)]
    modes += [("rs", f"capped{cap}", C, cap, False) for cap in (8, 16, 32, 64)]
    modes += [("rs", f"bulk_tma_capped{cap}", B, cap, False) for cap in (8, 16, 32, 64)]
    modes += [("rs", "bulk_tma_uncapped", B, 0, False), ("rs", "bulk_tma_uncapped_lowprio", B, 0, True)]
    modes += [("ag", "uncapped", U, 0, False), ("ag", "uncapped_lowprio", U, 0, True),
              ("ag", "bulk_tma", B, 0, False), ("ag", "bulk_tma_lowprio", B, 0, True),
              ("ag", "capped16", C, 16, False), ("ag", "copy_engine", CE, 0, False)]
    sampler = ClockSampler(smi_dev)
    sampler.start()
    time.sleep(0.2)
    for kind, name, mode, cap, prio in modes:
        sg, sr = streams[prio]
        layout.set_mode(mode, cap)
        if kind == "rs":
            def op():
                layout.reduce_scatter(gptr, sptr, wl.scale, sr)
            nbytes = wl.rs_bytes()
            opname = tide.TIDE_OP_RS
        else:
            def op():
                layout.place(job.gathered, pptr, sr)
            nbytes = wl.ag_bytes()
            opname = tide.TIDE_OP_AG
        with torch.cuda.stream(sr):
            op()
            torch.cuda.synchronize()
            x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            x0.record(sr)
            for _ in range(3):
                op()
            x1.record(sr)
        torch.cuda.synchronize()
        alone_ms = x0.elapsed_time(x1) / 3
        # a short probe sizes the op loop of the long windows: it must cover the GEMMs
        base_p = gemm_alone(sg, 8)
        t1_p, _, _ = concurrent(sg, sr, op, 8, max(2, int(2 * 8 * base_p * 5 / max(alone_ms, 1e-3)) + 2), nbytes)
        reps = []
        for _ in range(repeats):
            h0 = time.time()
            base = gemm_alone(sg, count)
            h1 = time.time()
            launches = max(2, math.ceil(1.3 * count * t1_p / max(alone_ms, 1e-3)) + 2)
            t1, during, loop_ms = concurrent(sg, sr, op, count, launches, nbytes)
            h2 = time.time()
            cb, cc = sampler.summary(h0, h1), sampler.summary(h1, h2)
            r = {"gemm_ms_alone": base, "gemm_ms_concurrent": t1, "during": during, "loop_ms": loop_ms,
                 "slowdown": 100.0 * (t1 / base - 1.0), "mhz_alone": cb["sm_mhz"], "mhz_concurrent": cc["sm_mhz"],
                 "samples": (cb.get("samples") or 0) + (cc.get("samples") or 0),
                 "reasons": sorted(set(cb["reasons"]) | set(cc["reasons"]))}
            if cb["sm_mhz"] and cc["sm_mhz"]:
                r["slowdown_cycles"] = 100.0 * (t1 * cc["sm_mhz"] / (base * cb["sm_mhz"]) - 1.0)
            reps.append(r)
        grid, _ = layout.launch_shape(opname)
        sm_used = min(grid, props.multi_processor_count) if grid else 0
        sl = [r["slowdown"] for r in reps]
        cyc = [r["slowdown_cycles"] for r in reps if "slowdown_cycles" in r]
        med = lambda xs, k=None: statistics.median(xs) if xs else None  # noqa: E731
        res["modes"].append({
            "op": kind, "mode": name, "grid": grid,
            "priority": "gemm high, op low" if prio else "equal",
            "op_ms_alone": round(alone_ms, 4),
            "op_GB/s_alone": round(nbytes / (alone_ms * 1e-3) / 1e9, 1),
            "op_ms_concurrent": round(med([r["loop_ms"] for r in reps]), 4),
            "op_GB/s_during_gemm": round(med([r["during"] for r in reps]), 1),
            "gemm_ms_alone": round(med([r["gemm_ms_alone"] for r in reps]), 4),
            "gemm_ms_concurrent": round(med([r["gemm_ms_concurrent"] for r in reps]), 4),
            "gemm_slowdown_pct": round(med(sl), 2),
            "gemm_slowdown_pct_range": [round(min(sl), 2), round(max(sl), 2)],
            "gemm_slowdown_cycles_pct": round(med(cyc), 2) if cyc else None,
            "sm_ms": round(alone_ms * sm_used, 2),
            "clocks": {"sm_mhz_alone": med([r["mhz_alone"] for r in reps if r["mhz_alone"]]),
                       "sm_mhz_concurrent": med([r["mhz_concurrent"] for r in reps if r["mhz_concurrent"]]),
                       "samples": sum(r["samples"] for r in reps),
                       "reasons": sorted(set().union(*[r["reasons"] for r in reps]))},
        })
    res["clocks"] = sampler.stop()
    layout.set_mode(tide.TIDE_MODE_UNCAPPED, 0)
    del a, b, c
    return res


def interference_summary(res):
    """One short row per mode, for the end of the JSON line."""
    short = {"sw_power_cap": "pcap", "hw_slowdown": "HW", "hw_thermal_slowdown": "HWT",
             "sw_thermal_slowdown": "SWT"}
    rows = []
    for m in res["modes"]:
        if m["op"] == "ag" and m["mode"] not in ("uncapped_lowprio", "copy_engine"):
            continue
        c = m["clocks"]
        rows.append([f"{m['op']} {m['mode']}", m["grid"], m["gemm_slowdown_pct"], m["gemm_slowdown_pct_range"],
                     m["gemm_slowdown_cycles_pct"], round(m["op_GB/s_during_gemm"]),
                     round(c["sm_mhz_concurrent"] or 0), round(c["sm_mhz_alone"] or 0), c["samples"],
                     "+".join(short.get(x, x) for x in c["reasons"])])
    return {"gemm_ms_alone": res["gemm_ms_alone"],
            "cols": "mode, grid, GEMM slowdown % (median), [min, max] over repeats, slowdown % in cycles, "
                    "op GB/s during GEMM, SM MHz beside op, SM MHz GEMM alone, clock samples, reasons",
            "rows": rows}


def run_ipc(args):
    """One process per rank (N = world size) over peer memory: rank r keeps its
    own gradients of every parameter and its rank-major buffer, maps its
    peers' (CUDA IPC), and each step runs the single-rank reduce-scatter on
    the pointer table of every rank's gradients, packs its shard into its own
    block, waits on the host for every rank's pack, places every block
    straight from its rank's buffer, and waits again.  Ranks map to devices
    round-robin; handles, barriers and the max-over-ranks time go over gloo.
    With fewer GPUs than ranks the processes share GPUs: a functional run of
    the multi-process path, not a multi-GPU measurement."""
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    ndev = torch.cuda.device_count()
    torch.cuda.set_device(local % ndev)
    if world > 1:
        dist.init_process_group("gloo")
    import layout_aware_collectives_gb300 as tide
    from layout_aware_collectives_gb300 import ipc
    import synth
    from synth.device import fill_bf16

    base = synth.WORKLOADS[args.config]()
    wl = synth.Workload(f"{base.name}_ipc{world}", world, base.shapes, base.names, base.sigma, base.seed,
                        base.outlier_every, base.outlier_mult, base.zero_groups, base.zero_pct)
    lay = tide.Layout(wl.shapes, world)
    P = wl.num_params
    numels = [synth.numel(s) for s in wl.shapes]
    offs, total = ipc.arena_offsets(numels, 2)
    arena = torch.empty(total // 2, dtype=torch.int16, device="cuda")
    for p, (o, n) in enumerate(zip(offs, numels)):
        if n and not wl.zero_grad(rank, p):
            fill_bf16(arena[o // 2: o // 2 + n], wl.grad_key(rank, p), 0, wl.sigma, wl.outlier_every,
                      wl.outlier_mult)
        elif n:
            arena[o // 2: o // 2 + n].zero_()
    S = lay.block_numel
    gathered = torch.zeros(world * S, dtype=torch.int16, device="cuda")
    shards = [torch.empty(lay.shard_numel(p), dtype=torch.float32, device="cuda") for p in range(P)]
    params = [torch.empty(n, dtype=torch.int16, device="cuda") for n in numels]
    torch.cuda.synchronize()
    mine = {"grads": tide.tide_ipc_export(arena), "gathered": tide.tide_ipc_export(gathered)}
    ex = ipc.exchange(mine) if world > 1 else [mine]
    peers = ipc.PeerMap()
    gtab = tide.PointerTable(ipc.grad_table(ipc.rank_addresses(ex, rank, "grads", arena.data_ptr(), peers), offs))
    btab = tide.PointerTable(ipc.rank_addresses(ex, rank, "gathered", gathered.data_ptr(), peers))
    stab, ptab = tide.PointerTable(shards), tide.PointerTable(params)
    stream = torch.cuda.Stream()

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        lay.reduce_scatter_rank(rank, gtab, stab, wl.scale, stream)
        if ev:
            ev[1].record(stream)
        lay.pack(rank, stab, gathered, stream)
        stream.synchronize()
        barrier(world)  # every rank's block is packed before anyone reads it
        if ev:
            ev[2].record(stream)
        lay.place_ranks(btab, ptab, stream)
        if ev:
            ev[3].record(stream)
        stream.synchronize()
        barrier(world)  # every peer has read this rank's block before it is packed again

    for _ in range(max(3, args.warmup)):
        step()
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K):
        step(evs[i])
    torch.cuda.synchronize()
    barrier(world)
    step_ms = reduce_max((time.perf_counter() - t0) * 1e3 / K, world)
    rs_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    ag_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    # each rank in turn, the others waiting at a barrier: its kernels alone on
    # the GPU, reading its peers' memory through the IPC mappings
    dims = [synth.dim0_inner(s) for s in wl.shapes]
    valid_r = sum(lay.valid_rows(p, rank) * inner for p, (_, inner) in enumerate(dims))
    turns = {}
    for turn in range(world):
        barrier(world)
        if turn == rank:
            with torch.cuda.stream(stream):
                lay.reduce_scatter_rank(rank, gtab, stab, wl.scale, stream)
                lay.place_ranks(btab, ptab, stream)
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                reps = 10
                ev[0].record(stream)
                for _ in range(reps):
                    lay.reduce_scatter_rank(rank, gtab, stab, wl.scale, stream)
                ev[1].record(stream)
                for _ in range(reps):
                    lay.place_ranks(btab, ptab, stream)
                ev[2].record(stream)
            torch.cuda.synchronize()
            rs_t = ev[0].elapsed_time(ev[1]) / reps
            pl_t = ev[1].elapsed_time(ev[2]) / reps
            turns = {"rs_ms": round(rs_t, 4),
                     "rs_GB/s": round((2 * world + 4) * valid_r / (rs_t * 1e-3) / 1e9, 1),
                     "place_ms": round(pl_t, 4), "place_GB/s": round(4 * wl.psi / (pl_t * 1e-3) / 1e9, 1)}
        barrier(world)
    if world > 1:
        every = [None] * world
        dist.all_gather_object(every, turns)
    else:
        every = [turns]
    # bytes every rank moves per step: its reduce-scatter (N bf16 reads and one
    # fp32 write per valid element of its shards), its pack (6 bytes per
    # padded shard element) and the placement of every parameter (4 bytes per
    # element)
    total_bytes = 0
    for r in range(world):
        valid = sum(lay.valid_rows(p, r) * inner for p, (_, inner) in enumerate(dims))
        padded = sum(lay.shard_numel(p) for p in range(P))
        total_bytes += (2 * world + 4) * valid + 6 * padded + 4 * wl.psi
    value = total_bytes / (step_ms * 1e-3) / 1e9
    if rank == 0:
        emit({"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": min(world, ndev),
              "steps": K, "warmup": max(3, args.warmup), "ms_per_step": round(step_ms, 4),
              "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
              "data": "synthetic", "collective": "ipc",
              "config": {"workload": wl.name, "num_ranks": world, "num_params": P, "psi": wl.psi,
                         "parallelism": f"ipc ranks x{world} on {min(world, ndev)} GPU(s)",
                         "step": "RS of this rank over every rank's gradients + pack + host barrier + "
                                 "placement from every rank's buffer + host barrier"},
              "rank0_kernels": {"rs_ms": round(rs_ms, 4), "place_ms": round(ag_ms, 4)},
              "ranks_in_turn": every,
              "ranks_in_turn_note": "each rank's single-rank reduce-scatter (over every rank's gradients, its "
                                    "peers' through CUDA IPC) and per-rank placement timed alone on the GPU "
                                    "while the other ranks wait",
              "note": "ranks share GPUs when there are fewer GPUs than ranks: a functional run of the "
                      "multi-process path, not a multi-GPU measurement"}, args)
    barrier(world)
    peers.close()
    barrier(world)
    lay.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.collective == "ipc":
        return run_ipc(args)
    if args.hbm_mix_only:
        import torch

        torch.cuda.set_device(0)
        emit({"hbm_mix": run_hbm_mix([1, 2, 4, 8, 16], smi_device(0)), "device": torch.cuda.get_device_name(0),
              "peak_copy_gbs": measured_peaks()[0]}, args)
        return 0
    return run_tide(args)


if __name__ == "__main__":
    sys.exit(main())
