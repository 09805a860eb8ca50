"""Benchmark of the fused residual-add + RMSNorm + FP8 / NVFP4 / MXFP4 path on GB300.

One step is one pass of the whole hot path over one batch of each of the three large workloads,
at their stated shapes and distributions, each resident in HBM:
  fp8    fp8_gemma        16384 x 8192 fp16 + residual, weight_offset 1, scale_ub 10
  nvfp4  nvfp4            32768 x 7168 bf16, no residual, global scale from the device pre-pass
                          (run once, before the timed region)
  mxfp4  mxfp4_residual   65536 x 16384 bf16 + residual (the largest shape of the sweep)
A step reads about 5 GB of distinct inputs -- far more than the 129 MB L2 -- so every launch
streams from HBM and no flush is needed.

Prints one JSON line:
  value      whole-job GB/s of algorithmic bytes (each launch's reads + writes counted once),
             inputs resident in HBM, CUDA-event timed over exactly K steps
  per_mode   each kernel's average launch time and GB/s (events on the launching stream around
             its launches in every 5th timed step, from step 2 on)
  rooflines  per kernel: those GB/s against the measured HBM copy bandwidth, the DRAM bytes of
             one launch from the committed ncu capture (when taken on the current kernel
             sources), and what a plain device copy of the same bytes reaches
  roofline   the entry of the dominant kernel (the longest launch)
  e2e        the same metric through the public API with host buffers: pinned host -> device
             copies of the step's inputs and device -> host copies of its outputs inside the
             timed region, overlapped with the kernels on separate copy streams; beside it, the
             same copies timed alone (the floor the host link sets)
  cpu_baseline  the oracle on a bounded row sample of the same three workloads, on this host's
             cores

--impl reference times the oracle itself as the reference arm, on the same config. --report runs
every workload (fp8_small ... the MXFP4 sweep) and prints one JSON line per workload with its
GB/s. Multi-GPU (torchrun): every rank runs an independent replica (the path has no exchange
step); value is the sum of all ranks' bytes over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "achieved HBM GB/s & rows/s, fused RMSNorm+FP8/FP4 quant, % of GB300 8 TB/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
MODES = ("fp8", "nvfp4", "mxfp4")
# the step: one batch per quantisation mode, at the workload's stated shape
STEP_WORKLOADS = {
    "fp8": W.config("fp8_gemma"),
    "nvfp4": W.config("nvfp4"),
    "mxfp4": W.config("mxfp4_residual", rows=65536, hidden=16384),
}
KERNEL_NAMES = {"fp8": "rmsnorm_quant_fp8", "nvfp4": "rmsnorm_quant_nvfp4",
                "mxfp4": "rmsnorm_quant_mxfp4"}
# largest row sample of each workload the oracle is timed on (a fraction of its rows)
ORACLE_MAX_FRACTION = 1.0 / 8


# ------------------------------------------------------------------------------------------
# helpers
# ------------------------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_sha():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "rmsnorm_precision_activation_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def workload_label(w):
    return "%s %dx%d" % (w.name, w.rows, w.hidden)


def recorded_traffic(mode, w):
    """Per-launch DRAM bytes (read + write) of the `mode` kernel on workload w from the committed
    ncu summary, if it was taken on the current kernel sources and on that workload; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("source_sha") != kernel_source_sha():
        return None
    e = d.get("kernels", {}).get(mode)
    if e is None or e.get("workload") != workload_label(w):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def parse_step_workloads(spec):
    """`mode=name[:rows:hidden],...` -> {mode: Workload}, over STEP_WORKLOADS (for experiments
    on other shapes; the default step is STEP_WORKLOADS)."""
    out = dict(STEP_WORKLOADS)
    if not spec:
        return out
    out = {}
    for item in spec.split(","):
        mode, rest = item.split("=", 1)
        parts = rest.split(":")
        rows = int(parts[1]) if len(parts) > 1 else None
        hidden = int(parts[2]) if len(parts) > 2 else None
        w = W.config(parts[0], rows=rows, hidden=hidden)
        if w.mode != mode:
            raise SystemExit("workload %s is not a %s workload" % (parts[0], mode))
        out[mode] = w
    return out


def step_config(workloads, world):
    """The `config` object of the JSON line (identical in both arms)."""
    inputs = sum(w.rows * w.hidden * 2 * (2 if w.residual else 1) for w in workloads.values())
    desc = []
    for m, w in workloads.items():
        d = "%s %s %dx%d %s%s" % (m, w.name, w.rows, w.hidden, w.dtype,
                                  " +residual" if w.residual else "")
        if m == "fp8":
            d += " offset %g ub %g" % (w.weight_offset, w.scale_ub)
        desc.append(d)
    return {
        "workload": "fused residual-add + RMSNorm + quantisation, one batch per mode: "
                    + "; ".join(desc),
        "workloads": {m: {"name": w.name, "rows": w.rows, "hidden": w.hidden,
                          "io_dtype": w.dtype, "residual": w.residual,
                          "weight_offset": w.weight_offset,
                          **({"scale_ub": w.scale_ub} if m == "fp8" else {}),
                          **({"global_scale": "device pre-pass, before the timed region"}
                             if m == "nvfp4" else {})}
                      for m, w in workloads.items()},
        "l2": "inputs larger than L2: %d MiB of distinct inputs per step, no flush"
              % (inputs // (1 << 20)),
        "parallelism": "replicas" if world > 1 else "single GPU",
    }


# ------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------

class Step:
    """Resident buffers for one step: one batch per mode at its workload's shape, outputs, the
    NVFP4 global scale (device pre-pass, computed once here), and the launches."""

    def __init__(self, rq, device, workloads=None, seed=0):
        self.rq = rq
        self.workloads = dict(STEP_WORKLOADS if workloads is None else workloads)
        self.batches, self.out = {}, {}
        dev = device
        for k, (mode, w) in enumerate(self.workloads.items()):
            d = W.generate(w, seed=seed + k, device=dev)
            self.batches[mode] = d
            rows, hidden = w.rows, w.hidden
            ro = torch.empty(rows, hidden, dtype=w.torch_dtype, device=dev) if w.residual else None
            if mode == "fp8":
                self.out[mode] = (torch.empty(rows, hidden, dtype=torch.float8_e4m3fn, device=dev),
                                  torch.empty(rows, dtype=torch.float32, device=dev), ro)
            elif mode == "nvfp4":
                self.out[mode] = (torch.empty(rows, hidden // 2, dtype=torch.uint8, device=dev),
                                  torch.empty(rows, hidden // 16, dtype=torch.float8_e4m3fn,
                                              device=dev), ro)
            else:
                self.out[mode] = (torch.empty(rows, hidden // 2, dtype=torch.uint8, device=dev),
                                  torch.empty(rows, hidden // 32, dtype=torch.uint8, device=dev),
                                  ro)
        self.gs = None
        if "nvfp4" in self.workloads:
            w, nb = self.workloads["nvfp4"], self.batches["nvfp4"]
            self.gs = rq.rmsnorm_nvfp4_global_scale(nb["input"], nb["gamma"],
                                                    residual=nb["residual"], epsilon=w.eps,
                                                    weight_offset=w.weight_offset)
        self.modes = tuple(self.workloads)
        self.bytes = {m: w.algorithmic_bytes() for m, w in self.workloads.items()}
        self.step_bytes = sum(self.bytes.values())
        self.step_rows = sum(w.rows for w in self.workloads.values())

    def launch(self, mode, stream=None, rows=None):
        """Queue mode's kernel on its batch, or on rows [r0, r1) of it (rows=(r0, r1))."""
        d, o, w, rq = self.batches[mode], self.out[mode], self.workloads[mode], self.rq
        if rows is not None:
            r0, r1 = rows
            d = {k: (v if v is None or k == "gamma" else v[r0:r1]) for k, v in d.items()}
            o = tuple(None if t is None else t[r0:r1] for t in o)
        if mode == "fp8":
            rq.rmsnorm_quant_fp8(d["input"], d["gamma"], residual=d["residual"], residual_output=o[2],
                                 epsilon=w.eps, weight_offset=w.weight_offset, scale_ub=w.scale_ub,
                                 output=o[0], scale_output=o[1], stream=stream)
        elif mode == "nvfp4":
            rq.rmsnorm_quant_nvfp4(d["input"], d["gamma"], global_scale=self.gs,
                                   residual=d["residual"], residual_output=o[2], epsilon=w.eps,
                                   weight_offset=w.weight_offset, output=o[0], block_scale=o[1],
                                   stream=stream)
        else:
            rq.rmsnorm_quant_mxfp4(d["input"], d["gamma"], residual=d["residual"],
                                   residual_output=o[2], epsilon=w.eps,
                                   weight_offset=w.weight_offset, output=o[0], block_scale=o[1],
                                   stream=stream)


def barrier_max(value, world):
    """The maximum of `value` over all ranks (NCCL on the GPUs, or gloo on the CPU)."""
    if world == 1:
        return value
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(step_bytes, steps, world, local_ms):
    """Whole-job GB/s of `world` independent replicas, each moving step_bytes per step: all
    ranks' bytes over the slowest rank's time. Returns (GB/s, slowest rank's ms)."""
    ms = barrier_max(local_ms, world)
    return step_bytes * steps * world / (ms * 1e-3) / 1e9, ms


def same_bytes_copy_gbs(nbytes, device, reps=10):
    """GB/s of a plain device-to-device copy that moves `nbytes` (half read, half written), the
    size of one launch. L2 is filled with clean lines by a 256 MiB read before each copy, so the
    copy reads from DRAM as the kernels do. Median of `reps` event-timed copies after 3
    warm-ups. Reported beside each roofline: what a copy reaches at the launch's size."""
    n = nbytes // 2 // 16 * 16
    src = torch.full((n,), 3, dtype=torch.uint8, device=device)
    dst = torch.empty_like(src)
    flush = torch.ones(64 << 20, dtype=torch.float32, device=device)
    times = []
    for i in range(reps + 3):
        flush.amax()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src)
        b.record()
        torch.cuda.synchronize()
        if i >= 3:
            times.append(a.elapsed_time(b))
    del src, dst, flush
    return 2 * n / statistics.median(times) / 1e6


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def probed_steps(K):
    """The timed steps whose launches get their own events: every 5th from step 2. An event
    recorded between two kernels ends the programmatic overlap of the second with the first, so
    the other steps run without them; the first steps are left out because the GPU can still be
    waiting for the host there."""
    return [i for i in range(K) if i % 5 == 2] or [K - 1]


def roofline_entry(mode, w, us, peak, peak_src, copy_gbs):
    gbs = w.algorithmic_bytes() / (us * 1e-6) / 1e9
    return {"bound": "hbm", "kernel": KERNEL_NAMES[mode], "workload": workload_label(w),
            "achieved": round(gbs, 1), "peak": peak,
            "peak_source": peak_src + " (MEASURED_PEAKS hbm_gbs, copy)", "unit": "GB/s",
            "frac": round(gbs / peak, 4), "traffic": recorded_traffic(mode, w),
            "algorithmic_bytes_per_launch": w.algorithmic_bytes(), "us": round(us, 2),
            "copy_same_bytes_gbs": round(copy_gbs, 1)}


def run_ours(args):
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    from rmsnorm_precision_activation_gb300 import build as B
    B.build()
    import rmsnorm_precision_activation_gb300 as rq
    if args.no_pdl:
        rq.rmsq_set_pdl(False)

    device = torch.device("cuda", local)
    step = Step(rq, device, parse_step_workloads(args.step_workloads))
    modes = step.modes
    stream = torch.cuda.current_stream(device)

    for _ in range(args.warmup):
        for m in modes:
            step.launch(m)
    torch.cuda.synchronize()

    K = args.steps
    probed = probed_steps(K)
    ev = {m: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in probed] for m in modes}
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = rq.rmsq_launch_count()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t0.record(stream)
        j = 0
        for i in range(K):
            probe = i in probed
            for m in modes:
                if probe:
                    ev[m][j][0].record(stream)
                step.launch(m)
                if probe:
                    ev[m][j][1].record(stream)
            j += probe
        t1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    launches = rq.rmsq_launch_count() - launches0
    value, total_ms = replica_throughput(step.step_bytes, K, world, t0.elapsed_time(t1))
    per_mode_ms = {m: statistics.mean(a.elapsed_time(b) for a, b in ev[m]) for m in modes}
    assert rq.rmsq_device_status() == 0

    # ---- end to end through the public API with host buffers -------------------------------
    e2e = run_e2e(step, device, max(3, min(K, 10)), world)

    peak, peak_src = measured_peak()
    rooflines = {}
    for m in modes:
        copy_gbs = same_bytes_copy_gbs(step.bytes[m], device)
        rooflines[m] = roofline_entry(m, step.workloads[m], per_mode_ms[m] * 1e3, peak,
                                      peak_src, copy_gbs)
    dom = max(per_mode_ms, key=per_mode_ms.get)
    roof = dict(rooflines[dom])
    roof["timing"] = ("CUDA events on the launching stream around each launch of timed steps %s"
                      % ",".join(str(i) for i in probed))
    rows_per_s = step.step_rows * K * world / (total_ms * 1e-3)
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / K, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded; each workload's stated distributions)",
        "config": step_config(step.workloads, world),
        "rows_per_s": round(rows_per_s),
        "pct_of_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "per_mode": {m: {"workload": workload_label(step.workloads[m]),
                         "us": round(per_mode_ms[m] * 1e3, 2),
                         "gbs": round(step.bytes[m] / (per_mode_ms[m] * 1e-3) / 1e9, 1),
                         "algorithmic_bytes": step.bytes[m]} for m in modes},
        "roofline": roof,
        "rooflines": rooflines,
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": clocks.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(step.workloads, seconds=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


E2E_CHUNK_BYTES = 512 << 20


def e2e_chunks(w, chunk_bytes=E2E_CHUNK_BYTES, row_align=16):
    """Row ranges [r0, r1) that split workload w's batch into pieces of about chunk_bytes of
    input each. Every piece starts on a multiple of row_align rows, so the pointers an entry
    point gets for it stay 16-byte aligned (an FP8 row scale is 4 bytes, or 2)."""
    per_row = w.hidden * torch.tensor([], dtype=w.torch_dtype).element_size() * (2 if w.residual else 1)
    n = max(1, min(w.rows, -(-w.rows * per_row // chunk_bytes)))
    bounds = [w.rows * i // n // row_align * row_align for i in range(n)] + [w.rows]
    return [(a, b) for a, b in zip(bounds, bounds[1:]) if b > a]


def run_e2e(step, device, K, world):
    """Same step through the public API, inputs from pinned host memory and outputs back to
    pinned host memory inside the timed region.

    The batches move through three streams, the way a caller overlaps transfers with compute:
    one stream copies inputs in (pinned host -> device), the launch stream runs the kernels, and
    one stream copies outputs back (device -> pinned host). Each batch goes in row chunks of
    about 512 MB of input (rows are independent, so a chunk is one call of the entry point on
    those rows): a chunk's kernel starts once its rows are in, and its outputs leave while the
    next chunk comes in, so the link is busy in both directions from the first chunk to the
    last. Events order each chunk's copy-in, kernel and copy-out. They also stop a copy-in from
    overwriting inputs that the chunk's previous kernel still reads, and a kernel from
    overwriting outputs that are still being copied out."""
    modes = step.modes

    def pinned_like(t):
        return torch.empty(t.shape, dtype=t.dtype, pin_memory=True)

    host_in = {}
    for m in modes:
        host_in[m] = {}
        for k, v in step.batches[m].items():
            if v is not None:
                h = pinned_like(v)
                h.copy_(v)
                host_in[m][k] = h
    host_out = {m: tuple(pinned_like(t) for t in step.out[m] if t is not None) for m in modes}
    dev_out = {m: tuple(t for t in step.out[m] if t is not None) for m in modes}
    h2d = sum(t.numel() * t.element_size() for d in host_in.values() for t in d.values())
    d2h = sum(t.numel() * t.element_size() for o in host_out.values() for t in o)
    chunks = [(m, r0, r1) for m in modes for r0, r1 in e2e_chunks(step.workloads[m])]
    compute = torch.cuda.current_stream(device)
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    in_done = {c: torch.cuda.Event() for c in chunks}
    ker_done = {c: torch.cuda.Event() for c in chunks}
    out_done = {c: torch.cuda.Event() for c in chunks}
    for c in chunks:
        ker_done[c].record(compute)
        out_done[c].record(compute)

    def one():
        for c in chunks:
            m, r0, r1 = c
            s_in.wait_event(ker_done[c])
            with torch.cuda.stream(s_in):
                for k, t in host_in[m].items():
                    if k == "gamma":
                        if r0 == 0:
                            step.batches[m][k].copy_(t, non_blocking=True)
                    else:
                        step.batches[m][k][r0:r1].copy_(t[r0:r1], non_blocking=True)
            in_done[c].record(s_in)
            compute.wait_event(in_done[c])
            compute.wait_event(out_done[c])
            step.launch(m, stream=compute, rows=(r0, r1))
            ker_done[c].record(compute)
            s_out.wait_event(ker_done[c])
            with torch.cuda.stream(s_out):
                for dst, src in zip(host_out[m], dev_out[m]):
                    dst[r0:r1].copy_(src[r0:r1], non_blocking=True)
            out_done[c].record(s_out)

    one()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    a.record(compute)
    s_in.wait_event(a)
    s_out.wait_event(a)
    for _ in range(K):
        one()
    compute.wait_stream(s_out)
    b.record(compute)
    torch.cuda.synchronize()
    value, ms = replica_throughput(step.step_bytes, K, world, a.elapsed_time(b))

    # The same copies with no kernels and no ordering between the two directions: the floor the
    # host link sets under the end-to-end step. Timed after the step, outside its timed region.
    def copies_only():
        for m in modes:
            with torch.cuda.stream(s_in):
                for k, t in host_in[m].items():
                    step.batches[m][k].copy_(t, non_blocking=True)
            with torch.cuda.stream(s_out):
                for dst, src in zip(host_out[m], dev_out[m]):
                    dst.copy_(src, non_blocking=True)

    copies_only()
    torch.cuda.synchronize()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(compute)
    s_in.wait_event(c0)
    s_out.wait_event(c0)
    for _ in range(K):
        copies_only()
    compute.wait_stream(s_in)
    compute.wait_stream(s_out)
    c1.record(compute)
    torch.cuda.synchronize()
    copy_ms = c0.elapsed_time(c1) / K
    del host_in, host_out
    return {"value": round(value, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms / K, 4), "steps": K,
            "copies_only_ms_per_step": round(copy_ms, 4),
            "copies_only_GBs": round((h2d + d2h) / copy_ms / 1e6, 1)}


# ------------------------------------------------------------------------------------------
# the oracle on the host cores
# ------------------------------------------------------------------------------------------

def sample_workloads(workloads, fraction):
    """The same workloads cut to `fraction` of their rows (at least one row each)."""
    import dataclasses
    return {m: dataclasses.replace(w, rows=max(1, int(round(w.rows * fraction))))
            for m, w in workloads.items()}


def oracle_sample(workloads, fraction, seed=0):
    """A callable that runs the oracle, as it stands, over a `fraction` row sample of every
    workload of the step (inputs drawn with the workloads' own recipes), and the sample's
    algorithmic bytes and rows."""
    import numpy as np
    import oracle
    sample = sample_workloads(workloads, fraction)
    calls = []
    for k, (m, w) in enumerate(sample.items()):
        d = W.generate(w, seed=seed + k)
        x, g = W.bits(d["input"]), W.bits(d["gamma"])
        r = None if d["residual"] is None else W.bits(d["residual"])
        odt = {"bf16": oracle.BF16, "fp16": oracle.FP16}[w.dtype]
        kw = dict(dtype=odt, eps=w.eps, weight_offset=w.weight_offset)
        if m == "fp8":
            calls.append(lambda x=x, r=r, g=g, ub=w.scale_ub, kw=kw:
                         oracle.quant_fp8(x, r, g, scale_ub=ub, **kw))
        elif m == "nvfp4":
            y = oracle.rmsnorm(x, r, g, **kw)["y"]
            gs = float(oracle.nvfp4_global_scale(np.abs(y).max()))
            calls.append(lambda x=x, r=r, g=g, gs=gs, kw=kw: oracle.quant_nvfp4(x, r, g, gs, **kw))
        else:
            calls.append(lambda x=x, r=r, g=g, kw=kw: oracle.quant_mxfp4(x, r, g, **kw))

    def run():
        for c in calls:
            c()

    nbytes = sum(w.algorithmic_bytes() for w in sample.values())
    rows = sum(w.rows for w in sample.values())
    return run, nbytes, rows, sample


def describe_sample(sample):
    return ", ".join("%s %d of %d rows" % (w.name, w.rows, STEP_ROWS.get(w.name, w.rows))
                     for w in sample.values())


STEP_ROWS = {w.name: w.rows for w in STEP_WORKLOADS.values()}


def size_oracle_sample(workloads, seconds_per_pass):
    """The row fraction whose oracle pass takes about `seconds_per_pass`, from a timed probe on a
    small fraction; at most ORACLE_MAX_FRACTION."""
    probe = 1.0 / 1024
    run, nb, _, _ = oracle_sample(workloads, probe, seed=900)
    t = time.perf_counter()
    run()
    dt = max(time.perf_counter() - t, 1e-3)
    return min(ORACLE_MAX_FRACTION, probe * seconds_per_pass / dt)


def cpu_baseline(workloads, seconds=15.0):
    import oracle
    oracle.build()
    cores = oracle.cores()
    frac = size_oracle_sample(workloads, seconds / 4)
    run, nb, rows, sample = oracle_sample(workloads, frac, seed=100)
    # Whole passes over the sample until about `seconds` of wall time.
    passes, dt = 0, 0.0
    while passes == 0 or dt < seconds:
        t = time.perf_counter()
        run()
        dt += time.perf_counter() - t
        passes += 1
    return {"value": round(passes * nb / dt / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": "%d pass(es) over %s (%.1f s)" % (passes, describe_sample(sample), dt),
            "rows_per_s": round(rows * passes / dt, 1)}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    cores = oracle.cores()
    workloads = parse_step_workloads(getattr(args, "step_workloads", ""))
    budget = 100.0 / max(1, args.steps + args.warmup)      # whole run within about 2 minutes
    frac = size_oracle_sample(workloads, budget)
    run, nb, rows, sample = oracle_sample(workloads, frac, seed=200)
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        run()
        times.append(time.perf_counter() - t)
    total = sum(times)
    value = nb * args.steps / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; each workload's stated distributions)",
        "config": step_config(workloads, world),
        "rows_per_s": round(rows * args.steps / total, 1),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle",
                         "sample": "each step one pass over %s" % describe_sample(sample)},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------
# per-workload report
# ------------------------------------------------------------------------------------------

def oracle_rate(w, seconds, threads=None):
    """The oracle, as it stands, on a bounded row sample of workload w: GB/s of the sample's
    algorithmic bytes and rows/s, on all host cores unless `threads` is given. The sample is
    grown until it runs for about `seconds`; it is timed best of 3 when it moves under 1 GB, once
    otherwise."""
    import dataclasses
    import numpy as np
    import oracle
    oracle.build()
    odt = {"bf16": oracle.BF16, "fp16": oracle.FP16}[w.dtype]
    kw = dict(dtype=odt, eps=w.eps, weight_offset=w.weight_offset, threads=threads)

    def sample(n):
        ws = dataclasses.replace(w, rows=n)
        d = W.generate(ws, seed=0)
        x, g = W.bits(d["input"]), W.bits(d["gamma"])
        r = None if d["residual"] is None else W.bits(d["residual"])
        if w.mode == "fp8":
            return ws, lambda: oracle.quant_fp8(x, r, g, scale_ub=w.scale_ub, **kw)
        if w.mode == "nvfp4":
            y = oracle.rmsnorm(x, r, g, dtype=odt, eps=w.eps, weight_offset=w.weight_offset)["y"]
            gs = float(oracle.nvfp4_global_scale(np.abs(y).max()))
            return ws, lambda: oracle.quant_nvfp4(x, r, g, gs, **kw)
        return ws, lambda: oracle.quant_mxfp4(x, r, g, **kw)

    def timed(fn):
        t = time.perf_counter()
        fn()
        return time.perf_counter() - t

    n = min(w.rows, 16)
    while True:                      # grow the sample until it runs for about `seconds`
        ws, fn = sample(n)
        dt = timed(fn)
        if dt >= seconds / 2 or n >= w.rows:
            break
        n = int(min(w.rows, max(2 * n, n * seconds / max(dt, 1e-4))))
    nbytes = ws.algorithmic_bytes()
    if nbytes < 1e9:
        dt = min([dt] + [timed(fn) for _ in range(2)])
    return {"gbs": round(nbytes / dt / 1e9, 4), "rows_per_s": round(n / dt, 1),
            "threads": threads or oracle.cores(), "sample_rows": n, "seconds": round(dt, 3)}


def host_cpu():
    """CPU model name and usable cores of this host, for the oracle columns."""
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return {"model": model or os.uname().machine, "cores": len(os.sched_getaffinity(0))}


def report_workloads():
    names = [("fp8_small", None, None), ("fp8_residual", None, None), ("fp8_gemma", None, None),
             ("nvfp4", None, None)]
    names += [("mxfp4_residual", r, h) for r in W.MXFP4_ROWS for h in W.MXFP4_HIDDEN]
    return names


class L2Flush:
    """Evicts L2 between timed repetitions with a 256 MiB pass over a device buffer, about twice
    the 129 MB L2. `write` fills it (the timing rules' flush: the timed launch then also pays
    for writing those dirty lines back); `read` reads it, which leaves only clean lines, for
    kernels that read far more than they write (the global-scale pre-pass writes 4 bytes)."""

    def __init__(self, kind="write"):
        self.kind = kind
        self.buf = (torch.empty(256 << 20, dtype=torch.uint8, device="cuda") if kind == "write"
                    else torch.ones(64 << 20, dtype=torch.float32, device="cuda"))

    def __call__(self):
        if self.kind == "write":
            self.buf.fill_(1)
        else:
            self.buf.amax()


def run_report(args):
    from rmsnorm_precision_activation_gb300 import build as B
    B.build()
    import rmsnorm_precision_activation_gb300 as rq
    torch.cuda.set_device(0)
    peak, _ = measured_peak()
    cpu = host_cpu()
    flush = L2Flush(args.flush)
    only = set(args.only.split(",")) if args.only else None
    for name, rows, hidden in report_workloads():
        if only and name not in only and "%s:%s:%s" % (name, rows, hidden) not in only:
            continue
        w = W.config(name, rows=rows, hidden=hidden)
        d = W.generate(w, seed=0, device="cuda")
        x, r, g = d["input"], d["residual"], d["gamma"]
        if w.mode == "fp8":
            fn = lambda: rq.rmsnorm_quant_fp8(x, g, residual=r, epsilon=w.eps,
                                              weight_offset=w.weight_offset, scale_ub=w.scale_ub)
        elif w.mode == "nvfp4":
            gs = rq.rmsnorm_nvfp4_global_scale(x, g, residual=r, epsilon=w.eps)
            fn = lambda: rq.rmsnorm_quant_nvfp4(x, g, global_scale=gs, residual=r, epsilon=w.eps)
        else:
            fn = lambda: rq.rmsnorm_quant_mxfp4(x, g, residual=r, epsilon=w.eps)
        outs = fn()        # warm + allocate
        for _ in range(3):
            fn()
        times = []
        for _ in range(args.report_reps):
            flush()                             # evict L2 between repetitions
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            times.append(a.elapsed_time(b))
        us = statistics.median(times) * 1e3
        gbs = w.algorithmic_bytes() / (us * 1e-6) / 1e9
        line = {"workload": name, "shape": [w.rows, w.hidden], "io_dtype": w.dtype,
                "mode": w.mode, "residual": w.residual, "us": round(us, 2),
                "algorithmic_bytes": w.algorithmic_bytes(), "gbs": round(gbs, 1),
                "rows_per_s": round(w.rows / (us * 1e-6)),
                "frac_of_measured": round(gbs / peak, 4),
                "pct_of_8tbs": round(100 * gbs / NOMINAL_HBM_GBS, 2), "l2_flush": args.flush}
        del outs, d
        if args.oracle_seconds > 0:
            # the oracle beside the GPU figure: a reported baseline, not the target
            line["oracle"] = {"all_cores": oracle_rate(w, args.oracle_seconds), "cpu": cpu}
            if name in ("fp8_small", "fp8_residual"):
                line["oracle"]["one_thread"] = oracle_rate(w, args.oracle_seconds, threads=1)
        print(json.dumps(line), flush=True)


def next_row_cases():
    """The widened rows, each as (row, case, workload, options). Options: `swizzled` (128x4
    scale layout), `prepass` (time the NVFP4 global-scale pre-pass instead of the quantiser),
    `dtype` (input dtype other than the workload's), `scale_dtype` (FP8 scale output type)."""
    nv = W.config("nvfp4")
    mx = W.config("mxfp4_residual", rows=65536, hidden=8192)
    f8 = W.config("fp8_residual")

    def wide(mode, rows, hidden):
        return W.Workload("wide_rows", mode, rows, hidden, "bf16", True, scale_ub=1200.0)

    return [
        ("NEXT-1", "swizzled_scales", nv, {"swizzled": True}),
        ("NEXT-1", "swizzled_scales", mx, {"swizzled": True}),
        ("NEXT-2", "global_scale_prepass", nv, {"prepass": True}),
        ("NEXT-2", "global_scale_prepass", W.Workload("nvfp4_residual", "nvfp4", 8192, 4096,
                                                      "bf16", True), {"prepass": True}),
        ("NEXT-2", "global_scale_prepass", wide("nvfp4", 4096, 65536), {"prepass": True}),
        ("NEXT-3", "fp32_input", f8, {"dtype": torch.float32}),
        ("NEXT-3", "fp32_input", W.config("mxfp4_residual", rows=4096, hidden=16384),
         {"dtype": torch.float32}),
        ("NEXT-3", "fp16_input", nv, {"dtype": torch.float16}),
        ("NEXT-3", "fp16_input", mx, {"dtype": torch.float16}),
        ("NEXT-3", "bf16_scale_output", f8, {"scale_dtype": torch.bfloat16}),
        ("NEXT-4", "cluster_rows", wide("fp8", 4096, 65536), {}),
        ("NEXT-4", "cluster_rows", wide("nvfp4", 4096, 65536), {}),
        ("NEXT-4", "cluster_rows", wide("mxfp4", 4096, 65536), {}),
        ("NEXT-4", "cluster_rows", wide("fp8", 2048, 131072), {}),
        ("NEXT-4", "cluster_rows", wide("nvfp4", 2048, 131072), {}),
        ("NEXT-4", "cluster_rows", wide("mxfp4", 2048, 131072), {}),
        ("NEXT-4", "cluster_rows_offset", W.config("fp8_gemma", rows=4096, hidden=65536), {}),
        ("NEXT-4", "cluster_rows_no_residual", W.Workload("wide_rows", "fp8", 4096, 65536, "bf16",
                                                          False, scale_ub=1200.0), {}),
        ("NEXT-4", "fp32_input", wide("fp8", 2048, 65536), {"dtype": torch.float32}),
    ]


def variant_bytes(w, opts):
    """Algorithmic bytes of one launch of workload w under `opts` (see next_row_cases): inputs
    read and outputs written once, gamma once per launch. The swizzled layout writes the same
    scale bytes when rows are a multiple of 128 and the scale columns a multiple of 4."""
    e = torch.tensor([], dtype=opts.get("dtype", w.torch_dtype)).element_size()
    n = w.rows * w.hidden
    read = n * e * (2 if w.residual else 1) + w.hidden * e
    if opts.get("prepass"):
        return read + 4                              # max |y| as one fp32 value
    write = n * e if w.residual else 0
    if w.mode == "fp8":
        sd = opts.get("scale_dtype", torch.float32)
        write += n + w.rows * torch.tensor([], dtype=sd).element_size()
    elif w.mode == "nvfp4":
        read += 4
        write += n // 2 + n // 16
    else:
        write += n // 2 + n // 32
    return read + write


def _time_launch(fn, flush, reps):
    fn()
    for _ in range(3):
        fn()
    times = []
    for _ in range(reps):
        flush()                                      # evict L2 between repetitions
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    return statistics.median(times) * 1e3


def run_report_next(args):
    """One JSON line per widened-row case: its event-timed duration and algorithmic GB/s, and
    beside it the same workload with the default options (`base_us`), where there is one."""
    from rmsnorm_precision_activation_gb300 import build as B
    B.build()
    import rmsnorm_precision_activation_gb300 as rq
    torch.cuda.set_device(0)
    peak, _ = measured_peak()
    flush = L2Flush(args.flush)

    def launcher(w, d, opts):
        x, r, g = d["input"], d["residual"], d["gamma"]
        sw = opts.get("swizzled", False)
        if opts.get("prepass"):
            return lambda: rq.rmsnorm_nvfp4_global_scale(x, g, residual=r, epsilon=w.eps)
        if w.mode == "fp8":
            sd = opts.get("scale_dtype", torch.float32)
            return lambda: rq.rmsnorm_quant_fp8(x, g, residual=r, epsilon=w.eps,
                                                weight_offset=w.weight_offset,
                                                scale_ub=w.scale_ub, scale_dtype=sd)
        if w.mode == "nvfp4":
            gs = torch.full((1,), 2.0, dtype=torch.float32, device="cuda")
            return lambda: rq.rmsnorm_quant_nvfp4(x, g, global_scale=gs, residual=r,
                                                  epsilon=w.eps, swizzled=sw)
        return lambda: rq.rmsnorm_quant_mxfp4(x, g, residual=r, epsilon=w.eps, swizzled=sw)

    only = set(args.only.split(",")) if args.only else None
    for row, case, w, opts in next_row_cases():
        key = "%s:%s:%d:%d" % (case, w.mode, w.rows, w.hidden)
        if only and case not in only and key not in only:
            continue
        d = W.generate(w, seed=0, device="cuda")
        if "dtype" in opts:
            d = {k: (None if v is None else v.to(opts["dtype"])) for k, v in d.items()}
        us = _time_launch(launcher(w, d, opts), flush, args.report_reps)
        nb = variant_bytes(w, opts)
        io = {torch.float32: "fp32", torch.float16: "fp16", torch.bfloat16: "bf16"}[d["input"].dtype]
        line = {"row": row, "case": case, "workload": w.name, "shape": [w.rows, w.hidden],
                "mode": w.mode, "io_dtype": io, "residual": w.residual,
                "options": {k: (str(v).replace("torch.", "") if isinstance(v, torch.dtype) else v)
                            for k, v in opts.items()},
                "us": round(us, 2), "algorithmic_bytes": nb, "gbs": round(nb / (us * 1e-6) / 1e9, 1),
                "frac_of_measured": round(nb / (us * 1e-6) / 1e9 / peak, 4), "l2_flush": args.flush}
        if case in ("fp32_input", "fp16_input"):
            db = W.generate(w, seed=0, device="cuda")
            line["base_us"] = round(_time_launch(launcher(w, db, {}), flush, args.report_reps), 2)
            line["base"] = "%s input" % w.dtype
            del db
        elif not case.startswith("cluster_rows"):
            line["base_us"] = round(_time_launch(launcher(w, d, {}), flush, args.report_reps), 2)
            line["base"] = {"swizzled_scales": "row-major scales",
                            "global_scale_prepass": "the NVFP4 quantiser on the same input",
                            "bf16_scale_output": "fp32 scale output"}[case]
        print(json.dumps(line), flush=True)
        del d
        torch.cuda.empty_cache()
    assert rq.rmsq_device_status() == 0


# ------------------------------------------------------------------------------------------
# ncu-backed per-workload table
# ------------------------------------------------------------------------------------------

NCU_UNITS = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "ns": 1e-9, "nsecond": 1e-9, "us": 1e-6,
             "usecond": 1e-6, "msecond": 1e-3, "second": 1.0, "%": 1.0}


def ncu_table(args):
    """Markdown table of DRAM figures per workload from the ncu CSV of a `--report` run.

    The CSV is ncu's long format (one row per metric per launch) of `bench.py --report` with the
    same --only / --report-reps, captured with `-k regex:rmsq_row_kernel`. Launches are assigned
    to workloads in the order the report runs them: per workload one launch that allocates the
    outputs, three warm-ups and --report-reps timed ones (NVFP4's global-scale pre-pass,
    template mode 3, is dropped). The figures are the medians over the timed launches."""
    import csv
    with open(args.ncu_table) as f:
        rows = [ln for ln in f if ln.startswith('"')]
    launches = {}
    for r in csv.DictReader(rows):
        e = launches.setdefault(int(r["ID"]), {"name": r["Kernel Name"]})
        v = float(r["Metric Value"].replace(",", ""))
        e[r["Metric Name"]] = v * NCU_UNITS.get(r["Metric Unit"], 1.0)
    seq = []
    for _, e in sorted(launches.items()):
        targs = re.search(r"<([^>]*)>", e["name"]).group(1).split(",")
        e["mode"] = int(targs[2])
        if e["mode"] != 3:
            seq.append(e)
    only = set(args.only.split(",")) if args.only else None
    per = 4 + args.report_reps
    mode_id = {"fp8": 0, "nvfp4": 1, "mxfp4": 2}
    print("| workload | rows x hidden | ncu duration (us) | DRAM read + write (MB) | algorithmic "
          "MB | DRAM throughput (% of peak) | min - max over launches (%) | algorithmic GB/s at "
          "ncu duration |")
    print("|---|---|---|---|---|---|---|---|")
    k = 0
    for name, rws, hid in report_workloads():
        if only and name not in only and "%s:%s:%s" % (name, rws, hid) not in only:
            continue
        w = W.config(name, rows=rws, hidden=hid)
        chunk = seq[k:k + per]
        k += per
        if len(chunk) < per or any(e["mode"] != mode_id[w.mode] for e in chunk):
            raise SystemExit("ncu CSV does not match the report's launch sequence at %s" % name)
        timed = chunk[4:]
        med = lambda m: statistics.median(e[m] for e in timed)
        dur = med("gpu__time_duration.sum")
        traffic = med("dram__bytes_read.sum") + med("dram__bytes_write.sum")
        pcts = [e["dram__throughput.avg.pct_of_peak_sustained_elapsed"] for e in timed]
        pct = statistics.median(pcts)
        algo = w.algorithmic_bytes()
        print("| %s | %d x %d | %.1f | %.1f | %.1f | %.1f | %.1f - %.1f | %.0f |"
              % (name, w.rows, w.hidden, dur * 1e6, traffic / 1e6, algo / 1e6, pct, min(pcts),
                 max(pcts), algo / dur / 1e9))
    if k != len(seq):
        raise SystemExit("ncu CSV has %d launches left over" % (len(seq) - k))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--report", action="store_true", help="per-workload GB/s lines")
    ap.add_argument("--report-reps", type=int, default=20)
    ap.add_argument("--report-next", action="store_true",
                    help="time the widened rows (swizzled scales, global-scale pre-pass, other "
                         "dtypes, cluster rows), one JSON line each")
    ap.add_argument("--flush", choices=["write", "read"], default="write",
                    help="--report / --report-next: evict L2 between repetitions by writing a "
                         "256 MiB buffer (default) or by reading one (clean lines only)")
    ap.add_argument("--only", default="", help="--report: comma-separated workload names "
                    "(or name:rows:hidden for one MXFP4 sweep point); --report-next: case names "
                    "(or case:mode:rows:hidden)")
    ap.add_argument("--step-workloads", default="",
                    help="replace the step's batches: mode=name[:rows:hidden],... (experiments; "
                         "the default is the three large workloads)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-pdl", action="store_true",
                    help="launch without programmatic dependent launch (for comparison)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--oracle-seconds", type=float, default=0.3,
                    help="--report: time the oracle on a row sample of each workload for about "
                         "this long (0: skip)")
    ap.add_argument("--ncu-table", default="", metavar="CSV",
                    help="print the per-workload DRAM table from the ncu CSV of a --report run "
                         "(same --only / --report-reps); needs no GPU")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)       # at least 3 untimed warm-up steps, always
    if args.ncu_table:
        ncu_table(args)
    elif args.impl == "reference":
        run_reference(args)
    elif args.report_next:
        run_report_next(args)
    elif args.report:
        run_report(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
