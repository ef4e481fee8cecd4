"""Benchmark: causal attention forward, B=2, M=Mkv=2048, H=32, K=Kv=128, bf16.

One step = one mslk_attn_fwd call (the whole hot path for this workload: every key tile,
online softmax, output and LSE) on resident inputs.  Prints ONE JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

`--impl reference` times the fp64 CPU oracle (the only reference this project has) on a
bounded sample of the same workload.  Under torchrun (N > 1) every rank runs its own
copy of the workload (weak scaling, no collective on the data path); rank 0 prints.
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

METRIC = "attn fwd TFLOP/s (causal-adjusted) & % BF16 tensor peak; merge GB/s % HBM"
WORKLOAD = "causal_fwd"
# This pool's measured GB300 peaks (copied from the driver's probe); the file, when
# present, takes precedence.
PEAKS_FALLBACK = {"bf16_tflops": 1887.2, "bf16_tflops_sustained": 1710.7, "hbm_gbs": 6788.6}
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SRC = os.path.join(ROOT, "attention_fmha_fwd_gb300", "csrc", "fmha_tc.cu")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in PEAKS_FALLBACK}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(PEAKS_FALLBACK), "measured (pool probe, copied)"


def causal_pairs(M, Mkv, kv_offset=0):
    """Allowed (query, key) pairs of a top-left causal mask."""
    total = 0
    for i in range(M):
        last = min(Mkv - 1, i - kv_offset)
        if last >= 0:
            total += last + 1
    return total


def fwd_flops(w):
    """Exact causal-adjusted FLOPs: 2*(K + Kv) per allowed (query, key) pair."""
    return causal_pairs(w.M, w.Mkv) * 2 * (w.K + w.Kv) * w.B * w.H


def check_device(fa, what):
    """A kernel that gave up on a bounded wait leaves its output incomplete: no number
    measured over it is reported."""
    st = fa.device_status()
    if st != 0:
        raise RuntimeError(f"device error word set during the {what} (status {st}): "
                           "a kernel timed out on a bounded wait; the measurement is void")


def kernel_sha():
    with open(KERNEL_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def traffic_for(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current source."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            d = json.load(f)
        e = d[kernel_key]
        if e.get("source_sha") != kernel_sha():
            return None
        return float(e["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (SM clock, max clock, throttle reasons) while the GPU works."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        if not self.samples:
            return None
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        # a timed region shorter than the sampling period: the samples nearest to it
        near = sorted(self.samples, key=lambda ts: min(abs(ts[0] - t0), abs(ts[0] - t1)))[:3]
        win = inside or [s for _, s in near]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(s[0]) for s in win if num(s[0]) is not None]
        mx = [num(s[1]) for s in win if num(s[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in win for n, v in zip(names, s[4:8]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(win), "samples_in_timed_region": len(inside)}


class NvmlClocks:
    """SM clock and throttle reasons read through NVML (the driver's libnvidia-ml) between
    the launches of the timed steps: the host queues steps ahead of the GPU, so each read
    sees the GPU while it runs timed work.  Reading only; no setting is changed."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device):
        import ctypes
        self.samples = []
        self.ok = False
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            self.lib, self.h = lib, ctypes.c_void_p()
            bus = None
            try:
                import torch
                pr = torch.cuda.get_device_properties(torch_device)
                bus = "%08x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
            except Exception:  # noqa: BLE001 - fall back to the index
                bus = None
            if bus is not None and lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.h)) == 0:
                self.ok = True
            elif lib.nvmlDeviceGetHandleByIndex_v2(torch_device.index or 0, ctypes.byref(self.h)) == 0:
                self.ok = True
            self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint(0)
            self.max_mhz = float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0 else None
            if self.max_mhz is not None:
                self.max_mhz = float(mx.value)
        except OSError:
            self.ok = False

    def read(self):
        if not self.ok:
            return
        import ctypes
        mhz, rs = ctypes.c_uint(0), ctypes.c_ulonglong(0)
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz)) == 0 and \
                self.reasons_fn(self.h, ctypes.byref(rs)) == 0:
            self.samples.append((float(mhz.value), int(rs.value)))

    def summary(self):
        if not self.samples:
            return None
        reasons = sorted({n for _, r in self.samples for bit, n in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(m for m, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples_in_timed_region": len(self.samples), "source": "nvml"}


# ---------------------------------------------------------------------------- helpers

def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def aggregate(per_rank_seconds: float, per_rank_units: float, world: int, backend_reduce):
    """Whole-job throughput: all ranks' units / the slowest rank's time."""
    t_max = backend_reduce(per_rank_seconds)
    return per_rank_units * world / t_max, t_max


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle_sample(q, k, v, w, budget_s, max_heads=None):
    """The fp64 oracle on whole (batch, head) pairs of the workload until ~budget_s."""
    import oracle

    qf, kf, vf = q.float().numpy(), k.float().numpy(), v.float().numpy()
    pairs_per_head = causal_pairs(w.M, w.Mkv)
    flops = 0.0
    heads = 0
    t0 = time.perf_counter()
    for b in range(w.B):
        for h in range(w.H):
            oracle.attention_head(qf, kf, vf, b, h, w.scale, oracle.MASK_CAUSAL)
            flops += pairs_per_head * 2 * (w.K + w.Kv)
            heads += 1
            if (max_heads and heads >= max_heads) or time.perf_counter() - t0 >= budget_s:
                return flops, time.perf_counter() - t0, heads
    return flops, time.perf_counter() - t0, heads


# ---------------------------------------------------------------------------- reference arm

REF_BUDGET_S = 90.0  # oracle seconds for a whole --impl reference run


def run_reference(args):
    rank, world, _ = dist_info()
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    from attention_fmha_fwd_gb300 import inputs

    w = inputs.WORKLOADS[WORKLOAD]
    q, k, v = inputs.qkv(w.B, w.M, w.Mkv, w.H, w.K, seed=0)
    qf, kf, vf = q.float().numpy(), k.float().numpy(), v.float().numpy()
    # Each step is a bounded sample of the workload, sized so that warm-up + steps take
    # about REF_BUDGET_S: whole (batch, head) pairs when one fits a step's share, else a
    # block of R consecutive query rows of one head (passed as a slice of q with the
    # causal offset -r0, the same arithmetic); blocks rotate over all rows and heads, and
    # FLOPs are counted for exactly the (row, key) pairs each step's rows allow.
    n_runs = args.warmup + args.steps
    share = REF_BUDGET_S / max(1, n_runs)
    t0 = time.perf_counter()
    oracle.attention_head(qf, kf, vf, 0, 0, w.scale, oracle.MASK_CAUSAL)
    t_head = time.perf_counter() - t0
    if t_head <= share:
        heads, block = max(1, min(w.B * w.H, int(share / t_head))), w.M
    else:
        heads, block = 1, max(64, min(w.M, int(w.M * share / t_head) // 64 * 64))
    n_blocks = (w.M + block - 1) // block
    times, flops_total = [], 0.0
    for s in range(n_runs):
        f = 0.0
        t0 = time.perf_counter()
        for hh in range(heads):
            u = s * heads + hh
            bh, blk = divmod(u, n_blocks)
            b, h = divmod(bh % (w.B * w.H), w.H)
            r0 = blk * block
            r1 = min(w.M, r0 + block)
            oracle.attention_head(qf[:, r0:r1], kf, vf, b, h, w.scale, oracle.MASK_CAUSAL,
                                  kv_offset=-r0)
            f += float(np.minimum(np.arange(r0, r1) + 1, w.Mkv).sum()) * 2 * (w.K + w.Kv)
        if s >= args.warmup:
            times.append(time.perf_counter() - t0)
            flops_total += f
    flops = flops_total / max(1, len(times))
    per_step_heads = heads
    mean_t = sum(times) / len(times)
    value = flops / mean_t / 1e12  # mean FLOPs per timed step / mean step time
    sample = (f"{per_step_heads} of {w.B * w.H} (batch, head) pairs per step, all 2048 rows"
              if block == w.M else
              f"one block of {block} consecutive query rows of one (batch, head) per step, "
              f"blocks rotating over all rows and heads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": mean_t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "causal_fwd B=2 M=Mkv=2048 H=32 K=Kv=128 causal (top-left)",
                   "sample": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------- GPU arm

def make_collectives(world, device):
    """(reduce_max, barrier) over the ranks of the initialised process group (identity and
    no-op for one rank): the slowest rank's time and the step fences around the timed
    region.  ``device`` is where the reduced scalar lives ("cuda" for NCCL, "cpu" for gloo)."""
    if world <= 1:
        return (lambda x: x), (lambda: None)
    import torch
    import torch.distributed as dist

    def reduce_max(x):
        t = torch.tensor([x], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    def barrier():
        dist.barrier()

    return reduce_max, barrier


def run_gpu(args):
    import torch

    rank, world, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        reduce_max, barrier = make_collectives(world, "cuda")
    else:
        torch.cuda.set_device(0)
        reduce_max, barrier = make_collectives(1, "cuda")

    import attention_fmha_fwd_gb300 as fa
    from attention_fmha_fwd_gb300 import build, inputs

    build.build()
    peaks, peak_src = load_peaks()
    dev = torch.device("cuda", torch.cuda.current_device())
    w = inputs.WORKLOADS[WORKLOAD]
    q, k, v = inputs.qkv(w.B, w.M, w.Mkv, w.H, w.K, seed=0)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out = torch.empty((w.B, w.M, w.H, w.Kv), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, w.M), dtype=torch.float32, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)  # > 129 MB L2
    flops = fwd_flops(w)
    stream = torch.cuda.current_stream()

    def step():
        fa.attn_fwd(qd, kd, vd, mask="causal", scale=w.scale, out=out, lse=lse)

    sampler = ClockSampler(dev.index) if (rank == 0 and not args.profile_mode) else None
    for _ in range(args.warmup):
        step()
    if not args.profile_mode:
        # keep the GPU busy briefly so the clock sampler sees load before the timed region
        t_end = time.time() + 0.3
        while time.time() < t_end:
            step()
    torch.cuda.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    nvml = NvmlClocks(dev) if (rank == 0 and not args.profile_mode) else None
    # CUDA creates an event when it is first recorded: record every timing event once here,
    # so that no host-side creation delays a timed step's launch after its start event.
    for e in starts + ends:
        e.record(stream)
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(args.steps):
        flush.zero_()                       # L2 flushed between timed steps
        starts[i].record(stream)
        step()
        ends[i].record(stream)
        if nvml is not None and i % 2 == 1:
            nvml.read()                     # the GPU is running the steps queued so far
    torch.cuda.synchronize()
    barrier()
    t1 = time.time()
    per = [s.elapsed_time(e) * 1e-3 for s, e in zip(starts, ends)]
    t_step = sum(per) / len(per)
    check_device(fa, "timed steps")
    value, t_max = aggregate(t_step, flops, world, reduce_max)
    value /= 1e12
    clocks = sampler.summary(t0, t1) if sampler else None
    if sampler:
        sampler.stop()
    in_region = nvml.summary() if nvml is not None else None
    if in_region is not None:
        # NVML reads taken between the timed launches; nvidia-smi's samples around them
        clocks = dict(in_region, nvidia_smi=clocks)

    if args.profile_mode:
        if rank == 0:
            print(json.dumps({"profile_mode": True, "ms_per_step": t_step * 1e3,
                              "value": value, "unit": "TFLOP/s"}))
        return 0

    # ---- end to end through the public call: pinned host in, host out, every step.
    # Steps are pipelined the way a serving loop would run them: step i's host->device
    # copies (one stream per input tensor), its attention call and its device->host copy
    # of (out, lse) are ordered by events, with device buffers double-buffered so step
    # i+1's inputs can arrive while step i computes and step i-1's results drain.
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    nbuf = 2
    dq = [qd] + [torch.empty_like(qd) for _ in range(nbuf - 1)]
    dk = [kd] + [torch.empty_like(kd) for _ in range(nbuf - 1)]
    dv = [vd] + [torch.empty_like(vd) for _ in range(nbuf - 1)]
    dout = [out] + [torch.empty_like(out) for _ in range(nbuf - 1)]
    dlse = [lse] + [torch.empty_like(lse) for _ in range(nbuf - 1)]
    out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(nbuf)]
    lse_h = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(nbuf)]
    s_in = [torch.cuda.Stream() for _ in range(3)]
    s_out = torch.cuda.Stream()
    ev_in = [[torch.cuda.Event() for _ in range(3)] for _ in range(nbuf)]
    ev_done = [torch.cuda.Event() for _ in range(nbuf)]
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]
    used = [False] * nbuf
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step(i):
        b = i % nbuf
        for j, (src, dst) in enumerate(((qh, dq[b]), (kh, dk[b]), (vh, dv[b]))):
            with torch.cuda.stream(s_in[j]):
                if used[b]:
                    s_in[j].wait_event(ev_done[b])   # step i-2 finished reading this buffer
                dst.copy_(src, non_blocking=True)
                ev_in[b][j].record(s_in[j])
        for j in range(3):
            stream.wait_event(ev_in[b][j])
        if used[b]:
            stream.wait_event(ev_out[b])             # step i-2's results have left this buffer
        fa.attn_fwd(dq[b], dk[b], dv[b], mask="causal", scale=w.scale, out=dout[b], lse=dlse[b])
        ev_done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[b])
            out_h[b].copy_(dout[b], non_blocking=True)
            lse_h[b].copy_(dlse[b], non_blocking=True)
            ev_out[b].record(s_out)
        used[b] = True

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)  # (created here, recorded again below as the start mark)
    e1.record(stream)
    torch.cuda.synchronize()
    e0.record(stream)
    for j in range(3):
        s_in[j].wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_stream(s_out)
    e1.record(stream)
    torch.cuda.synchronize()
    t_e2e = e0.elapsed_time(e1) * 1e-3 / e2e_steps
    e2e_value, _ = aggregate(t_e2e, flops, world, reduce_max)
    h2d = sum(t.numel() * t.element_size() for t in (q, k, v))
    d2h = out.numel() * out.element_size() + lse.numel() * lse.element_size()

    check_device(fa, "end-to-end steps")
    secondary = measure_secondary(fa, inputs, dev, flush, peaks) if (rank == 0 and not args.no_secondary) else None
    if secondary is not None:
        check_device(fa, "secondary measurements")

    if rank == 0:
        achieved = flops / t_step / 1e12
        traffic = traffic_for("fmha_tc_kernel<128, false, false> causal_fwd")
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "causal_fwd B=2 M=Mkv=2048 H=32 K=Kv=128 causal (top-left)",
                       "flops_per_step": flops, "flop_count": "exact causal pairs x 2(K+Kv)",
                       "l2": "flushed (256 MB write) between timed steps",
                       "inputs": "seeded N(0,1) bf16, seed 0", "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "tensor", "achieved": achieved,
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": achieved / peaks["bf16_tflops"], "traffic": traffic,
                         "frac_sustained": achieved / peaks["bf16_tflops_sustained"],
                         "kernel": "fmha_tc_kernel<128, false, false>", "peak_source": peak_src + " bf16 burst"},
            "e2e": {"value": e2e_value / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e * 1e3,
                    "pipeline": "pinned host q/k/v -> device (3 copy streams), attn_fwd, "
                                "out+lse -> pinned host (1 stream); steps overlap, device "
                                "buffers double-buffered"},
            "gpu_launches": args.steps,
            "step_ms": {"mean": t_step * 1e3, "median": statistics.median(per) * 1e3,
                        "min": min(per) * 1e3, "max": max(per) * 1e3,
                        "each": [round(x * 1e3, 5) for x in per],
                        "note": "per-step CUDA-event times of the timed steps on this rank; "
                                "value uses the mean"},
            "clocks": clocks,
            "secondary": secondary,
        }
        if not args.no_cpu_baseline:
            f, t, heads = time_oracle_sample(q, k, v, w, budget_s=args.cpu_budget)
            line["cpu_baseline"] = {
                "value": f / t / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(),
                "kind": "oracle",
                "sample": f"{heads} of {w.B * w.H} (batch, head) pairs, all 2048 rows, fp64 numpy"}
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def _time_it(fn, reps, stream, flush):
    import torch
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)  # created on first record, before any timed interval
    b.record(stream)
    ts = []
    for _ in range(reps):
        flush.zero_()
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) * 1e-3)
    return statistics.median(ts)


def measure_secondary(fa, inputs, dev, flush, peaks):
    """Merge roofline shape, decode split-KV and varlen throughput (context numbers)."""
    import torch
    stream = torch.cuda.current_stream()
    res = {}
    # tiny forward [1, 128, 2, 64], scale 1/8 (launch-latency bound: microseconds only)
    w = inputs.WORKLOADS["tiny_fwd"]
    qt, kt, vt = (t.to(dev) for t in inputs.qkv(w.B, w.M, w.Mkv, w.H, w.K, seed=0))
    tiny = lambda: fa.attn_fwd(qt, kt, vt, scale=w.scale)  # noqa: E731
    for _ in range(10):
        tiny()
    res["tiny_fwd_1x128x2x64"] = {"us": _time_it(tiny, 50, stream, flush) * 1e6, "launches": 1}
    # split-KV: q [1, 128, 16, 128] against k/v [1, 1024, 16, 128] in n equal chunks
    # (strided views, no copies): n partial launches (fp32 out) + one merge, timed apart
    w = inputs.WORKLOADS["split_kv"]
    qs, ks, vs = (t.to(dev) for t in inputs.qkv(w.B, w.M, w.Mkv, w.H, w.K, seed=0))
    for n in (2, 8):
        bounds = inputs.equal_chunks(w.Mkv, n)
        po = torch.empty((n, w.B, w.M, w.H, w.Kv), dtype=torch.float32, device=dev)
        pl = torch.empty((n, w.B, w.H, w.M), dtype=torch.float32, device=dev)
        mo = torch.empty((w.B, w.M, w.H, w.Kv), dtype=torch.bfloat16, device=dev)
        ml = torch.empty((w.B, w.H, w.M), dtype=torch.float32, device=dev)

        kvs = [(ks[:, a0:b0], vs[:, a0:b0]) for a0, b0 in bounds]

        def parts(independent=False, kvs=kvs, po=po, pl=pl):
            for c, (kc_, vc_) in enumerate(kvs):
                fa.attn_partial(qs, kc_, vc_, scale=w.scale, out=po[c], lse=pl[c],
                                independent=independent and c > 0)

        merge = lambda po=po, pl=pl, mo=mo, ml=ml: fa.merge_attentions(po, pl, out=mo, lse=ml)  # noqa: E731
        for _ in range(10):
            parts()
            merge()
        entry = {"eager_partials_us": _time_it(parts, 50, stream, flush) * 1e6,
                 "merge_us": _time_it(merge, 50, stream, flush) * 1e6, "launches": n + 1}
        for key, ind in (("graph_partials_us", False), ("graph_independent_partials_us", True)):
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                parts(ind)
            stream.wait_stream(side)
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr):
                parts(ind)
            gr.replay()
            torch.cuda.synchronize()
            entry[key] = _time_it(gr.replay, 50, stream, flush) * 1e6
            del gr
        # the same split in one library call (partials + merge, workspace given): the
        # host cost of n + 1 Python calls becomes one
        ws = torch.empty(fa.split_kv_workspace_bytes(qs, ks, vs, n_chunks=n), dtype=torch.uint8, device=dev)
        one_call = lambda n=n, ws=ws, mo=mo, ml=ml: fa.attn_split_kv(  # noqa: E731
            qs, ks, vs, n_chunks=n, scale=w.scale, out=mo, lse=ml, workspace=ws)
        for _ in range(10):
            one_call()
        entry["one_call_us"] = _time_it(one_call, 50, stream, flush) * 1e6
        res[f"split_kv_{n}_chunks_1x128x1024x16x128"] = entry
    # merge: 8 chunks of [2, 2048, 32, 128] fp32 -> bf16 out + fp32 lse
    n, B, M, H, Kv = 8, 2, 2048, 32, 128
    g = torch.Generator(device=dev).manual_seed(0)
    outs = torch.randn((n, B, M, H, Kv), generator=g, device=dev)
    lses = torch.randn((n, B, H, M), generator=g, device=dev)
    mo = torch.empty((B, M, H, Kv), dtype=torch.bfloat16, device=dev)
    ml = torch.empty((B, H, M), dtype=torch.float32, device=dev)
    for _ in range(3):
        fa.merge_attentions(outs, lses, out=mo, lse=ml)
    t = _time_it(lambda: fa.merge_attentions(outs, lses, out=mo, lse=ml), 20, stream, flush)
    nbytes = outs.numel() * 4 + lses.numel() * 4 + mo.numel() * 2 + ml.numel() * 4
    res["merge_8x[2,2048,32,128]"] = {"us": t * 1e6, "GB/s": nbytes / t / 1e9,
                                      "frac_hbm": nbytes / t / 1e9 / peaks["hbm_gbs"],
                                      "bytes": nbytes}
    del outs, lses
    # decode split-KV: 16 x 1 query, 32768 keys, 8 heads, 16 chunks of 2048 + merge
    w = inputs.WORKLOADS["decode_split_kv"]
    q, k, v = inputs.qkv(w.B, w.M, w.Mkv, w.H, w.K, seed=0)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    bounds = inputs.equal_chunks(w.Mkv, 16)
    po = torch.empty((16, w.B, w.M, w.H, w.Kv), dtype=torch.float32, device=dev)
    pl = torch.empty((16, w.B, w.H, w.M), dtype=torch.float32, device=dev)
    fo = torch.empty((w.B, w.M, w.H, w.Kv), dtype=torch.bfloat16, device=dev)
    fl = torch.empty((w.B, w.H, w.M), dtype=torch.float32, device=dev)

    # chunk views and output slots are made once (inputs resident, as in a decode loop)
    kc = [kd[:, a:b] for a, b in bounds]
    vc = [vd[:, a:b] for a, b in bounds]
    pos = [po[c] for c in range(len(bounds))]
    pls = [pl[c] for c in range(len(bounds))]

    def partials():
        for c in range(len(bounds)):
            fa.attn_partial(qd, kc[c], vc[c], scale=w.scale, out=pos[c], lse=pls[c])

    for _ in range(2):
        partials()
    t_eager = _time_it(partials, 10, stream, flush)
    # the 16 launches captured once in a CUDA graph: device time without host launch gaps
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        partials()
    stream.wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        partials()
    graph.replay()
    torch.cuda.synchronize()
    t_p = _time_it(graph.replay, 10, stream, flush)
    del graph

    # the same 16 partials declared independent of each other (programmatic dependent
    # launch: each may start while the previous finishes), one CUDA graph
    def partials_ind():
        for c in range(len(bounds)):
            fa.attn_partial(qd, kc[c], vc[c], scale=w.scale, out=pos[c], lse=pls[c],
                            independent=c > 0)

    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        partials_ind()
    stream.wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        partials_ind()
    graph.replay()
    torch.cuda.synchronize()
    t_pi = _time_it(graph.replay, 10, stream, flush)
    t_m = _time_it(lambda: fa.merge_attentions(po, pl, out=fo, lse=fl), 10, stream, flush)
    kv_bytes = (kd.numel() + vd.numel()) * 2
    res["decode_split_kv_16x2048"] = {"partials_us": t_p * 1e6, "merge_us": t_m * 1e6,
                                      "partial_GB/s": kv_bytes / t_p / 1e9,
                                      "frac_hbm": kv_bytes / t_p / 1e9 / peaks["hbm_gbs"],
                                      "partials": "16 launches replayed from one CUDA graph",
                                      "independent_partials_us": t_pi * 1e6,
                                      "independent_partial_GB/s": kv_bytes / t_pi / 1e9,
                                      "independent_frac_hbm": kv_bytes / t_pi / 1e9 / peaks["hbm_gbs"],
                                      "eager_partials_us": t_eager * 1e6,
                                      "eager_partial_GB/s": kv_bytes / t_eager / 1e9,
                                      "launches": 17}
    del graph
    # the 16-chunk split in one library call (partials + merge into bf16 out, workspace given)
    ws = torch.empty(fa.split_kv_workspace_bytes(qd, kd, vd, n_chunks=16), dtype=torch.uint8, device=dev)
    one_call = lambda: fa.attn_split_kv(qd, kd, vd, n_chunks=16, scale=w.scale, out=fo, lse=fl,  # noqa: E731
                                        workspace=ws)
    for _ in range(3):
        one_call()
    t_oc = _time_it(one_call, 10, stream, flush)
    res["decode_split_kv_16x2048"].update({"one_call_us": t_oc * 1e6,
                                           "one_call_GB/s": kv_bytes / t_oc / 1e9,
                                           "one_call_frac_hbm": kv_bytes / t_oc / 1e9 / peaks["hbm_gbs"]})
    # the same step as one call over all 32768 keys (the kernel splits keys on-chip)
    fo32 = torch.empty((w.B, w.M, w.H, w.Kv), dtype=torch.float32, device=dev)
    one = lambda: fa.attn_partial(qd, kd, vd, scale=w.scale, out=fo32, lse=fl)  # noqa: E731
    for _ in range(3):
        one()
    t_one = _time_it(one, 10, stream, flush)
    res["decode_single_launch_16x32768"] = {"us": t_one * 1e6, "GB/s": kv_bytes / t_one / 1e9,
                                            "frac_hbm": kv_bytes / t_one / 1e9 / peaks["hbm_gbs"],
                                            "launches": 1}
    # few heads: 1 x 1 query, 131072 keys, 8 heads (the keys of each head split over a cluster)
    q1, k1, v1 = inputs.qkv(1, 1, 131072, 8, 128, seed=5)
    q1, k1, v1 = q1.to(dev), k1.to(dev), v1.to(dev)
    o1 = torch.empty((1, 1, 8, 128), dtype=torch.float32, device=dev)
    l1 = torch.empty((1, 8, 1), dtype=torch.float32, device=dev)
    few = lambda: fa.attn_partial(q1, k1, v1, scale=w.scale, out=o1, lse=l1)  # noqa: E731
    for _ in range(3):
        few()
    t_few = _time_it(few, 10, stream, flush)
    b_few = (k1.numel() + v1.numel()) * 2
    res["decode_single_launch_1x131072x8"] = {"us": t_few * 1e6, "GB/s": b_few / t_few / 1e9,
                                              "frac_hbm": b_few / t_few / 1e9 / peaks["hbm_gbs"],
                                              "launches": 1}
    del q1, k1, v1
    # the same decode step over a paged cache: 16 lanes of 32768 keys in shuffled 256-key
    # pages (one launch; rows come from the page table)
    ps = 256
    lk = [w.Mkv] * w.B
    table, n_pages, _ = inputs.page_table(lk, ps, seed=0)
    pad = n_pages * ps - w.B * w.Mkv  # the spare page
    kp = torch.cat([kd.reshape(-1, w.H, w.K), kd.new_zeros((pad, w.H, w.K))]).view(n_pages, ps, w.H, w.K)
    vp = torch.cat([vd.reshape(-1, w.H, w.Kv), vd.new_zeros((pad, w.H, w.Kv))]).view(n_pages, ps, w.H, w.Kv)
    qp = qd.reshape(1, w.B, w.H, w.K)
    tbl, sk = table.to(dev), torch.tensor(lk, dtype=torch.int32, device=dev)
    cq = torch.arange(w.B + 1, dtype=torch.int32, device=dev)
    op = torch.empty((1, w.B, w.H, w.Kv), dtype=torch.bfloat16, device=dev)
    lp = torch.empty((1, w.H, w.B), dtype=torch.float32, device=dev)
    paged = lambda: fa.attn_fwd_lanes(qp, kp, vp, seqlen_k=sk, cu_seqlens_q=cq, max_seqlen_q=1,  # noqa: E731
                                      max_seqlen_k=w.Mkv, block_table=tbl, page_size=ps,
                                      scale=w.scale, bottom_right=True, out=op, lse=lp)
    for _ in range(3):
        paged()
    t_pg = _time_it(paged, 10, stream, flush)
    b_pg = sum(lk) * w.H * (w.K + w.Kv) * 2
    res["decode_paged_16x32768_page256"] = {"us": t_pg * 1e6, "GB/s": b_pg / t_pg / 1e9,
                                            "frac_hbm": b_pg / t_pg / 1e9 / peaks["hbm_gbs"],
                                            "launches": 1}
    del kp, vp
    # the same decode step with an E4M3 cache (per-head descales): half the bytes
    k8, dk8 = inputs.quantize_e4m3(kd)
    v8, dv8 = inputs.quantize_e4m3(vd)
    q8, dq8 = inputs.quantize_e4m3(qd)
    dk8, dv8, dq8 = dk8.to(dev), dv8.to(dev), dq8.to(dev)
    o8 = torch.empty((w.B, w.M, w.H, w.Kv), dtype=torch.bfloat16, device=dev)
    fp8_dec = lambda: fa.attn_fwd_fp8(q8, k8, v8, dq8, dk8, dv8, scale=w.scale, out=o8, lse=fl)  # noqa: E731
    for _ in range(3):
        fp8_dec()
    t_f8 = _time_it(fp8_dec, 10, stream, flush)
    b_f8 = k8.numel() + v8.numel()
    res["fp8_decode_single_launch_16x32768"] = {"us": t_f8 * 1e6, "GB/s": b_f8 / t_f8 / 1e9,
                                                "frac_hbm": b_f8 / t_f8 / 1e9 / peaks["hbm_gbs"],
                                                "speedup_vs_bf16": t_one / t_f8, "launches": 1}
    del k8, v8
    # grouped-query decode: 32 query heads on the same 8 K/V heads (group 4), one launch;
    # each K/V head is streamed once for its 4 query heads
    qg = torch.randn((w.B, 1, 32, w.K), device=dev).to(torch.bfloat16)
    og = torch.empty((w.B, 1, 32, w.Kv), dtype=torch.float32, device=dev)
    lg = torch.empty((w.B, 32, 1), dtype=torch.float32, device=dev)
    gqa = lambda: fa.attn_partial(qg, kd, vd, scale=w.scale, out=og, lse=lg)  # noqa: E731
    for _ in range(3):
        gqa()
    t_g = _time_it(gqa, 10, stream, flush)
    res["decode_gqa_16x32768_32q_8kv"] = {"us": t_g * 1e6, "GB/s": kv_bytes / t_g / 1e9,
                                          "frac_hbm": kv_bytes / t_g / 1e9 / peaks["hbm_gbs"],
                                          "query_heads_per_kv_head": 4, "launches": 1}
    del qg
    del kd, vd, k, v
    # varlen packed block-diagonal causal
    w = inputs.WORKLOADS["varlen_packed"]
    lens = inputs.varlen_seqlens(w.n_seqs, w.M, seed=0)
    cu = torch.tensor(inputs.cu_seqlens(lens), dtype=torch.int32, device=dev)
    q, k, v = inputs.qkv(1, w.M, w.Mkv, w.H, w.K, seed=0)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    vo = torch.empty((1, w.M, w.H, w.Kv), dtype=torch.bfloat16, device=dev)
    vl = torch.empty((1, w.H, w.M), dtype=torch.float32, device=dev)

    def vstep():
        fa.attn_fwd(qd, kd, vd, mask="blockdiag_causal", scale=w.scale, cu_seqlens_q=cu,
                    cu_seqlens_k=cu, max_seqlen_q=max(lens), max_seqlen_k=max(lens),
                    out=vo, lse=vl)

    for _ in range(3):
        vstep()
    t_v = _time_it(vstep, 10, stream, flush)
    vflops = sum(L * (L + 1) // 2 for L in lens) * 2 * (w.K + w.Kv) * w.H
    res["varlen_packed_12seq_16384"] = {"us": t_v * 1e6, "TFLOP/s": vflops / t_v / 1e12,
                                        "frac_bf16": vflops / t_v / 1e12 / peaks["bf16_tflops"],
                                        "seqlens": lens}
    del qd, kd, vd
    # local window and bottom-right alignment (key tiles outside every row's band skipped)
    import numpy as np

    def band_pairs(M, Mkv, shift, wl):
        i = np.arange(M, dtype=np.int64)
        hi = np.minimum(i + shift, Mkv - 1)
        lo = np.zeros_like(i) if wl is None else np.maximum(i + shift - wl, 0)
        return int(np.maximum(hi - lo + 1, 0).sum())

    for name, (M, Mkv, br, wl) in (("causal_window1024_1x8192x32x128", (8192, 8192, False, 1023)),
                                    ("causal_bottom_right_1x2048x8192x32x128", (2048, 8192, True, None))):
        q, k, v = inputs.qkv(1, M, Mkv, 32, 128, seed=6)
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        bo = torch.empty((1, M, 32, 128), dtype=torch.bfloat16, device=dev)
        bl = torch.empty((1, 32, M), dtype=torch.float32, device=dev)

        def bstep():
            fa.attn_fwd(qd, kd, vd, mask="causal", scale=w.scale, out=bo, lse=bl, bottom_right=br,
                        window_left=wl)

        for _ in range(3):
            bstep()
        t_b = _time_it(bstep, 10, stream, flush)
        bflops = band_pairs(M, Mkv, Mkv - M if br else 0, wl) * 2 * 256 * 32
        res[name] = {"us": t_b * 1e6, "TFLOP/s": bflops / t_b / 1e12,
                     "frac_bf16": bflops / t_b / 1e12 / peaks["bf16_tflops"]}
        if br:
            # the same chunked prefill over a paged cache: 8192 keys in shuffled 256-key pages
            ps = 256
            table, n_pages, _ = inputs.page_table([Mkv], ps, seed=6)
            pad = n_pages * ps - Mkv
            kp = torch.cat([kd[0], kd.new_zeros((pad, 32, 128))]).view(n_pages, ps, 32, 128)
            vp = torch.cat([vd[0], vd.new_zeros((pad, 32, 128))]).view(n_pages, ps, 32, 128)
            tbl = table.to(dev)
            sk = torch.tensor([Mkv], dtype=torch.int32, device=dev)
            cq = torch.tensor([0, M], dtype=torch.int32, device=dev)

            def pstep():
                fa.attn_fwd_lanes(qd, kp, vp, seqlen_k=sk, cu_seqlens_q=cq, max_seqlen_q=M,
                                  max_seqlen_k=Mkv, block_table=tbl, page_size=ps, scale=w.scale,
                                  bottom_right=True, out=bo, lse=bl)

            for _ in range(3):
                pstep()
            t_p = _time_it(pstep, 10, stream, flush)
            res["prefill_paged_1x2048x8192x32x128_page256"] = {
                "us": t_p * 1e6, "TFLOP/s": bflops / t_p / 1e12,
                "frac_bf16": bflops / t_p / 1e12 / peaks["bf16_tflops"]}
            del kp, vp
        del qd, kd, vd
    # E4M3 q/k/v on the tensor cores: the causal 2 x 2048 x 32 x 128 workload, per-head
    # descales; peak = measured bf16 x 2 (the nominal E4M3 : bf16 dense ratio, 4.5 : 2.25)
    w = inputs.WORKLOADS["causal_fwd"]
    q, k, v = inputs.qkv(w.B, w.M, w.Mkv, w.H, w.K, seed=0)
    q8, dq8 = inputs.quantize_e4m3(q.to(dev))
    k8, dk8 = inputs.quantize_e4m3(k.to(dev))
    v8, dv8 = inputs.quantize_e4m3(v.to(dev))
    fo = torch.empty((w.B, w.M, w.H, w.Kv), dtype=torch.bfloat16, device=dev)
    fl = torch.empty((w.B, w.H, w.M), dtype=torch.float32, device=dev)

    def f8step():
        fa.attn_fwd_fp8(q8, k8, v8, dq8, dk8, dv8, mask="causal", scale=w.scale, out=fo, lse=fl)

    for _ in range(3):
        f8step()
    t_c8 = _time_it(f8step, 20, stream, flush)
    fl8 = fwd_flops(w)
    res["fp8_causal_fwd_2x2048x32x128"] = {"us": t_c8 * 1e6, "TFLOP/s": fl8 / t_c8 / 1e12,
                                           "frac_fp8": fl8 / t_c8 / 1e12 / (2 * peaks["bf16_tflops"]),
                                           "peak": "2 x measured bf16"}
    return res


def run_profile_other(args):
    """Warm-up + timed steps of one secondary kernel's workload (for ncu captures)."""
    import torch

    import attention_fmha_fwd_gb300 as fa
    from attention_fmha_fwd_gb300 import build, inputs

    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if args.workload == "merge":
        n, B, M, H, Kv = 8, 2, 2048, 32, 128
        g = torch.Generator(device=dev).manual_seed(0)
        outs = torch.randn((n, B, M, H, Kv), generator=g, device=dev)
        lses = torch.randn((n, B, H, M), generator=g, device=dev)
        mo = torch.empty((B, M, H, Kv), dtype=torch.bfloat16, device=dev)
        ml = torch.empty((B, H, M), dtype=torch.float32, device=dev)

        def step():
            fa.merge_attentions(outs, lses, out=mo, lse=ml)
    elif args.workload == "decode_split_kv":
        w = inputs.WORKLOADS["decode_split_kv"]
        q, k, v = inputs.qkv(w.B, w.M, w.Mkv, w.H, w.K, seed=0)
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        bounds = inputs.equal_chunks(w.Mkv, 16)
        po = torch.empty((16, w.B, w.M, w.H, w.Kv), dtype=torch.float32, device=dev)
        pl = torch.empty((16, w.B, w.H, w.M), dtype=torch.float32, device=dev)

        def step():
            for c, (a, b) in enumerate(bounds):
                fa.attn_partial(qd, kd[:, a:b], vd[:, a:b], scale=w.scale, out=po[c], lse=pl[c])
            fa.merge_attentions(po, pl)
    elif args.workload == "fp8_causal_fwd":
        w = inputs.WORKLOADS["causal_fwd"]
        q, k, v = inputs.qkv(w.B, w.M, w.Mkv, w.H, w.K, seed=0)
        q8, dq = inputs.quantize_e4m3(q.to(dev))
        k8, dk = inputs.quantize_e4m3(k.to(dev))
        v8, dv = inputs.quantize_e4m3(v.to(dev))

        def step():
            fa.attn_fwd_fp8(q8, k8, v8, dq, dk, dv, mask="causal", scale=w.scale)
    elif args.workload in ("fp8_decode", "fp8_decode_tc"):
        # E4M3 decode, 16 x 8192 keys x 8 heads x 128 (268 MB of K/V: larger than L2):
        # fp8_decode on the CUDA-core kernel, fp8_decode_tc on the automatic choice (the
        # tensor cores with split units for these 128 units)
        fa.set_path_policy(2 if args.workload == "fp8_decode" else 0)
        g = torch.Generator(device=dev).manual_seed(0)
        k = torch.randn((16, 8192, 8, 128), generator=g, device=dev)
        v = torch.randn((16, 8192, 8, 128), generator=g, device=dev)
        q = torch.randn((16, 1, 8, 128), generator=g, device=dev)
        k8, dk = inputs.quantize_e4m3(k)
        v8, dv = inputs.quantize_e4m3(v)
        q8, dq = inputs.quantize_e4m3(q)
        del k, v

        def step():
            fa.attn_fwd_fp8(q8, k8, v8, dq, dk, dv, scale=128 ** -0.5)
    elif args.workload == "decode_single":
        # bf16 decode in one launch (keys split over a cluster), 16 x 8192 keys x 8 heads x
        # 128 (537 MB of K/V: larger than L2)
        q, k, v = inputs.qkv(16, 1, 8192, 8, 128, seed=0)
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)

        def step():
            fa.attn_fwd(qd, kd, vd, scale=128 ** -0.5)
    else:
        w = inputs.WORKLOADS["varlen_packed"]
        lens = inputs.varlen_seqlens(w.n_seqs, w.M, seed=0)
        cu = torch.tensor(inputs.cu_seqlens(lens), dtype=torch.int32, device=dev)
        q, k, v = inputs.qkv(1, w.M, w.Mkv, w.H, w.K, seed=0)
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)

        def step():
            fa.attn_fwd(qd, kd, vd, mask="blockdiag_causal", scale=w.scale, cu_seqlens_q=cu,
                        cu_seqlens_k=cu, max_seqlen_q=max(lens), max_seqlen_k=max(lens))
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        step()
    b.record()
    torch.cuda.synchronize()
    check_device(fa, "profiled steps")
    print(json.dumps({"profile_mode": True, "workload": args.workload,
                      "ms_per_step": a.elapsed_time(b) / args.steps}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--profile-mode", action="store_true",
                    help="only the warm-up and timed steps (for ncu); prints a short line")
    ap.add_argument("--workload", default="causal_fwd",
                    choices=["causal_fwd", "merge", "decode_split_kv", "varlen_packed", "fp8_causal_fwd",
                             "fp8_decode", "fp8_decode_tc", "decode_single"],
                    help="with --profile-mode: which kernel's workload to run")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.profile_mode and args.workload != "causal_fwd":
        return run_profile_other(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
