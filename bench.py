"""Benchmark of the MoE expert-parallel layout / dispatch / combine path on GB300.

One step on the prefill workload (32768 tokens = 8 logical ranks x 4096,
hidden 7168, 256 experts, top-8, expert_alignment 128, softmax weights):

    layout (bf16 handle) -> dispatch bf16 -> identity experts -> combine
    layout (fp8 handle)  -> dispatch FP8 e4m3 with per-128 scales

i.e. every step of the hot path once, on the routing of that step.  Inputs
are synthetic and seeded (synth module), resident in HBM before timing, and
larger than L2 (x is 470 MB, the receive buffers 4.2 GB and 2.1 GB), so no L2
flush is needed between steps.  Kernels are timed with CUDA events on the
stream they are launched on.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle instead
(test infrastructure used as the slow reference arm), on a bounded sample.
Multi-GPU: replicas only (one independent replica per GPU, no collective on
the data path); barrier + max-over-ranks timing.
"""
import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "dispatch & combine GB/s and tokens/s on 1 GB300; % of HBM roofline"
WORKLOAD = "prefill"
WORKLOAD_DESC = ("prefill: 8 logical ranks x 4096 tokens = 32768 tokens, hidden 7168 bf16 ~N(0,1), "
                 "256 experts (32/rank), top-8 uniform distinct, softmax weights, expert_alignment "
                 "128; dispatch bf16 and FP8 e4m3 (per-128 fp32 scales); combine bf16 with fp32 fma")
SHARED_SOURCES = ["ep_ptx.cuh", "ep_cfg.hpp", "ep_kernels.hpp", "ep_types.cuh"]
KERNEL_FILES = {"ep_dispatch_copy_kernel": ["ep_dispatch_body.cuh", "ep_dispatch.cu"],
                "ep_dispatch_fp8_kernel": ["ep_dispatch_body.cuh", "ep_dispatch.cu"],
                "ep_combine_kernel": ["ep_combine_body.cuh", "ep_combine.cu"],
                "ep_layout_count_kernel": ["ep_layout.cu"],
                "ep_layout_spine_kernel": ["ep_layout.cu"],
                "ep_layout_slots_kernel": ["ep_layout.cu"],
                "ep_layout_fused_kernel": ["ep_layout.cu"]}


# GPU cycles of the pre-roll sleep before each --all-configs step (~100 us at 2 GHz)
SLEEP_CYCLES = 200_000

# ----------------------------------------------------------------- helpers

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def reduce_over_ranks(ms, units, world):
    """Max of the per-rank elapsed time and the sum of the units processed."""
    if world <= 1:
        return ms, units
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def algorithmic_bytes(N, H, K, rcap, valid_entries=None):
    """Bytes each kernel must move (padding rows excluded)."""
    NK = N * K if valid_entries is None else valid_entries
    G = H // 128
    return {
        "layout": N * K * 8 + N * K * 4 + rcap * (K + 2) * 4,
        "dispatch_bf16": N * H * 2 + N * K * 4 + NK * H * 2,
        "dispatch_fp8": N * H * 2 + N * K * 4 + NK * H + NK * G * 4,
        "combine": NK * H * 2 + N * K * 4 + N * K * 4 + N * H * 2,
    }


def algorithmic_bytes_nonexpand(N, H, K, rows, rcap, fp8):
    """Bytes of the non-expand layout's kernels: `rows` (token, rank) rows received."""
    G = H // 128
    return {
        "layout": N * K * 8 + 2 * N * K * 4 + rcap * (K + 2) * 4,
        "dispatch": N * H * 2 + N * K * 4 + rows * (H + G * 4 if fp8 else 2 * H),
        "combine": rows * H * 2 + N * K * 4 + N * H * 2,
    }


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_source_digest(kernel):
    """Digest of the source file that holds `kernel` and the headers it includes."""
    h = hashlib.sha256()
    for n in KERNEL_FILES[kernel] + SHARED_SOURCES:
        with open(os.path.join(ROOT, "combine_ep_layout_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# The record's DRAM bytes are per launch of the 32768-token prefill batch.
TRAFFIC_TOKENS = 32768


def ncu_traffic(kernel, tokens=TRAFFIC_TOKENS):
    """DRAM bytes of one launch of `kernel` on `tokens` tokens of the prefill
    shape, from the committed ncu summary (scaled by the tokens processed), or
    None when the summary is missing or was taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            k = json.load(f).get("kernels", {}).get(kernel)
    except Exception:
        return None
    if k is None or k.get("source_digest") != kernel_source_digest(kernel):
        return None
    return int(round(k["dram_bytes_per_launch"] * tokens / TRAFFIC_TOKENS))


# NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*) reported by name
NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class NvmlClockSampler:
    """SM clock, its maximum, power and clock-event reasons read in-process
    through NVML (read-only queries of libnvidia-ml, loaded with ctypes) every
    `period_s` on a background thread, so that a timed region of a few tens of
    milliseconds still holds tens of samples.  `ok` is False when NVML or the
    device cannot be found; the caller then falls back to nvidia-smi."""

    def __init__(self, device_index, period_s=0.001):
        import ctypes
        self.period = period_s
        self.samples = []          # (sm_mhz, power_w, reasons bitmask)
        self.max_mhz = None
        self.ok = False
        self._stop = threading.Event()
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            import torch
            props = torch.cuda.get_device_properties(device_index)
            bus = "%08X:%02X:%02X.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
            if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
                return
            self.nv, self.h, self.ct = nv, h, ctypes
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:   # NVML_CLOCK_SM
                self.max_mhz = float(mx.value)
            self._reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self.ok = self._sample() is not None
        except (OSError, AttributeError, RuntimeError, AssertionError):
            self.ok = False

    def _sample(self):
        ct, nv, h = self.ct, self.nv, self.h
        mhz, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if nv.nvmlDeviceGetClockInfo(h, 1, ct.byref(mhz)) != 0:
            return None
        nv.nvmlDeviceGetPowerUsage(h, ct.byref(mw))
        self._reasons(h, ct.byref(rs))
        return (float(mhz.value), mw.value / 1000.0, int(rs.value))

    def _run(self):
        while not self._stop.is_set():
            v = self._sample()
            if v is not None:
                self.samples.append(v)
            time.sleep(self.period)

    def __enter__(self):
        self.samples = []
        self.t = threading.Thread(target=self._run, daemon=True)
        self.t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        self.t.join(timeout=5)

    def summary(self):
        sm = [v[0] for v in self.samples]
        bits = 0
        for v in self.samples:
            bits |= v[2]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(n for b, n in NVML_REASONS.items() if bits & b),
                "samples": len(sm), "sm_mhz_min": min(sm) if sm else None,
                "power_w_max": round(max(v[1] for v in self.samples), 1) if sm else None,
                "source": "NVML in-process, every %.0f ms" % (self.period * 1e3)}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms; entering the
    context waits (up to 5 s) for the first sample so that the sampler is
    running when the timed region starts."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            t0 = time.time()
            while not self.lines and time.time() - t0 < 5.0 and self.proc.poll() is None:
                time.sleep(0.01)
            self.skip = len(self.lines)     # samples taken before the timed region
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines[getattr(self, "skip", 0):]:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm),
                "source": "nvidia-smi every 20 ms"}


# ------------------------------------------------------------- GPU arm

def arm_config(wl, world):
    """The `config` object of both arms' JSON lines."""
    N = wl.num_tokens
    return {"workload": WORKLOAD_DESC if N == 32768 else
            WORKLOAD_DESC.replace("4096 tokens = 32768", "%d tokens = %d" % (N // 8, N)),
            "tokens": N, "hidden": wl.hidden, "experts": wl.num_experts,
            "world_size_logical": wl.world_size, "topk": wl.topk,
            "expert_alignment": wl.alignment, "recv_capacity": wl.recv_capacity,
            "step": "layout + dispatch bf16 + combine (identity experts) + dispatch fp8 "
                    "(the FP8 handle shares the step's layout)",
            "l2": "no flush: every step's inputs/outputs exceed L2 (x 470 MB, recv_x "
                  "4.2 GB, recv_x fp8 2.1 GB)",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def host_cpu():
    """Model name of the host CPU and its hardware threads (for the CPU-baseline record)."""
    model = platform.processor() or platform.machine()
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name:"):
                return {"cpu_model": line.split(":", 1)[1].strip(), "host_threads": os.cpu_count()}
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu part", "hardware"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return {"cpu_model": model, "host_threads": os.cpu_count()}


def prefill_workload(tokens=None):
    """The prefill workload, or the same shape with fewer tokens (a smaller case
    for profiler captures: 8 logical ranks x tokens/8)."""
    import synth
    wl = synth.WORKLOADS["prefill_bf16"]
    if tokens is None or tokens == wl.num_tokens:
        return wl
    assert tokens % wl.world_size == 0
    return wl.with_(num_tokens=tokens, max_tok_per_rank=tokens // wl.world_size)


def run_ours(args, rank, local_rank, world):
    import numpy as np
    import torch

    import combine_ep_layout_gb300 as ep
    import synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = prefill_workload(args.tokens)
    N, H, K, R = wl.num_tokens, wl.hidden, wl.topk, wl.recv_capacity
    cfg16 = ep.make_cfg(wl.world_size, H, wl.max_tok_per_rank, wl.num_expert_per_rank, K,
                        wl.alignment, "bf16", True)
    cfg8 = ep.make_cfg(wl.world_size, H, wl.max_tok_per_rank, wl.num_expert_per_rank, K,
                       wl.alignment, "fp8", True)
    # one layout per step: the FP8 handle reads the bf16 handle's routing
    h16 = ep.EpHandle(cfg16)
    h8 = ep.EpHandle(cfg8, layout_of=h16)
    topk_cpu = synth.gen_topk(wl)
    w_cpu = synth.gen_weights(wl)
    x = synth.gen_x(wl, device=dev)
    topk, w = topk_cpu.to(dev), w_cpu.to(dev)
    recv = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
    recv8 = torch.empty((R, H), dtype=torch.uint8, device=dev)
    scales = torch.empty((R, H // 128), dtype=torch.float32, device=dev)
    out = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    names = ["layout", "dispatch_bf16", "combine", "dispatch_fp8"]

    nvtx = torch.cuda.nvtx

    def step(ev=None):
        # NVTX ranges name each call for profilers that read them (ncu --nvtx)
        if ev is not None:
            ev[0].record(stream)
        nvtx.range_push("layout")
        h16.layout(topk, stream=stream)
        nvtx.range_pop()
        if ev is not None:
            ev[1].record(stream)
        nvtx.range_push("dispatch_bf16")
        h16.dispatch(x, recv, stream=stream)
        nvtx.range_pop()
        if ev is not None:
            ev[2].record(stream)
        nvtx.range_push("combine")
        h16.combine(recv, w, out, stream=stream)   # identity experts: y = recv
        nvtx.range_pop()
        if ev is not None:
            ev[3].record(stream)
        nvtx.range_push("dispatch_fp8")
        h8.dispatch(x, recv8, scales, stream=stream)
        nvtx.range_pop()
        if ev is not None:
            ev[4].record(stream)

    import torch.distributed as dist
    for _ in range(args.warmup):
        step()
    stream.synchronize()
    assert h16.status() == 0 and h8.status() == 0
    # kernels per step: the layout is one cluster launch for small batches, else three
    # the layout is one launch (cluster or fused kernel) or three
    single = "_cluster_" in h16.variant(0) or "_fused_" in h16.variant(0)
    launches_per_step = (1 if single else 3) + 3   # timed steps only
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # the timed region: exactly K steps, events only at its two ends, so that
    # each kernel's programmatic dependent launch overlaps its predecessor's tail
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    nvml = NvmlClockSampler(local_rank)
    with (nvml if nvml.ok else ClockSampler(local_rank)) as clk:
        start.record(stream)
        for i in range(args.steps):
            step()
        stop.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    total_ms = start.elapsed_time(stop)
    # per-kernel split: K more steps with an event between the kernels (the
    # events end each kernel's overlap with the next, so these steps run a
    # little longer than the timed ones)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    for i in range(args.steps):
        step(events[i])
    torch.cuda.synchronize()
    per_kernel = {n: [] for n in names}
    for ev in events:
        for j, n in enumerate(names):
            per_kernel[n].append(ev[j].elapsed_time(ev[j + 1]))
    avg = {n: sum(v) / len(v) for n, v in per_kernel.items()}
    split_ms = sum(ev[0].elapsed_time(ev[4]) for ev in events) / len(events)
    assert h16.status() == 0 and h8.status() == 0

    nbytes = algorithmic_bytes(N, H, K, R)
    step_bytes = nbytes["layout"] + nbytes["dispatch_bf16"] + nbytes["combine"] + \
        nbytes["dispatch_fp8"]
    ms, units = reduce_over_ranks(total_ms / args.steps, step_bytes, world)
    _, toks = reduce_over_ranks(total_ms / args.steps, N, world)
    peak, peak_kind = measured_peaks()
    kernels = {}
    for n in names:
        b = nbytes["layout" if n.startswith("layout") else n]
        us = avg[n] * 1e3
        gbs = b / (avg[n] * 1e-3) / 1e9
        kernels[n] = {"us": round(us, 2), "algorithmic_bytes": b, "gbs": round(gbs, 1),
                      "frac_of_peak": round(gbs / peak, 4),
                      "frac_of_8tbs": round(gbs / 8000.0, 4)}
    dom = max(["dispatch_bf16", "combine", "dispatch_fp8"], key=lambda n: avg[n])
    kname = {"dispatch_bf16": "ep_dispatch_copy_kernel", "combine": "ep_combine_kernel",
             "dispatch_fp8": "ep_dispatch_fp8_kernel"}[dom]
    variant = {"dispatch_bf16": h16.variant(1), "combine": h16.variant(2),
               "dispatch_fp8": h8.variant(1)}[dom]
    # the record holds the compiled register kernels' counters: none for the
    # TMA-staged or run-time specialised variants
    compiled = variant.startswith({"dispatch_bf16": "ep_dispatch_bf16_h", "combine": "ep_combine_w_h",
                                   "dispatch_fp8": "ep_dispatch_fp8_h"}[dom])
    roof = {"bound": "hbm", "kernel": dom, "variant": variant, "achieved": kernels[dom]["gbs"],
            "peak": peak, "peak_kind": peak_kind + " hbm_gbs (burst copy)", "unit": "GB/s",
            "frac": kernels[dom]["frac_of_peak"],
            "traffic": ncu_traffic(kname, N) if compiled else None,
            "algorithmic_bytes": nbytes[dom]}

    e2e = run_e2e(args, ep, torch, dev, wl, topk_cpu, w_cpu, x, (h16, h8), (recv, recv8, scales),
                  step_bytes, world) if not args.no_e2e else None
    # the other workloads (decode: 1024 tokens, the pages' small-batch shape;
    # tiny; skewed Zipf routing), each measured after the timed region as
    # --all-configs measures it: context, not `value`
    def summary(name):
        d = measure_workload(name, synth.WORKLOADS[name], False, 50, 5, cold)
        out = {k: d[k] for k in ("workload", "tokens", "hidden", "experts", "topk", "l2", "timing",
                                 "steps")}
        for k in ("layout", "dispatch", "combine", "layout_dispatch", "step"):
            keep = ("us_median", "gbs", "frac_of_8tbs", "frac_of_peak", "tokens_per_s")
            out[k] = {kk: d[k][kk] for kk in keep + (("variant",) if "variant" in d[k] else ())}
        return out
    decode, others = None, None
    if not args.no_decode:
        cold = ColdRegions(dev)
        decode = summary("decode")
        others = {name: summary(name) for name in ("tiny", "skewed")}
        del cold
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, topk_cpu, w_cpu, x, budget_s=args.cpu_seconds)

    if rank != 0:
        return None
    clocks = clk.summary()
    gbs = units / (ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; shapes and distributions of the prefill workload)",
        "config": arm_config(wl, world),
        "tokens_per_s": round(toks / (ms * 1e-3), 1),
        "kernels": kernels,
        "ms_per_step_with_kernel_events": round(split_ms, 4),
        "roofline": roof,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        # step time x median SM clock: thousands of SM cycles per step
        "ms_per_step_x_sm_mhz": round(ms * clocks["sm_mhz"], 1) if clocks.get("sm_mhz") else None,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "decode_workload": decode,
        "other_workloads": others,
    }
    return line


def run_e2e(args, ep, torch, dev, wl, topk_cpu, w_cpu, x, handles, bufs, step_bytes, world):
    """Same step through the public API, with this step's inputs copied from
    pinned host memory and the combined output read back, inside the timed
    region.  Steps are pipelined the way a serving loop runs them: inputs and
    outputs are double-buffered on the device, and three streams (host->device,
    compute, device->host) ordered by events let step i's read-back overlap
    step i+1's upload and kernels."""
    h16, h8 = handles
    recv, recv8, scales = bufs
    N, H = wl.num_tokens, wl.hidden
    x_h = x.cpu().pin_memory()
    topk_h = topk_cpu.pin_memory()
    w_h = w_cpu.pin_memory()
    nb = args.e2e_buffers
    out_h = [torch.empty((N, H), dtype=torch.bfloat16).pin_memory() for _ in range(nb)]
    x_d = [torch.empty_like(x) for _ in range(nb)]
    topk_d = [torch.empty(topk_cpu.shape, dtype=torch.int64, device=dev) for _ in range(nb)]
    w_d = [torch.empty(w_cpu.shape, dtype=torch.float32, device=dev) for _ in range(nb)]
    out_d = [torch.empty((N, H), dtype=torch.bfloat16, device=dev) for _ in range(nb)]
    s_in, s_cmp, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))

    def run(n):
        done = [None] * n     # compute of step i finished (its inputs may be overwritten)
        read = [None] * n     # step i's output is on the host (out_d[b] may be overwritten)
        for i in range(n):
            b = i % nb
            if i >= nb:
                s_in.wait_event(done[i - nb])
            with torch.cuda.stream(s_in):
                x_d[b].copy_(x_h, non_blocking=True)
                topk_d[b].copy_(topk_h, non_blocking=True)
                w_d[b].copy_(w_h, non_blocking=True)
            ready = torch.cuda.Event()
            ready.record(s_in)
            s_cmp.wait_event(ready)
            if i >= nb:
                s_cmp.wait_event(read[i - nb])
            h16.layout(topk_d[b], stream=s_cmp)
            h16.dispatch(x_d[b], recv, stream=s_cmp)
            h16.combine(recv, w_d[b], out_d[b], stream=s_cmp)
            h8.dispatch(x_d[b], recv8, scales, stream=s_cmp)
            done[i] = torch.cuda.Event()
            done[i].record(s_cmp)
            s_out.wait_event(done[i])
            with torch.cuda.stream(s_out):
                out_h[b].copy_(out_d[b], non_blocking=True)
            read[i] = torch.cuda.Event()
            read[i].record(s_out)

    run(max(3, args.warmup))
    torch.cuda.synchronize()
    n = max(1, args.steps)
    import torch.distributed as dist
    # three timed regions of n steps each; the median is reported (on shared
    # hosts an occasional region ran ~1.8x longer with the same link floor)
    reps = []
    for _ in range(3):
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        a.record(s_in)
        run(n)
        z.record(s_out)
        torch.cuda.synchronize()
        reps.append(a.elapsed_time(z) / n)
    ms, units = reduce_over_ranks(statistics.median(reps), step_bytes, world)
    h2d = x_h.numel() * 2 + topk_h.numel() * 8 + w_h.numel() * 4
    d2h = out_h[0].numel() * 2
    link = host_link(torch, x_h, x_d[0], out_d[0], out_h[0], s_in, s_out)
    link["floor_ms_per_step"] = round((h2d + d2h) / (link["bidir_gbs"] * 1e9) * 1e3, 4)
    return {"value": round(units / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "ms_per_step_regions": [round(r, 4) for r in reps],
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "host_link": link,
            "pipelining": "%d device buffers of inputs/outputs in rotation; upload, compute "
                          "and read-back on three streams ordered by events" % nb}


def host_link(torch, x_h, x_d, out_d, out_h, s_in, s_out, reps=5):
    """Copy-engine bandwidth of the host link on the e2e buffers: x up alone,
    the output down alone, and both at once (the floor under the e2e step)."""
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(up, down):
        torch.cuda.synchronize()
        a.record(s_in)
        s_out.wait_event(a)
        for _ in range(reps):
            if up:
                with torch.cuda.stream(s_in):
                    x_d.copy_(x_h, non_blocking=True)
            if down:
                with torch.cuda.stream(s_out):
                    out_h.copy_(out_d, non_blocking=True)
        done = torch.cuda.Event()
        done.record(s_out)
        s_in.wait_event(done)
        b.record(s_in)
        b.synchronize()
        return a.elapsed_time(b) / reps

    nb_up, nb_down = x_h.numel() * x_h.element_size(), out_d.numel() * out_d.element_size()
    timed(True, True)
    up, down, both = timed(True, False), timed(False, True), timed(True, True)
    return {"h2d_gbs": round(nb_up / up / 1e6, 1), "d2h_gbs": round(nb_down / down / 1e6, 1),
            "bidir_gbs": round((nb_up + nb_down) / both / 1e6, 1),
            "how": "cudaMemcpyAsync from / to the pinned e2e buffers, alone and both directions at once"}


# ------------------------------------------------------------- all configs

class ColdRegions:
    """The L2 flush (256 MB written, then 256 MB read) and the ~100 us GPU sleep
    that precede every region timed by measure_workload, on one stream."""

    def __init__(self, dev):
        import torch
        self.dev = dev
        self.flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.flush_read = torch.ones(256 << 20, dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.Stream(device=dev)

    def __call__(self, i):
        import torch
        with torch.cuda.stream(self.stream):
            self.flush.fill_(i & 0xFF)
            self.flush_read.sum(dtype=torch.int32)
            torch.cuda._sleep(SLEEP_CYCLES)


def measure_workload(name, wl, ne, steps, warmup, cold):
    """One workload's layout, dispatch, combine and step, each timed in its own
    region after cold(i) (see run_all_configs); returns the JSON line's dict."""
    import torch

    import combine_ep_layout_gb300 as ep
    import synth

    dev, s = cold.dev, cold.stream
    peak, peak_kind = measured_peaks()
    N, H, K = wl.num_tokens, wl.hidden, wl.topk
    cfg = ep.make_cfg(wl.world_size, H, wl.max_tok_per_rank, wl.num_expert_per_rank, K,
                      wl.alignment, wl.dispatch_dtype, wl.use_weights and not ne, no_expand=ne)
    R = ep.ep_recv_capacity(cfg)
    h = ep.EpHandle(cfg)
    topk = synth.gen_topk(wl).to(dev)
    w = synth.gen_weights(wl).to(dev)
    x = synth.gen_x(wl, device=dev)
    fp8 = wl.dispatch_dtype == "fp8"
    recv = torch.empty((R, H), dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev)
    scales = torch.empty((R, H // 128), dtype=torch.float32, device=dev) if fp8 else None
    # combine reads bf16 expert outputs: the dispatched rows (identity experts), or
    # for the FP8 workload an independent bf16 N(0,1) [Rcap, H]
    y = synth.gen_y(wl, device=dev) if fp8 else recv
    out = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
    wc = None if ne else w
    regions = {
        "layout": lambda: h.layout(topk, stream=s),
        "dispatch": lambda: h.dispatch(x, recv, scales, stream=s),
        "combine": lambda: h.combine(y, wc, out, stream=s),
        "layout_dispatch": lambda: (h.layout(topk, stream=s), h.dispatch(x, recv, scales, stream=s)),
        "step": lambda: (h.layout(topk, stream=s), h.dispatch(x, recv, scales, stream=s),
                         h.combine(y, wc, out, stream=s)),
    }
    times = {k: [] for k in regions}
    for i in range(warmup + steps):
        ev = []
        for k, fn in regions.items():
            cold(i)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            fn()
            b.record(s)
            ev.append((k, a, b))
        s.synchronize()
        if i >= warmup:
            for k, a, b in ev:
                times[k].append(a.elapsed_time(b) * 1e3)
    assert h.status() == 0
    if ne:
        rows = int(h.field(ep.FIELD_NUM_RECV).cpu()[0])
        nb = algorithmic_bytes_nonexpand(N, H, K, rows, R, fp8)
        dkey = "dispatch"
    else:
        nb = algorithmic_bytes(N, H, K, R)
        dkey = "dispatch_fp8" if fp8 else "dispatch_bf16"
    line = {"workload": name, "layout_kind": "non-expand" if ne else "expand",
            "tokens": N, "hidden": H, "experts": wl.num_experts, "topk": K,
            "alignment": wl.alignment, "dispatch_dtype": wl.dispatch_dtype,
            "routing": wl.routing,
            "l2": "flushed before every timed region (256 MB write, then 256 MB read)",
            "timing": "device: each region enqueued behind a 100 us GPU sleep",
            "steps": steps, "peak_gbs": peak, "peak_kind": peak_kind}
    step_bytes = nb["layout"] + nb[dkey] + nb["combine"]
    for k, b in (("layout", nb["layout"]), ("dispatch", nb[dkey]), ("combine", nb["combine"]),
                 ("layout_dispatch", nb["layout"] + nb[dkey]), ("step", step_bytes)):
        us = statistics.median(times[k])
        line[k] = {"us_median": round(us, 2), "us_mean": round(statistics.mean(times[k]), 2),
                   "us_min": round(min(times[k]), 2),
                   "us_max": round(max(times[k]), 2), "algorithmic_bytes": b,
                   "gbs": round(b / (us * 1e-6) / 1e9, 1),
                   "frac_of_peak": round(b / (us * 1e-6) / 1e9 / peak, 4),
                   "frac_of_8tbs": round(b / (us * 1e-6) / 1e9 / 8000.0, 4),
                   "tokens_per_s": round(N / (us * 1e-6), 1)}
        if k in ("layout", "dispatch", "combine"):
            line[k]["variant"] = h.variant({"layout": 0, "dispatch": 1, "combine": 2}[k])
    h.free()
    del recv, scales, y, out, x
    torch.cuda.empty_cache()
    return line


def run_all_configs(args):
    """Per workload (tiny, decode, prefill bf16, prefill FP8, skewed) and layout
    (expand, then non-expand: one row per (token, rank), unweighted combine),
    one JSON line each with four timed regions per step, each after its own L2
    flush and GPU sleep (below):
      layout    the layout alone;
      dispatch  the dispatch alone (on the layout just computed);
      combine   the combine alone (on the rows just dispatched, or y);
      layout_dispatch  layout -> dispatch back to back (dispatch with its layout);
      step      layout -> dispatch -> combine back to back, events only at its
                two ends, so that the kernels' programmatic dependent launch
                (each scheduled while its predecessor drains) is counted.
    Medians (and means) over args.steps steps.  The flush writes a 256 MB
    buffer (twice L2) and then reads another 256 MB buffer: the write alone
    leaves L2 full of the flush's own dirty lines, which the next write-heavy
    kernel would then have to write back to DRAM on top of its own traffic
    (decode dispatch measured 24.8 us after a write-only flush and 20.8 us
    after write + read); flushing before each kernel likewise keeps a kernel
    from paying for the write-back of its predecessor's output.  Each region
    starts behind a ~100 us device-side sleep, so that the host has enqueued it
    before the GPU reaches it: the events then time device work, not Python's
    launch latency, which is longer than a small workload's kernels."""
    import torch

    import synth

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    only = set(args.workload.split(",")) if args.workload else None
    cold = ColdRegions(dev)
    for name, wl, ne in [(n, w, ne) for ne in (False, True) for n, w in synth.WORKLOADS.items()
                         if only is None or n in only]:
        print(json.dumps(measure_workload(name, wl, ne, args.steps, args.warmup, cold)), flush=True)
    return 0


# Probe kernels for --mix-ceilings: the memory traffic of the data kernels
# with no routing (no index loads, contiguous destinations, xor instead of the
# fold), so that their times are what the memory system gives these byte mixes.
MIX_PROBE_CU = r"""
#include <cstdint>
#include <cuda_runtime.h>
struct V8 { uint32_t w[8]; };
__device__ __forceinline__ void ld8(const uint8_t* p, V8& v) {
  asm volatile("ld.global.cg.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]),
                 "=r"(v.w[5]), "=r"(v.w[6]), "=r"(v.w[7]) : "l"(p));
}
__device__ __forceinline__ void st8(uint8_t* p, const V8& v) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" :: "l"(p), "r"(v.w[0]),
               "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]),
               "r"(v.w[7]) : "memory");
}
// grid-stride over n32 32-byte vectors
__global__ void write_only(uint8_t* dst, int64_t n32) {
  V8 v;
  for (int j = 0; j < 8; ++j) v.w[j] = 0x3f803f80u + j;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n32; i += stride)
    st8(dst + i * 32, v);
}
__global__ void read_only(const uint8_t* src, int64_t n32, uint32_t* sink) {
  uint32_t acc = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n32; i += 4 * stride) {
    V8 a, b, c, d;
    ld8(src + i * 32, a); ld8(src + (i + stride) * 32, b);
    ld8(src + (i + 2 * stride) * 32, c); ld8(src + (i + 3 * stride) * 32, d);
    for (int j = 0; j < 8; ++j) acc ^= a.w[j] ^ b.w[j] ^ c.w[j] ^ d.w[j];
  }
  for (; i < n32; i += stride) {
    V8 a;
    ld8(src + i * 32, a);
    for (int j = 0; j < 8; ++j) acc ^= a.w[j];
  }
  if (acc == 0x9e3779b9u) sink[0] = acc;  // keeps the loads
}
__global__ void copy_1to1(const uint8_t* src, uint8_t* dst, int64_t n32) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n32; i += stride) {
    V8 a;
    ld8(src + i * 32, a);
    st8(dst + i * 32, a);
  }
}
// a CTA per row of `vecs` 32-byte vectors, 2 per thread (blockDim = vecs / 2):
// row t read once and written to rows t*K .. t*K+K-1 (dispatch's mix), or rows
// t*K .. t*K+K-1 read and their xor written to row t (combine's mix)
template <int K>
__global__ void bcast(const uint8_t* x, uint8_t* big, int row) {
  const int64_t t = blockIdx.x;
  const int T = blockDim.x;
  V8 a, b;
  ld8(x + t * row + threadIdx.x * 32, a);
  ld8(x + t * row + (threadIdx.x + T) * 32, b);
  for (int k = 0; k < K; ++k) {
    uint8_t* d = big + (t * K + k) * row;
    st8(d + threadIdx.x * 32, a);
    st8(d + (threadIdx.x + T) * 32, b);
  }
}
template <int K>
__global__ void reduce(const uint8_t* big, uint8_t* out, int row) {
  const int64_t t = blockIdx.x;
  const int T = blockDim.x;
  V8 a[K], b[K];
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const uint8_t* s = big + (t * K + k) * row;
    ld8(s + threadIdx.x * 32, a[k]);
    ld8(s + (threadIdx.x + T) * 32, b[k]);
  }
#pragma unroll
  for (int k = 1; k < K; ++k)
    for (int j = 0; j < 8; ++j) { a[0].w[j] ^= a[k].w[j]; b[0].w[j] ^= b[k].w[j]; }
  st8(out + t * row + threadIdx.x * 32, a[0]);
  st8(out + t * row + (threadIdx.x + T) * 32, b[0]);
}
extern "C" int mix_write(void* d, long long n32, int g, int b, void* s) {
  write_only<<<g, b, 0, (cudaStream_t)s>>>((uint8_t*)d, n32); return (int)cudaGetLastError();
}
extern "C" int mix_read(const void* x, long long n32, void* sink, int g, int b, void* s) {
  read_only<<<g, b, 0, (cudaStream_t)s>>>((const uint8_t*)x, n32, (uint32_t*)sink);
  return (int)cudaGetLastError();
}
extern "C" int mix_copy(const void* x, void* d, long long n32, int g, int b, void* s) {
  copy_1to1<<<g, b, 0, (cudaStream_t)s>>>((const uint8_t*)x, (uint8_t*)d, n32);
  return (int)cudaGetLastError();
}
extern "C" int mix_bcast8(const void* x, void* big, int n, int row, void* s) {
  bcast<8><<<n, row / 64, 0, (cudaStream_t)s>>>((const uint8_t*)x, (uint8_t*)big, row);
  return (int)cudaGetLastError();
}
extern "C" int mix_reduce8(const void* big, void* out, int n, int row, void* s) {
  reduce<8><<<n, row / 64, 0, (cudaStream_t)s>>>((const uint8_t*)big, (uint8_t*)out, row);
  return (int)cudaGetLastError();
}
"""


def run_mix_ceilings(args):
    """What the memory system gives the data kernels' byte mixes on the prefill
    shape (32768 tokens, or --tokens; rows of 7168 bf16 = 14336 bytes, top-8): probe kernels
    (MIX_PROBE_CU, compiled here with nvcc) that move the same bytes as the data
    kernels with no routing, each timed in its own region after the same L2
    flush and GPU sleep as --all-configs:
      write_only   fill the [N*K] rows                   (dispatch's write volume)
      read_only    read the [N*K] rows                   (combine's read volume)
      copy_1to1    copy [N] rows                         (the measured-peak copy)
      bcast_1to8   row t -> rows t*K..t*K+K-1, a CTA per row      (dispatch's mix)
      reduce_8to1  rows t*K..t*K+K-1 -> row t, a CTA per row      (combine's mix)
    The grid-stride cases run several grids (SMs x 2..16 CTAs of 256 or 512
    threads); the best is reported with its geometry.  GB/s = bytes read +
    written / device time; best and median over args.steps."""
    import ctypes

    import torch

    from combine_ep_layout_gb300 import build as native_build

    out_dir = os.path.join(ROOT, "_build")
    os.makedirs(out_dir, exist_ok=True)
    src, so = os.path.join(out_dir, "mix_probe.cu"), os.path.join(out_dir, "mix_probe.so")
    with open(src, "w") as f:
        f.write(MIX_PROBE_CU)
    subprocess.check_call([native_build.nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                           "-shared", "-Xcompiler", "-fPIC", "-o", so, src])
    lib = ctypes.CDLL(so)
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    cold = ColdRegions(dev)
    s = cold.stream
    sp = ctypes.c_void_p(s.cuda_stream)
    N, K, H = args.tokens or 32768, 8, 7168
    row = H * 2
    big = torch.empty(N * K * row, dtype=torch.uint8, device=dev)
    x = torch.randint(0, 255, (N * row,), dtype=torch.uint8, device=dev)
    out = torch.empty(N * row, dtype=torch.uint8, device=dev)
    sink = torch.zeros(4, dtype=torch.int32, device=dev)
    P = ctypes.c_void_p
    nbig, nx = big.numel() // 32, x.numel() // 32
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    grids = [(sms * c, b) for c in (2, 4, 8, 16) for b in (256, 512)]
    cases = []
    for g, b in grids:
        cases.append(("write_only", "%d x %d" % (g, b), big.numel(),
                      lambda g=g, b=b: lib.mix_write(P(big.data_ptr()), ctypes.c_longlong(nbig), g, b, sp)))
        cases.append(("read_only", "%d x %d" % (g, b), big.numel(),
                      lambda g=g, b=b: lib.mix_read(P(big.data_ptr()), ctypes.c_longlong(nbig),
                                                    P(sink.data_ptr()), g, b, sp)))
        cases.append(("copy_1to1", "%d x %d" % (g, b), 2 * x.numel(),
                      lambda g=g, b=b: lib.mix_copy(P(x.data_ptr()), P(out.data_ptr()),
                                                    ctypes.c_longlong(nx), g, b, sp)))
    cases.append(("bcast_1to8", "%d x %d" % (N, row // 64), (K + 1) * N * row,
                  lambda: lib.mix_bcast8(P(x.data_ptr()), P(big.data_ptr()), N, row, sp)))
    cases.append(("reduce_8to1", "%d x %d" % (N, row // 64), (K + 1) * N * row,
                  lambda: lib.mix_reduce8(P(big.data_ptr()), P(out.data_ptr()), N, row, sp)))
    peak, peak_kind = measured_peaks()
    line = {"mix_ceilings": "probe kernels moving the prefill data kernels' bytes with no routing",
            "tokens": N, "row_bytes": row, "topk": K,
            "l2": "flushed before every timed region (256 MB write, then 256 MB read)",
            "steps": args.steps, "peak_gbs": peak, "peak_kind": peak_kind, "cases": {}}
    for name, geom, nbytes, fn in cases:
        ts = []
        for i in range(args.warmup + args.steps):
            cold(i)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            rc = fn()
            b.record(s)
            s.synchronize()
            if rc != 0:
                raise RuntimeError("mix probe %s launch failed: %d" % (name, rc))
            if i >= args.warmup:
                ts.append(a.elapsed_time(b) * 1e3)
        best, med = min(ts), statistics.median(ts)
        r = {"grid": geom, "bytes": nbytes, "us_best": round(best, 1), "us_median": round(med, 1),
             "gbs_best": round(nbytes / best / 1e3, 1), "gbs_median": round(nbytes / med / 1e3, 1)}
        prev = line["cases"].get(name)
        if prev is None or r["gbs_median"] > prev["gbs_median"]:
            line["cases"][name] = r
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- CPU oracle

def oracle_bufs(wl, block):
    """Receive buffers for one oracle sub-batch of `block` tokens."""
    import numpy as np
    import oracle
    R = oracle.recv_capacity(block, wl.topk, wl.num_experts, wl.alignment)
    H = wl.hidden
    return (np.zeros((R, H), np.uint16), np.zeros((R, H), np.uint8),
            np.zeros((R, H // 128), np.float32))


def oracle_step_sample(wl, topk_np, w_np, x_bits, tok0, ntok, bufs):
    """One oracle pass of the whole step (layout, dispatch bf16, combine, dispatch
    fp8) over the sub-batch of tokens [tok0, tok0+ntok) of the prefill workload,
    taken as a batch of its own (ntok / W tokens per logical rank), so that the
    layout and the data movement keep the step's per-token proportions.
    Returns (algorithmic bytes, tokens)."""
    import oracle
    W = wl.world_size
    tk = topk_np[tok0:tok0 + ntok]
    recv16, recv8, scales = bufs
    lay = oracle.layout(tk, W, ntok // W, wl.num_expert_per_rank, wl.alignment,
                        rcap=recv16.shape[0])
    sl = lay["dst_slot"]
    xs = x_bits[tok0:tok0 + ntok]
    oracle.dispatch_bf16(xs, sl, recv16)
    oracle.combine(recv16, sl, w_np[tok0:tok0 + ntok])
    oracle.dispatch_fp8(xs, sl, recv8, scales)
    nb = algorithmic_bytes(ntok, wl.hidden, wl.topk, lay["rcap"])
    return nb["layout"] + nb["dispatch_bf16"] + nb["combine"] + nb["dispatch_fp8"], ntok


def cpu_baseline(wl, topk_cpu, w_cpu, x, budget_s=15.0, block=512):
    """The oracle as it stands (single-threaded C), on a bounded sample: sub-batches
    of `block` tokens until ~budget_s seconds of CPU work."""
    import synth
    x_bits = synth.bits16(x)
    topk_np, w_np = topk_cpu.numpy(), w_cpu.numpy()
    bufs = oracle_bufs(wl, block)
    t0 = time.perf_counter()
    nbytes, ntoks, tok = 0, 0, 0
    while time.perf_counter() - t0 < budget_s and tok + block <= wl.num_tokens:
        b, n = oracle_step_sample(wl, topk_np, w_np, x_bits, tok, block, bufs)
        nbytes += b
        ntoks += n
        tok += block
    dt = time.perf_counter() - t0
    return {"value": round(nbytes / dt / 1e9, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
            **host_cpu(),
            "tokens_per_s": round(ntoks / dt, 1),
            "sample": "%d of %d tokens as sub-batches of %d (each: layout, dispatch bf16, "
                      "combine, dispatch fp8 of the sub-batch), %.1f s" %
                      (ntoks, wl.num_tokens, block, dt)}


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle, timed on the host, same metric and unit."""
    if rank != 0:
        return None
    import numpy as np

    import synth
    wl = synth.WORKLOADS["prefill_bf16"]
    topk_cpu, w_cpu = synth.gen_topk(wl), synth.gen_weights(wl)
    block = args.ref_block
    nblk = wl.num_tokens // block
    # x for the sub-batches the run visits (cycling through the batch)
    x = synth.gen_bf16_normal(block * min(nblk, args.steps + args.warmup), wl.hidden,
                              wl.seed * 16 + 3)
    x_bits = synth.bits16(x)
    bufs = oracle_bufs(wl, block)
    topk_np, w_np = topk_cpu.numpy(), w_cpu.numpy()
    xb_full = np.zeros((wl.num_tokens, wl.hidden), np.uint16)
    xb_full[:x_bits.shape[0]] = x_bits
    for i in range(args.warmup):
        oracle_step_sample(wl, topk_np, w_np, xb_full, (i % nblk) * block, block, bufs)
    t0 = time.perf_counter()
    nbytes = ntok = 0
    for i in range(args.steps):
        b, n = oracle_step_sample(wl, topk_np, w_np, xb_full, ((args.warmup + i) % nblk) * block,
                                  block, bufs)
        nbytes += b
        ntok += n
    dt = time.perf_counter() - t0
    v = round(nbytes / dt / 1e9, 3)
    return {"metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / max(1, args.steps) * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "impl": "reference",
            "config": dict(arm_config(wl, 1),
                           sample="each step: the whole path (layout, dispatch bf16, combine, "
                                  "dispatch fp8) over a sub-batch of %d of the 32768 tokens" % block),
            "cpu_baseline": {"value": v, "unit": "GB/s", "kind": "oracle", "cores": 1, **host_cpu(),
                             "sample": "%d tokens per step, %d steps, %.1f s" %
                                       (block, args.steps, dt)},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-buffers", type=int, default=2,
                    help="device input/output buffers the end-to-end loop rotates through")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true",
                    help="skip the decode, tiny and skewed measurements added to the step line")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-block", type=int, default=256)
    ap.add_argument("--tokens", type=int, default=None,
                    help="tokens of a smaller case of the prefill shape (profiling, --mix-ceilings)")
    ap.add_argument("--all-configs", action="store_true",
                    help="time layout / dispatch / combine on every workload (one line each)")
    ap.add_argument("--workload", default=None,
                    help="with --all-configs: comma-separated workload names (default: all)")
    ap.add_argument("--mix-ceilings", action="store_true",
                    help="time probe kernels that move the data kernels' bytes with no routing")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0
    if args.mix_ceilings:
        return run_mix_ceilings(args)
    if args.all_configs:
        import __graft_entry__
        __graft_entry__.build()
        return run_all_configs(args)
    import torch
    import torch.distributed as dist
    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    import __graft_entry__
    __graft_entry__.build()
    line = run_ours(args, rank, local_rank, world)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
