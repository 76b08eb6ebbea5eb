#!/usr/bin/env python
"""Throughput of the clustered, compressed MoE layer forward pass (tokens/s) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

One step = one whole forward pass (route, permute, gate/up GEMM with the residual/SwiGLU epilogue,
down GEMM, combine) over the workload's T tokens, inputs resident in HBM.  The timed steps replay
a CUDA graph captured from one moe_hier_forward call (the same kernels, without the host's
per-call launch work); the end-to-end figure calls moe_hier_forward directly every step, with the
host-to-device copy of x and the device-to-host copy of y inside the timed region.  Between timed
steps the L2 is flushed (a 256 MiB write).  Per-kernel times come from CUDA events that the
library records between its launches, in a pass whose launches are queued behind a sleep kernel
so that the intervals hold device time only.  Multi-GPU (torchrun): every rank runs an
independent replica on its own GPU (tokens are independent; no collective on the data path),
weak scaling.
The oracle is only imported by the CPU-baseline leg and by --impl reference.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer fwd tokens/s on 1 B300; % of BF16 tensor or HBM roofline"
DEFAULT_CONFIG = "mixtral_prefill"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--prepared", action="store_true",
                    help="residual stacks built once (moe_hier_prepare), steps call moe_hier_forward_prepared")
    ap.add_argument("--tokens", type=int, default=0,
                    help="profiling aid: run the workload's layer on this many tokens instead of its T")
    return ap.parse_args()


def workload_config(args):
    from synth import CONFIGS
    cfg = CONFIGS[args.config]
    return cfg.replace(T=args.tokens) if args.tokens > 0 else cfg


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def recorded_traffic(config: str, kernel: str):
    """DRAM bytes (read + write) per launch of `kernel` on `config` from the committed ncu summary
    profiles/dram_traffic.json, or None when the source file that defines the kernel changed since
    the counters were taken (each entry records that file and its SHA-256)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        rec = json.load(fh)
    ent = rec.get("traffic", {}).get(config, {}).get(kernel)
    if not isinstance(ent, dict):
        return None
    src = os.path.join(ROOT, "compressed_expert_two_b300", "csrc", ent.get("source", ""))
    if not os.path.isfile(src):
        return None
    with open(src, "rb") as fh:
        if hashlib.sha256(fh.read()).hexdigest() != ent.get("sha256"):
            return None
    return ent.get("bytes")


def workload_name(cfg) -> str:
    return (f"{cfg.name}: T={cfg.T} d_model={cfg.d} d_ff={cfg.f} E={cfg.E} G={cfg.G} "
            f"top{cfg.kg} group(s) then top{cfg.ke} "
            f"{'over their union' if cfg.route == 'across' else 'in group'}, r={cfg.r} {cfg.resid} residual, "
            f"{cfg.dtype} base, SwiGLU")


# ------------------------------------------------------------------ clocks during the timed region
class _Nvml:
    """The few read-only NVML calls the clock sampler needs: the pynvml module when installed,
    else the driver's libnvidia-ml through ctypes."""
    SM = 1                                                  # NVML_CLOCK_SM

    def __init__(self):
        try:
            import pynvml
            pynvml.nvmlInit()
            self.py = pynvml
            return
        except Exception:
            self.py = None
        import ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        self.ct = ctypes
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def handle_by_uuid(self, uuid):
        if self.py:
            return self.py.nvmlDeviceGetHandleByUUID(uuid)
        h = self.ct.c_void_p()
        if self.lib.nvmlDeviceGetHandleByUUID(self.ct.c_char_p(uuid.encode()), self.ct.byref(h)) != 0:
            raise RuntimeError("nvmlDeviceGetHandleByUUID failed")
        return h

    def _uint(self, fn, h, kind):
        v = self.ct.c_uint()
        if fn(h, self.ct.c_int(kind), self.ct.byref(v)) != 0:
            raise RuntimeError("NVML clock query failed")
        return v.value

    def max_sm_mhz(self, h):
        if self.py:
            return self.py.nvmlDeviceGetMaxClockInfo(h, self.py.NVML_CLOCK_SM)
        return self._uint(self.lib.nvmlDeviceGetMaxClockInfo, h, self.SM)

    def sm_mhz(self, h):
        if self.py:
            return self.py.nvmlDeviceGetClockInfo(h, self.py.NVML_CLOCK_SM)
        return self._uint(self.lib.nvmlDeviceGetClockInfo, h, self.SM)

    def reasons(self, h):
        if self.py:
            try:
                return self.py.nvmlDeviceGetCurrentClocksEventReasons(h)
            except AttributeError:
                return self.py.nvmlDeviceGetCurrentClocksThrottleReasons(h)
        v = self.ct.c_ulonglong()
        if self.reasons_fn(h, self.ct.byref(v)) != 0:
            raise RuntimeError("NVML reasons query failed")
        return v.value


class Clocks:
    """SM clock and clock-event reasons sampled while the timed steps run.

    NVML is polled from a thread (about every 0.5 ms: the timed region can be a few ms); the GPU is
    found by its UUID because NVML does not follow CUDA_VISIBLE_DEVICES.  Without NVML the
    nvidia-smi sampler (200 ms) is used instead."""
    REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40}
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        import threading
        self.device = device
        self.samples = []
        self.stop_flag = threading.Event()
        self.thread = None
        self.handle = None
        self.proc = None
        self.file = None
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            self.nvml = _Nvml()
            self.handle = self.nvml.handle_by_uuid(uuid if uuid.startswith("GPU-") else "GPU-" + uuid)
            self.max_mhz = self.nvml.max_sm_mhz(self.handle)
        except Exception as exc:                      # no NVML: the nvidia-smi sampler below
            self.handle = None
            self.nvml_error = str(exc)[:120]

    def _poll(self):
        nv = self.nvml
        while not self.stop_flag.is_set():
            try:
                self.samples.append((nv.sm_mhz(self.handle), nv.reasons(self.handle)))
            except Exception:
                pass
            time.sleep(0.0005)

    def start(self):
        import threading
        if self.handle is not None:
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device.index or 0), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.thread is not None:
            self.stop_flag.set()
            self.thread.join()
            sm = [m for m, _ in self.samples]
            reasons = sorted(n for n, bit in self.REASONS.items() if any(r & bit for _, r in self.samples))
            return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                    "samples": len(sm), "source": "nvml, polled during the timed steps", "reasons": reasons}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock source"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        with open(self.file.name) as fh:
            lines = [ln.strip() for ln in fh if ln.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "samples": len(sm),
                "source": "nvidia-smi, 200 ms", "reasons": sorted(reasons)}


# ------------------------------------------------------------------ CPU oracle timing (rank 0 only)
def oracle_tokens_per_s(inp, seconds: float, chunk: int):
    """Runs the oracle (route + FFN of each chunk of tokens) until `seconds` elapsed."""
    import numpy as np

    import oracle
    from oracle.moe import _np
    cfg = inp["cfg"]
    x = _np(inp["x"]).astype(np.float32)
    wgp, bgp, wep = _np(inp["w_group"]), _np(inp["b_group"]), _np(inp["w_expert"])
    gm = _np(inp["group_map"])
    done, t0 = 0, time.perf_counter()
    start = 0
    while True:
        toks = np.arange(start, min(start + chunk, cfg.T))
        routing = oracle.route(x[toks], wgp, bgp, wep, gm, cfg.kg, cfg.ke, cfg.route)
        sub = dict(inp)
        sub["x"] = inp["x"][toks[0]:toks[-1] + 1]
        sub["cfg"] = cfg.replace(T=len(toks))
        oracle.forward_tokens(sub, routing=routing)
        done += len(toks)
        start = (start + chunk) % cfg.T
        el = time.perf_counter() - t0
        if el >= seconds:
            return done / el, done, el


CPU_CHUNK = {"tiny_f32": 256, "small_bf16_int4": 1024, "mixtral_prefill": 16,
             "finegrained_skewed": 512, "finegrained_across": 512, "decode": 4}


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ multi-rank aggregation
def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time, on every rank: the job is done when its last rank is.  Ranks are
    independent replicas, so this reduction of one number is the only cross-rank exchange."""
    if world == 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_rank: int, steps: int, ms: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank * steps / (ms / 1e3)


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from compressed_expert_two_b300 import _lib as L
    from compressed_expert_two_b300 import workload
    from compressed_expert_two_b300.layer import DeviceLayer
    from synth import make_inputs

    cfg = workload_config(args)
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    inp = make_inputs(cfg)
    layer = DeviceLayer(inp, device=dev)
    out = layer.new_outputs()
    stream = torch.cuda.current_stream(dev)
    if args.prepared:
        layer.prepare()
        layer.forward = layer.forward_prepared       # every step below runs the prepared path

    for _ in range(max(args.warmup, 3)):
        layer.forward(out=out)
    torch.cuda.synchronize(dev)
    if layer.status() != 0:
        raise RuntimeError("device status after warm-up: %d" % layer.status())

    # kernels of one forward and the groups/experts the workload hits (for the byte count)
    probe = [torch.cuda.Event(enable_timing=True) for _ in range(64)]
    for e in probe:
        e.record(stream)
    arr = L.moe_hier_profile_begin([e.cuda_event for e in probe])
    layer.forward(out=out)
    names = L.moe_hier_profile_end()
    del arr
    n_k = len(names)
    torch.cuda.synchronize(dev)
    eidx = out["eidx"].cpu()
    experts_hit = int(torch.unique(eidx).numel())
    groups_hit = int(torch.unique(out["gidx"].cpu()).numel())
    load = workload.load_stats(out["gidx"].cpu().numpy(), eidx.numpy(), cfg.G, cfg.E,
                               active=(out["gate"] > 0).cpu().numpy())

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    # ---- per-kernel device times: launches queued behind a sleep kernel, events between them
    n_prof = max(3, min(args.steps, 10))
    pev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_k + 1)] for _ in range(n_prof)]
    for row in pev:
        for e in row:
            e.record(stream)
    torch.cuda.synchronize(dev)
    for i in range(n_prof):
        flush.fill_(i & 0xFF)
        torch.cuda._sleep(2_000_000)               # ~1 ms: the host queues the whole forward meanwhile
        arr = L.moe_hier_profile_begin([e.cuda_event for e in pev[i]])
        layer.forward(out=out, routing_out=False)
        L.moe_hier_profile_end()
    torch.cuda.synchronize(dev)
    kern_ms = {}
    for i in range(n_prof):
        for j, nm in enumerate(names):
            kern_ms.setdefault(nm, []).append(pev[i][j].elapsed_time(pev[i][j + 1]))

    # ---- the timed steps: replays of a CUDA graph of one forward call
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        layer.forward(out=out, routing_out=False)          # outside capture: attributes, maps
        torch.cuda.synchronize(dev)
        with torch.cuda.graph(graph, stream=cap):
            layer.forward(out=out, routing_out=False)
    stream.wait_stream(cap)
    for _ in range(max(args.warmup, 3)):
        graph.replay()
    torch.cuda.synchronize(dev)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    clocks = Clocks(dev) if rank == 0 else None
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    if clocks:
        clocks.start()
    wall0 = time.perf_counter()
    for i in range(K):
        flush.fill_(i & 0xFF)                      # evict the weights from L2 between steps
        ev[i][0].record(stream)
        graph.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    if layer.status() != 0:
        raise RuntimeError("device status after timed steps: %d" % layer.status())

    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    value = job_tokens_per_s(world, cfg.T, K, total_ms)

    # ---- end to end through the C ABI with host buffers (copies inside the timed region).  Every
    # step copies its x from pinned host memory, runs moe_hier_forward and copies its y back; the
    # copies run on two copy streams (host->device, device->host) so that step i+1's input and
    # step i-1's output move while step i computes (two device buffers of each), as a serving
    # loop would run it.  The L2 is flushed before every forward, inside the timed region.
    x_h = inp["x"].pin_memory()
    y_h = [torch.empty(cfg.T, cfg.d, dtype=layer.act_dtype).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(layer.x) for _ in range(2)]
    outs = [layer.new_outputs() for _ in range(2)]
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    fwd_done = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]

    def e2e_steps(n):
        for i in range(n):
            b = i & 1
            h2d_s.wait_event(fwd_done[b])            # forward i-2 has read x_d[b]
            with torch.cuda.stream(h2d_s):
                x_d[b].copy_(x_h, non_blocking=True)
            h2d_done[b].record(h2d_s)
            stream.wait_event(h2d_done[b])
            stream.wait_event(d2h_done[b])           # step i-2's y has left outs[b]
            flush.fill_(i & 0xFF)
            layer.forward(x=x_d[b], out=outs[b], routing_out=False)
            fwd_done[b].record(stream)
            d2h_s.wait_event(fwd_done[b])
            with torch.cuda.stream(d2h_s):
                y_h[b].copy_(outs[b]["y"], non_blocking=True)
            d2h_done[b].record(d2h_s)

    for b in range(2):
        for e in (h2d_done[b], fwd_done[b], d2h_done[b]):
            e.record(stream)
    e2e_steps(4)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    h2d_s.wait_stream(stream)
    d2h_s.wait_stream(stream)
    e2e_steps(K)
    stream.wait_stream(h2d_s)
    stream.wait_stream(d2h_s)
    e_end.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e_start.elapsed_time(e_end)
    if not torch.equal(y_h[(K - 1) & 1], outs[(K - 1) & 1]["y"].cpu()):
        raise RuntimeError("end-to-end output differs from the device result")
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    e2e_value = job_tokens_per_s(world, cfg.T, K, e2e_ms)
    act_b = 2 if cfg.dtype == "bf16" else 4

    # ---- roofline of the dominant kernel (its own algorithmic work / its mean event time)
    peaks, peak_src = load_peaks()
    dom = max(kern_ms, key=lambda n: sum(kern_ms[n]))
    dom_ms = statistics.mean(kern_ms[dom])
    dom_flops, dom_bytes = workload.kernel_work(cfg, dom, groups_hit, experts_hit)
    traffic = recorded_traffic(args.config, dom)
    if cfg.T >= 512:       # prefill-sized batches: the contraction bounds the time
        achieved = dom_flops / (dom_ms / 1e3) / 1e12
        peak = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 2),
                "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "peak_source": f"{peak_src} bf16_tflops (burst: kernel timed within one step)",
                "algorithmic_flops_per_launch": dom_flops, "algorithmic_bytes_per_launch": dom_bytes,
                "traffic": traffic}
    else:                  # decode-sized batches: streaming the weights bounds the time
        achieved = dom_bytes / (dom_ms / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_source": f"{peak_src} hbm_gbs",
                "algorithmic_bytes_per_launch": dom_bytes, "traffic": traffic}
    step_mean = statistics.mean(step_ms)

    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(step_mean, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if cfg.dtype == "bf16" else "f32",
        "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": {"workload": workload_name(cfg), "T": cfg.T, "d_model": cfg.d, "d_ff": cfg.f,
                   "E": cfg.E, "G": cfg.G, "top_k_group": cfg.kg, "top_k_expert": cfg.ke,
                   "rank": cfg.r, "parallelism": "replicas" if world > 1 else "single",
                   "l2": "flushed between timed steps (256 MiB write)",
                   "groups_hit": groups_hit, "experts_hit": experts_hit,
                   "load_max_over_mean": {"group": round(load["group"]["max_over_mean"], 3),
                                          "expert": round(load["expert"]["max_over_mean"], 3)}},
        "roofline": roof,
        "achieved_tflops_step": round(workload.flops(cfg) / (step_mean / 1e3) / 1e12, 2),
        "kernels_ms": {n: round(statistics.mean(v), 5) for n, v in kern_ms.items()},
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s",
                "h2d_bytes_per_step": cfg.T * cfg.d * act_b, "d2h_bytes_per_step": cfg.T * cfg.d * act_b,
                "schedule": "per step: pinned x -> device, moe_hier_forward (direct call), y -> pinned host; "
                            "copies on their own streams overlap the neighbouring steps' forwards; L2 "
                            "flushed before every forward"},
        "gpu_launches": n_k * K,
        "timing": ("graph replay of one moe_hier_forward_prepared per step (residual stacks built once "
                   "before the timed region)" if args.prepared else "graph replay of one moe_hier_forward per step")
                  + " (kernels_ms: per-kernel device time, launches queued behind a sleep kernel)",
        "clocks": clk,
        "wall_s_timed": round(wall, 3),
    }
    return res, inp


# ------------------------------------------------------------------ the compression step (--config compress_*)
def run_compress(args):
    """Times moe_hier_compress on every matrix kind of the dense experts (gate, up, down), inputs
    resident; reports matrices compressed per second and the FP32 rate of the tall-skinny
    products (the bulk of the work) against the CUDA cores' FP32 peak (148 SMs x 128 FMA lanes x 2
    FLOP x the maximum SM clock)."""
    import torch

    from compressed_expert_two_b300 import _lib as L
    from synth import COMPRESS_CONFIGS, make_dense_experts
    cfg = COMPRESS_CONFIGS[args.config]
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = load_peaks()
    sm_mhz = peaks.get("sm_max_mhz", 2032.0)
    fp32_peak = 148 * 128 * 2 * sm_mhz * 1e6 / 1e12
    inp = make_dense_experts(cfg)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    per_kind, kern_ms, tot_ms, tsmm_flops, errs = {}, {}, 0.0, 0.0, []
    for kind in ("gate", "up", "down"):
        d_in, d_out = (cfg.d, cfg.f) if kind != "down" else (cfg.f, cfg.d)
        E, G, r = cfg.E, cfg.G, cfg.r
        desc = L.MoeHierCompressDesc(E=E, G=G, d_out=d_out, d_in=d_in, rank=r, sketch=cfg.l,
                                     power_iters=cfg.power_iters)
        W = inp[kind]["W"].to(dev)
        om = inp[kind]["omega"].to(dev)
        gm = inp["group_map"].to(torch.int32)
        o = [torch.empty(G, d_out, d_in, dtype=torch.bfloat16, device=dev),
             torch.empty(E, r, d_in // 2, dtype=torch.uint8, device=dev),
             torch.empty(E, r, d_in // 64, dtype=torch.float16, device=dev),
             torch.empty(E, r, d_out // 2, dtype=torch.uint8, device=dev),
             torch.empty(E, r, d_out // 64, dtype=torch.float16, device=dev),
             torch.empty(E, r, dtype=torch.float32, device=dev), torch.empty(E, dtype=torch.float64, device=dev)]
        nws = L.moe_hier_compress_workspace_size(desc)
        ws = torch.empty(nws, dtype=torch.uint8, device=dev)

        def call():
            L.moe_hier_compress(desc, W, gm, om, *o, None, None, ws, nws, stream.cuda_stream)

        for _ in range(max(args.warmup, 3)):
            call()
        torch.cuda.synchronize(dev)
        probe = [torch.cuda.Event(enable_timing=True) for _ in range(64)]
        for e in probe:
            e.record(stream)
        arr = L.moe_hier_profile_begin([e.cuda_event for e in probe])
        call()
        names = L.moe_hier_profile_end()
        del arr
        torch.cuda.synchronize(dev)
        for j, nm in enumerate(names[:63]):
            kern_ms[nm] = kern_ms.get(nm, 0.0) + probe[j].elapsed_time(probe[j + 1])
        K = max(1, min(args.steps, 20))
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for i in range(K):
            flush.fill_(i & 0xFF)
            ev[i][0].record(stream)
            call()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        tot_ms += ms
        passes = 2 * cfg.power_iters + 2
        tsmm_flops += passes * 2.0 * 64 * d_out * d_in * E
        errs += o[6].cpu().tolist()
        per_kind[kind] = {"ms": round(ms, 3), "d_out": d_out, "d_in": d_in}
    tsmm_ms = sum(v for k, v in kern_ms.items() if k.startswith("cmp_tsmm"))
    achieved = tsmm_flops / (tsmm_ms / 1e3) / 1e12 if tsmm_ms > 0 else 0.0
    n_mat = 3 * cfg.E
    res = {"metric": "compression: dense expert matrices compressed per second (group-mean base, rank-r TSVD, "
                     "INT4 g64 factors)",
           "value": round(n_mat / (tot_ms / 1e3), 2), "unit": "matrices/s", "n_gpus": 1,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_ms, 3), "higher_is_better": True,
           "dtype": "f32", "data": "synthetic dense experts (shared group part + rank-r deviation + 1% noise)",
           "config": {"workload": f"{cfg.name}: E={cfg.E} G={cfg.G} d_model={cfg.d} d_ff={cfg.f} r={cfg.r} "
                                  f"sketch={cfg.l} power_iters={cfg.power_iters}", "per_kind": per_kind,
                      "l2": "flushed between timed calls (256 MiB write)"},
           "roofline": {"bound": "alu", "kernel": "cmp_tsmm (tall-skinny products, FP32 CUDA cores)",
                        "achieved": round(achieved, 2), "peak": round(fp32_peak, 1), "unit": "TFLOP/s",
                        "frac": round(achieved / fp32_peak, 4),
                        "peak_source": "148 SMs x 128 FP32 lanes x 2 FLOP x sm_max_mhz (derived, not measured)"},
           "kernels_ms": {k: round(v, 4) for k, v in kern_ms.items()},
           "reconstruction_error": {"mean": round(statistics.mean(errs), 5), "max": round(max(errs), 5)},
           "gpu_launches": len(names)}
    if not args.no_cpu_baseline:
        import numpy as np

        from oracle import compress as C
        W0 = inp["gate"]["W"][:cfg.K].float().numpy()
        t0 = time.perf_counter()
        C.compress_matrix(W0, np.zeros(cfg.K, dtype=np.int64), 1, cfg.r)
        el = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": round(cfg.K / el, 3), "unit": "matrices/s", "cores": cpu_cores(),
                               "kind": "oracle", "sample": f"the gate matrices of one group ({cfg.K} experts, "
                                                           f"FP64 SVD each) in {el:.1f} s"}
    return res


# ------------------------------------------------------------------ idle-group offload (--config decode_offload)
def run_offload(args, slots: int = 4):
    """Steps of a few tokens each over distinct inputs, the group bases in pinned host memory and
    `slots` of the G groups cached on the device; batch i+1 is routed and its missing groups
    copied while batch i's FFN runs.  Reports tokens/s (wall clock over the steps, the host's
    per-step synchronisation included), the resident-weight rate on the same inputs, the cache hit
    rate, bytes copied per step and the host-to-device rate against a pinned 1 GiB copy."""
    import torch

    from compressed_expert_two_b300 import _lib as L
    from compressed_expert_two_b300.layer import DeviceLayer
    from synth import CONFIGS, make_inputs
    cfg = CONFIGS[args.config]
    dev = torch.device("cuda", 0)
    inp = make_inputs(cfg)
    layer = DeviceLayer(inp, device=dev)
    host = {m: inp["w_" + m].contiguous().pin_memory() for m in ("gate", "up", "down")}
    cache = {m: torch.empty((slots,) + tuple(inp["w_" + m].shape[1:]), dtype=torch.bfloat16, device=dev)
             for m in ("gate", "up", "down")}
    off = L.Offload(layer.desc, host["gate"], host["up"], host["down"], cache["gate"], cache["up"],
                    cache["down"], slots)
    gen = torch.Generator().manual_seed(99)
    n = max(args.steps, 8)
    xs = [torch.randn(cfg.T, cfg.d, generator=gen).to(torch.bfloat16).to(dev) for _ in range(n + args.warmup)]
    copy = torch.cuda.Stream(dev)
    streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    wss = [layer.ws, torch.zeros_like(layer.ws)]
    keep = []

    def step(i, x):
        s = streams[i & 1]
        ws = wss[i & 1]
        o = layer.new_outputs()
        pr = {"row_asg": torch.empty(cfg.T * cfg.kg, dtype=torch.int32, device=dev),
              "row_begin": torch.empty(cfg.G + 1, dtype=torch.int32, device=dev)}
        y = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16, device=dev)
        L.moe_hier_route(layer.desc, x, layer.w_group, layer.b_group, layer.w_expert, layer.group_map, o["gidx"],
                         o["eidx"], o["gate"], ws, layer.ws_bytes, s.cuda_stream)
        L.moe_hier_permute(layer.desc, layer.group_map, o["eidx"], None, None, None, None, None, pr["row_asg"],
                           None, pr["row_begin"], ws, layer.ws_bytes, s.cuda_stream)
        hit = off.groups_hit(pr["row_begin"], s.cuda_stream)
        off.require(hit, copy.cuda_stream)
        off.ffn(layer.desc, x, layer.group_map, layer.resid, o["eidx"], o["gate"], pr["row_asg"], pr["row_begin"],
                y, ws, layer.ws_bytes, s.cuda_stream)
        keep.append((o, pr, y))
        return int(hit.sum())

    for i in range(args.warmup):
        step(i, xs[n + i])
    torch.cuda.synchronize(dev)
    st0 = off.stats()
    t0 = time.perf_counter()
    hits_per_step = [step(i, xs[i]) for i in range(n)]
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t0
    st1 = off.stats()
    keep.clear()
    # the same inputs with every base resident (the layer's own forward, graph-free, same host loop)
    for i in range(3):
        layer.forward(x=xs[i])
    torch.cuda.synchronize(dev)
    t1 = time.perf_counter()
    for i in range(n):
        layer.forward(x=xs[i], routing_out=False)
    torch.cuda.synchronize(dev)
    wall_res = time.perf_counter() - t1
    # pinned host -> device copy rate (1 GiB, best of 3)
    hbuf = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    best = 0.0
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dbuf.copy_(hbuf, non_blocking=True)
        b.record()
        torch.cuda.synchronize(dev)
        best = max(best, (1 << 30) / (a.elapsed_time(b) / 1e3) / 1e9)
    off.close()
    cpu = None
    if not args.no_cpu_baseline:
        tps, n_tok, el = oracle_tokens_per_s(inp, args.cpu_seconds, cfg.T)
        cpu = {"value": round(tps, 3), "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{n_tok} tokens of the same layer ({cfg.T} per step; route + FP64 FFN with every W~ "
                         f"materialised) in {el:.1f} s"}
    copied = st1["bytes_copied"] - st0["bytes_copied"]
    misses, hits = st1["misses"] - st0["misses"], st1["hits"] - st0["hits"]
    group_bytes = 3 * cfg.d * cfg.f * 2
    return {"metric": "idle-group offload: MoE-layer fwd tokens/s with the group bases in pinned host memory",
            "value": round(cfg.T * n / wall, 1), "unit": "tokens/s", "n_gpus": 1, "steps": n, "warmup": args.warmup,
            "ms_per_step": round(wall / n * 1e3, 3), "higher_is_better": True, "dtype": "bf16",
            "data": "synthetic (seeded; distinct inputs per step)",
            "config": {"workload": workload_name(cfg) + f", {slots} of {cfg.G} group bases cached on the device",
                       "T": cfg.T, "slots": slots, "G": cfg.G,
                       "device_bytes_bases": slots * group_bytes, "resident_bytes_bases": cfg.G * group_bytes},
            "resident": {"value": round(cfg.T * n / wall_res, 1), "unit": "tokens/s",
                         "ms_per_step": round(wall_res / n * 1e3, 3)},
            "cache": {"groups_hit_per_step": round(statistics.mean(hits_per_step), 2),
                      "hit_rate": round(hits / max(hits + misses, 1), 4),
                      "bytes_copied_per_step": round(copied / n), "h2d_gbs": round(copied / wall / 1e9, 2),
                      "pinned_h2d_peak_gbs": round(best, 2), "h2d_frac": round(copied / wall / 1e9 / best, 4)},
            "timing": "wall clock over the steps (host synchronisation per step for the hit groups included)",
            "cpu_baseline": cpu}


def main():
    args = parse()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))

    if args.impl == "reference":
        if rank != 0:
            return 0
        return run_reference(args)

    if args.config.startswith("compress_") or args.config == "decode_offload":
        if world > 1 and rank != 0:
            return 0
        res = run_compress(args) if args.config.startswith("compress_") else run_offload(args)
        print(json.dumps(res), flush=True)
        return 0

    import torch
    import torch.distributed as dist
    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    res, inp = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            tps, n, el = oracle_tokens_per_s(inp, args.cpu_seconds, CPU_CHUNK.get(args.config, 256))
            res["cpu_baseline"] = {"value": round(tps, 2), "unit": "tokens/s", "cores": cpu_cores(),
                                   "kind": "oracle",
                                   "sample": f"{n} tokens of the same workload (chunks of "
                                             f"{CPU_CHUNK.get(args.config, 256)}; route + FP64 FFN with "
                                             f"every W~ materialised) in {el:.1f} s"}
        print(json.dumps(res), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_reference(args):
    """The oracle as the reference arm, on the host cores, each step a bounded token sample."""
    from synth import make_inputs
    cfg = workload_config(args)
    inp = make_inputs(cfg)
    chunk = CPU_CHUNK.get(args.config, 256)
    per_step = []
    for i in range(args.warmup + args.steps):
        tps, n, el = oracle_tokens_per_s(inp, 0.0, chunk)
        if i >= args.warmup:
            per_step.append((n, el))
    tok = sum(n for n, _ in per_step)
    sec = sum(e for _, e in per_step)
    value = tok / sec
    res = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(1e3 * sec / max(len(per_step), 1), 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded; shapes and distributions of the workload)",
           "config": {"workload": workload_name(cfg), "T": cfg.T, "sample_tokens_per_step": chunk},
           "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": cpu_cores(),
                            "kind": "oracle",
                            "sample": f"{chunk} tokens per step (route + FP64 FFN, every W~ materialised)"},
           "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
