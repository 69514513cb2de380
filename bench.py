#!/usr/bin/env python3
"""Benchmark of the NVFP4 W4A16 linear layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-extras]

Prints ONE JSON line.  A step is one pass of the layer over one batch of the
headline workload (decode GEMV over the fused MLP gate+up projection:
M=1, K=5120, N=34816); ``value`` is algorithmic bytes per step / time per
step (GB/s), inputs resident in HBM, K steps replayed from CUDA graphs and
timed with CUDA events on the launching stream, between barriers + device
synchronisations (--eager: eager launches instead).  Weights are rotated over enough copies
that the rotated set exceeds twice the L2 cache, so every step streams its
weights from HBM.

The other workloads (verify, M=32 layer, prefill with and without SwiGLU)
are timed the same way and reported under "workloads".

--impl reference times the CPU oracle (the reference arm) on
the host cores, on a bounded sample of the same workload per step.

Multi-GPU (torchrun): every rank runs an independent replica on its own GPU
(the layer has no exchange step); value = all ranks' bytes / max rank time.
"""
import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NVFP4 W4A16 linear: GB/s (M≤32) & TFLOPS (M=8192), % of GB300 roofline"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
HEADLINE = "decode_gate_up"


# ----------------------------------------------------------------- helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(
            p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "nvfp4_block_scaled_linear_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        e = t[kernel][workload]
        if e.get("source_hash") == kernel_source_hash():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks/throttle sampler over the benchmark's lifetime."""
    FIELDS = ("clocks.sm,clocks.max.sm,utilization.gpu,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, period_ms=50):
        self.index = index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []
        self.windows = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=timestamp," + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._reader, daemon=True).start()
        except Exception:
            self.proc = None

    def _reader(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), float(parts[3]), parts[5:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        inwin = [r for r in rows if any(a - 0.05 <= r[0] <= b + 0.05 for a, b in self.windows)]
        loaded = [r for r in inwin if r[3] > 0] or inwin or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in loaded:
            for n, v in zip(names, r[4][1:5]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median([r[1] for r in loaded])),
                "sm_max_mhz": float(max(r[2] for r in loaded)),
                "reasons": sorted(reasons), "samples": len(loaded)}


# ----------------------------------------------------------------- distributed
def dist_setup(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate_max(value, world):
    """Max of a float over ranks (the slowest rank's time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) \
        if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(units_per_rank, max_seconds, world):
    return units_per_rank * world / max_seconds


def workload_config(name, linears, swiglu):
    """The `config` of the JSON line: the workload alone (its name, shapes and
    epilogue), identical in both arms; measurement notes go elsewhere."""
    return {"workload": name, "shapes": [[int(t.M), int(t.N), int(t.K)] for t in linears],
            "swiglu": bool(swiglu)}


def compute_dtype(kernel, M):
    """The arithmetic the launched kernel multiplies in (fp32 accumulation in
    every kernel): the warp-MMA kernel at M <= 8 multiplies f16 operands (exact
    code * scale, activations scaled by a power of two; bf16 for a row's stage
    beyond the f16 window), every other path bf16."""
    return "f16" if kernel == "smallm" and M <= 8 else "bf16"


# ----------------------------------------------------------------- GPU arm
class Case:
    """Device-resident inputs of one workload, with rotated weight copies."""

    def __init__(self, name, lib, dev, min_rotated_bytes=2 * L2_BYTES, max_rows=None):
        import torch
        from nvfp4_block_scaled_linear_gb300.inputs import WORKLOADS, algorithmic_bytes, flops
        self.w = WORKLOADS[name]
        self.name = name
        self.lib = lib
        self.flags = lib.FLAG_SWIGLU if self.w.swiglu else 0
        self.linears = self.w.draw(max_rows)
        self.bytes = sum(algorithmic_bytes(t.M, t.N, t.K, self.w.swiglu) for t in self.linears)
        self.flops = sum(flops(t.M, t.N, t.K) for t in self.linears)
        per_copy = sum(t.w_packed.nbytes + t.w_scale.nbytes for t in self.linears)
        act = sum(t.x_bits.nbytes for t in self.linears)
        total = per_copy + act
        self.copies = 1 if total >= min_rotated_bytes else int(np.ceil(min_rotated_bytes / total))
        self.x = [torch.from_numpy(t.x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
                  for t in self.linears]
        self.wp = [[torch.from_numpy(t.w_packed).to(dev) for t in self.linears]
                   for _ in range(self.copies)]
        self.ws = [[torch.from_numpy(t.w_scale).to(dev) for t in self.linears]
                   for _ in range(self.copies)]
        n_out = [t.N // 2 if self.w.swiglu else t.N for t in self.linears]
        self.y = [torch.empty((t.M, n), dtype=torch.bfloat16, device=dev)
                  for t, n in zip(self.linears, n_out)]
        self.rotated_bytes = self.copies * per_copy + act
        self.launches_per_step = len(self.linears)
        self.only = None          # restrict a step to one linear (per-linear timing)
        self.kernel = lib.choose_plan(self.linears[0].M, self.linears[0].N, self.linears[0].K,
                                      self.flags)

    def indices(self):
        return range(len(self.linears)) if self.only is None else (self.only,)

    def step(self, i, stream):
        c = i % self.copies
        for j in self.indices():
            t = self.linears[j]
            self.lib.linear_ex(self.x[j], self.wp[c][j], self.ws[c][j], float(t.global_scale),
                               self.flags, out=self.y[j], stream=stream)

    def l2_note(self):
        if self.copies > 1:
            return "rotating %d weight copies (%d MB > 2x L2)" % (self.copies,
                                                                  self.rotated_bytes >> 20)
        return "inputs larger than L2 (%d MB)" % (self.rotated_bytes >> 20)


def _capture(case, n_steps, stream):
    """A CUDA graph of n_steps consecutive steps (weight copies rotating from
    copy 0), captured on `stream`."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for i in range(n_steps):
                case.step(i, stream)
    return g


# Device-side delay enqueued ahead of a timed region's start event: while it
# runs, the host enqueues the start event and the work, so the timed region
# starts with the work already queued and holds no host launch latency (a
# 20-step region otherwise counts ~20 us of it).  ~60 us at 2 GHz.
GATE_CYCLES = 120_000


def _gate(stream):
    import torch
    with torch.cuda.stream(stream):
        torch.cuda._sleep(GATE_CYCLES)


def _replay_steps(stream, steps, chunk_graph, chunk, tail_graph):
    import torch
    with torch.cuda.stream(stream):
        for _ in range(steps // chunk):
            chunk_graph.replay()
        if tail_graph is not None:
            tail_graph.replay()


def _timed_graph(case, steps, warmup, stream, world, sampler):
    """Time exactly `steps` steps, replayed from CUDA graphs of `chunk`
    steps (a multiple of the weight-copy count, so the rotation runs on
    across replays) plus one graph for the remainder."""
    import torch
    for i in range(max(warmup, 1)):          # eager warm-up: descriptors, attributes
        case.step(i, stream)
    torch.cuda.synchronize()
    chunk = case.copies * max(1, 32 // case.copies)
    chunk = min(chunk, max(case.copies, steps))
    g = _capture(case, chunk, stream)
    tail = _capture(case, steps % chunk, stream) if steps % chunk else None
    _replay_steps(stream, max(warmup, chunk), g, chunk, None)   # graph warm-up
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.time()
    _gate(stream)
    t0.record(stream)
    _replay_steps(stream, steps, g, chunk, tail)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall1 = time.time()
    if sampler:
        sampler.mark(wall0, wall1)
    return t0.elapsed_time(t1)


def time_case(case, steps, warmup, stream, world, sampler=None, graph=True):
    """(total ms of `steps` steps, [mean ms per launch of each linear]).

    graph=True: steps are replayed from CUDA graphs (the way a decode loop
    runs); the per-linear launch time comes from timing, the same way, a
    step restricted to that linear (for one-linear workloads it is the step
    time).  graph=False: eager launches with CUDA events around each."""
    import torch
    n_l = case.launches_per_step
    if graph:
        total_ms = _timed_graph(case, steps, warmup, stream, world, sampler)
        if n_l == 1:
            return total_ms, [total_ms / steps]
        launch_ms = []
        for j in range(n_l):
            case.only = j
            try:
                launch_ms.append(_timed_graph(case, steps, warmup, stream, world, None) / steps)
            finally:
                case.only = None
        return total_ms, launch_ms
    for i in range(warmup):
        case.step(i, stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps * n_l)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.time()
    _gate(stream)
    t_start.record(stream)
    for i in range(steps):
        c = i % case.copies
        for j, t in enumerate(case.linears):
            a, b = ev[i * n_l + j]
            a.record(stream)
            case.lib.linear_ex(case.x[j], case.wp[c][j], case.ws[c][j], float(t.global_scale),
                               case.flags, out=case.y[j], stream=stream)
            b.record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall1 = time.time()
    if sampler:
        sampler.mark(wall0, wall1)
    launch_ms = [float(np.mean([ev[i * n_l + j][0].elapsed_time(ev[i * n_l + j][1])
                                for i in range(steps)])) for j in range(n_l)]
    return t_start.elapsed_time(t_end), launch_ms


def e2e_case(case, steps, stream, dev):
    """Same workload through the public API with the step's data in host
    memory: every step calls nvfp4_linear_host (through its Python binding),
    which moves the activations in from pinned host memory, runs the layer
    and moves the result out to pinned host memory, all inside the timed
    region (for these page-locked, aligned buffers the transfers are the
    library's zero-copy staging kernels).  The packed weights and scales are the model's resident
    parameters (rotated over the same copies as the device-timed loop, so
    they stream from HBM), not step inputs."""
    import torch
    hx = [x.cpu().pin_memory() for x in case.x]
    hy = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for y in case.y]
    dx = [torch.empty_like(x) for x in case.x]
    h2d = sum(t.nbytes for t in hx)
    d2h = sum(t.nbytes for t in hy)

    def one(i):
        c = i % case.copies
        for j, t in enumerate(case.linears):
            case.lib.linear_host(hx[j], dx[j], case.wp[c][j], case.ws[c][j],
                                 float(t.global_scale), case.y[j], hy[j], case.flags,
                                 stream=stream)

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    _gate(stream)
    a.record(stream)
    for i in range(steps):
        one(i)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    return ms, h2d, d2h


def quantize_case(lib, dev, stream, hbm_peak, N=34816, K=5120, steps=20):
    """The load-time quantiser (bf16 -> NVFP4) on the decode projection's
    weight shape: bytes = bf16 in + codes + scales out (HBM-bound)."""
    import torch
    from nvfp4_block_scaled_linear_gb300.inputs import quantizer_weight
    w = quantizer_weight(N, K).to(dev)
    with torch.cuda.stream(stream):
        for _ in range(3):
            lib.quantize(w, stream=stream)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(steps):
            lib.quantize(w, stream=stream)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    nbytes = N * K * 2 + N * K // 2 + N * K // 16 + 4
    gbs = nbytes / (ms / 1e3) / 1e9
    del w
    return {"ms_per_step": round(ms, 5), "kernel": "quantize", "shape": [N, K],
            "GB/s": round(gbs, 1), "frac_hbm_peak": round(gbs / hbm_peak, 4)}


def quantize_fp8_case(lib, dev, stream, hbm_peak, N=34816, K=5120, block=128, steps=20):
    """The load-time FP8 -> NVFP4 conversion on the same weight shape:
    bytes = e4m3 codes and block scales in + codes + scales out."""
    import torch
    from nvfp4_block_scaled_linear_gb300.inputs import fp8_checkpoint_tensor
    w8, sinv = fp8_checkpoint_tensor(N, K, block)
    w8, sinv = w8.to(dev), sinv.to(dev)
    with torch.cuda.stream(stream):
        for _ in range(3):
            lib.quantize_fp8(w8, sinv, block, stream=stream)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(steps):
            lib.quantize_fp8(w8, sinv, block, stream=stream)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    nbytes = N * K + sinv.numel() * 4 + N * K // 2 + N * K // 16 + 4
    gbs = nbytes / (ms / 1e3) / 1e9
    del w8, sinv
    return {"ms_per_step": round(ms, 5), "kernel": "quantize_fp8", "shape": [N, K],
            "block": block, "GB/s": round(gbs, 1), "frac_hbm_peak": round(gbs / hbm_peak, 4)}


def run_ours(args):
    import torch
    from nvfp4_block_scaled_linear_gb300 import build as cuda_build

    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    cuda_build.build()
    from nvfp4_block_scaled_linear_gb300 import _lib as lib
    lib.load_library()
    hbm_peak, tc_peak, tc_sustained, peak_src = measured_peaks()
    sampler = ClockSampler(dev.index if world == 1 else local)
    sampler.start()
    stream = torch.cuda.Stream(dev)

    head = Case(args.workload, lib, dev, max_rows=args.max_rows)
    total_ms, launch_ms = time_case(head, args.steps, args.warmup, stream, world, sampler,
                                    graph=not args.eager)
    step_s = total_ms / 1e3 / args.steps
    max_step_s = aggregate_max(step_s, world)
    tensor_bound = head.linears[0].M > 32
    if tensor_bound:
        value = whole_job_value(head.flops / 1e12, max_step_s, world)
        unit = "TFLOP/s"
    else:
        value = whole_job_value(head.bytes / 1e9, max_step_s, world)
        unit = "GB/s"

    # dominant kernel = the longest launch of the step
    j_dom = int(np.argmax(launch_ms))
    t_dom = head.linears[j_dom]
    from nvfp4_block_scaled_linear_gb300.inputs import algorithmic_bytes, flops
    if tensor_bound:
        achieved = flops(t_dom.M, t_dom.N, t_dom.K) / (launch_ms[j_dom] / 1e3) / 1e12
        peak, runit, bound = tc_peak, "TFLOP/s", "tensor"
    else:
        achieved = algorithmic_bytes(t_dom.M, t_dom.N, t_dom.K, head.w.swiglu) / (
            launch_ms[j_dom] / 1e3) / 1e9
        peak, runit, bound = hbm_peak, "GB/s", "hbm"
    roofline = {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": runit,
                "frac": round(achieved / peak, 4), "peak_source": peak_src,
                "kernel": head.kernel, "launch_us": round(launch_ms[j_dom] * 1e3, 3),
                "traffic": profiled_traffic(head.kernel, head.name)}

    line = {"metric": METRIC, "value": round(value, 2), "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(max_step_s * 1e3, 6), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": compute_dtype(head.kernel, head.linears[0].M),
            "data": "synthetic (seeded; checkpoint-schema layouts, random codes/scales/"
                    "activations)",
            "config": workload_config(head.name, head.linears, head.w.swiglu),
            "l2": head.l2_note(),
            "parallelism": "replicas" if world > 1 else "single GPU",
            "roofline": roofline, "gpu_launches": args.steps * head.launches_per_step,
            "timing": ("CUDA graphs of consecutive steps, CUDA events on the launching "
                       "stream around the replays" if not args.eager else
                       "eager launches, CUDA events around each launch") +
                      "; after the barrier and synchronisation a short device-side delay "
                      "precedes the start event, so that the timed work is already queued "
                      "(no host launch latency inside the region)"}
    if args.max_rows is not None:
        line["max_rows"] = args.max_rows

    if not args.no_extras:
        e2e_ms, h2d, d2h = e2e_case(head, max(3, min(500, args.steps)), stream, dev)
        e2e_val = (head.flops / 1e12 if tensor_bound else head.bytes / 1e9) / (e2e_ms / 1e3)
        line["e2e"] = {"value": round(e2e_val * world, 2), "unit": unit,
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": round(e2e_ms, 4)}
        extras = {}
        for name, steps in (("verify_down", 2000), ("layer_m32", 500), ("prefill", 10),
                            ("prefill_swiglu", 10)):
            if name == head.name:
                continue
            c = Case(name, lib, dev)
            tot, lms = time_case(c, steps, 5, stream, world, sampler, graph=not args.eager)
            ms = tot / steps
            ent = {"ms_per_step": round(ms, 5), "kernel": c.kernel,
                   "dtype": compute_dtype(c.kernel, c.linears[0].M),
                   "launch_us": [round(v * 1e3, 2) for v in lms]}
            if c.linears[0].M > 32:
                tf = c.flops / (ms / 1e3) / 1e12
                ent.update({"TFLOP/s": round(tf, 1), "frac_bf16_peak": round(tf / tc_peak, 4)})
            else:
                gb = c.bytes / (ms / 1e3) / 1e9
                ent.update({"GB/s": round(gb, 1), "frac_hbm_peak": round(gb / hbm_peak, 4)})
            extras[name] = ent
            del c
            torch.cuda.empty_cache()
        if not args.eager:
            # the same headline steps launched eagerly, for comparison (host
            # launch overhead included)
            e_tot, _ = time_case(head, min(args.steps, 500), 5, stream, world, None,
                                 graph=False)
            line["eager_ms_per_step"] = round(e_tot / min(args.steps, 500), 6)
        extras["quantize"] = quantize_case(lib, dev, stream, hbm_peak)
        extras["quantize_fp8"] = quantize_fp8_case(lib, dev, stream, hbm_peak)
        line["workloads"] = extras
        line["gpu_launches_extras"] = "not in the headline timed region"
    sampler.stop()
    line["clocks"] = sampler.summary()
    if rank == 0 and not args.no_extras:
        line["cpu_baseline"] = cpu_baseline(head, budget_s=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ----------------------------------------------------------------- CPU (oracle)
def _oracle_step(t, rows, threads):
    import oracle
    return oracle.linear_f64(t.x_bits, t.w_packed[rows], t.w_scale[rows], t.global_scale,
                             threads=threads)


def _oracle_rate(t, threads, budget_s):
    """(GB/s, passes, rows, seconds) of the oracle on `threads` threads:
    repeated passes over a row sample sized at ~1 s per pass."""
    rows = slice(0, min(t.N, 2048))
    t0 = time.time()
    _oracle_step(t, rows, threads)
    one = time.time() - t0
    n_rows = int(min(t.N, max(128, (rows.stop - rows.start) * 1.0 / max(one, 1e-3))))
    rows = slice(0, n_rows)
    done, t0 = 0, time.time()
    while time.time() - t0 < budget_s:
        _oracle_step(t, rows, threads)
        done += 1
    el = time.time() - t0
    frac = n_rows / t.N
    byts = (t.N * t.K // 2 + t.N * t.K // 16) * frac + 2 * t.M * t.K + 2 * t.M * n_rows
    return byts * done / el / 1e9, done, n_rows, el


def _cpu_model():
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


# Oracle timing per configuration: every output on all cores; on one core,
# every output for the small configurations and a labelled prefix of the
# activation rows (time scaled by M / rows) for the M = 32 layer and prefill,
# whose full oracle takes minutes there.
ORACLE_TIMING_ROWS = {"layer_m32": (32, 4), "prefill": (16, 2)}   # (all cores, one core)


def oracle_timings(threads):
    import oracle
    from nvfp4_block_scaled_linear_gb300.inputs import WORKLOADS
    out = {}
    for name in ("tiny", "decode_gate_up", "verify_down", "layer_m32", "prefill"):
        linears = WORKLOADS[name].draw()
        ent = {}
        for label, thr, pick in (("all_cores", threads, 0), ("one_core", 1, 1)):
            total, notes = 0.0, []
            for t in linears:
                rows = min(t.M, ORACLE_TIMING_ROWS.get(name, (t.M, t.M))[pick])
                t0 = time.perf_counter()
                oracle.linear_f64(t.x_bits[:rows], t.w_packed, t.w_scale, t.global_scale,
                                  threads=thr)
                el = time.perf_counter() - t0
                total += el * t.M / rows
                if rows < t.M:
                    notes.append("%s: rows [0,%d) of %d, time x %g" % (t.name, rows, t.M,
                                                                        t.M / rows))
            ent[label] = {"ms": round(total * 1e3, 2), "threads": thr,
                          "sample": "; ".join(notes) if notes else "every output"}
        out[name] = ent
        del linears
    return out


def cpu_baseline(case, budget_s=10.0):
    """The oracle, as it stands, on the host cores (all of them, and one):
    repeated passes over a row sample of the headline workload for about
    budget_s (and budget_s / 3) seconds."""
    import oracle
    threads = oracle.default_threads()
    t = case.linears[0]
    value, done, n_rows, el = _oracle_rate(t, threads, budget_s)
    value1, done1, n_rows1, el1 = _oracle_rate(t, 1, budget_s / 3.0)
    return {"value": round(value, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": "%d passes over rows [0,%d) of %s (M=%d K=%d), %.1f s" % (
                done, n_rows, case.name, t.M, t.K, el),
            "one_core": {"value": round(value1, 4), "sample": "%d passes over rows [0,%d), %.1f s"
                         % (done1, n_rows1, el1)},
            "cpu": _cpu_model(),
            "oracle_ms_per_workload": oracle_timings(threads)}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from nvfp4_block_scaled_linear_gb300.inputs import WORKLOADS, algorithmic_bytes, flops
    w = WORKLOADS[args.workload]
    linears = w.draw()
    t = linears[0]
    threads = oracle.default_threads()
    # Size one step so that warmup + steps end within ~2 minutes.
    probe_rows = min(t.N, 512)
    t0 = time.time()
    _oracle_step(t, slice(0, probe_rows), threads)
    per_row = (time.time() - t0) / probe_rows
    budget = 120.0 / max(1, args.steps + args.warmup)
    n_rows = int(max(1, min(t.N, budget / max(per_row, 1e-9))))
    if t.M > 32:
        # large-M: sample activation rows too
        pass
    rows = slice(0, n_rows)
    for _ in range(args.warmup):
        _oracle_step(t, rows, threads)
    t0 = time.time()
    for _ in range(args.steps):
        _oracle_step(t, rows, threads)
    el = time.time() - t0
    frac = n_rows / t.N
    tensor_bound = t.M > 32
    if tensor_bound:
        units = flops(t.M, n_rows, t.K) / 1e12
        unit = "TFLOP/s"
    else:
        units = ((t.N * t.K // 2 + t.N * t.K // 16) * frac + 2 * t.M * t.K
                 + 2 * t.M * n_rows) / 1e9
        unit = "GB/s"
    value = units * args.steps / el
    sample = "rows [0,%d) of %d per step (M=%d K=%d)" % (n_rows, t.N, t.M, t.K)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": unit,
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)",
            "config": workload_config(w.name, linears, w.swiglu),
            "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--no-extras", action="store_true",
                    help="headline only: no e2e, other workloads or CPU baseline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--eager", action="store_true",
                    help="time eager launches instead of CUDA-graph replays")
    ap.add_argument("--max-rows", type=int, default=None,
                    help="cap the activation rows of each linear (small profiling cases)")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
