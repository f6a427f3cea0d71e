#!/usr/bin/env python3
"""Benchmark of the fused tensor-parallel matmul + collective operators.

One step = one pass over every fused operator on its TP8 layer shape (8
emulated ranks), i.e. every step of the hot path:

  bloom7b_ar          MATMUL_ALL_REDUCE   m 2048, K 16384 (8 x 2048), n 4096, bf16, chunks 4
  llama70b_ag_v2      ALL_GATHER_MATMUL_V2  8 x (512 x 8192) gathered, W 8192 x (8 x 7168), bf16
  llama70b_rs         MATMUL_REDUCE_SCATTER  m 4096, K 28672 (8 x 3584), n 8192, bf16
  w8a16_ar_{tensor,channel,group}  w8A16 MATMUL_ALL_REDUCE  m 4096, K 8192 (8 x 1024), n 8192, fp16 x int8
                      (dequantisation pre-pass + AllReduce kernel at this m)
  bloom176b_det_ar    deterministic MATMUL_ALL_REDUCE  m 2048, K 57344 (8 x 7168), n 14336, bf16
  bloom176b_det_rs    deterministic MATMUL_REDUCE_SCATTER, same shapes

value = algorithmic FLOPs (2 m n K per operator) of all steps on all ranks /
wall time of the timed steps (CUDA events, max over ranks), in TFLOP/s.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --case ar|rs|ag|ag_v2|w8a16|plain|moe --m M --n N --k K [...]   (one operator)

Under torchrun (N > 1) every rank runs the whole suite on its own GPU
(replicas; the path has no cross-GPU exchange), rank 0 prints the line.
--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused matmul+AR/RS/AG TFLOP/s and % of GB300 dense bf16 peak, 8 emulated TP shards"
UNIT = "TFLOP/s"
WORKLOAD = ("tp8_suite: bloom7b_ar + llama70b_ag_v2 + llama70b_rs + w8a16_ar x {tensor,channel,group} "
            "+ bloom176b_det_ar + bloom176b_det_rs (8 emulated TP ranks each)")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    # the end-to-end leg runs as many steps as the timed region (30 at least),
    # so that both legs see a power-capped GPU settle the same way
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-context", action="store_true")
    # --case: one operator on seeded synthetic data of a chosen size, timed
    # over --iters calls (the command the profiles/ captures run)
    ap.add_argument("--case", choices=["ar", "rs", "ag", "ag_v2", "w8a16", "plain", "moe"], default=None)
    ap.add_argument("--R", type=int, default=8)
    ap.add_argument("--m", type=int, help="rows (ar/rs/w8a16/plain: m; ag/ag_v2: m_shard; moe: tokens per rank)")
    ap.add_argument("--n", type=int, help="columns (ag/ag_v2: n_shard; moe: f)")
    ap.add_argument("--k", type=int, help="contraction per shard (ag/ag_v2: full k; moe: h)")
    ap.add_argument("--dtype", choices=["bf16", "fp16"], default="bf16")
    ap.add_argument("--chunks", type=int, default=1)
    ap.add_argument("--gran", choices=["tensor", "channel", "group"], default="group")
    ap.add_argument("--group", type=int, default=128)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--zero", action="store_true", help="w8a16: int8 zero points")
    ap.add_argument("--eloc", type=int, default=1, help="moe: experts per rank")
    ap.add_argument("--topk", type=int, default=1, help="moe: routing slots (gated combine if > 1)")
    ap.add_argument("--deterministic", action="store_true")
    a = ap.parse_args()
    if a.e2e_steps is None:
        a.e2e_steps = max(30, a.steps)
    return a


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, dist, device) -> float:
    """The largest value of x over all ranks (x itself without a process group)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(step_flops: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job TFLOP/s: every rank ran `steps` steps of `step_flops`; the job
    took as long as its slowest rank."""
    return world * step_flops * steps / (max_ms / 1e3) / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "sustained_sm_mhz": (d.get("clocks_under_load") or {}).get("sm_mhz_median"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sustained_sm_mhz": None,
            "source": "fallback"}


def kernel_source_hash() -> str:
    """Hash of the kernel and of the host code that sets its launch (tile
    order, L2 grouping): DRAM traffic taken on other sources is stale."""
    h = hashlib.sha256()
    for f in ("coc_kernel.cu", "coc_internal.h", "coc_api.cu", "coc_dequant.cuh", "coc_w8_prepass.cu", "coc_moe.cu"):
        h.update(open(os.path.join(ROOT, "tensor_matmul_collective_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:12]


def load_traffic(op: str, chunks: int):
    """DRAM bytes per launch of `op` at `chunks` from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want, key = kernel_source_hash(), f"{op}@c{chunks}"
    for line in open(path):
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == key and parts[2] == want:
            return float(parts[1])
    return None


# ------------------------------------------------------------------ clocks ---

class NvmlSampler:
    """SM clock, power draw and clock-event reasons of one GPU, sampled
    through NVML (libnvidia-ml, reached with ctypes; read-only queries)
    every `period_s` seconds by a background thread while the timed region
    runs.  Falls back to `nvidia-smi -lms 100` where NVML cannot be loaded."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, bus_id: str | None, index: int = 0, period_s: float = 0.005):
        self.bus, self.index, self.period = bus_id, index, period_s
        self.samples, self.thread, self.stop_evt, self.lib, self.handle = [], None, None, None, None
        self.fallback = None
        self.max_mhz = None

    def _open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        h = ctypes.c_void_p()
        ok = False
        if self.bus:
            for fmt in (self.bus, "0000" + self.bus):
                if lib.nvmlDeviceGetHandleByPciBusId_v2(fmt.encode(), ctypes.byref(h)) == 0:
                    ok = True
                    break
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        self.lib, self.handle = lib, h
        self.reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")

    def _loop(self):
        import ctypes
        mhz, mw, mask = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        i = 0
        while not self.stop_evt.is_set():
            t = time.perf_counter()
            a = self.lib.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(mhz))
            b = self.reason_fn(self.handle, ctypes.byref(mask))
            p = self.lib.nvmlDeviceGetPowerUsage(self.handle, ctypes.byref(mw)) if i % 10 == 0 else 1
            self.samples.append((t, mhz.value if a == 0 else None, mask.value if b == 0 else None,
                                 mw.value / 1000.0 if p == 0 else None))
            i += 1
            self.stop_evt.wait(self.period)

    def start(self):
        import threading
        try:
            self._open()
        except (OSError, AttributeError):
            self.fallback = SmiSampler(self.bus)
            self.fallback.start()
            return
        self.samples, self.stop_evt = [], threading.Event()
        self.thread = threading.Thread(target=self._loop, daemon=True)
        self.thread.start()

    def stop(self):
        if self.fallback is not None:
            return self.fallback.stop()
        if self.thread is None:
            return None
        self.stop_evt.set()
        self.thread.join()
        try:
            self.lib.nvmlShutdown()
        except Exception:
            pass
        sm = [x[1] for x in self.samples if x[1] is not None]
        reasons = sorted({name for x in self.samples if x[2] is not None
                          for bit, name in self.REASONS.items() if x[2] & bit})
        power = [x[3] for x in self.samples if x[3] is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(sm), "sm_mhz_min": min(sm) if sm else None, "sm_mhz_max": max(sm) if sm else None,
                "power_w_max": max(power) if power else None,
                "sampler": f"NVML in-process, every {self.period * 1e3:.0f} ms"}


class SmiSampler:
    FIELDS = ("pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.bus = (bus_id or "").lower()
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [[c.strip() for c in ln.split(",")] for ln in out.splitlines() if ln.count(",") >= 8]
        if self.bus:
            mine = [r for r in rows if self.bus in r[0].lower()]
            rows = mine or rows
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None,
                "sampler": "nvidia-smi -lms 100"}


# ------------------------------------------------------------------- suite ---

class Op:
    def __init__(self, name, kind, flops, run, inputs, outputs, shape, gran=None):
        self.name, self.kind, self.flops, self.run = name, kind, flops, run
        self.inputs, self.outputs, self.shape, self.gran = inputs, outputs, shape, gran
        self.shares_prev_inputs = False   # reads the inputs uploaded for the operator before it
        self.launches = 1                 # kernels one call launches

    def step_inputs(self):
        """The operator's per-step input as a user feeds it: the activation
        shards X_r (the first R input tensors).  Weights, scales and zero
        points are model state, uploaded once and resident, as a training
        step's parameters are; an operator that reads the previous one's
        inputs has none of its own."""
        return [] if self.shares_prev_inputs else self.inputs[:self.shape.R]

    def readback(self):
        """The operator's result as the host reads it: every distinct output
        tensor.  AllReduce (and w8A16) write the same tile to all R rank
        outputs and V2 the same gathered X to all R gather buffers (bitwise
        equal, which the tests check), so one copy of each is the whole
        result; per-rank results (ReduceScatter blocks, AllGather products)
        are all read."""
        R = self.shape.R
        if self.kind in ("ar", "w8a16_ar"):
            return self.outputs[:1]
        if self.kind == "ag_v2":
            return self.outputs[:R] + self.outputs[R:R + 1]
        return self.outputs


def algorithmic_bytes(op) -> int:
    """Inputs read once plus outputs written once (every rank copy), bytes."""
    s = op.shape
    if op.kind in ("ar", "rs"):
        out = s.R * s.m * s.n if op.kind == "ar" else s.m * s.n
        return 2 * (s.m * s.K + s.K * s.n + out)
    if op.kind == "ag_v2":
        return 2 * (s.m * s.k + s.R * s.k * s.n_shard + s.R * s.m * s.n_shard + s.R * s.m * s.k)
    if op.kind == "w8a16_ar":
        scales = {"tensor": s.R, "channel": s.n, "group": (s.K // s.group) * s.n}[op.gran]
        return 2 * s.m * s.K + s.K * s.n + 2 * scales + 2 * s.R * s.m * s.n
    raise ValueError(op.kind)


def build_suite(dev):
    """Device inputs/outputs for every operator of one step (inputs drawn on
    the host from the seeded generators, uploaded once)."""
    import torch

    from tensor_matmul_collective_gb300 import coc
    from tensor_matmul_collective_gb300 import workloads as wl

    ops, host = [], {}
    C = {w.name: w.chunks for w in wl.TP8_SUITE}

    def up(ts):
        return [t.to(dev) for t in ts]

    s = wl.BLOOM7B_AR
    xs, ws = s.make()
    host["bloom7b"] = (xs, ws)
    dx, dw = up(xs), up(ws)
    out7 = [torch.empty(s.m, s.n, dtype=s.dtype, device=dev) for _ in range(s.R)]
    ops.append(Op("bloom7b_ar", "ar", s.flops(), lambda dx=dx, dw=dw, o=out7: coc.matmul_all_reduce(dx, dw, o, chunks=C["bloom7b_ar"]),
                  dx + dw, out7, s))

    s = wl.LLAMA70B_AG
    xs, ws = s.make()
    host["llama_ag"] = (xs, ws)
    dx, dw = up(xs), up(ws)
    outg = [torch.empty(s.m, s.n_shard, dtype=s.dtype, device=dev) for _ in range(s.R)]
    gat = [torch.empty(s.m, s.k, dtype=s.dtype, device=dev) for _ in range(s.R)]
    ops.append(Op("llama70b_ag_v2", "ag_v2", s.flops(),
                  lambda dx=dx, dw=dw, o=outg, g=gat: coc.all_gather_matmul_v2(dx, dw, o, g, chunks=C["llama70b_ag_v2"]),
                  dx + dw, outg + gat, s))

    s = wl.LLAMA70B_RS
    xs, ws = s.make()
    host["llama_rs"] = (xs, ws)
    dx, dw = up(xs), up(ws)
    outr = [torch.empty(s.m // s.R, s.n, dtype=s.dtype, device=dev) for _ in range(s.R)]
    ops.append(Op("llama70b_rs", "rs", s.flops(),
                  lambda dx=dx, dw=dw, o=outr: coc.matmul_reduce_scatter(dx, dw, o, chunks=C["llama70b_rs"]),
                  dx + dw, outr, s))

    s = wl.W8A16_AR
    xs8 = wqs = None
    for gran in wl.SCALE_GRANS:
        x_, w_, scales = s.make(gran)
        if xs8 is None:
            xs8, wqs = x_, w_
            dx8, dwq = up(xs8), up(wqs)
        host[f"w8_{gran}"] = (xs8, wqs, scales)
        if gran == "group":
            dsc = up(scales)
            uniq = dsc
        else:                       # one scale tensor shared by every rank
            d0 = scales[0].to(dev)
            dsc, uniq = [d0] * s.R, [d0]
        out8 = [torch.empty(s.m, s.n, dtype=torch.float16, device=dev) for _ in range(s.R)]
        op = Op(f"w8a16_ar_{gran}", "w8a16_ar", s.flops(),
                lambda dx=dx8, dw=dwq, sc=dsc, o=out8, g=gran, grp=s.group: coc.matmul_all_reduce_w8a16(
                    dx, dw, sc, g, grp, o, chunks=C["w8a16_ar"]),
                (dx8 + dwq if gran == "tensor" else []) + uniq, out8, s, gran)
        op.shares_prev_inputs = gran != "tensor"
        # from 2048 rows the library dequantises the weight in a pre-pass kernel
        # and then runs the AllReduce kernel (COC_W8_PATH forces a path)
        path = os.environ.get("COC_W8_PATH", "")
        op.launches = 2 if path == "prepass" or (path != "fused" and s.m >= 2048) else 1
        ops.append(op)

    s = wl.BLOOM176B
    xs, ws = s.make()
    host["bloom176b"] = (xs, ws)
    dx, dw = up(xs), up(ws)
    outa = [torch.empty(s.m, s.n, dtype=s.dtype, device=dev) for _ in range(s.R)]
    outs = [torch.empty(s.m // s.R, s.n, dtype=s.dtype, device=dev) for _ in range(s.R)]
    ops.append(Op("bloom176b_det_ar", "ar", s.flops(),
                  lambda dx=dx, dw=dw, o=outa: coc.matmul_all_reduce(dx, dw, o, chunks=C["bloom176b_det_ar"],
                                                                    deterministic=True),
                  dx + dw, outa, s))
    op = Op("bloom176b_det_rs", "rs", s.flops(),
            lambda dx=dx, dw=dw, o=outs: coc.matmul_reduce_scatter(dx, dw, o, chunks=C["bloom176b_det_rs"],
                                                                deterministic=True),
            [], outs, s)
    op.shares_prev_inputs = True
    ops.append(op)
    return ops, host


def time_device(ops, steps, warmup, dist, sampler):
    import torch
    from tensor_matmul_collective_gb300 import coc

    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        for op in ops:
            op.run()
    torch.cuda.synchronize()
    coc.sync_status()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(ops) + 1)] for _ in range(steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    for i in range(len(ops)):
        coc.clock_read(i)            # clear the in-kernel clock slots
    t_start.record(stream)
    for s in range(steps):
        ev[s][0].record(stream)
        for i, op in enumerate(ops):
            coc.clock_probe(i)       # host-side flag: this operator's kernels record into slot i
            op.run()
            ev[s][i + 1].record(stream)
    t_end.record(stream)
    coc.clock_probe(-1)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    mhz = [coc.clock_mhz(i) for i in range(len(ops))]
    if clocks is not None:
        clocks["sm_mhz_in_kernel"] = {op.name: m for op, m in zip(ops, mhz)}
    if dist is not None:
        dist.barrier()
    coc.sync_status()
    total_ms = t_start.elapsed_time(t_end)
    # every operator's time in every timed step (events recorded between launches)
    per_op = [[ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(steps)] for i in range(len(ops))]
    return total_ms, per_op, clocks


def time_e2e(ops, steps, dev):
    """Same suite through the public API from pinned host buffers: each step
    copies every operator's activations host->device (Op.step_inputs; the
    weights are resident model state), runs it and copies its result
    device->host (Op.readback: every distinct output tensor).  Copies run on
    their own streams so one operator's transfers overlap another's
    compute."""
    import torch

    from tensor_matmul_collective_gb300 import coc

    h_in = [[t.to("cpu").pin_memory() for t in op.step_inputs()] for op in ops]
    h_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in op.readback()] for op in ops]
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    n = len(ops)
    in_ready = [torch.cuda.Event() for _ in range(n)]
    done = [torch.cuda.Event() for _ in range(n)]
    out_done = [torch.cuda.Event() for _ in range(n)]
    h2d = sum(t.numel() * t.element_size() for hs in h_in for t in hs)
    d2h = sum(t.numel() * t.element_size() for hs in h_out for t in hs)

    # the last operator of each run of operators that read the same inputs
    last_reader = list(range(n))
    for i in range(n - 1, 0, -1):
        if ops[i].shares_prev_inputs:
            last_reader[i - 1] = last_reader[i]

    def step(first):
        for i, op in enumerate(ops):
            with torch.cuda.stream(s_in):
                if not first and op.step_inputs():
                    s_in.wait_event(done[last_reader[i]])   # previous step finished reading these inputs
                for d, h in zip(op.step_inputs(), h_in[i]):
                    d.copy_(h, non_blocking=True)
                in_ready[i].record(s_in)
            comp.wait_event(in_ready[i])
            if i > 0:
                comp.wait_event(in_ready[i - 1])
            if not first:
                comp.wait_event(out_done[i])          # previous step's outputs are back on the host
            op.run()
            done[i].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done[i])
                for h, d in zip(h_out[i], op.readback()):
                    h.copy_(d, non_blocking=True)
                out_done[i].record(s_out)

    step(True)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        step(False)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    coc.sync_status()
    del h_in, h_out
    return wall, h2d, d2h


def interleaved(fns: dict, it: int = 20, warm: int = 3) -> dict:
    """The one timing protocol of every context figure: each call of `fns`
    (name -> callable) is bracketed by its own CUDA events on the current
    stream, and the calls are taken round-robin (a, b, c, a, b, c, ...) so
    that clock and power drift under the power cap hit every variant alike.
    Returns {name: {"median_ms", "min_ms", "max_ms"}} over `it` calls each,
    after `warm` untimed rounds."""
    import torch

    from tensor_matmul_collective_gb300 import coc

    names = list(fns)
    for _ in range(warm):
        for n in names:
            fns[n]()
    torch.cuda.synchronize()
    probe = len(names) <= 8          # one in-kernel clock slot per variant
    if probe:
        for j in range(len(names)):
            coc.clock_read(j)
    ev = {n: [] for n in names}
    for i in range(it):
        order = names if i % 2 == 0 else names[::-1]
        for n in order:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            if probe:
                coc.clock_probe(names.index(n))
            a.record()
            fns[n]()
            b.record()
            ev[n].append((a, b))
    coc.clock_probe(-1)
    torch.cuda.synchronize()
    out = {}
    for j, n in enumerate(names):
        ts = [a.elapsed_time(b) for a, b in ev[n]]
        out[n] = {"median_ms": round(statistics.median(ts), 4), "min_ms": round(min(ts), 4),
                  "max_ms": round(max(ts), 4)}
        if probe:
            out[n]["sm_mhz_in_kernel"] = coc.clock_mhz(j)
    return out


def time_context(ops, dev, bus=None, index=0):
    """Context numbers measured outside the timed region, all with the same
    protocol (interleaved, per-call CUDA events, median and min): each
    operator against the same kernel with a plain one-buffer epilogue (fused
    overhead) and against the unfused torch sequence (per-shard torch.matmul,
    then a separate reduction / copy); the Python-script chunking against the
    fused kernel at C = 1/2/4/8; a decode-sized AllReduce; the suite as one
    CUDA graph; and the rows built beyond the suite."""
    import torch

    from tensor_matmul_collective_gb300 import coc

    sampler = NvmlSampler(bus, index)
    sampler.start()
    out = {"protocol": "interleaved round-robin calls, each between its own CUDA events; median / min of 20 "
                       "calls per variant after 3 untimed rounds (torch and Python-chunked sequences: 6 calls)"}
    for op in ops:
        if op.kind not in ("ar", "rs"):
            continue
        s = op.shape
        dx, dw = op.inputs[:s.R], op.inputs[s.R:2 * s.R]
        if not dx:   # bloom176b_det_rs shares the AR inputs
            prev = [o for o in ops if o.name == "bloom176b_det_ar"][0]
            dx, dw = prev.inputs[:s.R], prev.inputs[s.R:2 * s.R]
        plain = torch.empty(s.m, s.n, dtype=s.dtype, device=dev)

        def unfused(dx=dx, dw=dw, R=s.R, kind=op.kind, m=s.m):
            acc = torch.stack([torch.matmul(a, b) for a, b in zip(dx, dw)]).sum(0, dtype=torch.float32).to(dx[0].dtype)
            if kind == "ar":
                return [acc.clone() for _ in range(R)]
            return [acc[r * (m // R):(r + 1) * (m // R)].clone() for r in range(R)]
        r = interleaved({"fused": op.run, "plain": lambda dx=dx, dw=dw, o=plain: coc.matmul(dx, dw, o)})
        u = interleaved({"torch": unfused}, it=6)
        out[op.name] = {"fused_ms": r["fused"], "plain_epilogue_ms": r["plain"],
                        "fused_overhead": round(r["fused"]["median_ms"] / r["plain"]["median_ms"] - 1.0, 4),
                        "torch_unfused_ms": u["torch"]}
    ag = [o for o in ops if o.kind == "ag_v2"]
    if ag:
        op = ag[0]
        s = op.shape
        dx, dw = op.inputs[:s.R], op.inputs[s.R:]
        outs = op.outputs[:s.R]
        xg = op.outputs[s.R]
        r = interleaved({"fused_v2": op.run,
                         "plain": lambda: [coc.matmul([xg], [dw[q]], outs[q]) for q in range(s.R)],
                         "all_gather_matmul": lambda: coc.all_gather_matmul(dx, dw, outs, chunks=1)})
        u = interleaved({"torch": lambda: [torch.matmul(torch.cat(dx, 0), dw[q]) for q in range(s.R)]}, it=6)
        out[op.name] = {"fused_ms": r["fused_v2"], "all_gather_matmul_ms": r["all_gather_matmul"],
                        "plain_epilogue_ms": r["plain"],
                        "fused_overhead": round(r["fused_v2"]["median_ms"] / r["plain"]["median_ms"] - 1.0, 4),
                        "torch_unfused_ms": u["torch"]}
    # the unfused torch sequence for w8A16 (explicit dequantisation, then the
    # AllReduce sequence), on the per-channel layer
    w8c = [o for o in ops if o.name == "w8a16_ar_channel"]
    w8t = [o for o in ops if o.name == "w8a16_ar_tensor"]
    if w8c and w8t:
        s = w8c[0].shape
        dx, dq = w8t[0].inputs[:s.R], w8t[0].inputs[s.R:2 * s.R]
        sc = w8c[0].inputs[0]

        def w8_unfused(dx=dx, dq=dq, sc=sc, R=s.R):
            wd = [(q.float() * sc.float()).half() for q in dq]
            acc = torch.stack([torch.matmul(a, b) for a, b in zip(dx, wd)]).sum(0, dtype=torch.float32).half()
            return [acc.clone() for _ in range(R)]
        r = interleaved({"fused": w8c[0].run})
        u = interleaved({"torch": w8_unfused}, it=6)
        out["w8a16_ar_channel"] = {"fused_ms": r["fused"], "torch_unfused_ms": u["torch"]}
    # the tiny AllReduce configuration (R = 2, 64 x 128 x 256 fp16, chunks 2):
    # latency-bound, reported in microseconds per call
    from tensor_matmul_collective_gb300 import workloads as wl
    ts = wl.TINY_AR
    txs, tws = ts.make()
    tx, tw = [x.to(dev) for x in txs], [w.to(dev) for w in tws]
    to = [torch.empty(ts.m, ts.n, dtype=ts.dtype, device=dev) for _ in range(ts.R)]
    r = interleaved({"det0": lambda: coc.matmul_all_reduce(tx, tw, to, chunks=2),
                     "det1": lambda: coc.matmul_all_reduce(tx, tw, to, chunks=2, deterministic=True)}, it=200)
    # per call between events, an eager call is bound by the host's launch;
    # the GPU time is taken from 100 calls replayed from a CUDA graph
    tg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(tg):
        for _ in range(100):
            coc.matmul_all_reduce(tx, tw, to, chunks=2)
    rg = interleaved({"graph": tg.replay}, it=10)
    out["tiny_ar_r2_64x128_k256"] = {"eager_us_per_call_median": round(1e3 * r["det0"]["median_ms"], 2),
                                     "eager_deterministic_us_per_call_median": round(1e3 * r["det1"]["median_ms"], 2),
                                     "graph_us_per_call_median": round(1e3 * rg["graph"]["median_ms"] / 100, 2)}
    del tg
    # The pages' Python-script CoC (CoC page, Python脚本层面实现), module
    # python_coc: each chunk's per-rank matmuls and reduction on a compute
    # stream, its collective (copies into the rank buffers) on a second
    # stream, 1 + 2R (AR/RS) or 2R + 1 (AG) host launches per chunk; against
    # the fused kernel at the same chunk count.
    from tensor_matmul_collective_gb300 import python_coc
    streams = (torch.cuda.Stream(), torch.cuda.Stream())

    def chunk_sweep(name, py, fused_call):
        r = interleaved({f"py{C}": (lambda C=C: py(C)) for C in (1, 2, 4, 8)}, it=6)
        f = interleaved({f"fused{C}": (lambda C=C: fused_call(C)) for C in (1, 2, 4, 8)})
        out[name] = {"python_chunked_ms": {str(C): r[f"py{C}"]["median_ms"] for C in (1, 2, 4, 8)},
                     "fused_ms": {str(C): f[f"fused{C}"]["median_ms"] for C in (1, 2, 4, 8)}}

    ar7 = [o for o in ops if o.name == "bloom7b_ar"]
    if ar7:
        op = ar7[0]
        s = op.shape
        dx, dw = op.inputs[:s.R], op.inputs[s.R:2 * s.R]
        outs = op.outputs
        chunk_sweep("bloom7b_ar_python_chunking",
                    lambda C: python_coc.all_reduce(dx, dw, outs, C, *streams),
                    lambda C: coc.matmul_all_reduce(dx, dw, outs, chunks=C))
    rs = [o for o in ops if o.name == "llama70b_rs"]
    if rs:
        op = rs[0]
        s = op.shape
        dx, dw = op.inputs[:s.R], op.inputs[s.R:2 * s.R]
        outs = op.outputs
        chunk_sweep("llama70b_rs_python_chunking",
                    lambda C: python_coc.reduce_scatter(dx, dw, outs, C, *streams),
                    lambda C: coc.matmul_reduce_scatter(dx, dw, outs, chunks=C))
    ag = [o for o in ops if o.kind == "ag_v2"]
    if ag:
        op = ag[0]
        s = op.shape
        dx, dw = op.inputs[:s.R], op.inputs[s.R:]
        outs, gath = op.outputs[:s.R], op.outputs[s.R:2 * s.R]
        chunk_sweep("llama70b_ag_v2_python_chunking",
                    lambda C: python_coc.all_gather(dx, dw, outs, C, gath, *streams),
                    lambda C: coc.all_gather_matmul_v2(dx, dw, outs, gath, chunks=C))
    # decode-sized AllReduce (8 ranks, n 8192, K 8 x 1024, bf16): weight-stream
    # bound, so reported as us per call (20 calls replayed from a CUDA graph)
    # and algorithmic HBM GB/s (W read once, X read, R output copies)
    graphs, keep, byts = {}, [], {}
    for m in (1, 16, 64, 128):
        ds_ = wl.RowParallel(R=8, m=m, n=8192, k_shard=1024, dtype=torch.bfloat16, x_dist="normal(0,1)",
                             w_dist="normal(0,0.02)", seed=1)
        dxs, dws = ds_.make()
        ddx, ddw = [x.to(dev) for x in dxs], [w.to(dev) for w in dws]
        dout = [torch.empty(m, ds_.n, dtype=ds_.dtype, device=dev) for _ in range(ds_.R)]
        coc.matmul_all_reduce(ddx, ddw, dout)
        torch.cuda.synchronize()
        gd = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gd):
            for _ in range(20):
                coc.matmul_all_reduce(ddx, ddw, dout)
        graphs[str(m)] = gd.replay
        keep.append((gd, ddx, ddw, dout))
        byts[str(m)] = 2 * (ds_.K * ds_.n + m * ds_.K + ds_.R * m * ds_.n)
    # the suite's other decode layers at m 16: BLOOM-7B (n 4096, K 8 x 2048) and
    # BLOOM-176B (n 14336, K 8 x 7168)
    for name, n_, ks_ in (("bloom7b_m16", 4096, 2048), ("bloom176b_m16", 14336, 7168)):
        ds_ = wl.RowParallel(R=8, m=16, n=n_, k_shard=ks_, dtype=torch.bfloat16, x_dist="normal(0,1)",
                             w_dist="normal(0,0.02)", seed=1)
        dxs, dws = ds_.make()
        ddx, ddw = [x.to(dev) for x in dxs], [w.to(dev) for w in dws]
        dout = [torch.empty(16, ds_.n, dtype=ds_.dtype, device=dev) for _ in range(ds_.R)]
        coc.matmul_all_reduce(ddx, ddw, dout)
        torch.cuda.synchronize()
        gd = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gd):
            for _ in range(20):
                coc.matmul_all_reduce(ddx, ddw, dout)
        graphs[name] = gd.replay
        keep.append((gd, ddx, ddw, dout))
        byts[name] = 2 * (ds_.K * ds_.n + 16 * ds_.K + ds_.R * 16 * ds_.n)
    r = interleaved(graphs, it=10)
    per_call = {m: {"us_per_call": round(1e3 * r[m]["median_ms"] / 20, 1),
                    "hbm_gbs": round(byts[m] / (1e3 * r[m]["median_ms"] / 20) / 1e3, 0)} for m in graphs}
    out["decode_ar_r8_n8192_k8192_cuda_graph"] = {m: v for m, v in per_call.items() if not m.startswith("bloom")}
    out["decode_ar_layers_cuda_graph"] = {m: v for m, v in per_call.items() if m.startswith("bloom")}
    del keep, graphs
    # w8A16 at the same decode shape (m 16, fp16, int8 weights: 64 MiB read)
    graphs, keep, byts = {}, [], {}
    for gran in ("channel", "group"):
        ws_ = wl.W8A16(R=8, m=16, n=8192, k_shard=1024, group=128, seed=3, dtype=torch.float16)
        wxs, wqs, wsc = ws_.make(gran)
        dxs, dqs, dsc = [x.to(dev) for x in wxs], [q.to(dev) for q in wqs], [t.to(dev) for t in wsc]
        dout = [torch.empty(16, 8192, dtype=torch.float16, device=dev) for _ in range(8)]
        call = (lambda dxs=dxs, dqs=dqs, dsc=dsc, dout=dout, gran=gran:
                coc.matmul_all_reduce_w8a16(dxs, dqs, dsc, gran, 128, dout))
        call()
        torch.cuda.synchronize()
        gd = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gd):
            for _ in range(20):
                call()
        graphs[gran] = gd.replay
        keep.append((gd, dxs, dqs, dsc, dout))
        byts[gran] = 8 * 1024 * 8192 + 2 * (16 * 8192 + 8 * 16 * 8192)
    r = interleaved(graphs, it=10)
    out["decode_w8a16_r8_m16_n8192_k8192_cuda_graph"] = {
        g: {"us_per_call": round(1e3 * r[g]["median_ms"] / 20, 1),
            "hbm_gbs": round(byts[g] / (1e3 * r[g]["median_ms"] / 20) / 1e3, 0)} for g in graphs}
    del keep, graphs
    # AllGather-V2 on the LLaMA2-70B layer (n_shard 7168, k 8192: 940 MB of
    # weights) at decode-sized m_shard 8 and 16 (column-slab kernel); bytes:
    # W, X, the R products and the R gathered copies
    graphs, keep, byts = {}, [], {}
    for ms in (8, 16):
        ag_ = wl.ColumnParallelSP(R=8, m_shard=ms, n_shard=7168, k=8192, dtype=torch.bfloat16, x_dist="normal(0,1)",
                                  w_dist="normal(0,0.02)", seed=2)
        axs, aws = ag_.make()
        dax, daw = [x.to(dev) for x in axs], [w.to(dev) for w in aws]
        m_ = 8 * ms
        dout = [torch.empty(m_, 7168, dtype=torch.bfloat16, device=dev) for _ in range(8)]
        dg = [torch.empty(m_, 8192, dtype=torch.bfloat16, device=dev) for _ in range(8)]
        call = lambda dax=dax, daw=daw, dout=dout, dg=dg: coc.all_gather_matmul_v2(dax, daw, dout, dg)  # noqa: E731
        call()
        torch.cuda.synchronize()
        gd = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gd):
            for _ in range(20):
                call()
        graphs[str(ms)] = gd.replay
        keep.append((gd, dax, daw, dout, dg))
        byts[str(ms)] = 2 * (8 * 8192 * 7168 + m_ * 8192 + 8 * m_ * 7168 + 8 * m_ * 8192)
    r = interleaved(graphs, it=10)
    out["decode_ag_v2_r8_ns7168_k8192_cuda_graph"] = {
        ms: {"us_per_call": round(1e3 * r[ms]["median_ms"] / 20, 1),
             "hbm_gbs": round(byts[ms] / (1e3 * r[ms]["median_ms"] / 20) / 1e3, 0)} for ms in graphs}
    del keep, graphs
    # the whole suite step captured once into a CUDA graph and replayed,
    # against the same step launched eagerly (the host's launch cost)
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for op in ops:
                op.run()
        r = interleaved({"graph": g.replay, "eager": lambda: [op.run() for op in ops]}, it=10)
        step_flops = sum(op.flops for op in ops)
        out["suite_cuda_graph"] = {"graph_ms_per_step": r["graph"]["median_ms"],
                                   "eager_ms_per_step": r["eager"]["median_ms"],
                                   "graph_tflops": round(step_flops / r["graph"]["median_ms"] / 1e9, 1)}
        del g
    except RuntimeError as e:   # reported, not hidden: the operators are meant to be capturable
        out["suite_cuda_graph"] = {"error": str(e)[:200]}
    out["next_rows"] = time_next_rows(ops, dev)
    out["clocks"] = sampler.stop()
    return out


def time_next_rows(ops, dev):
    """The rows built beyond the headline suite, on the suite's layer shapes:
    Megatron's n x k weight and the weight-gradient pass (LLaMA2-70B layers),
    the w8A16 extensions (bf16 activations, int8 zero points) and the MoE
    expert-parallel layer, each with the interleaved protocol."""
    import torch

    from tensor_matmul_collective_gb300 import coc
    from tensor_matmul_collective_gb300 import workloads as wl

    res = {}
    rs = [o for o in ops if o.name == "llama70b_rs"]
    if rs:
        op = rs[0]
        s = op.shape
        dx, dw = op.inputs[:s.R], op.inputs[s.R:2 * s.R]
        wnk = [w.t().contiguous() for w in dw]
        outs = [torch.empty(s.m // s.R, s.n, dtype=s.dtype, device=dev) for _ in range(s.R)]
        r = interleaved({"kn": op.run, "nk": lambda: coc.fused_matmul("reduce_scatter", dx, wnk, w_layout="nk",
                                                                      outs=outs)})
        res["llama70b_rs_weight_nk"] = {"kn_ms": r["kn"]["median_ms"], "nk_ms": r["nk"]["median_ms"],
                                        "nk_tflops": round(s.flops() / r["nk"]["median_ms"] / 1e9, 1)}
        del wnk, outs
    ag = [o for o in ops if o.kind == "ag_v2"]
    if ag:
        op = ag[0]
        s = op.shape
        dys = op.outputs[:s.R]                 # tokens x n_shard per rank (stands in for dY)
        xgs = op.outputs[s.R:2 * s.R]          # the gathered X V2 returned, per rank (tokens x k)
        dws = [torch.empty(s.n_shard, s.k, dtype=s.dtype, device=dev) for _ in range(s.R)]
        r = interleaved({"wgrad": lambda: coc.weight_grad(dys, xgs, dws)}, it=10)
        flops = 2.0 * s.m * s.n_shard * s.k * s.R
        res["llama70b_weight_grad"] = {"ms": r["wgrad"]["median_ms"],
                                       "tflops": round(flops / r["wgrad"]["median_ms"] / 1e9, 1)}
        del dws
    w8 = [o for o in ops if o.kind == "w8a16_ar"]
    if w8:
        base = w8[0].shape
        fns, flops, keep = {}, {}, []
        for dt, zero in ((torch.float16, False), (torch.float16, True), (torch.bfloat16, False), (torch.bfloat16, True)):
            s = wl.W8A16(R=base.R, m=base.m, n=base.n, k_shard=base.k_shard, group=base.group, seed=base.seed,
                         dtype=dt)
            xs, wqs, scales = s.make("channel")
            dx, dq, ds = [x.to(dev) for x in xs], [w.to(dev) for w in wqs], [c.to(dev) for c in scales]
            dz = [z.to(dev) for z in s.zeros("channel")] if zero else None
            outs = [torch.empty(s.m, s.n, dtype=dt, device=dev) for _ in range(s.R)]
            name = f"w8a16_ar_channel_{'bf16' if dt == torch.bfloat16 else 'fp16'}_{'zp' if zero else 'sym'}"
            fns[name] = lambda dx=dx, dq=dq, ds=ds, dz=dz, outs=outs, g=s.group: coc.matmul_all_reduce_w8a16(
                dx, dq, ds, "channel", g, outs, zeros=dz)
            flops[name] = s.flops()
            keep.append((dx, dq, ds, dz, outs))
        r = interleaved(fns, it=10)
        for name in fns:
            res[name] = {"ms": r[name]["median_ms"], "tflops": round(flops[name] / r[name]["median_ms"] / 1e9, 1)}
        del keep, fns
    # MoE dispatch + GroupedMatMul (EP form of the fused operators): a
    # Mixtral-style layer on 8 EP ranks, one expert each, 4096 tokens per rank,
    # against one plain GEMM over the same number of rows
    s = wl.MoEDispatch(R=8, T=4096, h=4096, f=14336, e_loc=1, seed=21)
    xs, idxs, ws = s.make()
    dx, di, w = [x.to(dev) for x in xs], [i.to(dev) for i in idxs], torch.stack(ws).to(dev)
    y, xd, cnt, off = coc.moe_dispatch_grouped_matmul(dx, di, w, s.e_loc)
    xg = torch.cat(dx, 0)
    og = torch.empty(xg.shape[0], s.f, dtype=s.dtype, device=dev)
    ti, tg = s.routing_topk(2)
    ti, tg = [i.to(dev) for i in ti], [g.to(dev) for g in tg]
    yt, y2, xd2, cnt2, off2 = coc.moe_topk_grouped_matmul_combine(dx, ti, tg, w, s.e_loc)
    r = interleaved({"moe": lambda: coc.moe_dispatch_grouped_matmul(dx, di, w, s.e_loc, xd=xd, y=y, counts=cnt,
                                                                    offsets=off),
                     "plain": lambda: coc.matmul([xg], [w[0]], og),
                     "top2": lambda: coc.moe_topk_grouped_matmul_combine(dx, ti, tg, w, s.e_loc, xd=xd2, y=y2,
                                                                         y_tok=yt, counts=cnt2, offsets=off2)},
                    it=10)
    res["moe_dispatch_grouped_matmul_mixtral_ep8"] = {
        "ms": r["moe"]["median_ms"], "tflops": round(s.flops() / r["moe"]["median_ms"] / 1e9, 1),
        "plain_gemm_same_rows_ms": r["plain"]["median_ms"],
        "tokens_per_expert": [int(v) for v in cnt.cpu().tolist()]}
    res["moe_top2_grouped_matmul_combine_mixtral_ep8"] = {
        "ms": r["top2"]["median_ms"], "tflops": round(2 * s.flops() / r["top2"]["median_ms"] / 1e9, 1),
        "entries_per_expert": [int(v) for v in cnt2.cpu().tolist()]}
    del dx, di, w, ti, tg, yt, y2, xd2, y, xd, xg, og
    return res


# --------------------------------------------------------- CPU oracle legs ---

def oracle_sample(host, rows: int, cols: int | None, seed: int = 1234):
    """Run the fp64 oracle on `rows` seeded output rows (and the first `cols`
    columns, None = all) of every operator.  Returns (seconds, flops, cores)."""
    import numpy as np

    from oracle import oracle as orc
    from tensor_matmul_collective_gb300 import workloads as wl

    def b(ts, c=None):
        return [wl.bits16(t) if c is None else np.ascontiguousarray(wl.bits16(t)[:, :c]) for t in ts]

    flops = 0.0
    t0 = time.perf_counter()
    xs, ws = host["bloom7b"]
    s = wl.BLOOM7B_AR
    c = cols or s.n
    r_ = wl.sample_rows(s.m, rows, seed)
    orc.matmul_all_reduce(orc.BF16, b(xs), b(ws, c), r_)
    flops += 2.0 * rows * c * s.K

    xs, ws = host["llama_ag"]
    s = wl.LLAMA70B_AG
    c = cols or s.n_shard
    r_ = wl.sample_rows(s.m, rows, seed)
    bx, bw = b(xs), b(ws, c)
    for r in range(s.R):
        orc.all_gather_matmul(orc.BF16, bx, bw, r, r_)
        flops += 2.0 * rows * c * s.k
    orc.all_gather(bx)

    xs, ws = host["llama_rs"]
    s = wl.LLAMA70B_RS
    c = cols or s.n
    bx, bw = b(xs), b(ws, c)
    r_ = wl.sample_rows(s.m // s.R, max(1, rows // s.R), seed)
    for r in range(s.R):
        orc.matmul_reduce_scatter(orc.BF16, bx, bw, r, r_)
        flops += 2.0 * r_.size * c * s.K

    s = wl.W8A16_AR
    for code, gran in enumerate(wl.SCALE_GRANS):
        xs, wqs, scales = host[f"w8_{gran}"]
        c = cols or s.n
        wq = [np.ascontiguousarray(w.numpy()[:, :c]) for w in wqs]
        sc = [wl.bits16(t) for t in scales]
        if gran != "tensor":
            sc = [np.ascontiguousarray(x.reshape(-1, s.n)[:, :c]) for x in sc]
        r_ = wl.sample_rows(s.m, rows, seed)
        orc.matmul_all_reduce_w8a16(b(xs), wq, sc, code, s.group, r_)
        flops += 2.0 * rows * c * s.K

    xs, ws = host["bloom176b"]
    s = wl.BLOOM176B
    c = cols or s.n
    bx, bw = b(xs), b(ws, c)
    r_ = wl.sample_rows(s.m, rows, seed)
    orc.matmul_all_reduce(orc.BF16, bx, bw, r_)
    flops += 2.0 * rows * c * s.K
    r2 = wl.sample_rows(s.m // s.R, max(1, rows // s.R), seed)
    for r in range(s.R):
        orc.matmul_reduce_scatter(orc.BF16, bx, bw, r, r2)
        flops += 2.0 * r2.size * c * s.K
    return time.perf_counter() - t0, flops, orc.max_threads()


def make_host_inputs():
    from tensor_matmul_collective_gb300 import workloads as wl
    host = {}
    host["bloom7b"] = wl.BLOOM7B_AR.make()
    host["llama_ag"] = wl.LLAMA70B_AG.make()
    host["llama_rs"] = wl.LLAMA70B_RS.make()
    for gran in wl.SCALE_GRANS:
        host[f"w8_{gran}"] = wl.W8A16_AR.make(gran)
    host["bloom176b"] = wl.BLOOM176B.make()
    return host


def suite_flops() -> float:
    from tensor_matmul_collective_gb300 import workloads as wl
    return (wl.BLOOM7B_AR.flops() + wl.LLAMA70B_AG.flops() + wl.LLAMA70B_RS.flops() + 3 * wl.W8A16_AR.flops()
            + 2 * wl.BLOOM176B.flops())


def base_line(n_gpus, steps, warmup):
    return {"metric": METRIC, "unit": UNIT, "n_gpus": n_gpus, "steps": steps, "warmup": warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; BLOOM-7B / LLaMA2-70B / BLOOM-176B TP8 layer shapes)"}


def config_dict(world):
    from tensor_matmul_collective_gb300 import workloads as wl
    return {"workload": WORKLOAD, "ranks_emulated": 8, "chunks": {w.name: w.chunks for w in wl.TP8_SUITE},
            "compute_types": "bf16 in / fp32 accumulate / bf16 out; w8A16: fp16 x int8 -> fp16",
            "l2": "no flush: every operator's operands exceed the 129 MB L2 and each step streams > 5 GB",
            "parallelism": f"replicas x{world} (no cross-GPU exchange on this path)"}


# -------------------------------------------------------------------- arms ---

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    host = make_host_inputs()
    rows, cols = 1, 64
    for _ in range(args.warmup):
        oracle_sample(host, rows, cols)
    secs, flops, cores = [], 0.0, 1
    for _ in range(args.steps):
        t, flops, cores = oracle_sample(host, rows, cols)
        secs.append(t)
    total = sum(secs)
    value = flops * args.steps / total / 1e12
    line = base_line(args.gpus, args.steps, args.warmup)
    line.update({"impl": "reference", "value": value, "ms_per_step": 1000.0 * total / args.steps,
                 "dtype": "f64", "config": config_dict(1),
                 "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                                  "sample": f"per step: {rows} seeded output row x first {cols} columns of every "
                                            f"operator of the suite ({flops / 1e9:.3f} GFLOP)"},
                 "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}})
    print(json.dumps(line), flush=True)
    return 0


def op_stats(op, ts, peaks):
    """Median / min / max of one operator's per-step times, its TFLOP/s at the
    median and min, fractions of the measured tensor peaks, and its achieved
    algorithmic HBM bandwidth."""
    med, lo, hi = statistics.median(ts), min(ts), max(ts)
    tf = op.flops / (med / 1e3) / 1e12
    ab = algorithmic_bytes(op)
    return {"ms_median": round(med, 4), "ms_min": round(lo, 4), "ms_max": round(hi, 4),
            "spread": round((hi - lo) / med, 4), "samples": len(ts),
            "tflops": round(tf, 1), "tflops_at_min": round(op.flops / (lo / 1e3) / 1e12, 1),
            "frac_burst": round(tf / peaks["bf16_tflops"], 4),
            "frac_sustained": round(tf / peaks["bf16_tflops_sustained"], 4),
            "algorithmic_gb": round(ab / 1e9, 4), "hbm_gbs": round(ab / (med / 1e3) / 1e9, 1),
            "hbm_frac": round(ab / (med / 1e3) / 1e9 / peaks["hbm_gbs"], 4)}


def roofline_obj(op, ts, peaks, clocks, traffic):
    """The dominant kernel against the dense bf16 tensor roofline.  frac (the
    headline) divides by the measured BURST peak, the right denominator for a
    sub-second timed region; frac_clock_normalised scales the measured
    sustained peak by the SM clock this kernel ran at (measured inside the
    kernel: SM cycles over %globaltimer ns) over the clock that peak was
    measured at, i.e. the kernel's per-clock efficiency against cuBLAS's."""
    med = statistics.median(ts)
    tf = op.flops / (med / 1e3) / 1e12
    burst, sus = peaks["bf16_tflops"], peaks["bf16_tflops_sustained"]
    kern_mhz = ((clocks or {}).get("sm_mhz_in_kernel") or {}).get(op.name)
    line_mhz, peak_mhz = (clocks or {}).get("sm_mhz"), peaks.get("sustained_sm_mhz")
    norm = None
    if kern_mhz and peak_mhz:
        norm = round(tf / (sus * kern_mhz / peak_mhz), 4)
    return {"bound": "tensor", "kernel": op.name, "achieved": round(tf, 1), "peak": burst, "unit": UNIT,
            "frac": round(tf / burst, 4), "traffic": traffic,
            "frac_burst": round(tf / burst, 4), "frac_sustained": round(tf / sus, 4),
            "frac_clock_normalised": norm,
            "sm_mhz_samples": (clocks or {}).get("samples"), "sm_mhz_line": line_mhz,
            "sm_mhz_in_kernel": kern_mhz, "sm_mhz_of_sustained_peak": peak_mhz,
            "headline": "frac = frac_burst (measured burst bf16 peak, of measured)",
            "achieved_from": f"median over {len(ts)} timed steps of the kernel's CUDA-event duration "
                             f"on the launching stream; algorithmic 2mnK FLOPs",
            "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json: burst {burst}, sustained {sus} TFLOP/s)"}


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local))
        dist = tdist
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from tensor_matmul_collective_gb300 import build as cbuild
    from tensor_matmul_collective_gb300 import coc
    cbuild.build()
    coc.lib()

    ops, host = build_suite(dev)
    bus = None
    try:
        props = torch.cuda.get_device_properties(dev)
        bus = "%04x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id, props.pci_device_id)
    except Exception:
        bus = None
    sampler = NvmlSampler(bus, local)
    total_ms, per_op, clocks = time_device(ops, args.steps, args.warmup, dist, sampler)

    total_ms = max_over_ranks(total_ms, dist, dev)
    step_flops = sum(op.flops for op in ops)
    value = job_value(step_flops, args.steps, world, total_ms)

    peaks = load_peaks()
    dom = max(range(len(ops)), key=lambda i: statistics.median(per_op[i]))
    from tensor_matmul_collective_gb300 import workloads as wl
    chunks_of = {w.name: w.chunks for w in wl.TP8_SUITE}
    traffic = load_traffic(ops[dom].name, chunks_of.get(ops[dom].name, chunks_of.get("w8a16_ar", 1)))
    per_op_json = {op.name: op_stats(op, ts, peaks) for op, ts in zip(ops, per_op)}
    for op in ops:
        per_op_json[op.name]["sm_mhz_in_kernel"] = ((clocks or {}).get("sm_mhz_in_kernel") or {}).get(op.name)

    e2e = None
    if args.e2e_steps > 0:
        e2e_sampler = NvmlSampler(bus, local)
        e2e_sampler.start()
        wall, h2d, d2h = time_e2e(ops, args.e2e_steps, dev)
        e2e_clocks = e2e_sampler.stop()
        wall_ms = max_over_ranks(wall * 1e3, dist, dev)
        e2e = {"value": job_value(step_flops, args.e2e_steps, world, wall_ms), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "h2d": "every operator's activation shards X_r from pinned host memory (weights resident)",
               "d2h": "every distinct result tensor to pinned host memory",
               # the SM clock of this leg (power-capped boxes settle differently per phase)
               "sm_mhz": e2e_clocks["sm_mhz"] if e2e_clocks else None}

    context = None if args.no_context else time_context(ops, dev, bus, local)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rows = 16
        t, flops, cores = oracle_sample(host, rows, None)
        cpu = {"value": flops / t / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
               "extrapolated_step_s": round(t * step_flops / flops, 1),
               "sample": f"{rows} seeded output rows (all columns) of every operator of one suite step "
                         f"({flops / 1e9:.1f} GFLOP in {t:.1f} s)"}

    if rank == 0:
        line = base_line(world, args.steps, args.warmup)
        line.update({
            "value": value, "ms_per_step": total_ms / args.steps, "config": config_dict(world),
            "pct_of_peak_burst": round(100.0 * value / world / peaks["bf16_tflops"], 2),
            "pct_of_peak_sustained": round(100.0 * value / world / peaks["bf16_tflops_sustained"], 2),
            "peak": {"bf16_tflops_burst": peaks["bf16_tflops"], "bf16_tflops_sustained": peaks["bf16_tflops_sustained"],
                     "hbm_gbs": peaks["hbm_gbs"], "source": peaks["source"]},
            "roofline": roofline_obj(ops[dom], per_op[dom], peaks, clocks, traffic),
            "per_op": per_op_json,
            "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": sum(o.launches for o in ops) * args.steps,
            "context": context,
        })
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_case(a):
    """One operator on seeded synthetic data, timed over a.iters calls (CUDA
    events, after one untimed call); prints one JSON line."""
    import torch

    from tensor_matmul_collective_gb300 import build as cbuild
    from tensor_matmul_collective_gb300 import coc
    from tensor_matmul_collective_gb300 import workloads as wl
    cbuild.build()
    dev = torch.device("cuda:0")
    dt = torch.bfloat16 if a.dtype == "bf16" else torch.float16
    if a.case in ("ag", "ag_v2"):
        s = wl.ColumnParallelSP(R=a.R, m_shard=a.m, n_shard=a.n, k=a.k, dtype=dt, x_dist="normal(0,1)",
                                w_dist="normal(0,0.02)", seed=2)
        xs, ws = s.make()
        dx, dw = [x.to(dev) for x in xs], [w.to(dev) for w in ws]
        outs = [torch.empty(s.m, s.n_shard, dtype=dt, device=dev) for _ in range(a.R)]
        if a.case == "ag_v2":
            g = [torch.empty(s.m, s.k, dtype=dt, device=dev) for _ in range(a.R)]
            run = lambda: coc.all_gather_matmul_v2(dx, dw, outs, g, chunks=a.chunks)  # noqa: E731
        else:
            run = lambda: coc.all_gather_matmul(dx, dw, outs, chunks=a.chunks)  # noqa: E731
        flops = s.flops()
    elif a.case == "moe":
        s = wl.MoEDispatch(R=a.R, T=a.m, h=a.k, f=a.n, e_loc=a.eloc, seed=21, dtype=dt)
        xs, idxs, ws = s.make()
        dx, w = [x.to(dev) for x in xs], torch.stack(ws).to(dev)
        if a.topk > 1:
            ti, tg = s.routing_topk(a.topk)
            ti, tg = [i.to(dev) for i in ti], [g.to(dev) for g in tg]
            run = lambda: coc.moe_topk_grouped_matmul_combine(dx, ti, tg, w, a.eloc)  # noqa: E731
        else:
            di = [i.to(dev) for i in idxs]
            run = lambda: coc.moe_dispatch_grouped_matmul(dx, di, w, a.eloc)  # noqa: E731
        flops = s.flops() * a.topk
    elif a.case == "w8a16":
        s = wl.W8A16(R=a.R, m=a.m, n=a.n, k_shard=a.k, group=a.group, seed=3, dtype=dt)
        xs, wqs, scales = s.make(a.gran)
        dx, dw, dsc = [x.to(dev) for x in xs], [w.to(dev) for w in wqs], [t.to(dev) for t in scales]
        dz = [z.to(dev) for z in s.zeros(a.gran)] if a.zero else None
        outs = [torch.empty(s.m, s.n, dtype=dt, device=dev) for _ in range(a.R)]
        run = lambda: coc.matmul_all_reduce_w8a16(dx, dw, dsc, a.gran, a.group, outs, chunks=a.chunks,  # noqa: E731
                                                  zeros=dz)
        flops = s.flops()
    else:
        s = wl.RowParallel(R=a.R, m=a.m, n=a.n, k_shard=a.k, dtype=dt, x_dist="normal(0,1)",
                           w_dist="normal(0,0.02)", seed=1)
        xs, ws = s.make()
        dx, dw = [x.to(dev) for x in xs], [w.to(dev) for w in ws]
        if a.case == "ar":
            outs = [torch.empty(s.m, s.n, dtype=dt, device=dev) for _ in range(a.R)]
            run = lambda: coc.matmul_all_reduce(dx, dw, outs, chunks=a.chunks,  # noqa: E731
                                                deterministic=a.deterministic)
        elif a.case == "rs":
            outs = [torch.empty(s.m // a.R, s.n, dtype=dt, device=dev) for _ in range(a.R)]
            run = lambda: coc.matmul_reduce_scatter(dx, dw, outs, chunks=a.chunks,  # noqa: E731
                                                    deterministic=a.deterministic)
        else:
            out = torch.empty(s.m, s.n, dtype=dt, device=dev)
            run = lambda: coc.matmul(dx, dw, out)  # noqa: E731
        flops = s.flops()
    run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(a.iters):
        run()
    e1.record()
    torch.cuda.synchronize()
    coc.sync_status()
    ms = e0.elapsed_time(e1) / a.iters
    print(json.dumps({"case": a.case, "R": a.R, "m": a.m, "n": a.n, "k": a.k, "chunks": a.chunks, "ms": ms,
                      "tflops": flops / (ms / 1e3) / 1e12}), flush=True)
    return 0


def main():
    args = parse_args()
    if args.case is not None:
        return run_case(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
