#!/usr/bin/env python
"""Benchmark of the NF4 weight-only linear hot path on one GB300 (or N replicas).

One step is one pass of the whole path over one batch of synthetic input on
the Gemma3-12B q_proj shape (W [4096, 3840] bf16 ~ N(0, 0.02), X [2048, 3840]
bf16 ~ N(0, 1) = 2 prompts x 1024 tokens):

    nf4_quantize(W) -> packed, absmax          blockwise absmax + nibble pack
    nf4_dequantize(packed, absmax) -> Wdeq      byte-LUT dequant (bulk path)
    nf4_linear(X, packed, absmax) -> Y          fused NF4 GEMM, M = 2048
    nf4_linear(X[:16], packed, absmax) -> Ys    skinny path, M = 16

`value` is the linear FLOPs of a step (2*M*N*K for both calls) divided by the
step time, summed over ranks (replicas, weak scaling).  Inputs are resident in
HBM; an L2 flush precedes every step, outside the events: a 512 MiB memset,
then a read of another 256 MiB so the step starts on clean L2 lines instead
of paying for the memset's write-backs.
Per-kernel times come from CUDA events around each call on the launching
stream (a separate pass).  `e2e` repeats the step through the public API with
W and X copied from pinned host memory and Y, Ys copied back every step,
pipelined over three streams and two buffer sets as a serving loop would.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

`--impl reference` times the CPU oracle (the plain C reference this library
is checked against) on a bounded sample of the same step: it is the baseline
arm, not a target.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import random
import re
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "nf4_linear TFLOP/s at M=2048 Gemma3-12B projections; dequant HBM GB/s vs peak"
CFG = workloads.Q_PROJ
SKINNY_M = 16
FLOPS_PER_STEP = 2 * CFG.m * CFG.n * CFG.k + 2 * SKINNY_M * CFG.n * CFG.k
# Algorithmic bytes per weight element: quantize reads 2 and writes 0.5 + 4/64;
# dequantize reads 0.5 + 4/64 and writes 2.
BYTES_PER_W_QUANT = 2.5625
BYTES_PER_W_DEQUANT = 2.5625
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
REF_STEP_ROWS = 128             # reference arm: rows of X per step


# ---------------------------------------------------------------- helpers


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        pk = {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"])}
        # the cuBLAS rate held for seconds under the power cap: the peak for a
        # GEMM timed inside a long pass
        pk["bf16_tflops_sustained"] = float(d.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
        return pk, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# what the roofline kernel (wide_kernel, the CTA-pair GEMM nf4_linear runs at
# M = 2048 on this shape) is built from
GEMM_SOURCES = ("nf4_device.cuh", "nf4_convert.cuh", "nf4_gemm_wide.cu", "nf4_launch.h")
ROOFLINE_KERNEL = "wide_kernel"


def code_tokens(text: str) -> str:
    """C++ source with comments removed and whitespace collapsed: what the
    compiler sees, so a comment edit does not change the hash."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash() -> str:
    """Hash of the code of the kernel the roofline reports (ROOFLINE_KERNEL)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "nf4_weight_quantized_quantize_gb300", "csrc")
    for fn in GEMM_SOURCES:
        with open(os.path.join(csrc, fn)) as f:
            h.update(fn.encode() + b"\0" + code_tokens(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` on this workload from the committed ncu
    summaries, if they were taken on the current kernel sources; else None."""
    prof = os.path.join(ROOT, "profiles")
    if not os.path.isdir(prof):
        return None
    want = kernel_source_hash()
    for fn in sorted(os.listdir(prof)):
        if not fn.endswith(".md"):
            continue
        text = open(os.path.join(prof, fn)).read()
        for m in re.finditer(r"^traffic\s+kernel=(\S+)\s+workload=(\S+)\s+bytes_per_launch=(\d+)\s+"
                             r"source_hash=(\w+)", text, flags=re.M):
            if m.group(1) == kernel and m.group(2) == CFG.name and m.group(4) == want:
                return int(m.group(3))
    return None


class ClockSampler:
    """Polls SM clock and clock-event reasons through NVML (read only) on a
    background thread while the timed region runs."""
    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, device_index: int, period_s: float = 0.002):
        self.samples = []
        self.max_mhz = None
        self.error = None
        self.period = period_s
        self._stop = threading.Event()
        self._thread = None
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit failed")
            import torch
            props = torch.cuda.get_device_properties(device_index)
            bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0".encode()
            self.handle = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(self.handle)) != 0:
                raise RuntimeError(f"no NVML handle for {bus!r}")
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._reasons_fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        except Exception as e:  # noqa: BLE001 - clocks are reported as unavailable
            self.error = str(e)

    def _run(self):
        clk = ctypes.c_uint()
        rsn = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk)) == 0 and \
                    self._reasons_fn(self.handle, ctypes.byref(rsn)) == 0:
                self.samples.append((clk.value, rsn.value))
            time.sleep(self.period)

    def start(self):
        if self.error is None:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
            if not self.samples:   # region shorter than one period: take one reading now
                self._stop.clear()
                clk, rsn = ctypes.c_uint(), ctypes.c_ulonglong()
                if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk)) == 0 and \
                        self._reasons_fn(self.handle, ctypes.byref(rsn)) == 0:
                    self.samples.append((clk.value, rsn.value))

    def summary(self):
        if self.error is not None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": f"nvml unavailable: {self.error}"}
        mhz = [s[0] for s in self.samples]
        bits = 0
        for _, r in self.samples:
            bits |= r
        reasons = sorted(n for b, n in self.REASONS.items() if bits & b and n != "gpu_idle")
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(mhz)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def allreduce_max(value: float, ws: int, device=None) -> float:
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def allreduce_sum(value: float, ws: int, device=None) -> float:
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def aggregate_tflops(flops_this_rank: float, step_ms_max: float, ws: int, device=None) -> float:
    """Whole-job throughput: the FLOPs every rank did (each rank counts its own
    work; replicas do the same amount on their own prompts), summed over ranks,
    over the slowest rank's time."""
    return allreduce_sum(flops_this_rank, ws, device) / (step_ms_max * 1e-3) / 1e12


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- CPU oracle arm


def oracle_sample(rows: int, x_bits, w_bits):
    """One bounded sample of the step on the CPU oracle; returns (flops, seconds)."""
    import oracle
    t0 = time.perf_counter()
    p, a = oracle.quantize(w_bits)
    oracle.dequantize(p, a, w_bits.size)
    oracle.linear(x_bits[:rows], p, a, CFG.n)
    oracle.linear(x_bits[:SKINNY_M], p, a, CFG.n)
    dt = time.perf_counter() - t0
    return 2 * (rows + SKINNY_M) * CFG.n * CFG.k, dt


# The oracle per workload, on one core and on all cores: (name, projections,
# X rows of each projection timed on all cores / on one core, W rows quantized
# and dequantized on all cores / on one core; None = all).  A sample smaller
# than the workload is timed and its rate reported as "extrapolated" (the
# oracle's time is linear in the rows of X and in the weight elements).  The
# stack is timed on layer 0's seven projections and stands for all 48.
CPU_CASES = (
    ("tiny", [workloads.TINY], (None, None), (None, None)),
    ("q_proj_m2048", [workloads.Q_PROJ], (None, 64), (None, None)),
    ("gate_up_m2048", [workloads.GATE_UP], (256, 16), (None, 4096)),
    ("down_proj_m2048", [workloads.DOWN], (256, 32), (None, None)),
    ("down_proj_m16", [workloads.DOWN_SKINNY], (None, None), (None, None)),
    ("stack_48x7_m8192", [workloads.stack_layer(0, i) for i in range(len(workloads.PROJECTIONS))],
     (64, 4), (None, 1024)),
)


def _oracle_case(inputs, lin_rows, w_rows, threads):
    """Time the oracle's quantize, dequantize and linear on the given samples
    of each projection's (config, W bits, X bits) with `threads` OpenMP
    threads; rates, and whether they were measured on less than the whole
    workload."""
    import oracle
    oracle.set_num_threads(threads)
    t_q = t_d = t_l = 0.0
    n_q = flop = 0
    part = False
    for c, w, x in inputs:
        ws = w if w_rows is None or w_rows >= c.n else w[:w_rows]
        part |= ws.shape[0] < c.n
        t0 = time.perf_counter()
        p, a = oracle.quantize(ws)
        t_q += time.perf_counter() - t0
        t0 = time.perf_counter()
        oracle.dequantize(p, a, ws.size)
        t_d += time.perf_counter() - t0
        n_q += ws.size
        if ws.shape[0] < c.n:
            p, a = oracle.quantize(w)
        rows = c.m if lin_rows is None else min(lin_rows, c.m)
        part |= rows < c.m
        t0 = time.perf_counter()
        oracle.linear(x[:rows], p, a, c.n)
        t_l += time.perf_counter() - t0
        flop += 2 * rows * c.n * c.k
    return {"linear_TFLOP/s": flop / t_l / 1e12, "quantize_GB/s": n_q * BYTES_PER_W_QUANT / t_q / 1e9,
            "dequantize_GB/s": n_q * BYTES_PER_W_DEQUANT / t_d / 1e9, "seconds": t_q + t_d + t_l,
            "extrapolated": part}


def cpu_baseline():
    """The oracle (fp64 accumulation, plain C) timed on the host cores of this
    box, per workload, once on one core and once on all cores.  The line's
    `value` is the headline workload's linear (q_proj, M = 2048) on all cores."""
    import oracle
    all_cores = oracle.num_threads()
    per = {}
    for name, projs, lin_rows, w_rows in CPU_CASES:
        inputs = [(c, workloads.bits(workloads.make_weight(c)), workloads.bits(workloads.make_activation(c)))
                  for c in projs]
        per[name] = {"all_cores": _oracle_case(inputs, lin_rows[0], w_rows[0], all_cores),
                     "one_core": _oracle_case(inputs, lin_rows[1], w_rows[1], 1)}
        del inputs
        per[name]["samples"] = {"x_rows_all_cores": lin_rows[0], "x_rows_one_core": lin_rows[1],
                                "w_rows_all_cores": w_rows[0], "w_rows_one_core": w_rows[1]}
    oracle.set_num_threads(all_cores)
    secs = sum(v[k]["seconds"] for v in per.values() for k in ("all_cores", "one_core"))
    head = per["q_proj_m2048"]["all_cores"]
    return {"value": head["linear_TFLOP/s"], "unit": "TFLOP/s", "cores": all_cores, "kind": "oracle",
            "sample": (f"q_proj linear on all {CFG.m} rows of X, {all_cores} threads; per workload below: "
                       f"quantize, dequantize and linear on one core and on all cores ({secs:.1f} s of CPU "
                       "work in all); 'extrapolated' marks a rate measured on a row sample of the workload"),
            "configs": per}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    w = workloads.bits(workloads.make_weight(CFG))
    x = workloads.bits(workloads.make_activation(CFG))
    for _ in range(args.warmup):
        oracle_sample(REF_STEP_ROWS, x, w)
    total_flops, total_s = 0, 0.0
    for _ in range(args.steps):
        f, dt = oracle_sample(REF_STEP_ROWS, x, w)
        total_flops += f
        total_s += dt
    value = total_flops / total_s / 1e12
    sample = (f"per step: quantize + dequantize of the full W [{CFG.n}, {CFG.k}], linear on "
              f"{REF_STEP_ROWS} of the {CFG.m} rows of X plus the {SKINNY_M}-row batch")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_s / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_block(args),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def config_block(args):
    return {"workload": CFG.name, "M": CFG.m, "N": CFG.n, "K": CFG.k, "skinny_M": SKINNY_M,
            "block": 64, "absmax": "fp32", "w_dist": "N(0,0.02) bf16", "x_dist": "N(0,1) bf16",
            "seeds": {"w": CFG.w_seed, "x": f"{CFG.x_seed} + 1000 x rank (each replica its own prompts)"},
            "l2": "flushed before every step: 512 MiB memset, then a 256 MiB read (clean lines)",
            "parallelism": f"replicas{args.gpus}"}


# ---------------------------------------------------------------- GPU arm


def run_ours(args):
    import torch
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    import nf4_weight_quantized_quantize_gb300 as nf4

    stream = torch.cuda.current_stream(dev)
    mine = workloads.for_replica(CFG, rank)    # this replica's prompts, the shared weight
    w = workloads.make_weight(mine, device=dev)
    x = workloads.make_activation(mine, device=dev)
    xs = x[:SKINNY_M].contiguous()
    numel = w.numel()
    packed = torch.empty(numel // 2, dtype=torch.uint8, device=dev)
    absmax = torch.empty(numel // 64, dtype=torch.float32, device=dev)
    wdeq = torch.empty(numel, dtype=torch.bfloat16, device=dev)
    y = torch.empty(CFG.m, CFG.n, dtype=torch.bfloat16, device=dev)
    ys = torch.empty(SKINNY_M, CFG.n, dtype=torch.bfloat16, device=dev)
    st, ws_bytes = nf4.nf4_linear_workspace_size(SKINNY_M, CFG.n, CFG.k)
    assert st == nf4.NF4_OK
    wsp = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_read = torch.zeros(256 << 20, dtype=torch.uint8, device=dev)

    def flush_l2():
        flush.zero_()
        flush_read.max()

    names = ["nf4_quantize", "nf4_dequantize", "nf4_linear_m2048", "nf4_linear_m16"]
    calls = [
        lambda: nf4.quantize(w, out=(packed, absmax)),
        lambda: nf4.dequantize(packed, absmax, numel, out=wdeq),
        lambda: nf4.linear(x, packed, absmax, CFG.n, out=y),
        lambda: nf4.linear(xs, packed, absmax, CFG.n, out=ys, workspace=wsp),
    ]

    def step(evs=None):
        for i, c in enumerate(calls):
            if evs is not None:
                evs[i][0].record(stream)
            c()
            if evs is not None:
                evs[i][1].record(stream)

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    if nf4.nf4_last_error(stream.cuda_stream) != nf4.NF4_OK:
        raise RuntimeError("a kernel reported a timeout during warm-up")

    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    step_ev = [(mk(), mk()) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    launches0 = nf4.nf4_launch_count()
    barrier(ws)
    torch.cuda.synchronize()
    sampler.start()
    t_wall = time.perf_counter()
    for k in range(args.steps):
        flush_l2()
        phase_jitter()
        step_ev[k][0].record(stream)
        step()
        step_ev[k][1].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    barrier(ws)
    sampler.stop()
    launches = nf4.nf4_launch_count() - launches0
    if nf4.nf4_last_error(stream.cuda_stream) != nf4.NF4_OK:
        raise RuntimeError("a kernel reported a timeout in the timed region")
    step_ms = sum(a.elapsed_time(b) for a, b in step_ev)
    step_ms = allreduce_max(step_ms, ws, dev)
    value = aggregate_tflops(FLOPS_PER_STEP * args.steps, step_ms, ws, dev)

    # ---- per-call breakdown: a second pass with events around every call
    # (kept out of the timed steps above, whose value they would inflate)
    call_steps = min(args.steps, 50)
    call_ev = [[(mk(), mk()) for _ in calls] for _ in range(call_steps)]
    for k in range(call_steps):
        flush_l2()
        phase_jitter()
        step(call_ev[k])
    torch.cuda.synchronize()
    per_call = [statistics.mean(call_ev[k][i][0].elapsed_time(call_ev[k][i][1]) for k in range(call_steps))
                for i in range(len(calls))]

    # ---- end to end through the public API, host buffers.  Every step copies
    # W and X from pinned host memory and reads Y, Ys back.  Pipelined the
    # way a serving loop would run it: three streams and two buffer sets, so
    # step k+1's host-to-device copies overlap step k's kernels and step
    # k-1's device-to-host copies; the timed region spans the first copy in
    # to the last copy out.
    w_h = w.cpu().pin_memory()
    x_h = x.cpu().pin_memory()
    sets = [dict(w=torch.empty_like(w), x=torch.empty_like(x), xs=torch.empty_like(xs),
                 packed=torch.empty_like(packed), absmax=torch.empty_like(absmax), wdeq=torch.empty_like(wdeq),
                 y=torch.empty_like(y), ys=torch.empty_like(ys), ws=torch.zeros_like(wsp),
                 y_h=torch.empty(CFG.m, CFG.n, dtype=torch.bfloat16).pin_memory(),
                 ys_h=torch.empty(SKINNY_M, CFG.n, dtype=torch.bfloat16).pin_memory()) for _ in range(2)]
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_done = [torch.cuda.Event() for _ in range(2)]
    cmp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def e2e_steps(nsteps, t0=None, t1=None):
        if t0 is not None:
            t0.record(s_in)
        for k in range(nsteps):
            b, i = sets[k % 2], k % 2
            with torch.cuda.stream(s_in):
                if k >= 2:
                    s_in.wait_event(cmp_done[i])          # step k-2 is done reading this set's W, X
                b["w"].copy_(w_h, non_blocking=True)
                b["x"].copy_(x_h, non_blocking=True)
                in_done[i].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(in_done[i])
                if k >= 2:
                    s_cmp.wait_event(out_done[i])         # step k-2's Y has been read back
                b["xs"].copy_(b["x"][:SKINNY_M])
                nf4.quantize(b["w"], out=(b["packed"], b["absmax"]))
                nf4.dequantize(b["packed"], b["absmax"], numel, out=b["wdeq"])
                nf4.linear(b["x"], b["packed"], b["absmax"], CFG.n, out=b["y"])
                nf4.linear(b["xs"], b["packed"], b["absmax"], CFG.n, out=b["ys"], workspace=b["ws"])
                cmp_done[i].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(cmp_done[i])
                b["y_h"].copy_(b["y"], non_blocking=True)
                b["ys_h"].copy_(b["ys"], non_blocking=True)
                out_done[i].record(s_out)
        if t1 is not None:
            t1.record(s_out)

    e2e_steps(args.warmup)
    torch.cuda.synchronize()
    barrier(ws)
    e0, e1 = mk(), mk()
    e2e_steps(args.steps, e0, e1)
    torch.cuda.synchronize()
    barrier(ws)
    if nf4.nf4_last_error(s_cmp.cuda_stream) != nf4.NF4_OK:
        raise RuntimeError("a kernel reported a timeout in the end-to-end steps")
    if not torch.equal(sets[(args.steps - 1) % 2]["y_h"], y.cpu()):
        raise RuntimeError("end-to-end result differs from the device-resident step's")
    e2e_ms = allreduce_max(e0.elapsed_time(e1), ws, dev)
    e2e_value = aggregate_tflops(FLOPS_PER_STEP * args.steps, e2e_ms, ws, dev)
    h2d = (w.numel() + x.numel()) * 2
    d2h = (y.numel() + ys.numel()) * 2

    if rank != 0:
        return 0
    pk, pk_kind = peaks()
    t_q, t_d, t_l, t_s = per_call
    lin_tflops = 2 * CFG.m * CFG.n * CFG.k / (t_l * 1e-3) / 1e12
    deq_gbs = numel * BYTES_PER_W_DEQUANT / (t_d * 1e-3) / 1e9
    q_gbs = numel * BYTES_PER_W_QUANT / (t_q * 1e-3) / 1e9
    sk_bytes = numel * 0.5625 + 2 * SKINNY_M * CFG.k + 2 * SKINNY_M * CFG.n
    sk_gbs = sk_bytes / (t_s * 1e-3) / 1e9
    clocks = sampler.summary()
    traffic = profiled_traffic(ROOFLINE_KERNEL)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "value_definition": ("composite: the linear FLOPs of a step (nf4_linear at M = 2048 and at M = 16) over "
                             "the time of the whole step, which also quantizes and dequantizes the weight; the "
                             "per-kernel figures are under 'kernels' and 'configs'"),
        "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_block(args),
        "roofline": {"bound": "tensor", "kernel": f"{ROOFLINE_KERNEL} (nf4_linear, M=2048)",
                     "achieved": lin_tflops, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": lin_tflops / pk["bf16_tflops"], "peak_source": f"bf16_tflops of {pk_kind}",
                     "traffic": traffic, "algorithmic": "2*M*N*K FLOP per launch"},
        "kernels": {
            "nf4_quantize": {"ms": t_q, "GB/s": q_gbs, "frac_hbm": q_gbs / pk["hbm_gbs"],
                             "bytes_per_weight": BYTES_PER_W_QUANT},
            "nf4_dequantize": {"ms": t_d, "GB/s": deq_gbs, "frac_hbm": deq_gbs / pk["hbm_gbs"],
                               "bytes_per_weight": BYTES_PER_W_DEQUANT},
            "nf4_linear_m2048": {"ms": t_l, "TFLOP/s": lin_tflops, "frac_bf16": lin_tflops / pk["bf16_tflops"]},
            "nf4_linear_m16": {"ms": t_s, "GB/s": sk_gbs, "frac_hbm": sk_gbs / pk["hbm_gbs"],
                               "bytes": sk_bytes},
        },
        "peaks": {"hbm_gbs": pk["hbm_gbs"], "bf16_tflops": pk["bf16_tflops"],
                  "bf16_tflops_sustained": pk["bf16_tflops_sustained"], "source": pk_kind},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms / args.steps,
                "mode": "pipelined: 3 streams, 2 buffer sets; step k+1's H2D overlaps step k's kernels "
                        "and step k-1's D2H; no L2 flush (inputs arrive by copy every step)"},
        "gpu_launches": launches,
        "clocks": clocks,
        "wall_s_timed": t_wall,
    }
    if not args.no_configs:
        line["configs"] = configs_block(dev)
    if not args.no_geglu:
        line["geglu"] = geglu_block(dev)
    if not args.no_dtypes:
        line["dtypes"] = dtypes_block(dev)
    if not args.no_stack:
        line["stack"] = stack_block(dev)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    print(json.dumps(line))
    return 0


_JITTER = random.Random(20261203)


def phase_jitter():
    """Spin the device for a random 0-4095 clocks (0-2 us) before a start
    event.  CUDA event timestamps on GB300 advance in steps of 2.048 us; with
    the phase of the start fixed (an L2 flush of constant length before every
    call) the mean of many short intervals keeps that quantisation, with a
    random phase it does not."""
    import torch
    if hasattr(torch.cuda, "_sleep"):
        torch.cuda._sleep(_JITTER.randrange(0, 4096))


def _timed_mean(fn, stream, reps: int, flush):
    """Mean CUDA-event time (ms) of `fn` over `reps` calls, L2 flushed before
    each (a memset larger than L2, then a read, so the lines are clean) and
    the start phase randomised (phase_jitter).  The mean, not the median:
    event timestamps on GB300 advance in steps of 2.048 us, so the median of a
    call of a few microseconds is a whole number of steps, while the mean of
    many calls with random phases is not."""
    import torch
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    fn()
    ts = []
    for _ in range(reps):
        flush[0].zero_()
        flush[1].max()
        phase_jitter()
        e0, e1 = mk(), mk()
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.mean(ts)


def _stream_per_call(x, p, a, n, y, wsp, stream, calls: int = 64, copy_x: bool = False):
    """Per-call time (ms) of back-to-back nf4_linear calls, the way a model
    issues them one after another: call i reads copy i % c of the weight (and,
    with copy_x, of the activations), with c copies holding more than three
    times the L2, so no call finds its inputs in L2.  The calls are captured
    once in a CUDA graph and replayed between one pair of CUDA events, so
    neither the host's per-call launch work (argument checks, tensor-map
    encoding) nor the per-call events' own launch latency paces the device;
    consecutive kernels overlap launch and prologue through programmatic
    dependent launch, as they do in a model."""
    import torch
    import nf4_weight_quantized_quantize_gb300 as nf4
    l2 = getattr(torch.cuda.get_device_properties(x.device), "L2_cache_size", 128 << 20) or (128 << 20)
    wbytes = p.numel() + 4 * a.numel() + (x.numel() * x.element_size() if copy_x else 0)
    copies = max(2, -(-3 * l2 // wbytes))
    ps = [p.clone() for _ in range(copies)]
    am = [a.clone() for _ in range(copies)]
    xs = [x.clone() for _ in range(copies)] if copy_x else [x] * copies

    def run():
        for i in range(calls):
            nf4.linear(xs[i % copies], ps[i % copies], am[i % copies], n, out=y, workspace=wsp)

    run()   # first calls on this device set up the library's per-device state
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    graph.replay()
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    e0, e1 = mk(), mk()
    torch.cuda.synchronize()
    phase_jitter()
    e0.record(stream)
    graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / calls
    del graph, ps, am, xs
    return ms, copies, calls


def configs_block(dev, reps: int = 50):
    """Each workload's own figures: nf4_quantize and nf4_dequantize of its
    weight (GB/s of 2.5625 B per weight against the HBM peak) and nf4_linear
    at its batch -- TFLOP/s against the bf16 peak for M >= 128, GB/s of the
    algorithmic bytes (0.5625 B per weight + X + Y) against the HBM peak for
    the skinny batches.  Mean of `reps` calls, L2 flushed before each; the
    batches of the large weights also as a stream of back-to-back calls over
    distinct input copies (`_stream_per_call`)."""
    import torch
    import nf4_weight_quantized_quantize_gb300 as nf4

    stream = torch.cuda.current_stream(dev)
    flush = (torch.empty(512 << 20, dtype=torch.uint8, device=dev),
             torch.zeros(256 << 20, dtype=torch.uint8, device=dev))
    pk, pk_kind = peaks()
    out = {"timing": f"mean of {reps} calls, CUDA events (2.048 us timestamp steps), L2 flushed before each "
                     "(512 MiB memset + 256 MiB read)",
           "peaks": f"{pk_kind}: HBM {pk['hbm_gbs']} GB/s, bf16 {pk['bf16_tflops']} TFLOP/s"}
    cases = [(workloads.TINY, (workloads.TINY.m,)), (workloads.Q_PROJ, (workloads.Q_PROJ.m, SKINNY_M)),
             (workloads.GATE_UP, (workloads.GATE_UP.m, SKINNY_M)), (workloads.DOWN, (workloads.DOWN.m, SKINNY_M))]
    for cfg, batches in cases:
        w = workloads.make_weight(cfg, device=dev)
        numel = w.numel()
        p = torch.empty(numel // 2, dtype=torch.uint8, device=dev)
        a = torch.empty(numel // 64, dtype=torch.float32, device=dev)
        wd = torch.empty(numel, dtype=torch.bfloat16, device=dev)
        t_q = _timed_mean(lambda: nf4.quantize(w, out=(p, a)), stream, reps, flush)
        t_d = _timed_mean(lambda: nf4.dequantize(p, a, numel, out=wd), stream, reps, flush)
        del w, wd
        q_gbs = numel * BYTES_PER_W_QUANT / (t_q * 1e-3) / 1e9
        d_gbs = numel * BYTES_PER_W_DEQUANT / (t_d * 1e-3) / 1e9
        ent = {"N": cfg.n, "K": cfg.k,
               "nf4_quantize": {"ms": t_q, "GB/s": q_gbs, "frac_hbm": q_gbs / pk["hbm_gbs"]},
               "nf4_dequantize": {"ms": t_d, "GB/s": d_gbs, "frac_hbm": d_gbs / pk["hbm_gbs"]}}
        x_all = workloads.make_activation(cfg, device=dev)
        for m in batches:
            x = x_all[:m].contiguous()
            y = torch.empty(m, cfg.n, dtype=torch.bfloat16, device=dev)
            _, wsb = nf4.nf4_linear_workspace_size(m, cfg.n, cfg.k)
            wsp = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=dev)
            t = _timed_mean(lambda: nf4.linear(x, p, a, cfg.n, out=y, workspace=wsp), stream, reps, flush)
            tf = 2 * m * cfg.n * cfg.k / (t * 1e-3) / 1e12
            byts = numel * 0.5625 + 2 * m * cfg.k + 2 * m * cfg.n
            gbs = byts / (t * 1e-3) / 1e9
            e = {"ms": t, "TFLOP/s": tf, "GB/s": gbs, "bytes": byts}
            if m >= 128:
                e["frac_bf16"] = tf / pk["bf16_tflops"]
                if cfg.m >= 2048:
                    ms_s, copies, ncalls = _stream_per_call(x, p, a, cfg.n, y, wsp, stream, calls=32, copy_x=True)
                    tf_s = 2 * m * cfg.n * cfg.k / (ms_s * 1e-3) / 1e12
                    e["stream"] = {"ms_per_call": ms_s, "TFLOP/s": tf_s, "frac_bf16": tf_s / pk["bf16_tflops"],
                                   "input_copies": copies, "calls": ncalls,
                                   "how": "back-to-back calls over distinct weight and activation copies (> 3x "
                                          "L2 in all), replayed as one CUDA graph between one pair of events: "
                                          "the per-call time of layers run one after another, without the "
                                          "launch latency a lone call between events pays"}
            else:
                e["frac_hbm"] = gbs / pk["hbm_gbs"]
                if numel * 0.5625 >= 4e6:   # a weight L2 cannot hold three times over in a few copies
                    ms_s, copies, ncalls = _stream_per_call(x, p, a, cfg.n, y, wsp, stream)
                    g_s = byts / (ms_s * 1e-3) / 1e9
                    e["stream"] = {"ms_per_call": ms_s, "GB/s": g_s, "frac_hbm": g_s / pk["hbm_gbs"],
                                   "weight_copies": copies, "calls": ncalls,
                                   "how": "back-to-back calls over distinct weight copies (> 3x L2 in all), "
                                          "replayed as one CUDA graph between one pair of events: the "
                                          "per-call time of a decode loop"}
            ent[f"nf4_linear_m{m}"] = e
            del x, y, wsp
        out[cfg.name.replace(f"_m{cfg.m}", "")] = ent
        del x_all, p, a
        torch.cuda.empty_cache()
    if nf4.nf4_last_error(stream.cuda_stream) != nf4.NF4_OK:
        raise RuntimeError("a kernel reported a timeout in the per-workload measurement")
    del flush
    torch.cuda.empty_cache()
    return out


def geglu_block(dev, reps: int = 20):
    """The Gemma3 MLP's gate and up projections as one fused call
    (nf4_linear_geglu: [2F, K] NF4 weight, gelu_tanh(gate) * up written as
    [M, F]) against nf4_linear over the same stacked weight (both projections'
    outputs written, [M, 2F], the activation left to another kernel), at
    M = 2048 and M = 16.  Mean of `reps` calls, L2 flushed before each."""
    import torch
    import nf4_weight_quantized_quantize_gb300 as nf4

    cfg = workloads.GATE_UP
    F = cfg.n // 2
    stream = torch.cuda.current_stream(dev)
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    w = workloads.make_weight(cfg, device=dev)
    p, a = nf4.quantize(w)
    del w
    x = workloads.make_activation(cfg, device=dev)
    xs = x[:SKINNY_M].contiguous()
    y2 = torch.empty(cfg.m, 2 * F, dtype=torch.bfloat16, device=dev)
    y1 = torch.empty(cfg.m, F, dtype=torch.bfloat16, device=dev)
    _, wsb = nf4.nf4_linear_workspace_size(SKINNY_M, 2 * F, cfg.k)
    wsp = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    def timed(fn):
        fn()
        ev = [(mk(), mk()) for _ in range(reps)]
        for e0, e1 in ev:
            flush.zero_()
            phase_jitter()
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)

    t_fused = timed(lambda: nf4.linear_geglu(x, p, a, F, out=y1))
    t_plain = timed(lambda: nf4.linear(x, p, a, 2 * F, out=y2))
    t_fused_s = timed(lambda: nf4.linear_geglu(xs, p, a, F, out=y1[:SKINNY_M], workspace=wsp))
    t_plain_s = timed(lambda: nf4.linear(xs, p, a, 2 * F, out=y2[:SKINNY_M], workspace=wsp))
    if nf4.nf4_last_error(stream.cuda_stream) != nf4.NF4_OK:
        raise RuntimeError("a kernel reported a timeout in the gate/up measurement")
    pk, _ = peaks()
    flop = 2 * cfg.m * 2 * F * cfg.k
    tf = lambda ms: flop / (ms * 1e-3) / 1e12  # noqa: E731
    del p, a, x, xs, y1, y2, wsp, flush
    torch.cuda.empty_cache()
    return {
        "workload": f"gemma3_12b_gate_up_pair_F{F}_K{cfg.k}",
        "m2048": {"fused_ms": t_fused, "fused_TFLOP/s": tf(t_fused), "frac_bf16": tf(t_fused) / pk["bf16_tflops"],
                  "unfused_linear_ms": t_plain, "unfused_linear_TFLOP/s": tf(t_plain),
                  "output_bytes_fused": cfg.m * F * 2, "output_bytes_unfused": cfg.m * 2 * F * 2},
        "m16": {"fused_ms": t_fused_s, "unfused_linear_ms": t_plain_s},
        "timing": f"mean of {reps} calls, CUDA events, 512 MiB L2 flush before each",
    }


def dtypes_block(dev, reps: int = 20):
    """The three compute dtypes on the q_proj workload (W [4096, 3840], X
    [2048, 3840]): nf4_quantize_ex, nf4_dequantize_ex and nf4_linear_ex, mean
    of `reps` calls with the L2 flushed before each.  Bytes per weight:
    quantize e + 0.5625, dequantize 0.5625 + e (e = 2 for bf16 / fp16, 4 for
    fp32).  The fp32 linear runs on the tf32 tensor cores; its peak is the
    measured bf16 peak times the nominal dense tf32 : bf16 ratio 1.1 : 2.25."""
    import torch
    import nf4_weight_quantized_quantize_gb300 as nf4

    cfg = CFG
    stream = torch.cuda.current_stream(dev)
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    pk, pk_kind = peaks()
    out = {"workload": cfg.name, "timing": f"mean of {reps} calls, CUDA events, 512 MiB L2 flush before each"}

    def timed(fn):
        fn()
        ev = [(mk(), mk()) for _ in range(reps)]
        for e0, e1 in ev:
            flush.zero_()
            phase_jitter()
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)

    for name, dt in (("bf16", torch.bfloat16), ("f16", torch.float16), ("f32", torch.float32)):
        eb = torch.tensor([], dtype=dt).element_size()
        w = workloads.make_weight(cfg, device=dev, dtype=dt)
        x = workloads.make_activation(cfg, device=dev, dtype=dt)
        numel = w.numel()
        p = torch.empty(numel // 2, dtype=torch.uint8, device=dev)
        a = torch.empty(numel // 64, dtype=torch.float32, device=dev)
        wd = torch.empty(numel, dtype=dt, device=dev)
        y = torch.empty(cfg.m, cfg.n, dtype=dt, device=dev)
        t_q = timed(lambda: nf4.quantize(w, out=(p, a)))
        t_d = timed(lambda: nf4.dequantize(p, a, numel, out=wd))
        t_l = timed(lambda: nf4.linear(x, p, a, cfg.n, out=y))
        tf = 2 * cfg.m * cfg.n * cfg.k / (t_l * 1e-3) / 1e12
        peak = pk["bf16_tflops"] * (1.1 / 2.25 if name == "f32" else 1.0)
        out[name] = {
            "quantize": {"ms": t_q, "GB/s": numel * (eb + 0.5625) / (t_q * 1e-3) / 1e9},
            "dequantize": {"ms": t_d, "GB/s": numel * (0.5625 + eb) / (t_d * 1e-3) / 1e9},
            "linear_m2048": {"ms": t_l, "TFLOP/s": tf, "frac_peak": tf / peak,
                             "peak": ("tf32 = bf16 x 1.1/2.25 (nominal ratio), " if name == "f32" else "bf16, ")
                             + f"of {pk_kind}"},
        }
        for k in ("quantize", "dequantize"):
            out[name][k]["frac_hbm"] = out[name][k]["GB/s"] / pk["hbm_gbs"]
        del w, x, p, a, wd, y
    if nf4.nf4_last_error(stream.cuda_stream) != nf4.NF4_OK:
        raise RuntimeError("a kernel reported a timeout in the dtype measurement")
    del flush
    torch.cuda.empty_cache()
    return out


def stack_block(dev, passes: int = 2):
    """The 48-layer Gemma3-12B projection stack: every one of the 336 weights
    quantized once (the one-time cost the pages quote as 52 s), then timed
    passes of nf4_linear at M = 8192 over all 336 projections and of the bulk
    nf4_dequantize of all 336 weights.  Weights, their NF4 form and the seeded
    activations stay resident in HBM; outputs go to one reused buffer per kind."""
    import torch
    import nf4_weight_quantized_quantize_gb300 as nf4

    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    stream = torch.cuda.current_stream(dev)
    entries, q_ms, params = [], 0.0, 0
    for layer in range(workloads.LAYERS):
        for pi in range(len(workloads.PROJECTIONS)):
            cfg = workloads.stack_layer(layer, pi)
            w = workloads.make_weight(cfg, device=dev)
            p = torch.empty(w.numel() // 2, dtype=torch.uint8, device=dev)
            a = torch.empty(w.numel() // 64, dtype=torch.float32, device=dev)
            e0, e1 = mk(), mk()
            e0.record(stream)
            nf4.quantize(w, out=(p, a))
            e1.record(stream)
            x = workloads.make_activation(cfg, device=dev)
            entries.append((cfg, x, p, a, (e0, e1)))
            params += w.numel()
            del w
    torch.cuda.synchronize()
    q_ms = sum(e[4][0].elapsed_time(e[4][1]) for e in entries)
    y = torch.empty(max(c.m * c.n for c, *_ in entries), dtype=torch.bfloat16, device=dev)
    deq = torch.empty(max(c.n * c.k for c, *_ in entries), dtype=torch.bfloat16, device=dev)
    flops = sum(2 * c.m * c.n * c.k for c, *_ in entries)

    def linear_pass():
        for c, x, p, a, _ in entries:
            nf4.linear(x, p, a, c.n, out=y[: c.m * c.n].view(c.m, c.n))

    def dequant_pass():
        for c, x, p, a, _ in entries:
            nf4.dequantize(p, a, c.n * c.k, out=deq[: c.n * c.k])

    def timed(run):
        times = []
        for _ in range(passes):
            e0, e1 = mk(), mk()
            torch.cuda.synchronize()
            e0.record(stream)
            run()
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        return min(times)

    res, res_graph, clocks = {}, {}, {}
    for name, fn in (("linear", linear_pass), ("dequantize", dequant_pass)):
        fn()                                  # warm: descriptors, kernel attributes
        res[name] = timed(fn)
        # the same 336 launches captured once as a CUDA graph and replayed:
        # no host launch gaps between the short kernels
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
        graph.replay()
        # clocks and clock-event reasons during the graph passes: a pass is
        # long enough (about 0.1 s for the linear) to meet the power cap
        sampler = ClockSampler(dev.index if dev.index is not None else 0)
        sampler.start()
        res_graph[name] = timed(graph.replay)
        sampler.stop()
        clocks[name] = sampler.summary()
        del graph
    if nf4.nf4_last_error(stream.cuda_stream) != nf4.NF4_OK:
        raise RuntimeError("a kernel reported a timeout in the stack passes")
    pk, _ = peaks()
    deq_bytes = params * BYTES_PER_W_DEQUANT
    lin_tf = lambda ms: flops / (ms * 1e-3) / 1e12  # noqa: E731
    deq_gbs = lambda ms: deq_bytes / (ms * 1e-3) / 1e9  # noqa: E731
    out = {
        "workload": f"gemma3_12b_48_layers_x_7_projections_m{workloads.STACK_M}",
        "weights": len(entries), "params": params,
        "linear": {"ms": res_graph["linear"], "TFLOP/s": lin_tf(res_graph["linear"]),
                   "frac_bf16": lin_tf(res_graph["linear"]) / pk["bf16_tflops"], "flop": flops,
                   "frac_bf16_sustained": lin_tf(res_graph["linear"]) / pk["bf16_tflops_sustained"],
                   "eager": {"ms": res["linear"], "TFLOP/s": lin_tf(res["linear"])},
                   "clocks": clocks["linear"]},
        "dequantize": {"ms": res_graph["dequantize"], "GB/s": deq_gbs(res_graph["dequantize"]),
                       "frac_hbm": deq_gbs(res_graph["dequantize"]) / pk["hbm_gbs"], "bytes": deq_bytes,
                       "eager": {"ms": res["dequantize"], "GB/s": deq_gbs(res["dequantize"])},
                       "clocks": clocks["dequantize"]},
        "quantize_once": {"ms": q_ms, "GB/s": params * BYTES_PER_W_QUANT / (q_ms * 1e-3) / 1e9,
                          "pages_one_time_s": 52.0},
        "timing": (f"best of {passes} passes, CUDA events around the whole pass; each pass is the 336 "
                   "calls replayed as one captured CUDA graph ('eager': the same calls launched one by "
                   "one from Python); working set > L2"),
    }
    del entries, y, deq
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="omit the CPU oracle timing")
    ap.add_argument("--no-stack", action="store_true", help="omit the 48-layer stack measurement")
    ap.add_argument("--no-configs", action="store_true", help="omit the per-workload measurement")
    ap.add_argument("--no-geglu", action="store_true", help="omit the fused gate/up measurement")
    ap.add_argument("--no-dtypes", action="store_true", help="omit the fp16 / fp32 measurement")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
