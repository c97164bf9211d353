"""Run one library call on a named synthetic workload a few times (for profiling).

    python run_case.py \
        --workload gemma3_12b_gate_up_m2048 --op linear --iters 3

--op is one of quantize, dequantize, linear, linear_geglu (the workload's
weight read as a stacked gate/up pair, F = N / 2); --dtype the compute dtype
of weights, activations and outputs (bf16, f16, f32); --m the number of activation
rows of a linear (default the workload's own, e.g. 16 for a skinny batch on a
larger weight).  The workloads are the seeded
Gemma3-12B projection shapes of workloads.py; inputs are generated on the
device.  Prints the median CUDA-event time of the calls.
"""
from __future__ import annotations

import argparse
import os
import statistics
import sys

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main(argv=None):
    import torch

    import workloads
    import nf4_weight_quantized_quantize_gb300 as nf4

    cases = {c.name: c for c in (workloads.TINY, workloads.Q_PROJ, workloads.GATE_UP, workloads.DOWN,
                                 workloads.DOWN_SKINNY)}
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", choices=sorted(cases), default=workloads.GATE_UP.name)
    ap.add_argument("--op", choices=["quantize", "dequantize", "linear", "linear_geglu"], default="linear")
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--dtype", choices=["bf16", "f16", "f32"], default="bf16")
    ap.add_argument("--m", type=int, default=None, help="activation rows (default: the workload's)")
    a = ap.parse_args(argv)
    cfg = cases[a.workload]
    m = cfg.m if a.m is None else a.m
    dev = torch.device("cuda", 0)
    dt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[a.dtype]
    w = workloads.make_weight(cfg, device=dev, dtype=dt)
    packed, absmax = nf4.quantize(w)
    if a.op == "quantize":
        fn = lambda: nf4.quantize(w, out=(packed, absmax))  # noqa: E731
    elif a.op == "dequantize":
        out = torch.empty(w.numel(), dtype=dt, device=dev)
        fn = lambda: nf4.dequantize(packed, absmax, w.numel(), out=out)  # noqa: E731
    elif a.op == "linear_geglu":
        x = workloads.make_activation(cfg, device=dev, dtype=dt)[:m].contiguous()
        y = torch.empty(m, cfg.n // 2, dtype=dt, device=dev)
        _, wsb = nf4.nf4_linear_workspace_size(m, cfg.n, cfg.k)
        ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=dev)
        fn = lambda: nf4.linear_geglu(x, packed, absmax, cfg.n // 2, out=y, workspace=ws)  # noqa: E731
    else:
        x = workloads.make_activation(cfg, device=dev, dtype=dt)[:m].contiguous()
        y = torch.empty(m, cfg.n, dtype=dt, device=dev)
        _, wsb = nf4.nf4_linear_workspace_size(m, cfg.n, cfg.k)
        ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=dev)
        fn = lambda: nf4.linear(x, packed, absmax, cfg.n, out=y, workspace=ws)  # noqa: E731
    ts = []
    for _ in range(a.iters):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        torch.cuda.synchronize()
        ts.append(s.elapsed_time(e))
    st = nf4.nf4_last_error(torch.cuda.current_stream().cuda_stream)
    if st != nf4.NF4_OK:
        raise SystemExit(f"kernel error: {nf4.nf4_status_string(st)}")
    print(f"{cfg.name} {a.op} {a.dtype} M={m}: median {statistics.median(ts):.4f} ms over {a.iters}")
    return 0


if __name__ == "__main__":
    sys.exit(main())
