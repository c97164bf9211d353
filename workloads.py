"""Seeded synthetic inputs for the NF4 linear workloads.

This module only draws random tensors: it holds none of the quantization,
dequantization or matmul arithmetic, so both the CUDA path and the CPU oracle
may take their inputs from it.

The shapes are the Gemma3-12B text-encoder projections (hidden 3840, 48
layers, seven projections per layer: q 3840->4096, k and v 3840->2048,
o 4096->3840, gate and up 3840->15360, down 15360->3840).  Activation rows are
prompts x tokens: two prompts (classifier-free guidance, positive and
negative) of 1024 tokens give M = 2048; the stack workload uses eight prompts
(M = 8192).  Weights are N(0, 0.02) cast to bf16, activations N(0, 1) cast to
bf16.  No trained weights are involved.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

HIDDEN = 3840
LAYERS = 48
# (name, out_features N, in_features K) of one Gemma3-12B decoder layer.
PROJECTIONS = (
    ("q", 4096, 3840),
    ("k", 2048, 3840),
    ("v", 2048, 3840),
    ("o", 3840, 4096),
    ("gate", 15360, 3840),
    ("up", 15360, 3840),
    ("down", 3840, 15360),
)


@dataclass(frozen=True)
class Linear:
    """One NF4 linear problem: W [n, k] quantized, X [m, k], Y = X W^T [m, n]."""
    name: str
    m: int
    n: int
    k: int
    w_seed: int
    x_seed: int
    outlier_frac: float = 0.0   # fraction of W entries multiplied by 20 before the bf16 cast
    w_std: float = 0.02
    x_rows: int = 0             # rows drawn for X (0: m); X keeps the first m of them


# The five workloads, each described by what it is.
TINY = Linear("tiny_256x512_m16", 16, 256, 512, w_seed=0, x_seed=0)
Q_PROJ = Linear("gemma3_12b_q_proj_m2048", 2048, 4096, 3840, w_seed=1, x_seed=101)
GATE_UP = Linear("gemma3_12b_gate_up_m2048", 2048, 2 * 15360, 3840, w_seed=2, x_seed=102,
                 outlier_frac=0.001)
DOWN = Linear("gemma3_12b_down_proj_m2048", 2048, 3840, 15360, w_seed=3, x_seed=103)
# Skinny batch on the same weight: its 16 rows are the first 16 rows of DOWN's X.
DOWN_SKINNY = Linear("gemma3_12b_down_proj_m16", 16, 3840, 15360, w_seed=3, x_seed=103,
                     x_rows=2048)
STACK_M = 8192


def stack_layer(layer: int, proj_idx: int, m: int = STACK_M) -> Linear:
    """Projection `proj_idx` of decoder layer `layer` in the 48-layer stack."""
    name, n, k = PROJECTIONS[proj_idx]
    return Linear(f"gemma3_12b_l{layer}_{name}_m{m}", m, n, k,
                  w_seed=10000 + 10 * layer + proj_idx, x_seed=20000 + 10 * layer + proj_idx)


def for_replica(cfg: Linear, rank: int) -> Linear:
    """The workload as replica `rank` of a batch-parallel run draws it: the same
    weight (one model, replicated) and its own prompts (X seed + 1000 rank)."""
    return replace(cfg, name=f"{cfg.name}_rank{rank}" if rank else cfg.name, x_seed=cfg.x_seed + 1000 * rank)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_weight(cfg: Linear, device="cpu", rows: slice | None = None, dtype=torch.bfloat16) -> torch.Tensor:
    """W [n, k] for `cfg`, drawn in fp32 and cast to `dtype` (bf16 by default;
    the same tensor on every call with the same device)."""
    g = _gen(cfg.w_seed, device)
    w = torch.randn(cfg.n, cfg.k, generator=g, device=device, dtype=torch.float32)
    w.mul_(cfg.w_std)
    if cfg.outlier_frac > 0:
        mask = torch.rand(cfg.n, cfg.k, generator=g, device=device) < cfg.outlier_frac
        w[mask] *= 20.0
    w = w.to(dtype)
    return w if rows is None else w[rows].contiguous()


def make_activation(cfg: Linear, device="cpu", dtype=torch.bfloat16) -> torch.Tensor:
    """X [m, k] of `dtype` (bf16 by default): `x_rows` (default m) rows are drawn
    and the first m kept, so a skinny batch is a prefix of the full batch drawn
    with the same seed."""
    g = _gen(cfg.x_seed, device)
    rows = max(cfg.m, cfg.x_rows)
    x = torch.randn(rows, cfg.k, generator=g, device=device, dtype=torch.float32)
    x = x.to(dtype)
    return x[: cfg.m].contiguous()


def bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")


def from_bits(a, device="cpu") -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 tensor."""
    import numpy as np
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def host(t: torch.Tensor):
    """A tensor as the oracle takes it: numpy uint16 bit patterns for bf16 and
    fp16, float32 values for fp32 (host copy)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.float32:
        return t.numpy()
    return t.view(torch.int16).numpy().view("uint16")


def from_host(a, dtype, device="cpu") -> torch.Tensor:
    """The inverse of host(): numpy data of the oracle's storage -> tensor of `dtype`."""
    import numpy as np
    a = np.ascontiguousarray(a)
    if dtype == torch.float32:
        return torch.from_numpy(a.astype(np.float32)).to(device)
    return torch.from_numpy(a.view(np.int16)).view(dtype).to(device)
