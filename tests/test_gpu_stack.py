"""The 48-layer Gemma3-12B projection stack through nf4_linear.

Every one of the 336 projections (48 layers x q, k, v, o, gate, up, down) is
quantized on the GPU and multiplied by its own seeded activations at
M = 8192 (eight 1024-token prompts).  Each product is checked on 8 x 8
seeded (row, column) samples against the oracle, which quantizes the sampled
weight rows itself from the generator's weights: since a block never
straddles a row (K % 64 == 0), the oracle's bytes for those rows are the
bytes the GPU multiplies.  The bound per element is bf16 output rounding plus
fp32 summation error.  (The bulk quantize/dequantize of all 336 weights is
checked in test_gpu_quant.)
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import nf4_weight_quantized_quantize_gb300 as nf4

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def f32_of_bits(b):
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def test_stack_linear_sampled():
    rs = np.random.default_rng(48)
    worst = 0.0
    for layer in range(workloads.LAYERS):
        for pi in range(len(workloads.PROJECTIONS)):
            cfg = workloads.stack_layer(layer, pi)
            w = workloads.make_weight(cfg, device=DEV)
            x = workloads.make_activation(cfg, device=DEV)
            p, a = nf4.quantize(w)
            y = nf4.linear(x, p, a, cfg.n)
            mi = np.sort(rs.choice(cfg.m, 8, replace=False))
            ni = np.sort(rs.choice(cfg.n, 8, replace=False))
            wb = workloads.bits(w[torch.from_numpy(ni).to(DEV)])
            xb = workloads.bits(x[torch.from_numpy(mi).to(DEV)])
            pr, ar = oracle.quantize(wb)
            yref = oracle.linear(xb, pr, ar, 8)
            yg = y[torch.from_numpy(mi).to(DEV)][:, torch.from_numpy(ni).to(DEV)].float().cpu().numpy()
            wd = f32_of_bits(oracle.dequantize(pr, ar, wb.size)).astype(np.float64).reshape(8, cfg.k)
            mag = np.abs(f32_of_bits(xb).astype(np.float64)) @ np.abs(wd).T
            bound = 2.0 ** -8 * np.abs(yref) + cfg.k * 2.0 ** -23 * mag + 1e-30
            err = np.abs(yg - yref)
            assert np.all(err <= bound), (layer, pi, float(np.max(err / bound)))
            worst = max(worst, float(np.max(err / bound)))
            del w, x, p, a, y
    assert nf4.nf4_last_error(torch.cuda.current_stream().cuda_stream) == nf4.NF4_OK
    assert worst <= 1.0
