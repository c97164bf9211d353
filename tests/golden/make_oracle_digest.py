"""Write oracle_digest.json: SHA-256 digests of the oracle's outputs on small
seeded inputs, so that a later change in the oracle's results, or a platform
on which it computes differently, shows up as a failed test.

It calls only the oracle (and numpy/torch to draw and cast inputs).  Run it
from the repository root:  python tests/golden/make_oracle_digest.py
"""
import hashlib
import json
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402

CASES = [  # (name, n, k, m, seed, w_std)
    ("w64x256_m8", 64, 256, 8, 1234, 0.02),
    ("w96x192_m5", 96, 192, 5, 4321, 1.0),
]


def inputs(n, k, m, seed, w_std):
    rs = np.random.default_rng(seed)
    w = torch.from_numpy((rs.standard_normal((n, k)) * w_std).astype(np.float32))
    x = torch.from_numpy(rs.standard_normal((m, k)).astype(np.float32))
    wb = w.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xb = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return wb, xb


def digest(a):
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def compute():
    out = {}
    for name, n, k, m, seed, std in CASES:
        w, x = inputs(n, k, m, seed, std)
        p, a = oracle.quantize(w)
        y = oracle.dequantize(p, a, w.size)
        lin = oracle.linear(x, p, a, n)
        out[name] = {
            "input_w": digest(w), "input_x": digest(x),
            "packed": digest(p), "absmax": digest(a), "dequant": digest(y),
            # fp64 sums may differ in the last bits across compilers: store rounded values
            "linear_first_row": [float(f"{v:.12e}") for v in lin[0, :8]],
        }
    return out


if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_digest.json")
    with open(path, "w") as f:
        json.dump(compute(), f, indent=1, sort_keys=True)
    print("wrote", path)
