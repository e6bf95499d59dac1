"""Seeded random shapes through the dispatcher against the oracle.

Each case draws a storage type, M, K (aligned or not to the type's 16-byte chunk,
K = 0 included), B (up to 16, and up to 64 for fp16/bf16) and a bias, runs the
library's default plan, and checks y against the oracle and a repeat bit for bit.
The draws are fixed by the seed, so a failure names a reproducible case.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import decode_linear_layers_gb300 as g
import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

VEC = {"f32": 4, "f16": 8, "bf16": 8, "w8": 16, "w4": 32}


def _cases(n=192, seed=2027):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        dt = ["f32", "f16", "bf16", "w8", "w4"][int(rng.integers(5))]
        M = int(rng.choice([rng.integers(1, 64), rng.integers(64, 1500), rng.integers(1500, 6000)]))
        vec = VEC[dt]
        if dt == "w4":
            K = 128 * int(rng.integers(0, 40))
        else:
            K = int(rng.integers(0, 700)) * vec
            if rng.random() < 0.25:
                K += int(rng.integers(1, vec))  # rows no longer 16-byte aligned
        bmax = 64 if dt in ("f16", "bf16") else 16
        B = int(rng.choice([rng.integers(1, 5), rng.integers(1, 17), rng.integers(1, bmax + 1)]))
        if rng.random() < 0.06:
            K = 0  # the empty sum: y = bias
        if B > 16:
            K -= K % vec  # more than 16 vectors: the tensor cores need 16-byte rows
        # keep the oracle quick: at most ~40 M multiply-adds per case
        while M * max(K, 1) * B > 40_000_000 and M > 1:
            M //= 2
        out.append((i, dt, M, K, B, bool(rng.random() < 0.5)))
    return out


@pytest.mark.parametrize("case", _cases(), ids=lambda c: f"{c[0]}-{c[1]}-{c[2]}x{c[3]}-B{c[4]}")
def test_random_shape(case):
    _, dtype, M, K, B, bias = case
    w = W.small(dtype, M, K, B, bias, seed=case[0] + 9000)
    inp = W.make_inputs(w)
    y_ref, absdot = U.oracle_for(dtype, inp)
    d = U.to_device(inp)
    y1 = U.run_gpu(dtype, d, M, K, B)
    plan = g.last_plan()
    y2 = U.run_gpu(dtype, d, M, K, B)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2), "results differ between two identical calls"
    U.assert_close(dtype, y1, y_ref, absdot, with_rounding=True,
                   what=f"{dtype} {M}x{K} B={B} bias={bias} [{plan['kernel_name']}/{plan['variant']}]")
