"""Helpers shared by the GPU parity tests: run libgemv and the oracle on one input.

The oracle runs on the CPU over the same stored values the GPU reads; the GPU
result is compared element by element under the tolerance the spec gives:

    fp32:            |y - y_ref| <= 1e-5 * sum_k |s_m A_mk x_k| + 1e-6
    fp16/bf16/w8:    |y - y_ref| <= 2e-3 * sum_k |s_m A_mk x_k| + 1e-3

(the bound covers fp32 accumulation and the final rounding to the output type).
For small edge cases whose rows can be dominated by the bias, ``with_rounding``
adds the output type's unit roundoff times |y_ref| (2^-11 for fp16, 2^-8 for
bf16, 2^-24 for fp32): the bound above has no |bias| term.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import decode_linear_layers_gb300 as g
import oracle
import workloads as W

TOL = {"f32": (1e-5, 1e-6), "f16": (2e-3, 1e-3), "bf16": (2e-3, 1e-3), "w8": (2e-3, 1e-3),
       "w4": (2e-3, 1e-3)}
U_OUT = {"f32": 2.0 ** -24, "f16": 2.0 ** -11, "bf16": 2.0 ** -8, "w8": 2.0 ** -8, "w4": 2.0 ** -8}


def threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def oracle_for(w_dtype: str, inp: dict):
    return oracle.gemv(w_dtype, W.storage_bits(inp["A"]), W.storage_bits(inp["x"]),
                       W.storage_bits(inp["bias"]), None if inp["scale"] is None else inp["scale"].numpy(),
                       nthreads=threads())


def to_device(inp: dict, dev="cuda") -> dict:
    return {k: (None if v is None else v.to(dev)) for k, v in inp.items()}


def out_dtype(dtype: str):
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16, "w8": torch.bfloat16,
            "w4": torch.bfloat16}[dtype]


def call(dtype: str, d: dict, y: torch.Tensor, M: int, K: int, B: int, stream=None):
    if dtype == "w8":
        g.gemv_w8(d["A"], d["scale"], d["x"], d["bias"], y, M, K, B, stream)
    elif dtype == "w4":
        g.gemv_w4(d["A"], d["scale"], d["x"], d["bias"], y, M, K, B, stream)
    else:
        getattr(g, f"gemv_{dtype}")(d["A"], d["x"], d["bias"], y, M, K, B, stream)


def run_gpu(dtype: str, d: dict, M: int, K: int, B: int, stream=None) -> torch.Tensor:
    y = torch.empty((B, M), dtype=out_dtype(dtype), device="cuda")
    call(dtype, d, y, M, K, B, stream)
    return y


def assert_close(dtype: str, y: torch.Tensor, y_ref: np.ndarray, absdot: np.ndarray,
                 with_rounding: bool = False, what: str = ""):
    got = y.detach().double().cpu().numpy().reshape(y_ref.shape)
    rel, ab = TOL[dtype]
    bound = rel * absdot + ab
    if with_rounding:
        bound = bound + U_OUT[dtype] * np.abs(y_ref)
    nan_ref = np.isnan(y_ref)
    assert np.array_equal(np.isnan(got), nan_ref), f"{what}: NaN positions differ"
    inf_ref = np.isinf(y_ref)
    assert np.array_equal(got[inf_ref], y_ref[inf_ref]), f"{what}: infinities differ"
    fin = ~(nan_ref | inf_ref)
    err = np.abs(got[fin] - y_ref[fin])
    bad = err > bound[fin]
    if bad.any():
        i = int(np.argmax(err - bound[fin]))
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outputs out of tolerance; worst err "
            f"{err[i]:.3e} > bound {bound[fin][i]:.3e} (got {got[fin][i]!r}, ref {y_ref[fin][i]!r})")
    return float((err / bound[fin]).max()) if err.size else 0.0


SILU_LIP = 1.1  # max |d silu / dv| is 1.0998 (at v ~ 2.40)
F32_SLACK = 4e-7  # fp32 expf and division in the GPU's silu, relative


def assert_close_ex(dtype, y, y_ref, absdot, act: int, what: str = ""):
    """Fused epilogue: the GEMV bound through SiLU's Lipschitz constant, plus the
    output rounding and the fp32 activation's own rounding."""
    rel, ab = TOL[dtype]
    bound = (SILU_LIP if act else 1.0) * (rel * absdot + ab)
    bound = bound + (U_OUT[dtype] + F32_SLACK) * np.abs(y_ref)
    _compare(y, y_ref, bound, what)


def assert_close_swiglu(dtype, y, y_ref, gate, up, adg, adu, what: str = ""):
    """silu(g) * u with g, u each within the GEMV bound: |d| <= L tg (|u| + tu) + |silu(g)| tu."""
    rel, ab = TOL[dtype]
    tg, tu = rel * adg + ab, rel * adu + ab
    sg = gate / (1.0 + np.exp(-gate))
    bound = SILU_LIP * tg * (np.abs(up) + tu) + np.abs(sg) * tu
    bound = bound + (U_OUT[dtype] + F32_SLACK) * np.abs(y_ref)
    _compare(y, y_ref, bound, what)


def _compare(y, y_ref, bound, what):
    got = y.detach().double().cpu().numpy().reshape(y_ref.shape)
    assert np.array_equal(np.isnan(got), np.isnan(y_ref)), f"{what}: NaN positions differ"
    fin = np.isfinite(y_ref)
    err = np.abs(got[fin] - y_ref[fin])
    bad = err > bound[fin]
    if bad.any():
        i = int(np.argmax(err - bound[fin]))
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} out of tolerance; worst err "
                             f"{err[i]:.3e} > bound {bound[fin][i]:.3e} (got {got[fin][i]!r}, ref {y_ref[fin][i]!r})")
