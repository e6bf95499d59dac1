"""Seeded synthetic inputs and byte/flop accounting for dense GEMV workloads.

This module is shared by the GPU parity tests, the benchmark and the CPU oracle's
tests. It holds input recipes and roofline bookkeeping only: none of the
matrix-vector arithmetic lives here, and it imports neither the CUDA binding nor
the oracle.

Operation being fed: y[b][m] = s_m * sum_k A[m][k] * x[b][k] + bias[m], A row-major
M x K, x B x K row-major, y B x M row-major ("16-sgemv" notes, problem definition;
"GEMV and row-level parallelism" lesson, section 1, y = A x + bias).

Random numbers come from numpy's PCG64, cut into blocks of 2**22 elements; block j
of stream s under seed q is seeded with SeedSequence([q, s, j]), so the values do
not depend on the number of threads that fill them or on the machine. Draws are
made in fp32 and then rounded to the storage dtype with round-to-nearest-even.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

_BLOCK = 1 << 22

# stream ids: one independent stream per tensor role
_S_A, _S_X, _S_BIAS, _S_SCALE = 1, 2, 3, 4

DTYPES = ("f32", "f16", "bf16", "w8")
W4_GROUP = 128  # int4: elements of a row per scale

# storage element sizes in bytes: (A, x, y, bias)
ELEM_BYTES = {
    "f32": (4, 4, 4, 4),
    "f16": (2, 2, 2, 2),
    "bf16": (2, 2, 2, 2),
    "w8": (1, 2, 2, 2),
    "w4": (0.5, 2, 2, 2),   # two int4 per byte
}


def _threads() -> int:
    try:
        return max(1, min(16, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(16, os.cpu_count() or 1))


def _fill(n: int, seed: int, stream: int, draw) -> np.ndarray:
    """Fill an fp32 (or int8) array of n elements block by block."""
    out = None

    def one(j):
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, j])))
        s = j * _BLOCK
        e = min(n, s + _BLOCK)
        return draw(g, e - s, out[s:e])

    kind = draw(None, 0, None)  # returns the dtype to allocate
    out = np.empty(n, dtype=kind)
    nblk = (n + _BLOCK - 1) // _BLOCK
    if nblk <= 1:
        for j in range(nblk):
            one(j)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(one, range(nblk)))
    return out


def normal(n: int, sigma: float, seed: int, stream: int) -> np.ndarray:
    """n draws of N(0, sigma^2) as fp32 (sigma applied in fp32)."""
    def draw(g, m, o):
        if g is None:
            return np.float32
        g.standard_normal(m, dtype=np.float32, out=o)
        if sigma != 1.0:
            o *= np.float32(sigma)
    return _fill(n, seed, stream, draw)


def uniform(n: int, lo: float, hi: float, seed: int, stream: int) -> np.ndarray:
    """n draws of U[lo, hi) as fp32: lo + (hi - lo) * u with u in [0, 1)."""
    def draw(g, m, o):
        if g is None:
            return np.float32
        g.random(m, dtype=np.float32, out=o)
        o *= np.float32(hi - lo)
        o += np.float32(lo)
    return _fill(n, seed, stream, draw)


def int8_uniform(n: int, lo: int, hi: int, seed: int, stream: int) -> np.ndarray:
    """n integers uniform on [lo, hi] (inclusive) as int8."""
    def draw(g, m, o):
        if g is None:
            return np.int8
        o[:] = g.integers(lo, hi + 1, size=m, dtype=np.int8)
    return _fill(n, seed, stream, draw)


_TORCH_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def to_storage(a: np.ndarray, dt: str) -> torch.Tensor:
    """fp32 numpy -> torch CPU tensor in the storage dtype (RNE rounding)."""
    t = torch.from_numpy(a)
    return t if dt == "f32" else t.to(_TORCH_DT[dt])


@dataclasses.dataclass(frozen=True)
class Workload:
    """One GEMV problem: shapes, storage dtype and input distributions."""
    name: str
    dtype: str            # "f32" | "f16" | "bf16" | "w8" | "w4"
    M: int
    K: int
    B: int
    bias: bool
    a_dist: tuple         # ("normal", sigma) | ("uniform", lo, hi) | ("int8", lo, hi) | ("bytes",)
    x_dist: tuple
    bias_dist: tuple = ("normal", 1.0)
    scale_dist: tuple = ("uniform", 1e-3, 1e-2)   # w8 (per row), w4 (per group)
    seed: int = 0

    @property
    def qmin_bytes(self) -> int:
        return qmin_bytes(self.dtype, self.M, self.K, self.B)

    @property
    def full_bytes(self) -> int:
        return full_bytes(self.dtype, self.M, self.K, self.B, self.bias)

    @property
    def flops(self) -> int:
        return flops(self.M, self.K, self.B)


def _draw(dist: tuple, n: int, seed: int, stream: int) -> np.ndarray:
    kind = dist[0]
    if kind == "normal":
        return normal(n, dist[1], seed, stream)
    if kind == "uniform":
        return uniform(n, dist[1], dist[2], seed, stream)
    if kind == "int8":
        return int8_uniform(n, dist[1], dist[2], seed, stream)
    if kind == "bytes":  # uniform storage bytes: for int4, both nibbles uniform in [-8, 7]
        return int8_uniform(n, -128, 127, seed, stream).view(np.uint8)
    raise ValueError(f"unknown distribution {dist!r}")


def make_inputs(w: Workload) -> dict:
    """CPU tensors in storage dtype, drawn in the fixed order A, x, bias, scale.

    Returns {"A": (M,K), "x": (B,K), "bias": (M,) or None, "scale": (M,) fp32 or None}.
    For "w8", A is int8 and x / bias are bf16.  For "w4", A is (M, K/2) uint8 (two
    int4 per byte) and scale is (M, K/W4_GROUP) fp32.
    """
    xdt = "bf16" if w.dtype in ("w8", "w4") else w.dtype
    if w.dtype == "w4":
        a = _draw(w.a_dist, w.M * w.K // 2, w.seed, _S_A)
        A = torch.from_numpy(a.astype(np.uint8, copy=False)).reshape(w.M, w.K // 2)
    else:
        a = _draw(w.a_dist, w.M * w.K, w.seed, _S_A)
    if w.dtype == "w4":
        pass  # A is already the packed bytes
    elif w.dtype == "w8":
        A = torch.from_numpy(a.astype(np.int8, copy=False)).reshape(w.M, w.K)
    else:
        A = to_storage(a, w.dtype).reshape(w.M, w.K)
    x = to_storage(_draw(w.x_dist, w.B * w.K, w.seed, _S_X), xdt).reshape(w.B, w.K)
    bias = None
    if w.bias:
        bias = to_storage(_draw(w.bias_dist, w.M, w.seed, _S_BIAS), xdt)
    scale = None
    if w.dtype == "w8":
        scale = torch.from_numpy(_draw(w.scale_dist, w.M, w.seed, _S_SCALE))
    elif w.dtype == "w4":
        ng = w.K // W4_GROUP
        scale = torch.from_numpy(_draw(w.scale_dist, w.M * ng, w.seed, _S_SCALE)).reshape(w.M, ng)
    return {"A": A, "x": x, "bias": bias, "scale": scale}


def storage_bits(t: torch.Tensor | None) -> np.ndarray | None:
    """Raw storage of a CPU tensor as numpy (fp16/bf16 as uint16 bit patterns)."""
    if t is None:
        return None
    t = t.contiguous()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


# --------------------------------------------------------------------------
# byte / flop accounting (roofline bookkeeping, not the method's arithmetic)
# --------------------------------------------------------------------------

def qmin_bytes(dtype: str, M: int, K: int, B: int) -> int:
    """Minimum bytes moved: read A and x once, write y once.

    Q_min = M*K*s_A + B*K*s_x + B*M*s_y, the arithmetic-intensity page's
    "minimum bytes" model (m*k + k*n + m*n)*s with one element size per operand.
    """
    sa, sx, sy, _ = ELEM_BYTES[dtype]
    a_bytes = M * K // 2 if dtype == "w4" else M * K * sa
    return a_bytes + B * K * sx + B * M * sy


def full_bytes(dtype: str, M: int, K: int, B: int, bias: bool) -> int:
    """Q_min plus the side inputs: bias (M*s_bias), the w8 row scale (4*M) and the
    w4 group scales (4*M*K/W4_GROUP)."""
    _, _, _, sb = ELEM_BYTES[dtype]
    extra = (M * sb if bias else 0) + (4 * M if dtype == "w8" else 0)
    extra += 4 * M * (K // W4_GROUP) if dtype == "w4" else 0
    return qmin_bytes(dtype, M, K, B) + extra


def flops(M: int, K: int, B: int) -> int:
    """One multiply and one add per A element per vector: 2*M*K*B."""
    return 2 * M * K * B


# --------------------------------------------------------------------------
# the benchmark's and parity tests' workloads
# --------------------------------------------------------------------------

def _cfgs() -> list[Workload]:
    out = [
        Workload("f32_1024x128_b1", "f32", 1024, 128, 1, False,
                 ("uniform", -1.0, 1.0), ("uniform", -1.0, 1.0)),
    ]
    for K in (16, 32, 4096):
        out.append(Workload(f"f32_16384x{K}_b1_bias", "f32", 16384, K, 1, True,
                            ("normal", float(np.sqrt(1.0 / K))), ("normal", 1.0)))
    for B in (1, 16):
        out.append(Workload(f"f16_4096x4096_b{B}", "f16", 4096, 4096, B, False,
                            ("normal", 0.02), ("normal", 1.0)))
    for M, K in ((14336, 4096), (4096, 14336), (128256, 4096)):
        out.append(Workload(f"bf16_{M}x{K}_b1", "bf16", M, K, 1, False,
                            ("normal", 0.02), ("normal", 1.0)))
    for B in (1, 4):
        out.append(Workload(f"w8_8192x8192_b{B}_bias", "w8", 8192, 8192, B, True,
                            ("int8", -127, 127), ("normal", 1.0)))
    return out


CONFIGS: list[Workload] = _cfgs()

# int4 weights with group-wise scales (the next storage type after int8): the
# int8 shapes, and a Llama-3-8B FFN shape.
W4_CONFIGS: list[Workload] = [
    Workload("w4_8192x8192_b1_bias", "w4", 8192, 8192, 1, True, ("bytes",), ("normal", 1.0)),
    Workload("w4_8192x8192_b4_bias", "w4", 8192, 8192, 4, True, ("bytes",), ("normal", 1.0)),
    Workload("w4_14336x4096_b1", "w4", 14336, 4096, 1, False, ("bytes",), ("normal", 1.0)),
]
# More than 16 vectors (fp16/bf16 only): the tensor-core crossover, on the fp16
# 4096x4096 and bf16 decode shapes of the configurations.
TC_CONFIGS: list[Workload] = [
    Workload("f16_4096x4096_b32", "f16", 4096, 4096, 32, False, ("normal", 0.02), ("normal", 1.0)),
    Workload("f16_4096x4096_b64", "f16", 4096, 4096, 64, False, ("normal", 0.02), ("normal", 1.0)),
    Workload("f16_4096x4096_b256", "f16", 4096, 4096, 256, False, ("normal", 0.02), ("normal", 1.0)),
    Workload("bf16_14336x4096_b32", "bf16", 14336, 4096, 32, False, ("normal", 0.02), ("normal", 1.0)),
    Workload("bf16_14336x4096_b128", "bf16", 14336, 4096, 128, False, ("normal", 0.02), ("normal", 1.0)),
    Workload("bf16_4096x14336_b64", "bf16", 4096, 14336, 64, False, ("normal", 0.02), ("normal", 1.0)),
    Workload("bf16_128256x4096_b64", "bf16", 128256, 4096, 64, False, ("normal", 0.02), ("normal", 1.0)),
]

BY_NAME = {w.name: w for w in CONFIGS + W4_CONFIGS + TC_CONFIGS}

# The benchmark's headline workload: the largest single-GPU configuration, the
# bf16 vocabulary projection 128256 x 4096 (about 1.05 GB of weights) with one
# vector; one step is one GEMV.
HEADLINE = ("bf16_128256x4096_b1",)
# The fp32 sweep over K at M = 16384 with bias (rows per warp, warp per row and the
# long-row kernels), reported beside the headline as a three-GEMV step.
FP32_STEP = ("f32_16384x16_b1_bias", "f32_16384x32_b1_bias", "f32_16384x4096_b1_bias")


def small(dtype: str, M: int, K: int, B: int, bias: bool, seed: int = 0) -> Workload:
    """A small problem with the same value distributions as the configs."""
    if dtype == "f32":
        a = ("normal", float(np.sqrt(1.0 / max(K, 1))))
    elif dtype == "w8":
        a = ("int8", -127, 127)
    elif dtype == "w4":
        a = ("bytes",)
    else:
        a = ("normal", 0.02)
    return Workload(f"{dtype}_{M}x{K}_b{B}{'_bias' if bias else ''}_s{seed}", dtype,
                    M, K, B, bias, a, ("normal", 1.0), seed=seed)
