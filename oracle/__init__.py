"""CPU oracle for dense GEMV — test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package. It wraps ``gemv_oracle.c`` (plain C, fp64 accumulation
over the exactly decoded stored values, k ascending) through ctypes and shares no
code with the CUDA library.

The definition it follows: y[b][m] = s_m * sum_k A[m][k] * x[b][k] + bias[m]
("16-sgemv" notes, problem definition; "GEMV and row-level parallelism" lesson,
section 1; int8 weights with per-row scale from the NPU MatMul post, section 1.2);
int4 weights with one scale per group of consecutive elements of a row (the NPU
MatMul post, section 5.2): y[b][m] = sum_k s[m][k/group] * q[m][k] * x[b][k] + bias[m].

Pins (checked by ``tests/test_oracle.py`` against values fixed by the pages and by
mathematics, not by this code): exact-rational brute force on tiny inputs, the
identity and permutation matrices, one-hot x, linearity, bias == NULL, the all-ones
closed form, rank-1 matrices, exact integer results for int8 weights with unit
scale, and the fp16/bf16 decoders against independent decoders over all 65,536
bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemv_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_gemv.so")

KIND = {"f32": 0, "f16": 1, "bf16": 2, "w8": 3, "w4": 4}
W4_GROUP = 128  # the library's int4 group size (the oracle takes any group)


def build(force: bool = False) -> str:
    """Compile gemv_oracle.c into liboracle_gemv.so next to it (gcc, OpenMP)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-std=c11", _SRC, "-o", tmp]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:] + ["-lm"], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-lm"], check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        vp, i64 = ctypes.c_void_p, ctypes.c_int64
        L.oracle_gemv.argtypes = [ctypes.c_int, vp, vp, vp, vp, i64, i64, i64, vp, vp, ctypes.c_int]
        L.oracle_gemv.restype = ctypes.c_int
        L.oracle_gemv_g.argtypes = [ctypes.c_int, vp, vp, i64, vp, vp, i64, i64, i64, vp, vp, ctypes.c_int]
        L.oracle_gemv_g.restype = ctypes.c_int
        L.oracle_decode.argtypes = [ctypes.c_int, vp, i64, vp]
        L.oracle_decode.restype = ctypes.c_int
        L.oracle_max_threads.argtypes = []
        L.oracle_max_threads.restype = ctypes.c_int
        L.oracle_silu.argtypes = [ctypes.c_double]
        L.oracle_silu.restype = ctypes.c_double
        L.oracle_gemv_ex.argtypes = [ctypes.c_int, vp, vp, i64, vp, vp, vp, i64, i64, i64, ctypes.c_int,
                                     vp, vp, vp, ctypes.c_int]
        L.oracle_gemv_ex.restype = ctypes.c_int
        L.oracle_swiglu.argtypes = [ctypes.c_int, vp, vp, i64, vp, vp, i64, i64, i64, vp, vp, vp, vp, vp,
                                    ctypes.c_int]
        L.oracle_swiglu.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _storage(a, dtype_code):
    """Contiguous numpy array with the storage layout the C code expects."""
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    want = {0: np.float32, 1: np.uint16, 2: np.uint16, 3: np.int8, 4: np.uint8}[dtype_code]
    if a.dtype == np.float16 and want == np.uint16:
        a = a.view(np.uint16)
    if a.dtype != want:
        raise TypeError(f"expected storage {np.dtype(want)}, got {a.dtype}")
    return a


def _prep(dtype, A, x, bias, scale, group):
    """Storage arrays and sizes: (code, A, x, bias, scale, group, M, K, B)."""
    code = KIND[dtype]
    A = _storage(A, code)
    xcode = KIND["bf16"] if dtype in ("w8", "w4") else code
    x = _storage(x, xcode)
    bias = _storage(bias, xcode)
    M = A.shape[0]
    K = A.shape[1] * (2 if dtype == "w4" else 1)
    B = x.shape[0]
    if x.shape[1] != K or (bias is not None and bias.shape != (M,)):
        raise ValueError("shape mismatch")
    g = 0
    if dtype == "w4":
        g = W4_GROUP if group is None else int(group)
        if g <= 0 or K % g:
            raise ValueError("group must divide K")
        scale = np.ascontiguousarray(scale, dtype=np.float32)
        if scale.shape != (M, K // g):
            raise ValueError("int4 scales must be (M, K / group)")
    elif scale is not None:
        scale = np.ascontiguousarray(scale, dtype=np.float32)
    return code, A, x, bias, scale, g, M, K, B


def gemv(dtype: str, A, x, bias=None, scale=None, nthreads: int = 1, group=None):
    """Oracle GEMV on stored values.

    dtype: "f32" | "f16" | "bf16" | "w8" | "w4".  A: (M, K) storage (float32, uint16
    bit patterns of fp16/bf16, int8), or for "w4" (M, K/2) uint8 holding two int4
    per byte (even element in the low nibble); x: (B, K) storage (bf16 bits for
    "w8"/"w4"); bias: (M,) storage or None; scale: (M,) float32 for "w8", (M, K/group)
    float32 for "w4" (group defaults to W4_GROUP).
    Returns (y, absdot), both float64 of shape (B, M).
    """
    code, A, x, bias, scale, g, M, K, B = _prep(dtype, A, x, bias, scale, group)
    y = np.empty((B, M), dtype=np.float64)
    absdot = np.empty((B, M), dtype=np.float64)
    rc = lib().oracle_gemv_g(code, _ptr(A), _ptr(scale), g, _ptr(x), _ptr(bias), M, K, B,
                             _ptr(y), _ptr(absdot), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gemv rejected its arguments")
    return y, absdot


def silu(v: float) -> float:
    """The oracle's SiLU, v / (1 + e^-v), in double."""
    return float(lib().oracle_silu(float(v)))


def gemv_ex(dtype: str, A, x, bias=None, scale=None, residual=None, act: int = 0, nthreads: int = 1,
            group=None):
    """GEMV with the fused epilogue: y = act(s * sum_k A x + bias) + residual.

    act: 0 none, 1 SiLU.  residual: (B, M) in y's storage type (like x) or None.
    Returns (y, pre, absdot): y after the epilogue, pre the value before the
    activation, absdot = sum_k |s A x|; all float64 (B, M).
    """
    code, A, x, bias, scale, g, M, K, B = _prep(dtype, A, x, bias, scale, group)
    residual = _storage(residual, KIND["bf16"] if dtype in ("w8", "w4") else code)
    if residual is not None and residual.shape != (B, M):
        raise ValueError("residual must be (B, M)")
    y = np.empty((B, M)); pre = np.empty((B, M)); ad = np.empty((B, M))
    rc = lib().oracle_gemv_ex(code, _ptr(A), _ptr(scale), g, _ptr(x), _ptr(bias), _ptr(residual), M, K, B,
                              int(act), _ptr(y), _ptr(pre), _ptr(ad), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gemv_ex rejected its arguments")
    return y, pre, ad


def swiglu(dtype: str, A, x, bias=None, scale=None, nthreads: int = 1, group=None):
    """SwiGLU over A = [gate rows; up rows] (2I x K): y = silu(gate) * up.

    Returns (y, gate, up, absdot_gate, absdot_up), all float64 (B, I).
    """
    code, A, x, bias, scale, g, M2, K, B = _prep(dtype, A, x, bias, scale, group)
    if M2 % 2:
        raise ValueError("A must have an even number of rows (gate then up)")
    I = M2 // 2
    out = [np.empty((B, I)) for _ in range(5)]
    rc = lib().oracle_swiglu(code, _ptr(A), _ptr(scale), g, _ptr(x), _ptr(bias), I, K, B,
                             *[_ptr(o) for o in out], int(nthreads))
    if rc != 0:
        raise ValueError("oracle_swiglu rejected its arguments")
    return tuple(out)


def decode(kind: str, bits) -> np.ndarray:
    """Decode stored values ("f32", "f16", "bf16" bit patterns, "w8" int8, or "w4"
    bytes holding two int4 each, low nibble first) to float64."""
    code = KIND[kind]
    a = _storage(np.asarray(bits).reshape(-1), code)
    n = a.size * (2 if kind == "w4" else 1)
    out = np.empty(n, dtype=np.float64)
    if lib().oracle_decode(code, _ptr(a), n, _ptr(out)) != 0:
        raise ValueError("bad decode request")
    return out


def max_threads() -> int:
    return int(lib().oracle_max_threads())
