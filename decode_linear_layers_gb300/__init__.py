"""Python binding of libgemv (ctypes): argument marshalling only.

The names and argument order are those of ``include/gemv.h``:

    gemv_f32 (A, x, bias, y, M, K, B, stream=None)
    gemv_f16 (A, x, bias, y, M, K, B, stream=None)
    gemv_bf16(A, x, bias, y, M, K, B, stream=None)
    gemv_w8  (A, row_scale, x, bias, y, M, K, B, stream=None)

Buffers may be torch CUDA tensors (checked for device, contiguity, element size
and minimum length before the call) or raw device addresses (ints, unchecked).
``bias`` may be None.  ``stream`` may be None (torch's current stream), a
``torch.cuda.Stream`` or a raw ``cudaStream_t`` value.  Every computation runs in
the CUDA library; a status other than GEMV_SUCCESS raises ``GemvError``.  There is
no fallback: without ``libgemv.so`` (build it with ``build()``) nothing runs.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB as LIB_PATH, build

__all__ = [
    "gemv_f32", "gemv_f16", "gemv_bf16", "gemv_w8", "gemv_w4", "gemv_bf16_splitk_noalloc", "gemv_ex",
    "gemv_swiglu", "gemv_host", "set_launch_overlap", "ACT_NONE", "ACT_SILU", "GemvError", "Plan", "plan_for",
    "status_string", "launch_count", "last_cuda_error", "force_kernel", "last_plan",
    "KERNELS", "DTYPE_CODES", "lib", "build", "LIB_PATH", "device_status", "test_stall",
]

SUCCESS, ERR_INVALID_VALUE, ERR_UNSUPPORTED, ERR_CUDA, ERR_DEVICE_TIMEOUT = 0, 1, 2, 3, 4
MAX_BATCH, MAX_BATCH_TC = 16, 256
ACT_NONE, ACT_SILU = 0, 1
DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2, "w8": 3, "w4": 4}
W4_GROUP = 128  # elements of a row that share one int4 scale
KERNELS = {"auto": 0, "rows_per_warp": 1, "warp_per_row": 2, "block_per_row": 3,
           "split_k": 4, "batched": 5, "scalar": 6, "stream": 7, "xsplit": 8, "tc": 9}
X_STAGING = {0: "global", 1: "smem", 2: "smem_fp32", 3: "regs"}
# BATCHED kernel variants (plan "variant"; force_kernel("batched", variant + 1))
BATCHED_ROWPAIR, BATCHED_RING, BATCHED_RING_MIXED = 0, 1, 2
KERNEL_NAMES = {v: k for k, v in KERNELS.items()}


class Plan(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int), ("lanes_per_row", ctypes.c_int),
                ("rows_per_warp", ctypes.c_int), ("splits", ctypes.c_int), ("unroll", ctypes.c_int),
                ("x_staging", ctypes.c_int), ("nb", ctypes.c_int),
                ("threads", ctypes.c_int), ("grid", ctypes.c_int64), ("smem_bytes", ctypes.c_int),
                ("workspace_bytes", ctypes.c_int64), ("variant", ctypes.c_int)]

    def as_dict(self) -> dict:
        d = {f: getattr(self, f) for f, _ in self._fields_}
        d["kernel_name"] = KERNEL_NAMES.get(self.kernel, "?")
        return d


class GemvError(RuntimeError):
    def __init__(self, status: int, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        msg = status_string(status)
        if status == ERR_CUDA:
            msg += f" (cudaError {cuda_error})"
        super().__init__(msg)


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libgemv.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run decode_linear_layers_gb300.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        for n in ("gemv_f32", "gemv_f16", "gemv_bf16"):
            f = getattr(L, n)
            f.argtypes = [vp, vp, vp, vp, i64, i64, ci, vp]
            f.restype = ci
        L.gemv_w8.argtypes = [vp, vp, vp, vp, vp, i64, i64, ci, vp]
        L.gemv_w8.restype = ci
        L.gemv_w4.argtypes = [vp, vp, vp, vp, vp, i64, i64, ci, vp]
        L.gemv_w4.restype = ci
        L.gemv_bf16_splitk_noalloc.argtypes = [vp, vp, vp, vp, i64, i64, ci, vp]
        L.gemv_bf16_splitk_noalloc.restype = ci
        L.gemv_ex.argtypes = [ci, vp, vp, vp, vp, vp, vp, i64, i64, ci, ci, vp]
        L.gemv_ex.restype = ci
        L.gemv_swiglu.argtypes = [ci, vp, vp, vp, vp, vp, i64, i64, ci, vp]
        L.gemv_swiglu.restype = ci
        L.gemv_host.argtypes = [ci, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, ci, vp]
        L.gemv_host.restype = ci
        L.gemv_set_launch_overlap.argtypes = [ci]
        L.gemv_set_launch_overlap.restype = ci
        L.gemv_status_string.argtypes = [ci]
        L.gemv_status_string.restype = ctypes.c_char_p
        L.gemv_last_cuda_error.argtypes = []
        L.gemv_last_cuda_error.restype = ci
        L.gemv_launch_count.argtypes = []
        L.gemv_launch_count.restype = ctypes.c_uint64
        L.gemv_plan_for.argtypes = [ci, i64, i64, ci, ci, ci, ctypes.POINTER(Plan)]
        L.gemv_plan_for.restype = ci
        L.gemv_test_force_kernel.argtypes = [ci, ci]
        L.gemv_test_force_kernel.restype = ci
        L.gemv_test_last_plan.argtypes = [ctypes.POINTER(Plan)]
        L.gemv_test_last_plan.restype = ci
        L.gemv_get_device_status.argtypes = [vp, ctypes.POINTER(ci)]
        L.gemv_get_device_status.restype = ci
        L.gemv_test_stall.argtypes = [ci, i64]
        L.gemv_test_stall.restype = ci
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().gemv_status_string(int(status)).decode()


def last_cuda_error() -> int:
    return int(lib().gemv_last_cuda_error())


def launch_count() -> int:
    return int(lib().gemv_launch_count())


def plan_for(dtype: str, M: int, K: int, B: int, aligned16: bool = True, num_sms: int = 152) -> dict:
    p = Plan()
    st = lib().gemv_plan_for(DTYPE_CODES[dtype], int(M), int(K), int(B), int(bool(aligned16)),
                             int(num_sms), ctypes.byref(p))
    if st != SUCCESS:
        raise GemvError(st)
    return p.as_dict()


def device_status(stream=None) -> tuple:
    """Synchronise `stream` and read (then clear) the device status word of the
    kernels with bounded waits: (status, bits), status SUCCESS or
    ERR_DEVICE_TIMEOUT; raises GemvError on a CUDA failure."""
    bits = ctypes.c_int(0)
    st = lib().gemv_get_device_status(_stream(stream), ctypes.byref(bits))
    if st not in (SUCCESS, ERR_DEVICE_TIMEOUT):
        _check(st)
    return st, int(bits.value)


def test_stall(stall: bool, timeout_ns: int = 0) -> None:
    """TEST ONLY: make later tensor-core launches skip their first CTA's last MMA,
    so that CTA's wait runs out after timeout_ns (<= 0: 2 s)."""
    _check(lib().gemv_test_stall(int(bool(stall)), int(timeout_ns)))


def force_kernel(kernel, param: int = 0) -> None:
    """TEST ONLY: force a kernel family ("auto" restores dispatch)."""
    k = KERNELS[kernel] if isinstance(kernel, str) else int(kernel)
    st = lib().gemv_test_force_kernel(k, int(param))
    if st != SUCCESS:
        raise GemvError(st)


def last_plan() -> dict:
    """TEST ONLY: the plan of this thread's last successful call."""
    p = Plan()
    st = lib().gemv_test_last_plan(ctypes.byref(p))
    if st != SUCCESS:
        raise GemvError(st)
    return p.as_dict()


# ------------------------------------------------------------------ marshalling
def _addr(t, elem_size: int, min_elems: int, what: str):
    """Device address of a tensor (checked) or of a raw int pointer (unchecked)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not getattr(t, "is_cuda", False):
        raise ValueError(f"{what} must be a CUDA tensor or a device address")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if t.element_size() != elem_size:
        raise ValueError(f"{what}: element size {t.element_size()} != {elem_size}")
    if t.numel() < min_elems:
        raise ValueError(f"{what}: {t.numel()} elements < {min_elems} needed")
    return t.data_ptr()


_current_raw_stream = None  # (torch's current stream of the current device, as a handle)


def _stream(stream):
    global _current_raw_stream
    if stream is None:
        # the raw handle straight from torch (a Stream object per call costs microseconds)
        if _current_raw_stream is None:
            import torch
            get = getattr(torch._C, "_cuda_getCurrentRawStream", None)
            dev = torch._C._cuda_getDevice
            _current_raw_stream = ((lambda: get(dev())) if get is not None
                                   else (lambda: torch.cuda.current_stream().cuda_stream))
        return _current_raw_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int) -> None:
    if st != SUCCESS:
        raise GemvError(st, last_cuda_error() if st == ERR_CUDA else 0)


def _sizes(M, K, B):
    M, K, B = int(M), int(K), int(B)
    if min(M, K, B) < 0:
        return M, K, B, 0, 0, 0  # let the library report the bad size
    return M, K, B, M * K, B * K, B * M


_entry = {}  # entry points by name, looked up once


def _fn(name):
    f = _entry.get(name)
    if f is None:
        f = _entry[name] = getattr(lib(), name)
    return f


def _float_gemv(name, esize, A, x, bias, y, M, K, B, stream):
    M, K, B, na, nx, ny = _sizes(M, K, B)
    args = (_addr(A, esize, na, "A"), _addr(x, esize, nx, "x"),
            _addr(bias, esize, M if bias is not None else 0, "bias"),
            _addr(y, esize, ny, "y"))
    _check(_fn(name)(*args, M, K, B, _stream(stream)))


def gemv_f32(A, x, bias, y, M, K, B, stream=None) -> None:
    """y[b, m] = sum_k A[m, k] x[b, k] (+ bias[m]); fp32 storage and accumulation."""
    _float_gemv("gemv_f32", 4, A, x, bias, y, M, K, B, stream)


def gemv_f16(A, x, bias, y, M, K, B, stream=None) -> None:
    """fp16 storage (torch.float16), fp32 accumulation, fp16 output."""
    _float_gemv("gemv_f16", 2, A, x, bias, y, M, K, B, stream)


def gemv_bf16(A, x, bias, y, M, K, B, stream=None) -> None:
    """bf16 storage (torch.bfloat16), fp32 accumulation, bf16 output."""
    _float_gemv("gemv_bf16", 2, A, x, bias, y, M, K, B, stream)


def gemv_w8(A, row_scale, x, bias, y, M, K, B, stream=None) -> None:
    """int8 A with fp32 row_scale; bf16 x, bias and y; fp32 accumulation."""
    M, K, B, na, nx, ny = _sizes(M, K, B)
    args = (_addr(A, 1, na, "A"), _addr(row_scale, 4, M, "row_scale"), _addr(x, 2, nx, "x"),
            _addr(bias, 2, M if bias is not None else 0, "bias"), _addr(y, 2, ny, "y"))
    _check(_fn("gemv_w8")(*args, M, K, B, _stream(stream)))


OVERLAP = {"off": 0, "launch": 1, "weights": 2}


def set_launch_overlap(mode: str) -> None:
    """Launch overlap for this thread's later calls: "off", "launch" (programmatic
    dependent launches, every access after the previous kernel; the default) or
    "weights" (the first weight loads before that wait; only for weights the
    preceding work does not write)."""
    _check(lib().gemv_set_launch_overlap(OVERLAP[mode]))


def _host_addr(t, elem_size: int, min_elems: int, what: str):
    """Host address of a CPU tensor (checked) or of a raw int pointer (unchecked)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if getattr(t, "is_cuda", True):
        raise ValueError(f"{what} must be a CPU tensor (pinned for asynchronous copies) or a host address")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if t.element_size() != elem_size:
        raise ValueError(f"{what}: element size {t.element_size()} != {elem_size}")
    if t.numel() < min_elems:
        raise ValueError(f"{what}: {t.numel()} elements < {min_elems} needed")
    return t.data_ptr()


def gemv_host(dtype, h_A, h_scale, h_x, h_bias, h_y, d_A, d_scale, d_x, d_bias, d_y, M, K, B,
              stream=None) -> None:
    """The GEMV on host buffers: copies h_A, h_scale, h_x, h_bias (CPU tensors,
    pinned for asynchronous copies; None skips a copy) into the device buffers d_*,
    runs it there and copies y back into h_y, all enqueued on `stream`."""
    M, K, B, _, nx, ny = _sizes(M, K, B)
    sa = {"f32": 4, "f16": 2, "bf16": 2, "w8": 1, "w4": 1}[dtype]
    sx = 4 if dtype == "f32" else 2
    na, ns = _a_count(dtype, M, K)
    hs = (_host_addr(h_A, sa, na, "h_A"), _host_addr(h_scale, 4, ns, "h_scale"), _host_addr(h_x, sx, nx, "h_x"),
          _host_addr(h_bias, sx, M if h_bias is not None else 0, "h_bias"), _host_addr(h_y, sx, ny, "h_y"))
    ds = (_addr(d_A, sa, na, "d_A"), _addr(d_scale, 4, ns, "d_scale"), _addr(d_x, sx, nx, "d_x"),
          _addr(d_bias, sx, M if d_bias is not None else 0, "d_bias"), _addr(d_y, sx, ny, "d_y"))
    _check(lib().gemv_host(DTYPE_CODES[dtype], *hs, *ds, M, K, B, _stream(stream)))


NOALLOC_SCRATCH_BYTES = 4 * 1024 * 1024


def gemv_w4(A, group_scale, x, bias, y, M, K, B, stream=None) -> None:
    """int4 A, two per byte (torch.uint8, M x K/2, even element in the low nibble),
    with fp32 group_scale (M x K/W4_GROUP); bf16 x, bias and y; fp32 accumulation."""
    M, K, B, _, nx, ny = _sizes(M, K, B)
    na, ns = _a_count("w4", M, K)
    args = (_addr(A, 1, na, "A"), _addr(group_scale, 4, ns, "group_scale"), _addr(x, 2, nx, "x"),
            _addr(bias, 2, M if bias is not None else 0, "bias"), _addr(y, 2, ny, "y"))
    _check(_fn("gemv_w4")(*args, M, K, B, _stream(stream)))


def gemv_bf16_splitk_noalloc(A, x, bias, y, M, K, B, stream=None) -> None:
    """gemv_bf16 on the split-K path with its partial sums in the library's fixed
    device array (no device allocation).  For callers that cannot allocate while
    they run; calls that overlap on the GPU race on the shared array.  Raises
    GemvError(GEMV_ERR_UNSUPPORTED) when splits x B x M x 4 bytes exceed
    NOALLOC_SCRATCH_BYTES or the rows are not 16-byte aligned."""
    _float_gemv("gemv_bf16_splitk_noalloc", 2, A, x, bias, y, M, K, B, stream)


_ESIZE = {"f32": (4, 4), "f16": (2, 2), "bf16": (2, 2), "w8": (1, 2), "w4": (1, 2)}   # (A, x/bias/y)


def _a_count(dtype, M, K):
    """Elements of A's storage (bytes for int4, two values each) and of its scales."""
    if dtype == "w4":
        return max(0, M * K // 2), max(0, M * (K // W4_GROUP))
    return max(0, M * K), max(0, M)


def gemv_ex(dtype, A, row_scale, x, bias, residual, y, M, K, B, act=ACT_NONE, stream=None) -> None:
    """y = act(s_m * sum_k A x + bias) + residual, one launch, any storage type.

    row_scale: w8 only (else None).  residual: (B, M) in y's type, None, or y itself
    (in place)."""
    M, K, B, _, nx, ny = _sizes(M, K, B)
    na, ns = _a_count(dtype, M, K)
    sa, sx = _ESIZE[dtype]
    args = (_addr(A, sa, na, "A"), _addr(row_scale, 4, ns, "row_scale"), _addr(x, sx, nx, "x"),
            _addr(bias, sx, M if bias is not None else 0, "bias"),
            _addr(residual, sx, ny if residual is not None else 0, "residual"), _addr(y, sx, ny, "y"))
    _check(_fn("gemv_ex")(DTYPE_CODES[dtype], *args, M, K, B, int(act), _stream(stream)))


def gemv_swiglu(dtype, A, row_scale, x, bias, y, I, K, B, stream=None) -> None:
    """y[b][m] = silu(gate_m) * up_m over A = [gate rows; up rows] (2I x K)."""
    I, K, B = int(I), int(K), int(B)
    M2 = 2 * I if I >= 0 else 0
    sa, sx = _ESIZE[dtype]
    na, ns = _a_count(dtype, M2, K)
    args = (_addr(A, sa, na, "A"), _addr(row_scale, 4, ns, "row_scale"),
            _addr(x, sx, max(0, B * K), "x"), _addr(bias, sx, M2 if bias is not None else 0, "bias"),
            _addr(y, sx, max(0, B * I), "y"))
    _check(_fn("gemv_swiglu")(DTYPE_CODES[dtype], *args, I, K, B, _stream(stream)))
