"""gemv_bf16_splitk_noalloc through the C ABI on the GPU.

This entry point is for callers that cannot allocate device memory while they run
(memory reserved up front by their own allocator, real-time loops, hosts that
forbid the CUDA allocator): its split-K partial sums live in a fixed device array
inside the library.  Two calls in a row, with different shapes and data, must
agree with the regular gemv_bf16 entry point within the tolerance the parity
tests use; a request too large for the fixed array must be refused before any
launch.  The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

import decode_linear_layers_gb300 as g
import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    g.build()
    g.force_kernel("auto")


def _call_noalloc(d, y, M, K, B):
    """The raw C call: the entry point allocates nothing itself."""
    st = g.lib().gemv_bf16_splitk_noalloc(
        ctypes.c_void_p(d["A"].data_ptr()), ctypes.c_void_p(d["x"].data_ptr()),
        None if d["bias"] is None else ctypes.c_void_p(d["bias"].data_ptr()),
        ctypes.c_void_p(y.data_ptr()), M, K, B,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def test_two_calls_match_the_regular_entry_point():
    cases = [(64, 65536, 1, True, 11), (300, 8192, 3, False, 12)]
    for (M, K, B, bias, seed) in cases:
        w = W.small("bf16", M, K, B, bias, seed=seed)
        inp = W.make_inputs(w)
        y_ref, absdot = U.oracle_for("bf16", inp)
        d = U.to_device(inp)
        y_na = torch.full((B, M), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _call_noalloc(d, y_na, M, K, B) == 0
        y_reg = U.run_gpu("bf16", d, M, K, B)
        torch.cuda.synchronize()
        # against the existing entry point, within the parity tolerance
        U.assert_close("bf16", y_na, y_reg.double().cpu().numpy(), absdot, with_rounding=True,
                       what=f"noalloc vs gemv_bf16 M={M} K={K} B={B}")
        # and against the oracle
        U.assert_close("bf16", y_na, y_ref, absdot, what=f"noalloc vs oracle M={M} K={K} B={B}")


def test_refuses_requests_larger_than_its_array():
    M, K, B = 65536, 16, 16   # two K slices x 16 x 65536 x 4 bytes = 8 MiB > 4 MiB
    d = {"A": torch.zeros(M, K, dtype=torch.bfloat16, device="cuda"),
         "x": torch.zeros(B, K, dtype=torch.bfloat16, device="cuda"), "bias": None}
    y = torch.zeros(B, M, dtype=torch.bfloat16, device="cuda")
    assert _call_noalloc(d, y, M, K, B) == 2   # GEMV_ERR_UNSUPPORTED, nothing launched
    with pytest.raises(g.GemvError):
        g.gemv_bf16_splitk_noalloc(d["A"], d["x"], None, y, M, K, B)
