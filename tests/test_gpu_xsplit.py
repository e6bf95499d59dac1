"""The K-split kernel (GEMV_KERNEL_XSPLIT) against the oracle.

512 threads split each row; x lives in registers; rows are streamed by cp.async
into per-thread slots; warp partials meet every 16 rows.  The shapes cover every
B in 1..4, one, two and four chunks per thread (K up to 16384), a ragged chunk
count (513 chunks), row counts below, at and above the SM count, and blocks whose
last batch of 16 rows is partial; with and without bias, and the fused epilogue.
"""
from __future__ import annotations

import pytest
import torch

import decode_linear_layers_gb300 as g
import oracle
import workloads as W
from tests import gpu_util as U
from tests.test_gpu_parity import xsplit_feasible

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _auto_dispatch():
    g.force_kernel("auto")
    yield
    g.force_kernel("auto")


KS = {"f32": (2048, 4096, 8192, 2052), "f16": (4096, 8192, 16384, 4104), "bf16": (4096, 8192, 16384, 4104),
      "w8": (8192, 16384, 4112)}


@pytest.mark.parametrize("dtype", W.DTYPES)
@pytest.mark.parametrize("B", [1, 2, 3, 4])
def test_xsplit_parity(dtype, B):
    seed = 10 * B
    for K in KS[dtype]:
        for M in (1, 151, 153, 5000):
            if not xsplit_feasible(dtype, K, B):
                continue
            bias = (M + K) % 2 == 1
            w = W.small(dtype, M, K, B, bias, seed=seed)
            seed += 1
            inp = W.make_inputs(w)
            y_ref, absdot = U.oracle_for(dtype, inp)
            d = U.to_device(inp)
            g.force_kernel("xsplit")
            y1 = U.run_gpu(dtype, d, M, K, B)
            assert g.last_plan()["kernel_name"] == "xsplit", (dtype, M, K, B)
            y2 = U.run_gpu(dtype, d, M, K, B)
            torch.cuda.synchronize()
            assert torch.equal(y1, y2), "results differ between two identical calls"
            U.assert_close(dtype, y1, y_ref, absdot, with_rounding=True,
                           what=f"{dtype} xsplit M={M} K={K} B={B} bias={bias}")


@pytest.mark.parametrize("dtype", W.DTYPES)
def test_xsplit_epilogue(dtype):
    M, K, B = 3000, 8192 if dtype == "w8" else 4096, 4
    w = W.small(dtype, M, K, B, True, seed=77)
    inp = W.make_inputs(w)
    xdt = U.out_dtype(dtype)
    r = (torch.randn(B, M, generator=torch.Generator().manual_seed(3)) * 2).to(xdt)
    y_ref, _, absdot = oracle.gemv_ex(dtype, W.storage_bits(inp["A"]), W.storage_bits(inp["x"]),
                                      W.storage_bits(inp["bias"]),
                                      None if inp["scale"] is None else inp["scale"].numpy(),
                                      residual=W.storage_bits(r), act=1, nthreads=U.threads())
    d = U.to_device(inp)
    y = r.cuda()
    g.force_kernel("xsplit")
    g.gemv_ex(dtype, d["A"], d["scale"], d["x"], d["bias"], y, y, M, K, B, 1)
    assert g.last_plan()["kernel_name"] == "xsplit"
    U.assert_close_ex(dtype, y, y_ref, absdot, 1, what=f"{dtype} xsplit silu + residual in place")


# Shapes the dispatcher itself sends to the K-split kernel (no forcing): two long
# 16-bit rows per call, four long fp32 ones, the fp32 one- and two-vector ranges, and
# one vector of few long 16-bit rows.  A reordering of the dispatcher's rules that moved them elsewhere, or a
# fault on their launch configuration, fails here.
AUTO_XSPLIT = [("bf16", 1024, 16384, 2), ("f16", 4096, 8192, 2), ("f32", 2048, 8192, 4),
               ("f32", 4096, 4096, 1), ("f32", 8192, 4096, 2), ("bf16", 1024, 16384, 1), ("f16", 256, 8192, 1),
               ("bf16", 2048, 14336, 1)]


@pytest.mark.parametrize("dtype,M,K,B", AUTO_XSPLIT)
def test_auto_dispatch_takes_xsplit(dtype, M, K, B):
    w = W.small(dtype, M, K, B, True, seed=M + B)
    inp = W.make_inputs(w)
    y_ref, absdot = U.oracle_for(dtype, inp)
    d = U.to_device(inp)
    y = U.run_gpu(dtype, d, M, K, B)
    assert g.last_plan()["kernel_name"] == "xsplit", (dtype, M, K, B, g.last_plan()["kernel_name"])
    torch.cuda.synchronize()
    U.assert_close(dtype, y, y_ref, absdot, with_rounding=True, what=f"auto {dtype} {M}x{K} B={B}")


# The other kernels the dispatcher picks for few long rows: block per row for two
# fp32 vectors, the mixed-precision ring for four 16-bit vectors.
@pytest.mark.parametrize("dtype,M,K,B,kernel,variant", [("f32", 1024, 8192, 2, "block_per_row", None),
                                                        ("f32", 600, 12288, 2, "block_per_row", None),
                                                        ("bf16", 1024, 8192, 4, "batched", g.BATCHED_RING_MIXED),
                                                        ("f16", 2000, 4104, 3, "batched", g.BATCHED_RING_MIXED)])
def test_auto_dispatch_few_long_rows(dtype, M, K, B, kernel, variant):
    w = W.small(dtype, M, K, B, True, seed=M + K + B)
    inp = W.make_inputs(w)
    y_ref, absdot = U.oracle_for(dtype, inp)
    y = U.run_gpu(dtype, U.to_device(inp), M, K, B)
    p = g.last_plan()
    assert p["kernel_name"] == kernel and (variant is None or p["variant"] == variant), p
    torch.cuda.synchronize()
    U.assert_close(dtype, y, y_ref, absdot, with_rounding=True, what=f"auto {dtype} {M}x{K} B={B} {kernel}")

