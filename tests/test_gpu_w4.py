"""gemv_w4 (int4 weights, per-group scales) on the GPU against the oracle.

* the int4 workloads at full size through the default dispatch, twice (bitwise
  equal);
* every kernel family that runs int4, forced, on shapes with several tiles and
  ragged tails, B in 1..16, with and without bias;
* edges: K = 0, K not a multiple of the group (rejected), rows not 16-byte aligned
  (element-load kernel), guard bytes around y, closed forms;
* the fused epilogues: gemv_ex with SiLU and an in-place residual, SwiGLU with one
  and with three vectors.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import decode_linear_layers_gb300 as g
import oracle
import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _auto_dispatch():
    g.force_kernel("auto")
    yield
    g.force_kernel("auto")


def _bits(t):
    return t.view(torch.int16)


@pytest.mark.parametrize("name", [w.name for w in W.W4_CONFIGS])
def test_w4_config_full_size(name):
    w = W.BY_NAME[name]
    inp = W.make_inputs(w)
    y_ref, absdot = U.oracle_for("w4", inp)
    d = U.to_device(inp)
    y1 = U.run_gpu("w4", d, w.M, w.K, w.B)
    plan = g.last_plan()
    y2 = U.run_gpu("w4", d, w.M, w.K, w.B)
    torch.cuda.synchronize()
    assert torch.equal(_bits(y1), _bits(y2)), "results differ between two identical calls"
    U.assert_close("w4", y1, y_ref, absdot, what=f"{name} [{plan['kernel_name']}]")


SHAPES = [(1, 128), (37, 256), (300, 384), (1001, 1024), (77, 4224), (5, 20096)]
FORCED = [("rows_per_warp", 0), ("warp_per_row", 0), ("block_per_row", 0), ("split_k", 0),
          ("split_k", 3), ("scalar", 4), ("scalar", 32), ("stream", 0), ("stream", 2), ("batched", 2), ("auto", 0)]


@pytest.mark.parametrize("kernel,param", FORCED)
def test_w4_forced_kernel(kernel, param):
    seed = 0
    for (M, K) in SHAPES:
        for B in (1, 3, 16):
            if kernel == "rows_per_warp" and K > 512:
                continue  # more than 16 chunks per row: not a rows-per-warp shape
            bias = (B + M) % 2 == 0
            w = W.small("w4", M, K, B, bias, seed=seed)
            seed += 1
            inp = W.make_inputs(w)
            y_ref, absdot = U.oracle_for("w4", inp)
            d = U.to_device(inp)
            g.force_kernel(kernel, param)
            y = U.run_gpu("w4", d, M, K, B)
            plan = g.last_plan()
            g.force_kernel("auto")
            if kernel not in ("auto",) and not (kernel == "stream" and B > 1) and not (kernel == "batched" and B == 1):
                assert plan["kernel_name"] == kernel, (plan, kernel)
            U.assert_close("w4", y, y_ref, absdot, with_rounding=True,
                           what=f"w4 {kernel}/{param} M={M} K={K} B={B} bias={bias}")


@pytest.mark.parametrize("B", list(range(1, 17)))
def test_w4_all_batch_sizes(B):
    M, K = 700, 2048
    w = W.small("w4", M, K, B, True, seed=100 + B)
    inp = W.make_inputs(w)
    y_ref, absdot = U.oracle_for("w4", inp)
    y = U.run_gpu("w4", U.to_device(inp), M, K, B)
    U.assert_close("w4", y, y_ref, absdot, with_rounding=True, what=f"w4 B={B}")


def test_w4_unaligned_rows_use_element_loads():
    M, K, B = 257, 384, 2
    w = W.small("w4", M, K, B, True, seed=200)
    inp = W.make_inputs(w)
    y_ref, absdot = U.oracle_for("w4", inp)
    d = U.to_device(inp)
    # A one byte past a 16-byte boundary
    buf = torch.empty(M * K // 2 + 16, dtype=torch.uint8, device="cuda")
    A = buf[1:1 + M * K // 2]
    A.copy_(d["A"].reshape(-1))
    y = torch.empty(B, M, dtype=torch.bfloat16, device="cuda")
    g.gemv_w4(A, d["scale"], d["x"], d["bias"], y, M, K, B)
    assert g.last_plan()["kernel_name"] == "scalar"
    U.assert_close("w4", y, y_ref, absdot, with_rounding=True, what="w4 unaligned")


def test_w4_k_zero_and_bad_k():
    M = 9
    bias = torch.randn(M, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).cuda()
    y = torch.full((2, M), 7.0, dtype=torch.bfloat16, device="cuda")
    A = torch.empty(0, dtype=torch.uint8, device="cuda")
    x = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    g.gemv_w4(A, None, x, bias, y, M, 0, 2)
    torch.cuda.synchronize()
    assert torch.equal(y, bias.expand(2, M))
    A = torch.zeros(M * 100 // 2, dtype=torch.uint8, device="cuda")
    xs = torch.zeros(100, dtype=torch.bfloat16, device="cuda")
    sc = torch.ones(M, dtype=torch.float32, device="cuda")
    with pytest.raises(g.GemvError) as e:
        g.gemv_w4(A, sc, xs, None, y, M, 100, 1)   # K not a multiple of 128
    assert e.value.status == g.ERR_INVALID_VALUE
    with pytest.raises(g.GemvError):
        g.gemv_w4(torch.zeros(M * 64, dtype=torch.uint8, device="cuda"), None,
                  torch.zeros(128, dtype=torch.bfloat16, device="cuda"), None, y, M, 128, 1)  # no scales


def test_w4_guard_bytes_untouched():
    for kernel, param, B in (("auto", 0, 4), ("split_k", 4, 4), ("block_per_row", 0, 4), ("scalar", 32, 4),
                             ("stream", 0, 1), ("stream", 2, 1), ("warp_per_row", 0, 3), ("rows_per_warp", 2, 4),
                             ("batched", 2, 9),
                             ("batched", 2, 3)):
        M, K = 333, 256
        w = W.small("w4", M, K, B, False, seed=400)
        d = U.to_device(W.make_inputs(w))
        n = B * M
        buf = torch.full((n + 2048,), 7, dtype=torch.bfloat16, device="cuda")
        y = buf[1024:1024 + n]
        g.force_kernel(kernel, param)
        U.call("w4", d, y, M, K, B)
        g.force_kernel("auto")
        torch.cuda.synchronize()
        assert bool((buf[:1024] == 7).all()) and bool((buf[1024 + n:] == 7).all()), kernel


def test_w4_closed_forms():
    # every weight 1 (bytes 0x11), -8 (0x88) or 7 (0x77), x = 1, scale 0.5 per group:
    # y = 0.5 * q * K exactly in every kernel family
    M, K, B = 96, 4096, 2
    x = torch.ones(B, K, dtype=torch.bfloat16, device="cuda")
    sc = torch.full((M, K // 128), 0.5, dtype=torch.float32, device="cuda")
    for byte, qv in ((0x11, 1), (0x88, -8), (0x77, 7)):
        A = torch.full((M, K // 2), byte, dtype=torch.uint8, device="cuda")
        for kernel, param, b in (("auto", 0, B), ("warp_per_row", 0, B), ("block_per_row", 0, B),
                                 ("split_k", 5, B), ("scalar", 32, B), ("stream", 0, 1), ("batched", 2, B)):
            y = torch.empty(b, M, dtype=torch.bfloat16, device="cuda")
            g.force_kernel(kernel, param)
            g.gemv_w4(A, sc, x[:b], None, y, M, K, b)
            g.force_kernel("auto")
            assert bool((y.double() == 0.5 * qv * K).all()), (byte, kernel)


@pytest.mark.parametrize("act,res", [(0, "inplace"), (1, "none"), (1, "sep")])
def test_w4_epilogue(act, res):
    M, K, B = 1500, 4096, 1
    w = W.small("w4", M, K, B, True, seed=500 + act)
    inp = W.make_inputs(w)
    r = (torch.randn(B, M, generator=torch.Generator().manual_seed(5)) * 2).to(torch.bfloat16) \
        if res != "none" else None
    y_ref, _, absdot = oracle.gemv_ex("w4", W.storage_bits(inp["A"]), W.storage_bits(inp["x"]),
                                      W.storage_bits(inp["bias"]), inp["scale"].numpy(),
                                      residual=None if r is None else W.storage_bits(r), act=act,
                                      nthreads=U.threads())
    d = U.to_device(inp)
    rd = None if r is None else r.cuda()
    y = rd if res == "inplace" else torch.empty(B, M, dtype=torch.bfloat16, device="cuda")
    g.gemv_ex("w4", d["A"], d["scale"], d["x"], d["bias"], rd, y, M, K, B, act)
    U.assert_close_ex("w4", y, y_ref, absdot, act, what=f"w4 act={act} res={res}")


@pytest.mark.parametrize("I,K", [(777, 1024), (14336, 4096)])
def test_w4_swiglu(I, K):
    w = W.small("w4", 2 * I, K, 1, True, seed=600 + I)
    inp = W.make_inputs(w)
    yr, gate, up, adg, adu = oracle.swiglu("w4", W.storage_bits(inp["A"]), W.storage_bits(inp["x"]),
                                           W.storage_bits(inp["bias"]), inp["scale"].numpy(),
                                           nthreads=U.threads())
    d = U.to_device(inp)
    y = torch.empty(1, I, dtype=torch.bfloat16, device="cuda")
    g.gemv_swiglu("w4", d["A"], d["scale"], d["x"], d["bias"], y, I, K, 1)
    U.assert_close_swiglu("w4", y, yr, gate, up, adg, adu, what=f"w4 swiglu I={I} K={K}")
    # more than one vector: the batched ring kernel carries the gate/up row pairs
    w3 = W.small("w4", 2 * I, K, 3, True, seed=700 + I)
    inp3 = W.make_inputs(w3)
    yr3, gate3, up3, adg3, adu3 = oracle.swiglu("w4", W.storage_bits(inp3["A"]), W.storage_bits(inp3["x"]),
                                                W.storage_bits(inp3["bias"]), inp3["scale"].numpy(),
                                                nthreads=U.threads())
    d3 = U.to_device(inp3)
    y3 = torch.empty(3, I, dtype=torch.bfloat16, device="cuda")
    g.gemv_swiglu("w4", d3["A"], d3["scale"], d3["x"], d3["bias"], y3, I, K, 3)
    assert g.last_plan()["kernel_name"] == "batched"
    U.assert_close_swiglu("w4", y3, yr3, gate3, up3, adg3, adu3, what=f"w4 swiglu B=3 I={I} K={K}")
