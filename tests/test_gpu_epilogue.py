"""Fused epilogues on the GPU against the oracle: gemv_ex (SiLU and residual add)
and gemv_swiglu (silu(gate) * up over a concatenated gate/up projection).

These fold the elementwise steps a decode layer runs after its projections into
the GEMV's own epilogue (the NPU MatMul post, section 5.1, fuses bias, activation
and residual into the MatMul).
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
def _auto():
    g.force_kernel("auto")
    yield
    g.force_kernel("auto")


def _residual(dtype, B, M, seed):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((B, M)).astype(np.float32)
    t = torch.from_numpy(v)
    return t if dtype == "f32" else t.to(U.out_dtype(dtype))


SHAPES = [(300, 4096, 1), (300, 4096, 4), (5000, 64, 2), (100, 20000, 1), (257, 1040, 9)]


@pytest.mark.parametrize("dtype", W.DTYPES)
@pytest.mark.parametrize("act,res", [(0, "sep"), (1, "none"), (1, "sep"), (1, "inplace")])
def test_gemv_ex(dtype, act, res):
    for i, (M, K, B) in enumerate(SHAPES):
        w = W.small(dtype, M, K, B, i % 2 == 0, seed=1000 + i)
        inp = W.make_inputs(w)
        r = None if res == "none" else _residual(dtype, B, M, seed=2000 + i)
        y_ref, pre, absdot = oracle.gemv_ex(dtype, W.storage_bits(inp["A"]), W.storage_bits(inp["x"]),
                                            W.storage_bits(inp["bias"]),
                                            None if inp["scale"] is None else inp["scale"].numpy(),
                                            residual=W.storage_bits(r), act=act, nthreads=U.threads())
        d = U.to_device(inp)
        if res == "inplace":
            y = r.to("cuda").contiguous()
            rd = y
        else:
            y = torch.empty((B, M), dtype=U.out_dtype(dtype), device="cuda")
            rd = None if r is None else r.to("cuda")
        g.gemv_ex(dtype, d["A"], d["scale"], d["x"], d["bias"], rd, y, M, K, B, act)
        torch.cuda.synchronize()
        U.assert_close_ex(dtype, y, y_ref, absdot, act,
                          what=f"ex {dtype} act={act} res={res} {M}x{K} B={B} [{g.last_plan()['kernel_name']}]")


def test_gemv_ex_rejects_shifted_residual():
    A = torch.randn(64, 64, device="cuda")
    x = torch.randn(1, 64, device="cuda")
    buf = torch.zeros(128, device="cuda")
    with pytest.raises(g.GemvError) as e:
        g.gemv_ex("f32", A, None, x, None, buf[1:65], buf[0:64], 64, 64, 1)   # overlaps y, not equal
    assert e.value.status == 1
    with pytest.raises(g.GemvError) as e:
        g.gemv_ex("f32", A, None, x, None, None, buf[0:64], 64, 64, 1, act=7)
    assert e.value.status == 1


@pytest.mark.parametrize("dtype", W.DTYPES)
def test_swiglu(dtype):
    for B in (1, 2, 3, 4, 5, 8, 16):
        I, K = 777, 1024
        bias = B % 2 == 1
        w = W.small(dtype, 2 * I, K, B, bias, seed=3000 + B)
        inp = W.make_inputs(w)
        y_ref, gate, up, adg, adu = oracle.swiglu(dtype, W.storage_bits(inp["A"]), W.storage_bits(inp["x"]),
                                                  W.storage_bits(inp["bias"]),
                                                  None if inp["scale"] is None else inp["scale"].numpy(),
                                                  nthreads=U.threads())
        d = U.to_device(inp)
        y = torch.empty((B, I), dtype=U.out_dtype(dtype), device="cuda")
        g.gemv_swiglu(dtype, d["A"], d["scale"], d["x"], d["bias"], y, I, K, B)
        torch.cuda.synchronize()
        U.assert_close_swiglu(dtype, y, y_ref, gate, up, adg, adu,
                              what=f"swiglu {dtype} I={I} K={K} B={B} [{g.last_plan()['kernel_name']}]")


@pytest.mark.parametrize("dtype", W.DTYPES)
def test_swiglu_batched_variants(dtype):
    # every batched kernel variant (forced: variant + 1) carries SwiGLU's gate/up row pairs
    I, K = 1000, 2048
    for B in (2, 7, 16):
        w = W.small(dtype, 2 * I, K, B, True, seed=3100 + B)
        inp = W.make_inputs(w)
        y_ref, gate, up, adg, adu = oracle.swiglu(dtype, W.storage_bits(inp["A"]), W.storage_bits(inp["x"]),
                                                  W.storage_bits(inp["bias"]),
                                                  None if inp["scale"] is None else inp["scale"].numpy(),
                                                  nthreads=U.threads())
        d = U.to_device(inp)
        for param in (1, 2, 3):
            if param == 3 and dtype not in ("f16", "bf16"):
                continue
            g.force_kernel("batched", param)
            y = torch.empty((B, I), dtype=U.out_dtype(dtype), device="cuda")
            g.gemv_swiglu(dtype, d["A"], d["scale"], d["x"], d["bias"], y, I, K, B)
            plan = g.last_plan()
            g.force_kernel("auto")
            assert plan["kernel_name"] == "batched" and plan["variant"] == param - 1, plan
            U.assert_close_swiglu(dtype, y, y_ref, gate, up, adg, adu,
                                  what=f"swiglu {dtype} B={B} variant={param - 1}")


def test_swiglu_decode_size():
    # the gate/up projection of a Llama-3-8B-shaped layer: I = 14336, K = 4096
    I, K = 14336, 4096
    w = W.Workload("bf16_gate_up", "bf16", 2 * I, K, 1, False, ("normal", 0.02), ("normal", 1.0))
    inp = W.make_inputs(w)
    y_ref, gate, up, adg, adu = oracle.swiglu("bf16", W.storage_bits(inp["A"]), W.storage_bits(inp["x"]),
                                              nthreads=U.threads())
    d = U.to_device(inp)
    y = torch.empty((1, I), dtype=torch.bfloat16, device="cuda")
    g.gemv_swiglu("bf16", d["A"], None, d["x"], None, y, I, K, 1)
    y2 = torch.empty_like(y)
    g.gemv_swiglu("bf16", d["A"], None, d["x"], None, y2, I, K, 1)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    U.assert_close_swiglu("bf16", y, y_ref, gate, up, adg, adu, what="swiglu 14336x4096")


def test_swiglu_unsupported_cases():
    I, K = 64, 1040
    A = torch.randn(2 * I * K + 8, dtype=torch.bfloat16, device="cuda")
    x = torch.randn(1, K, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(1, I, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(g.GemvError) as e:     # rows not 16-byte aligned
        g.gemv_swiglu("bf16", A[1:1 + 2 * I * K], None, x, None, y, I, K, 1)
    assert e.value.status == 2
    Kb = 32768                                  # 16 x 32768 bf16 of x: too large to stage
    A2 = torch.zeros(2 * 8, Kb, dtype=torch.bfloat16, device="cuda")
    x2 = torch.zeros(16, Kb, dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty(16, 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(g.GemvError) as e:
        g.gemv_swiglu("bf16", A2, None, x2, None, y2, 8, Kb, 16)
    assert e.value.status == 2
