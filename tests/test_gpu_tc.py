"""The tensor-core kernel (GEMV_KERNEL_TC): fp16/bf16 with 17..256 vectors.

* every batch size class (N = B rounded up to 16 from 32 to 256, ragged B), both
  storage types, shapes with ragged M (partial 128-row tiles) and ragged K (partial
  64-column stages), with and without split-K, with and without bias;
* decode-size matrices on sampled rows (the oracle on a subset of A's rows);
* bit-identical repeats, K = 0, one row, the fused epilogue, guard bytes around y,
  CUDA-graph capture (the split-K scratch comes from the stream-ordered pool);
* the kernel forced for B <= 16 (N = 16);
* bounded waits: a launch that skips one MMA reports GEMV_ERR_DEVICE_TIMEOUT through
  gemv_get_device_status, without a fault or a hang, and the next launch is normal;
* the persistent form (one CTA per SM over its tiles, two accumulators) forced on
  small and ragged shapes and chosen by the dispatcher for many tiles, with its
  epilogue and its bounded waits.
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

HALF = ("f16", "bf16")


@pytest.fixture(autouse=True)
def _auto_dispatch():
    g.force_kernel("auto")
    g.test_stall(False)
    yield
    g.force_kernel("auto")
    g.test_stall(False)


def _bits(t):
    return t.view(torch.int16)


@pytest.mark.parametrize("dtype", HALF)
@pytest.mark.parametrize("B", [17, 24, 32, 48, 64, 100, 128, 200, 256])
def test_tc_parity(dtype, B):
    seed = B
    for (M, K) in ((128, 64), (300, 1000), (1, 4096), (1000, 520)):
        bias = (M + B) % 2 == 0
        w = W.small(dtype, M, K, B, bias, seed=seed)
        seed += 1
        inp = W.make_inputs(w)
        y_ref, absdot = U.oracle_for(dtype, inp)
        d = U.to_device(inp)
        y1 = U.run_gpu(dtype, d, M, K, B)
        p = g.last_plan()
        assert p["kernel_name"] == "tc" and p["nb"] == -(-B // 16) * 16, p
        y2 = U.run_gpu(dtype, d, M, K, B)
        torch.cuda.synchronize()
        assert torch.equal(_bits(y1), _bits(y2)), "results differ between two identical calls"
        U.assert_close(dtype, y1, y_ref, absdot, with_rounding=True,
                       what=f"{dtype} tc M={M} K={K} B={B} splits={p['splits']} bias={bias}")
    assert g.device_status() == (g.SUCCESS, 0)


@pytest.mark.parametrize("dtype,M,K,B", [("bf16", 14336, 4096, 32), ("bf16", 4096, 14336, 128),
                                         ("f16", 28672, 4096, 64), ("bf16", 6144, 4096, 256),
                                         ("f16", 40000, 4096, 48)])
def test_tc_decode_sizes_sampled_rows(dtype, M, K, B):
    w = W.small(dtype, M, K, B, True, seed=5)
    inp = W.make_inputs(w)
    d = U.to_device(inp)
    y = U.run_gpu(dtype, d, M, K, B)
    torch.cuda.synchronize()
    # more tiles than two CTAs per SM hold: the persistent form (192 threads)
    p = g.last_plan()
    assert (p["threads"] == 192) == (-(-M // 128) > 2 * torch.cuda.get_device_properties(0).multi_processor_count), p
    rows = np.sort(np.random.default_rng(0).choice(M, size=192, replace=False))
    sub = {"A": inp["A"][rows], "x": inp["x"], "bias": inp["bias"][rows], "scale": None}
    y_ref, absdot = U.oracle_for(dtype, sub)
    U.assert_close(dtype, y[:, rows], y_ref, absdot, what=f"{dtype} tc {M}x{K} B={B} sampled rows")


@pytest.mark.parametrize("name", [w.name for w in W.TC_CONFIGS])
def test_tc_configs_full_size_sampled_rows(name):
    # the benchmark's tensor-core workloads at full size, in the launch configuration
    # the bench times (split K in clusters, the deep ring, the persistent form):
    # repeats bitwise equal, 256 sampled rows (the last ones among them) against the oracle
    w = W.BY_NAME[name]
    inp = W.make_inputs(w)
    d = U.to_device(inp)
    y1 = U.run_gpu(w.dtype, d, w.M, w.K, w.B)
    p = g.last_plan()
    y2 = U.run_gpu(w.dtype, d, w.M, w.K, w.B)
    torch.cuda.synchronize()
    assert p["kernel_name"] == "tc", p
    assert torch.equal(_bits(y1), _bits(y2)), "results differ between two identical calls"
    rng = np.random.default_rng(w.M + w.B)
    rows = np.unique(np.concatenate([rng.choice(w.M, size=224, replace=False), np.arange(w.M - 32, w.M)]))
    sub = {"A": inp["A"][rows], "x": inp["x"], "bias": None if inp["bias"] is None else inp["bias"][rows],
           "scale": None}
    y_ref, absdot = U.oracle_for(w.dtype, sub)
    U.assert_close(w.dtype, y1[:, rows], y_ref, absdot, with_rounding=True,
                   what=f"{name} [threads {p['threads']}, splits {p['splits']}] sampled rows")


@pytest.mark.parametrize("dtype", HALF)
def test_tc_k_zero_and_one_row(dtype):
    M, B = 200, 40
    bias = torch.randn(M, generator=torch.Generator().manual_seed(1)).to(U.out_dtype(dtype)).cuda()
    y = torch.full((B, M), 3.0, dtype=U.out_dtype(dtype), device="cuda")
    empty = torch.empty(0, dtype=U.out_dtype(dtype), device="cuda")
    getattr(g, f"gemv_{dtype}")(empty, empty, bias, y, M, 0, B)
    torch.cuda.synchronize()
    assert torch.equal(y, bias.expand(B, M))


@pytest.mark.parametrize("dtype", HALF)
@pytest.mark.parametrize("B", [1, 5, 16])
def test_tc_forced_small_batches(dtype, B):
    M, K = 700, 2048
    w = W.small(dtype, M, K, B, True, seed=40 + B)
    inp = W.make_inputs(w)
    y_ref, absdot = U.oracle_for(dtype, inp)
    g.force_kernel("tc")
    y = U.run_gpu(dtype, U.to_device(inp), M, K, B)
    assert g.last_plan()["kernel_name"] == "tc" and g.last_plan()["nb"] == 16
    U.assert_close(dtype, y, y_ref, absdot, with_rounding=True, what=f"{dtype} tc forced B={B}")


@pytest.mark.parametrize("dtype", HALF)
def test_tc_epilogue(dtype):
    M, K, B = 1000, 4096, 64
    w = W.small(dtype, M, K, B, True, seed=77)
    inp = W.make_inputs(w)
    xdt = U.out_dtype(dtype)
    r = (torch.randn(B, M, generator=torch.Generator().manual_seed(3)) * 2).to(xdt)
    y_ref, _, absdot = oracle.gemv_ex(dtype, W.storage_bits(inp["A"]), W.storage_bits(inp["x"]),
                                      W.storage_bits(inp["bias"]), None, residual=W.storage_bits(r), act=1,
                                      nthreads=U.threads())
    d = U.to_device(inp)
    y = r.cuda()
    g.gemv_ex(dtype, d["A"], None, d["x"], d["bias"], y, y, M, K, B, 1)
    assert g.last_plan()["kernel_name"] == "tc"
    U.assert_close_ex(dtype, y, y_ref, absdot, 1, what=f"{dtype} tc silu + residual in place")


@pytest.mark.parametrize("dtype", HALF)
def test_tc_unsplit_epilogue_forms(dtype):
    # tiles enough to fill the SMs without a K split: the outputs leave through shared
    # memory, 8 rows of a vector per 16-byte store where M % 8 == 0 and y (and the
    # residual) are 16-byte aligned, element by element otherwise.  Both forms, with
    # the activation and a residual (separate and in place), against the oracle; the
    # bytes around y untouched
    K, B = 256, 40
    for M, off, inplace in ((19200, 0, False), (19200, 0, True), (19200, 1, False), (19196, 0, True)):
        w = W.small(dtype, M, K, B, True, seed=M + off)
        inp = W.make_inputs(w)
        xdt = U.out_dtype(dtype)
        r = (torch.randn(B, M, generator=torch.Generator().manual_seed(off + 9)) * 2).to(xdt)
        y_ref, _, absdot = oracle.gemv_ex(dtype, W.storage_bits(inp["A"]), W.storage_bits(inp["x"]),
                                          W.storage_bits(inp["bias"]), None, residual=W.storage_bits(r), act=1,
                                          nthreads=U.threads())
        d = U.to_device(inp)
        n = B * M
        buf = torch.full((n + 64,), 7, dtype=xdt, device="cuda")
        y = buf[8 + off:8 + off + n]
        res = r.cuda()
        if inplace:
            y.copy_(res.view(-1))
            res = y
        g.gemv_ex(dtype, d["A"], None, d["x"], d["bias"], res.view(-1) if res is not y else y, y, M, K, B, 1)
        p = g.last_plan()
        assert p["kernel_name"] == "tc" and p["splits"] == 1, p
        torch.cuda.synchronize()
        assert bool((buf[:8 + off] == 7).all()) and bool((buf[8 + off + n:] == 7).all())
        U.assert_close_ex(dtype, y.view(B, M), y_ref, absdot, 1,
                          what=f"{dtype} tc unsplit M={M} y offset {off} in place {inplace}")


PERSIST = 1_000_000  # force parameter: the persistent form


def _sampled(dtype, inp, y, rows, what):
    sub = {"A": inp["A"][rows], "x": inp["x"], "bias": None if inp["bias"] is None else inp["bias"][rows],
           "scale": None}
    y_ref, absdot = U.oracle_for(dtype, sub)
    U.assert_close(dtype, y[:, rows], y_ref, absdot, with_rounding=True, what=what)


@pytest.mark.parametrize("dtype", HALF)
@pytest.mark.parametrize("M,K,B", [(60001, 520, 17), (58368, 256, 64), (40000, 1000, 200), (300, 4096, 33)])
def test_tc_persistent(dtype, M, K, B):
    # one CTA per SM walking its tiles with two tensor-memory accumulators: several
    # tiles per CTA (both accumulators reused), a partial last tile, a partial last
    # k-tile, N from 32 to 208 (the two accumulators take all 512 columns), fewer tiles
    # than SMs; sampled rows (with the last ones) against the oracle, repeats bitwise equal
    w = W.small(dtype, M, K, B, (M + B) % 2 == 1, seed=M + B)
    inp = W.make_inputs(w)
    d = U.to_device(inp)
    g.force_kernel("tc", PERSIST)
    y1 = U.run_gpu(dtype, d, M, K, B)
    p = g.last_plan()
    y2 = U.run_gpu(dtype, d, M, K, B)
    g.force_kernel("auto")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert p["threads"] == 192 and p["splits"] == 1 and p["grid"] == min(-(-M // 128), sms), p
    torch.cuda.synchronize()
    assert torch.equal(_bits(y1), _bits(y2)), "results differ between two identical calls"
    rng = np.random.default_rng(M)
    rows = np.unique(np.concatenate([rng.choice(M, size=min(M, 160), replace=False), np.arange(max(0, M - 40), M)]))
    _sampled(dtype, inp, y1, rows, f"{dtype} tc persistent M={M} K={K} B={B}")
    assert g.device_status() == (g.SUCCESS, 0)


@pytest.mark.parametrize("dtype", HALF)
def test_tc_persistent_epilogue(dtype):
    M, K, B = 40000, 256, 40
    w = W.small(dtype, M, K, B, True, seed=78)
    inp = W.make_inputs(w)
    xdt = U.out_dtype(dtype)
    r = (torch.randn(B, M, generator=torch.Generator().manual_seed(4)) * 2).to(xdt)
    y_ref, _, absdot = oracle.gemv_ex(dtype, W.storage_bits(inp["A"]), W.storage_bits(inp["x"]),
                                      W.storage_bits(inp["bias"]), None, residual=W.storage_bits(r), act=1,
                                      nthreads=U.threads())
    d = U.to_device(inp)
    y = r.cuda()
    g.force_kernel("tc", PERSIST)
    g.gemv_ex(dtype, d["A"], None, d["x"], d["bias"], y, y, M, K, B, 1)
    assert g.last_plan()["threads"] == 192
    g.force_kernel("auto")
    U.assert_close_ex(dtype, y, y_ref, absdot, 1, what=f"{dtype} tc persistent silu + residual in place")


def test_tc_persistent_bounded_wait():
    M, K, B = 40000, 512, 32
    w = W.small("bf16", M, K, B, True, seed=991)
    inp = W.make_inputs(w)
    d = U.to_device(inp)
    assert g.device_status() == (g.SUCCESS, 0)
    # CTA 0 skips the MMAs of its last k-tile: its epilogue's wait for that tile's
    # accumulator runs out after 50 ms; the CTA drains and returns, the status word says
    # so, the other CTAs finish normally, and the next launch is normal
    g.force_kernel("tc", PERSIST)
    g.test_stall(True, 50_000_000)
    y = torch.zeros(B, M, dtype=torch.bfloat16, device="cuda")
    U.call("bf16", d, y, M, K, B)
    assert g.last_plan()["threads"] == 192
    st, bits = g.device_status()
    assert st == g.ERR_DEVICE_TIMEOUT and bits & 16, (st, bits)
    g.test_stall(False)
    y2 = U.run_gpu("bf16", d, M, K, B)
    g.force_kernel("auto")
    assert g.device_status() == (g.SUCCESS, 0)
    _sampled("bf16", inp, y2, np.arange(0, M, 97), "tc persistent after a timeout")


def test_tc_guard_bytes():
    M, K, B = 333, 256, 40
    w = W.small("bf16", M, K, B, False, seed=400)
    d = U.to_device(W.make_inputs(w))
    n = B * M
    buf = torch.full((n + 2048,), 7, dtype=torch.bfloat16, device="cuda")
    y = buf[1024:1024 + n]
    U.call("bf16", d, y, M, K, B)
    torch.cuda.synchronize()
    assert bool((buf[:1024] == 7).all()) and bool((buf[1024 + n:] == 7).all())


@pytest.mark.parametrize("M,K,B,persist", [(4096, 4096, 32, False), (40000, 512, 48, True)])
def test_tc_in_cuda_graph(M, K, B, persist):
    # split K (the slices summed in the kernel, one cluster per tile) and the persistent
    # form (two launches back to back: the second's tensor memory and stages after the
    # first's under the programmatic launch overlap), captured and replayed
    w = W.small("bf16", M, K, B, False, seed=991)
    d = U.to_device(W.make_inputs(w))
    y = torch.empty(B, M, dtype=torch.bfloat16, device="cuda")
    U.call("bf16", d, y, M, K, B)
    p = g.last_plan()
    assert (p["threads"] == 192 and p["splits"] == 1) if persist else p["splits"] > 1, p
    torch.cuda.synchronize()
    eager = y.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        U.call("bf16", d, y, M, K, B)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    y.zero_()
    y2 = torch.empty_like(y)
    with torch.cuda.graph(graph):
        U.call("bf16", d, y, M, K, B)
        U.call("bf16", d, y2, M, K, B)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(_bits(y), _bits(eager)) and torch.equal(_bits(y2), _bits(eager))
    assert g.device_status() == (g.SUCCESS, 0)


def test_tc_bounded_wait_reports_timeout_and_recovers():
    M, K, B = 1024, 2048, 32
    w = W.small("bf16", M, K, B, True, seed=990)
    inp = W.make_inputs(w)
    y_ref, absdot = U.oracle_for("bf16", inp)
    d = U.to_device(inp)
    assert g.device_status() == (g.SUCCESS, 0)
    # CTA (0, 0) skips its last MMA: the wait for that stage's commit runs out after
    # 50 ms; the CTA drains its other MMAs and copies, frees its tensor memory and
    # returns, and the status word says so.  The other CTAs finish normally.
    g.test_stall(True, 50_000_000)
    y = torch.zeros(B, M, dtype=torch.bfloat16, device="cuda")
    U.call("bf16", d, y, M, K, B)
    st, bits = g.device_status()
    assert st == g.ERR_DEVICE_TIMEOUT and bits & 16, (st, bits)
    assert g.device_status() == (g.SUCCESS, 0), "the status word is cleared by the read"
    g.test_stall(False)
    y2 = U.run_gpu("bf16", d, M, K, B)
    assert g.device_status() == (g.SUCCESS, 0)
    U.assert_close("bf16", y2, y_ref, absdot, with_rounding=True, what="tc after a timeout")


@pytest.mark.parametrize("S", [1, 2, 3, 4, 5, 6, 7, 8])
def test_tc_every_cluster_size(S):
    """The K slices of a row tile are summed inside one thread-block cluster: CTA r of
    S owns rows [ceil(128 r / S), ceil(128 (r + 1) / S)), uneven when S does not divide
    128.  Every size from 1 to 8, forced through the test hook, on a ragged last tile
    (333 rows), a ragged K (2 S k-tiles of 128, the last one 88 columns) and a batch
    that is not a multiple of 16 (40 vectors, N = 48), against the oracle and bitwise
    from call to call."""
    M, K, B = 333, 256 * S - 40, 40
    w = W.small("bf16", M, K, B, True, seed=500 + S)
    inp = W.make_inputs(w)
    y_ref, absdot = U.oracle_for("bf16", inp)
    d = U.to_device(inp)
    g.force_kernel("tc", S * 1000)
    y1 = U.run_gpu("bf16", d, M, K, B)
    p = g.last_plan()
    assert p["kernel_name"] == "tc" and p["splits"] == S, p
    y2 = U.run_gpu("bf16", d, M, K, B)
    torch.cuda.synchronize()
    assert torch.equal(_bits(y1), _bits(y2)), "results differ between two identical calls"
    U.assert_close("bf16", y1, y_ref, absdot, with_rounding=True, what=f"tc cluster of {S}")
    assert g.device_status() == (g.SUCCESS, 0)
