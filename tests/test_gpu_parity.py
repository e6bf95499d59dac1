"""libgemv on the GPU against the CPU oracle, element by element.

* every benchmark configuration at full size, through the default dispatch (the
  launch configuration the benchmark times), all outputs, twice (bitwise equal);
* every kernel family forced on small shapes that span several tiles and end in
  ragged tails, each storage type, B in 1..16, with and without bias;
* edge cases: K = 0, M or B = 0, unaligned rows, IEEE specials, guard bytes
  around y, rejected arguments on real buffers, a non-default stream.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import decode_linear_layers_gb300 as g
import oracle
import workloads as W
from tests import gpu_util as U
from tests import oracle_pins as P

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _auto_dispatch():
    g.force_kernel("auto")
    yield
    g.force_kernel("auto")


# ------------------------------------------------------------- full-size configs
@pytest.mark.parametrize("name", [w.name for w in W.CONFIGS])
def test_config_full_size(name):
    w = W.BY_NAME[name]
    inp = W.make_inputs(w)
    y_ref, absdot = U.oracle_for(w.dtype, inp)
    d = U.to_device(inp)
    y1 = U.run_gpu(w.dtype, d, w.M, w.K, w.B)
    plan = g.last_plan()
    y2 = U.run_gpu(w.dtype, d, w.M, w.K, w.B)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16) if y1.dtype != torch.float32 else y1.view(torch.int32),
                       y2.view(torch.int16) if y2.dtype != torch.float32 else y2.view(torch.int32)), \
        "results differ between two identical calls"
    worst = U.assert_close(w.dtype, y1, y_ref, absdot, what=f"{name} [{plan['kernel_name']}]")
    assert worst <= 1.0


# ------------------------------------------------------------- forced kernels
SHAPES = [  # (M, K) with several tiles and ragged tails for each kernel family
    (1, 16), (37, 48), (300, 160), (1001, 1024), (77, 4112), (5, 20000),
]
FORCED = [("rows_per_warp", 0), ("rows_per_warp", 1), ("rows_per_warp", 16),
          ("warp_per_row", 0), ("block_per_row", 0), ("split_k", 0), ("split_k", 3),
          ("split_k", 7), ("batched", 1), ("batched", 2), ("batched", 3), ("scalar", 4), ("scalar", 32),
          ("stream", 0), ("stream", 1), ("stream", 3), ("xsplit", 0)]


def xsplit_feasible(dtype, K, B):
    """Mirror of the dispatcher's XSPLIT rule: B <= 4, 16-byte chunks, at most 4
    chunks per thread of 512 and at most 64 fp32 x values per thread."""
    vec = {"f32": 4, "f16": 8, "bf16": 8, "w8": 16}[dtype]
    if K % vec or K == 0 or B > 4:
        return False
    nb = 1 << (B - 1).bit_length()
    per = -(-(K // vec) // 512)
    j = 1 << (per - 1).bit_length()
    return j <= 4 and j * nb * vec <= 64


def forced_feasible(dtype, kernel, param, K, B):
    """Mirror of the dispatcher's rules for honouring a forced kernel."""
    sa = {"f32": 4, "f16": 2, "bf16": 2, "w8": 1}[dtype]
    sx = 4 if dtype == "f32" else 2
    nb = 1 << (B - 1).bit_length()
    if kernel == "batched":
        # param = variant + 1: 1 the row-pair kernel (x as stored in 200 KB), 2 the
        # cp.async ring (x, or its share of one of at most 64 K slices, as stored
        # next to a 64 KB ring in 227 KB), 3 the mixed-precision ring
        vec = {"f32": 4, "f16": 8, "bf16": 8, "w8": 16}[dtype]
        nch = K // vec
        ring = any(nb * (-(-nch // s)) * vec * sx + 65536 <= 227 * 1024 for s in range(1, 65))
        rowpair = nb * K * sx <= 200 * 1024
        mixed = dtype in ("f16", "bf16") and ring
        ok = {0: ring or rowpair, 1: rowpair, 2: ring, 3: mixed}.get(param, False)
        return B >= 2 and ok
    if kernel == "split_k":
        return K * sa // 16 >= 2
    if kernel == "stream":
        return B == 1
    if kernel == "xsplit":
        return xsplit_feasible(dtype, K, B)
    return True


@pytest.mark.parametrize("dtype", W.DTYPES)
@pytest.mark.parametrize("kernel,param", FORCED)
def test_forced_kernel(dtype, kernel, param):
    seed = 0
    for (M, K) in SHAPES:
        if dtype == "w8" and K % 16:
            K += 16 - K % 16
        for B in (1, 3, 16):
            if kernel == "rows_per_warp" and K > 4096:
                continue  # rows of thousands of chunks on 1..16 lanes: slow, not a target
            bias = (B + M) % 2 == 0
            w = W.small(dtype, M, K, B, bias, seed=seed)
            seed += 1
            inp = W.make_inputs(w)
            y_ref, absdot = U.oracle_for(dtype, inp)
            d = U.to_device(inp)
            g.force_kernel(kernel, param)
            y = U.run_gpu(dtype, d, M, K, B)
            plan = g.last_plan()
            g.force_kernel("auto")
            if forced_feasible(dtype, kernel, param, K, B):
                assert plan["kernel"] == g.KERNELS[kernel], (plan, kernel)
                if kernel == "batched" and param > 0:
                    assert plan["variant"] == param - 1, (plan, param)
            U.assert_close(dtype, y, y_ref, absdot, with_rounding=True,
                           what=f"{dtype} {kernel}/{param} M={M} K={K} B={B} bias={bias}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_rowpair_four_rows(dtype):
    # 16 vectors of 16-bit rows: the row-pair kernel carries 4 rows per warp and sums
    # them in two reduce-scatter butterflies.  Row counts that leave 1..3 rows in the
    # last group, vectors 9..16 (the rest zero-padded), one chunk and a ragged chunk
    # count; forced and by the dispatcher; repeats bitwise equal
    seed = 500
    for M in (1, 3, 6, 4097):
        for K in (8, 4104):
            for B in (9, 13, 16):
                bias = (M + B) % 2 == 1
                w = W.small(dtype, M, K, B, bias, seed=seed)
                seed += 1
                inp = W.make_inputs(w)
                y_ref, absdot = U.oracle_for(dtype, inp)
                d = U.to_device(inp)
                for kernel, param in (("batched", 1), ("auto", 0)):
                    g.force_kernel(kernel, param)
                    y1 = U.run_gpu(dtype, d, M, K, B)
                    plan = g.last_plan()
                    y2 = U.run_gpu(dtype, d, M, K, B)
                    g.force_kernel("auto")
                    if kernel == "batched":
                        assert plan["variant"] == g.BATCHED_ROWPAIR and plan["rows_per_warp"] == 4, plan
                    torch.cuda.synchronize()
                    assert torch.equal(y1, y2), "results differ between two identical calls"
                    U.assert_close(dtype, y1, y_ref, absdot, with_rounding=True,
                                   what=f"{dtype} {kernel} M={M} K={K} B={B} bias={bias}")


@pytest.mark.parametrize("dtype,M,K,xs", [("w8", 7300, 8192, 2), ("w8", 7300, 32768, 1),
                                          ("w4", 2500, 8192, 2), ("w4", 2500, 32768, 1)])
def test_one_vector_ring(dtype, M, K, xs):
    # one vector of int8/int4 rows in the ring kernel (4 steps of 4 rows in flight per
    # warp), x staged as fp32 (xs = 2) or, for long rows, as stored (xs = 1); a ragged
    # last row group; sampled rows against the oracle, repeats bitwise equal
    w = W.small(dtype, M, K, 1, True, seed=M + K)
    inp = W.make_inputs(w)
    d = U.to_device(inp)
    y1 = U.run_gpu(dtype, d, M, K, 1)
    plan = g.last_plan()
    assert plan["kernel_name"] == "batched" and plan["variant"] == g.BATCHED_RING, plan
    assert plan["nb"] == 1 and plan["rows_per_warp"] == 4 and plan["unroll"] == 4 and plan["x_staging"] == xs, plan
    y2 = U.run_gpu(dtype, d, M, K, 1)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2), "results differ between two identical calls"
    rows = np.unique(np.append(np.random.default_rng(2).choice(M, size=150, replace=False), [M - 1]))
    sub = {k: (None if inp[k] is None else inp[k][rows]) for k in ("A", "bias", "scale")}
    sub["x"] = inp["x"]
    y_ref, absdot = U.oracle_for(dtype, sub)
    U.assert_close(dtype, y1[:, rows], y_ref, absdot, with_rounding=True, what=f"{dtype} {M}x{K} B=1 xs={xs}")


@pytest.mark.parametrize("dtype,M,K,B", [("bf16", 4096, 14336, 16), ("w8", 8192, 8192, 16),
                                         ("f16", 3000, 14336, 9), ("bf16", 2500, 30000, 5),
                                         ("f32", 1000, 20000, 12), ("bf16", 1024, 16384, 8)])
def test_batched_k_slices(dtype, M, K, B):
    # x[0..B) too large to stage whole: the ring over K slices, partial sums and a
    # fixed-order second pass (sampled rows against the oracle, with bias; repeats
    # bitwise equal; the fused epilogue through the second pass)
    if dtype == "w8":
        K -= K % 16
    w = W.small(dtype, M, K, B, True, seed=M + K)
    inp = W.make_inputs(w)
    d = U.to_device(inp)
    y1 = U.run_gpu(dtype, d, M, K, B)
    plan = g.last_plan()
    assert plan["kernel_name"] == "batched" and plan["splits"] > 1, plan
    y2 = U.run_gpu(dtype, d, M, K, B)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2), "results differ between two identical calls"
    rows = np.sort(np.random.default_rng(1).choice(M, size=min(M, 160), replace=False))
    sub = {"A": inp["A"][rows], "x": inp["x"], "bias": inp["bias"][rows],
           "scale": None if inp["scale"] is None else inp["scale"][rows]}
    y_ref, absdot = U.oracle_for(dtype, sub)
    U.assert_close(dtype, y1[:, rows], y_ref, absdot, with_rounding=True,
                   what=f"{dtype} {M}x{K} B={B} splits={plan['splits']} variant={plan['variant']}")
    # SiLU and an in-place residual, applied by the second pass
    xdt = U.out_dtype(dtype)
    r = (torch.randn(B, M, generator=torch.Generator().manual_seed(7)) * 2).to(xdt)
    sub_r = r[:, rows].contiguous()
    y_ref2, _, absdot2 = oracle.gemv_ex(dtype, W.storage_bits(sub["A"]), W.storage_bits(sub["x"]),
                                        W.storage_bits(sub["bias"]), None if sub["scale"] is None else sub["scale"].numpy(),
                                        residual=W.storage_bits(sub_r), act=1, nthreads=U.threads())
    y = r.cuda()
    g.gemv_ex(dtype, d["A"], d["scale"], d["x"], d["bias"], y, y, M, K, B, 1)
    assert g.last_plan()["splits"] > 1
    U.assert_close_ex(dtype, y[:, rows], y_ref2, absdot2, 1, what=f"{dtype} {M}x{K} B={B} k-slices silu+res")


@pytest.mark.parametrize("dtype", W.DTYPES)
def test_all_batch_sizes(dtype):
    for B in range(1, 17):
        w = W.small(dtype, 257, 512, B, True, seed=100 + B)
        inp = W.make_inputs(w)
        y_ref, absdot = U.oracle_for(dtype, inp)
        y = U.run_gpu(dtype, U.to_device(inp), w.M, w.K, B)
        U.assert_close(dtype, y, y_ref, absdot, with_rounding=True, what=f"{dtype} B={B}")


@pytest.mark.parametrize("dtype", W.DTYPES)
def test_small_k_sweep(dtype):
    # every K from 0 to 70: rows-per-warp lane counts, scalar tails, K = 0
    step = 16 if dtype == "w8" else 1
    for K in range(0, 71, step):
        w = W.small(dtype, 133, K, 2, K % 3 == 0, seed=200 + K)
        inp = W.make_inputs(w)
        y_ref, absdot = U.oracle_for(dtype, inp)
        y = U.run_gpu(dtype, U.to_device(inp), w.M, K, 2)
        U.assert_close(dtype, y, y_ref, absdot, with_rounding=True, what=f"{dtype} K={K}")


# ------------------------------------------------------------- edge cases
@pytest.mark.parametrize("dtype", W.DTYPES)
def test_unaligned_rows(dtype):
    # A and x start one element past a 16-byte boundary: the scalar kernel
    M, K, B = 211, 1040, 3
    w = W.small(dtype, M, K, B, True, seed=300)
    inp = W.make_inputs(w)
    y_ref, absdot = U.oracle_for(dtype, inp)
    d = U.to_device(inp)
    for key in ("A", "x"):
        flat = d[key].reshape(-1)
        buf = torch.empty(flat.numel() + 16, dtype=flat.dtype, device="cuda")
        buf[1:1 + flat.numel()] = flat
        d[key] = buf[1:1 + flat.numel()]
    y = U.run_gpu(dtype, d, M, K, B)
    assert g.last_plan()["kernel"] == g.KERNELS["scalar"]
    U.assert_close(dtype, y, y_ref, absdot, with_rounding=True, what=f"{dtype} unaligned")


@pytest.mark.parametrize("dtype", W.DTYPES)
def test_guard_bytes_untouched(dtype):
    for kernel, param, B in (("auto", 0, 4), ("split_k", 4, 4), ("batched", 1, 4), ("batched", 2, 9),
                             ("batched", 1, 9), ("batched", 3, 16), ("batched", 3, 2),
                             ("block_per_row", 0, 4), ("rows_per_warp", 2, 4), ("scalar", 32, 4),
                             ("stream", 0, 1), ("warp_per_row", 0, 3), ("xsplit", 0, 3), ("xsplit", 0, 1)):
        M, K = 333, 256
        w = W.small(dtype, M, K, B, False, seed=400)
        d = U.to_device(W.make_inputs(w))
        n = B * M
        buf = torch.full((n + 2048,), 7, dtype=U.out_dtype(dtype), device="cuda")
        y = buf[1024:1024 + n]
        g.force_kernel(kernel, param)
        U.call(dtype, d, y, M, K, B)
        g.force_kernel("auto")
        torch.cuda.synchronize()
        assert bool((buf[:1024] == 7).all()) and bool((buf[1024 + n:] == 7).all()), kernel


@pytest.mark.parametrize("dtype", W.DTYPES)
def test_k_zero_is_bias(dtype):
    M, B = 100, 3
    w = W.small(dtype, M, 0, B, True, seed=500)
    inp = W.make_inputs(w)
    d = U.to_device(inp)
    y = U.run_gpu(dtype, {"A": None, "x": None, "bias": d["bias"], "scale": d["scale"]}, M, 0, B)
    want = inp["bias"].to(U.out_dtype(dtype))
    assert torch.equal(y.cpu(), want.unsqueeze(0).expand(B, M))
    y = U.run_gpu(dtype, {"A": None, "x": None, "bias": None, "scale": d["scale"]}, M, 0, B)
    assert bool((y == 0).all())


def test_empty_problems():
    y = torch.full((4,), 3.0, device="cuda")
    a = torch.ones(4, 8, device="cuda")
    g.gemv_f32(a, a, None, y, 0, 8, 1)
    g.gemv_f32(a, a, None, y, 4, 8, 0)
    torch.cuda.synchronize()
    assert bool((y == 3.0).all())


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_ieee_specials(dtype):
    M, K = 64, 64
    A = np.zeros((M, K))
    A[np.arange(M), np.arange(M)] = 1.0       # identity
    xv = np.arange(1, K + 1, dtype=np.float64)
    xv[3] = np.inf
    xv[7] = -np.inf
    tdt = U.out_dtype(dtype)
    At = torch.tensor(A, dtype=tdt)
    xt = torch.tensor(xv[None, :], dtype=tdt)
    # identity x inf gives nan in the rows whose diagonal misses the inf (inf * 0)
    y = U.run_gpu(dtype, U.to_device({"A": At, "x": xt, "bias": None, "scale": None}), M, K, 1)
    yr, ad = U.oracle_for(dtype, {"A": At, "x": xt, "bias": None, "scale": None})
    U.assert_close(dtype, y, yr, ad, what="inf in x")
    xt2 = xt.clone()
    xt2[0, 5] = float("nan")
    y = U.run_gpu(dtype, U.to_device({"A": At, "x": xt2, "bias": None, "scale": None}), M, K, 1)
    assert bool(torch.isnan(y).all())


def test_rejected_arguments_on_real_buffers():
    A = torch.randn(64, 64, device="cuda")
    x = torch.randn(1, 64, device="cuda")
    with pytest.raises(g.GemvError) as e:
        g.gemv_f32(A, x, None, A.reshape(-1)[:64], 64, 64, 1)   # y overlaps A
    assert e.value.status == 1
    with pytest.raises(g.GemvError) as e:
        g.gemv_f32(A, torch.randn(17, 64, device="cuda"), None, torch.empty(64 * 17, device="cuda"),
                   64, 64, 17)
    assert e.value.status == 2
    with pytest.raises(ValueError):
        g.gemv_f32(A, x, None, torch.empty(10, device="cuda"), 64, 64, 1)  # y too small


def test_non_default_stream_and_launch_count():
    w = W.small("bf16", 4096, 1024, 1, True, seed=600)
    inp = W.make_inputs(w)
    y_ref, absdot = U.oracle_for("bf16", inp)
    d = U.to_device(inp)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    before = g.launch_count()
    with torch.cuda.stream(s):
        y = torch.empty((1, w.M), dtype=torch.bfloat16, device="cuda")
        U.call("bf16", d, y, w.M, w.K, 1, stream=s)
    s.synchronize()
    assert g.launch_count() == before + 1
    U.assert_close("bf16", y, y_ref, absdot, what="side stream")


@pytest.mark.parametrize("dtype", W.DTYPES)
def test_exact_closed_forms_on_gpu(dtype):
    # A = 1, x = 1 gives y = K exactly (times the w8 scale) in every kernel family
    xk = P.xkind(dtype)
    for kernel, param, B in (("auto", 0, 2), ("warp_per_row", 0, 2), ("block_per_row", 0, 2),
                             ("split_k", 5, 2), ("batched", 2, 2), ("batched", 2, 12), ("batched", 1, 2),
                             ("batched", 1, 12), ("batched", 3, 12), ("scalar", 32, 2),
                             ("stream", 0, 1), ("xsplit", 0, 2), ("xsplit", 0, 4)):
        M, K = 96, 4096
        A = torch.ones(M, K, dtype=torch.int8 if dtype == "w8" else U.out_dtype(dtype))
        x = torch.ones(B, K, dtype=U.out_dtype(xk if dtype != "w8" else "bf16"))
        scale = torch.full((M,), 0.5) if dtype == "w8" else None
        g.force_kernel(kernel, param)
        y = U.run_gpu(dtype, U.to_device({"A": A, "x": x, "bias": None, "scale": scale}), M, K, B)
        g.force_kernel("auto")
        want = 0.5 * K if dtype == "w8" else float(K)
        assert bool((y.double() == want).all()), (dtype, kernel)
