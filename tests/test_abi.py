"""libgemv on the host, without a GPU: exports, argument checks, dispatcher rules.

No test here makes a call that passes validation, so nothing reaches a device:
every call either returns before any CUDA work or is a host-only function.
"""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

import decode_linear_layers_gb300 as g
from decode_linear_layers_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemv.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    build()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gemv_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("gemv_f32", "gemv_f16", "gemv_bf16", "gemv_w8", "gemv_status_string",
              "gemv_last_cuda_error", "gemv_plan_for"):
        assert n in names


def test_every_declared_symbol_is_exported():
    out = subprocess.run(["nm", "-D", "--defined-only", g.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (\w+)$", out, flags=re.M))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    L = ctypes.CDLL(g.LIB_PATH)
    for n in declared_functions():
        assert getattr(L, n) is not None


def test_header_compiles_as_c():
    src = '#include "gemv.h"\nint main(void){ gemv_plan_t p; return (int)sizeof(p) > 0 ? 0 : 1; }\n'
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER),
                        "-x", "c", "-", "-fsyntax-only"], input=src, text=True, capture_output=True)
    assert r.returncode == 0, r.stderr


def test_status_strings():
    assert g.status_string(0) == "GEMV_SUCCESS"
    assert g.status_string(1) == "GEMV_ERR_INVALID_VALUE"
    assert g.status_string(2) == "GEMV_ERR_UNSUPPORTED"
    assert g.status_string(3) == "GEMV_ERR_CUDA"
    assert g.status_string(99) == "GEMV_ERR_UNKNOWN"


# --------------------------------------------------------- argument validation
# Fake addresses: every call below must be rejected before any device work.
P = 1 << 32


def call(fn, *a):
    L = g.lib()
    return getattr(L, fn)(*a)


def test_negative_sizes_and_big_batch():
    for fn in ("gemv_f32", "gemv_f16", "gemv_bf16"):
        assert call(fn, P, P + 4096, None, P + 8192, -1, 4, 1, None) == 1
        assert call(fn, P, P + 4096, None, P + 8192, 4, -1, 1, None) == 1
        assert call(fn, P, P + 4096, None, P + 8192, 4, 4, -1, None) == 1
    # more than 16 vectors: fp32 never; fp16/bf16 up to 256 (tensor cores)
    assert call("gemv_f32", P, P + 4096, None, P + 8192, 4, 4, 17, None) == 2
    for fn in ("gemv_f16", "gemv_bf16"):
        assert call(fn, P, P + 4096, None, P + 8192, 4, 8, 257, None) == 2
    assert g.lib().gemv_w8(P, P + 64, P + 4096, None, P + 8192, 4, 4, 17, None) == 2


def test_empty_problems_succeed_without_device():
    # M == 0 or B == 0: nothing to do, no device touched
    assert call("gemv_f32", None, None, None, None, 0, 5, 1, None) == 0
    assert call("gemv_bf16", None, None, None, None, 7, 5, 0, None) == 0
    assert g.lib().gemv_w8(None, None, None, None, None, 0, 3, 2, None) == 0


def test_null_pointers():
    assert call("gemv_f32", P, P + 4096, None, None, 4, 4, 1, None) == 1      # y
    assert call("gemv_f32", None, P + 4096, None, P + 8192, 4, 4, 1, None) == 1  # A with K > 0
    assert call("gemv_f32", P, None, None, P + 8192, 4, 4, 1, None) == 1      # x with K > 0
    assert g.lib().gemv_w8(P, None, P + 4096, None, P + 8192, 4, 16, 1, None) == 1  # scale


def test_misaligned_pointers():
    assert call("gemv_f32", P + 2, P + 4096, None, P + 8192, 4, 4, 1, None) == 1
    assert call("gemv_f32", P, P + 4097, None, P + 8192, 4, 4, 1, None) == 1
    assert call("gemv_f32", P, P + 4096, P + 6, P + 8192, 4, 4, 1, None) == 1
    assert call("gemv_f32", P, P + 4096, None, P + 8193, 4, 4, 1, None) == 1
    assert call("gemv_bf16", P + 1, P + 4096, None, P + 8192, 4, 4, 1, None) == 1
    assert g.lib().gemv_w8(P + 1, P + 66, P + 4096, None, P + 8192, 4, 16, 1, None) == 1


def test_overlapping_output():
    # y inside A, y over x, y over bias, y over the w8 scale
    assert call("gemv_f32", P, P + 4096, None, P + 16, 4, 4, 1, None) == 1
    assert call("gemv_f32", P, P + 4096, None, P + 4100, 4, 4, 1, None) == 1
    assert call("gemv_f32", P, P + 4096, P + 8192, P + 8196, 4, 4, 1, None) == 1
    assert g.lib().gemv_w8(P, P + 8192, P + 4096, None, P + 8192, 4, 16, 1, None) == 1
    # touching but not overlapping is fine up to the device step; not called here


def test_size_overflow():
    big = 1 << 62
    assert call("gemv_f32", P, P + 4096, None, P + 8192, big, 16, 1, None) == 1
    assert call("gemv_f32", P, P + 4096, None, P + 8192, 16, big, 1, None) == 1


def test_force_kernel_validation():
    with pytest.raises(g.GemvError):
        g.force_kernel(99)
    with pytest.raises(g.GemvError):
        g.force_kernel("split_k", -1)
    g.force_kernel("auto")


# ------------------------------------------------------------- dispatcher rules
def test_plan_config_shapes():
    K = g.KERNELS
    assert g.plan_for("f32", 1024, 128, 1)["kernel"] == K["warp_per_row"]
    p = g.plan_for("f32", 16384, 16, 1)
    assert p["kernel"] == K["rows_per_warp"] and p["lanes_per_row"] == 4
    p = g.plan_for("f32", 16384, 32, 1)
    assert p["kernel"] == K["rows_per_warp"] and p["lanes_per_row"] == 8
    p = g.plan_for("f32", 16384, 4096, 1)
    assert p["kernel"] == K["stream"] and p["unroll"] == 2 and p["x_staging"] == 0
    assert p["threads"] == 512 and p["grid"] == 4 * 152
    p = g.plan_for("f16", 4096, 4096, 1)
    assert p["kernel"] == K["stream"] and p["unroll"] == 4 and p["x_staging"] == 1
    assert p["smem_bytes"] == 4096 * 2 and p["grid"] == 2 * 152
    p = g.plan_for("f16", 4096, 4096, 16)   # 16 vectors of 16-bit rows: the row-pair kernel, 4 rows per warp
    assert p["kernel"] == K["batched"] and p["nb"] == 16 and p["x_staging"] == 1
    assert p["variant"] == g.BATCHED_ROWPAIR
    assert p["smem_bytes"] == 16 * 4096 * 2 and p["rows_per_warp"] == 4 and p["unroll"] == 1 and p["grid"] == 152
    p = g.plan_for("f16", 4096, 4096, 8)    # fewer vectors: 2 rows per warp, 2 chunks each
    assert p["variant"] == g.BATCHED_ROWPAIR and p["rows_per_warp"] == 2 and p["unroll"] == 2
    p = g.plan_for("f32", 32768, 2048, 16)  # 16 fp32 vectors: 2 rows per warp
    assert p["variant"] == g.BATCHED_ROWPAIR and p["rows_per_warp"] == 2
    for M, Kd in ((14336, 4096), (4096, 14336)):
        assert g.plan_for("bf16", M, Kd, 1)["kernel"] == K["stream"]
    p = g.plan_for("bf16", 128256, 4096, 1)
    assert p["kernel"] == K["warp_per_row"] and p["grid"] == 152 * 32
    # one vector of fp32 on long rows the streaming warps would share unevenly: warp per row
    assert g.plan_for("f32", 4096, 32768, 1)["kernel"] == K["warp_per_row"]
    assert g.plan_for("f32", 14336, 4096, 1)["kernel"] == K["warp_per_row"]
    # long rows, few of them: the K-split kernel for 2 16-bit or 4 fp32 vectors
    assert g.plan_for("bf16", 1024, 16384, 2)["kernel"] == K["xsplit"]
    assert g.plan_for("f32", 8192, 8192, 4)["kernel"] == K["xsplit"]
    assert g.plan_for("bf16", 4096, 4096, 2)["kernel"] == K["batched"]
    # ... and up to 12288 rows of at most 8192 elements: the K-split kernel
    for M in (2048, 4096, 8192, 12288):
        assert g.plan_for("f32", M, 8192, 1)["kernel"] == K["xsplit"]
    assert g.plan_for("f32", 16384, 4096, 1)["kernel"] == K["stream"]
    # one vector of 16-bit or int8 rows from 12 rows per SM: the streaming kernel
    assert g.plan_for("bf16", 2048, 8192, 1)["kernel"] == K["stream"]
    # fp32 with 2 vectors from 8 rows per SM: the K-split kernel
    assert g.plan_for("f32", 2048, 8192, 2)["kernel"] == K["xsplit"]
    # one vector of int8 with fewer than 48 rows per SM: the streaming kernel
    assert g.plan_for("w8", 4096, 16384, 1)["kernel"] == K["stream"]
    p = g.plan_for("w8", 8192, 8192, 1)     # one vector of int8: the ring, 4 rows per warp, 4 steps
    assert p["kernel"] == K["batched"] and p["variant"] == g.BATCHED_RING and p["nb"] == 1
    assert p["x_staging"] == 2 and p["rows_per_warp"] == 4 and p["unroll"] == 4
    assert p["smem_bytes"] == 8192 * 4 + 128 * 1024  # one vector: a 16-slot (128 KB) ring
    p = g.plan_for("w8", 8192, 8192, 4)     # at most one ring row group per warp: the row pairs
    assert p["kernel"] == K["batched"] and p["variant"] == g.BATCHED_ROWPAIR and p["x_staging"] == 1
    assert p["rows_per_warp"] == 2 and p["smem_bytes"] == 4 * 8192 * 2
    p = g.plan_for("w8", 16384, 8192, 4)    # the ring: fp32 x (128 KB) + the 64 KB ring
    assert p["kernel"] == K["batched"] and p["variant"] == g.BATCHED_RING and p["x_staging"] == 2
    assert p["rows_per_warp"] == 4 and p["unroll"] == 2 and p["smem_bytes"] == 4 * 8192 * 4 + 64 * 1024


def test_plan_stream_needs_one_vector():
    # more than one vector never goes to the one-row streaming kernel
    for B in range(2, 17):
        assert g.plan_for("bf16", 8192, 32768, B)["kernel"] != g.KERNELS["stream"]
    # x larger than the streaming kernel's shared-memory budget is read through L1
    p = g.plan_for("bf16", 8192, 65536, 1)
    assert p["kernel"] == g.KERNELS["stream"] and p["x_staging"] == 0 and p["smem_bytes"] == 0


def test_plan_xsplit():
    K = g.KERNELS
    # fp32 with 2 vectors whose x slice fits 64 registers per thread
    for Kd, J in ((4096, 2), (8192, 4), (2048, 1)):
        p = g.plan_for("f32", 14336, Kd, 2)
        assert p["kernel"] == K["xsplit"] and p["unroll"] == J, (Kd, p)
        assert p["smem_bytes"] == 128 * 1024 and p["grid"] == 152
    # 16-bit and int8 types, and fp32 with 3..4 vectors, take the ring kernel; one
    # vector the streaming kernel
    for dt, Kd, B in (("f16", 4096, 4), ("bf16", 8192, 4), ("bf16", 14336, 2), ("f32", 4096, 3), ("w8", 8192, 4)):
        p = g.plan_for(dt, 14336, Kd, B)
        assert p["kernel"] == K["batched"], (dt, Kd, B, p)
        assert p["variant"] == (g.BATCHED_RING_MIXED if (dt, B) == ("bf16", 2) else g.BATCHED_RING), (dt, B, p)
    assert g.plan_for("bf16", 14336, 4096, 1)["kernel"] == K["stream"]
    assert g.plan_for("f32", 16384, 4096, 1)["kernel"] == K["stream"]
    # few rows per SM, or very many rows -> not the K-split kernel
    assert g.plan_for("f32", 1000, 4096, 2)["kernel"] != K["xsplit"]
    assert g.plan_for("f32", 128256, 4096, 2)["kernel"] != K["xsplit"]


def test_plan_batched_staging():
    K = g.KERNELS
    ring = 64 * 1024
    # the ring: fp32 x when x and the 64 KB ring fit in 227 KB, else x as stored
    p = g.plan_for("w8", 16384, 8192, 4)
    assert p["variant"] == g.BATCHED_RING and p["x_staging"] == 2 and p["smem_bytes"] == 4 * 8192 * 4 + ring
    p = g.plan_for("bf16", 16384, 16384, 4)
    assert p["variant"] == g.BATCHED_RING and p["x_staging"] == 1 and p["smem_bytes"] == 4 * 16384 * 2 + ring
    assert p["rows_per_warp"] == 4 and p["unroll"] == 2
    # at most one row pair per warp (M <= 2 x 16 warps x 152 SMs) and 4..16 vectors:
    # the row-pair kernel, x as stored
    p = g.plan_for("bf16", 4096, 14336, 4)
    assert p["variant"] == g.BATCHED_ROWPAIR and p["x_staging"] == 1 and p["smem_bytes"] == 4 * 14336 * 2
    assert g.plan_for("f16", 4096, 4096, 2)["variant"] == g.BATCHED_RING_MIXED
    assert g.plan_for("w8", 4096, 4096, 2)["variant"] == g.BATCHED_ROWPAIR  # up to one ring group per warp
    assert g.plan_for("w8", 14336, 4096, 2)["variant"] == g.BATCHED_RING
    p = g.plan_for("bf16", 16384, 4096, 8)  # vector pairs, 4 rows per warp, 2-step ring
    assert p["variant"] == g.BATCHED_RING and p["x_staging"] == 2 and p["rows_per_warp"] == 4 and p["unroll"] == 2
    # up to one ring row group per warp (M <= 4 x 16 x 152), 8 vectors of fp16/bf16 and
    # 4 of int8: the row pairs
    assert g.plan_for("bf16", 8192, 4096, 8)["variant"] == g.BATCHED_ROWPAIR
    assert g.plan_for("f32", 8192, 4096, 8)["variant"] == g.BATCHED_RING
    # 8 vectors of fp16/bf16 whose ring would read x as stored (fp32 x 192 KB): row pairs
    assert g.plan_for("f16", 16384, 6144, 8)["variant"] == g.BATCHED_ROWPAIR
    # 9..16 vectors of fp16/bf16/fp32 wherever x fits: the row pairs (int8 keeps the ring)
    p = g.plan_for("bf16", 14336, 4096, 16)
    assert p["variant"] == g.BATCHED_ROWPAIR and p["x_staging"] == 1 and p["smem_bytes"] == 16 * 4096 * 2
    p = g.plan_for("f16", 4866, 4096, 9)
    assert p["variant"] == g.BATCHED_ROWPAIR and p["smem_bytes"] == 16 * 4096 * 2
    assert g.plan_for("f32", 32768, 2048, 16)["variant"] == g.BATCHED_ROWPAIR
    assert g.plan_for("w8", 14336, 4096, 16)["variant"] == g.BATCHED_RING
    # x too large for the ring but within 200 KB: the row-pair kernel
    p = g.plan_for("bf16", 20000, 6144, 16)
    assert p["kernel"] == K["batched"] and p["variant"] == g.BATCHED_ROWPAIR and p["smem_bytes"] == 16 * 6144 * 2
    # x too large to stage whole (and for the row-pair kernel): the ring over K
    # slices, one CTA per SM in all, partial sums [slice][b][m] and a second pass
    p = g.plan_for("w8", 8192, 8192, 16)
    assert p["kernel"] == K["batched"] and p["variant"] == g.BATCHED_RING and p["splits"] == 2
    assert p["x_staging"] == 1 and p["smem_bytes"] == 16 * 4096 * 2 + ring and p["grid"] == 76
    assert p["workspace_bytes"] == 2 * 16 * 8192 * 4
    p = g.plan_for("bf16", 4096, 14336, 16)   # 1792 chunks in 3 slices of 598
    assert p["variant"] == g.BATCHED_RING_MIXED and p["splits"] == 3 and p["grid"] == 50
    assert p["smem_bytes"] == 16 * 598 * 8 * 2 + ring and p["workspace_bytes"] == 3 * 16 * 4096 * 4
    p = g.plan_for("bf16", 4096, 14336, 8)    # 8 x 14336 bf16 (229 KB): two slices, mixed FMAs
    assert p["variant"] == g.BATCHED_RING_MIXED and p["splits"] == 2 and p["x_staging"] == 1
    assert p["smem_bytes"] == 8 * 7168 * 2 + ring
    p = g.plan_for("bf16", 1024, 16384, 8)
    assert p["variant"] == g.BATCHED_RING_MIXED and p["splits"] == 2
    p = g.plan_for("bf16", 4096, 14336, 4)    # the row-pair kernel's x fits (115 KB)
    assert p["variant"] == g.BATCHED_ROWPAIR and p["splits"] == 1
    # padded vectors are staged too (zeros): B = 3 and B = 9 stage 4 and 16 vectors
    assert g.plan_for("w8", 16384, 4096, 3)["smem_bytes"] == 4 * 4096 * 4 + ring
    assert g.plan_for("f16", 4096, 4096, 9)["smem_bytes"] == 16 * 4096 * 2
    # int4: the ring with a group-scale ring (16 KB) beside it, 2 rows per warp
    p = g.plan_for("w4", 8192, 8192, 4)
    assert p["kernel"] == K["batched"] and p["variant"] == g.BATCHED_RING and p["rows_per_warp"] == 2
    assert p["x_staging"] == 2 and p["smem_bytes"] == 4 * 8192 * 4 + ring + 16 * 1024
    # one or two vectors of int4 (and fp32 with 4 vectors, 2 rows): rows per warp as measured
    # (one vector: 16 ring slots per thread, so 4 steps)
    for B in (1, 2):
        p = g.plan_for("w4", 14336, 4096, B)
        assert p["variant"] == g.BATCHED_RING and p["rows_per_warp"] == 4 and p["unroll"] == (4 if B == 1 else 2)
    p = g.plan_for("f32", 8192, 4096, 4)
    assert p["variant"] == g.BATCHED_RING and p["rows_per_warp"] == 2 and p["unroll"] == 4


def test_plan_small_k_lanes():
    # K <= 16 chunks of 16 bytes: lanes per row = next power of two of the chunks
    for dt, vec in (("f32", 4), ("f16", 8), ("bf16", 8), ("w8", 16)):
        for chunks, lanes in ((1, 1), (2, 2), (3, 4), (5, 8), (9, 16), (16, 16)):
            p = g.plan_for(dt, 1000, chunks * vec, 1)
            assert p["kernel"] == g.KERNELS["rows_per_warp"], (dt, chunks)
            assert p["lanes_per_row"] == lanes, (dt, chunks)
            assert p["grid"] == min(-(-1000 // (256 // lanes)), 152 * 32)


def test_plan_unaligned_goes_scalar():
    assert g.plan_for("f32", 100, 4096, 1, aligned16=False)["kernel"] == g.KERNELS["scalar"]
    assert g.plan_for("f32", 100, 4095, 1)["kernel"] == g.KERNELS["scalar"]   # K % 4 != 0
    assert g.plan_for("w8", 100, 4104, 1)["kernel"] == g.KERNELS["scalar"]    # K % 16 != 0
    p = g.plan_for("f16", 100, 3, 1)
    assert p["kernel"] == g.KERNELS["scalar"] and p["lanes_per_row"] == 4


def test_plan_few_rows_long_k():
    p = g.plan_for("bf16", 8, 1 << 20, 1)
    assert p["kernel"] == g.KERNELS["split_k"]
    assert p["splits"] >= 2
    assert p["workspace_bytes"] == p["splits"] * 1 * 8 * 4
    nch = (1 << 20) // 8
    per = -(-nch // p["splits"])
    assert (p["splits"] - 1) * per < nch  # no empty slice
    p = g.plan_for("bf16", 600, 1 << 16, 1)   # 2..16 rows per SM: a CTA per row
    assert p["kernel"] == g.KERNELS["block_per_row"] and p["grid"] == 600


def test_plan_batch_too_big_for_smem():
    # 16 vectors of 16384 bf16 = 512 KB of x: staged in 4 K slices of 128 KB
    p = g.plan_for("bf16", 8192, 16384, 16)
    assert p["kernel"] == g.KERNELS["batched"] and p["nb"] == 16 and p["splits"] == 4 and p["grid"] == 38
    # beyond 64 slices (x of more than ~10 MB): warp per row, x through L1
    p = g.plan_for("bf16", 8192, 1 << 20, 16)
    assert p["kernel"] == g.KERNELS["warp_per_row"] and p["nb"] == 16


def test_plan_nb_rounding_and_degenerate():
    for B, nb in ((1, 1), (2, 2), (3, 4), (5, 8), (9, 16), (16, 16)):
        assert g.plan_for("f32", 4096, 4096, B)["nb"] == nb
    p = g.plan_for("f32", 0, 10, 1)
    assert p["kernel"] == 0 and p["grid"] == 0
    p = g.plan_for("f32", 10, 0, 1)   # K = 0: epilogue only
    assert p["kernel"] == g.KERNELS["rows_per_warp"] and p["lanes_per_row"] == 1
    with pytest.raises(g.GemvError):
        g.plan_for("f32", 10, 10, 17)
    with pytest.raises(g.GemvError):
        g.plan_for("f32", -1, 10, 1)


def test_plan_grid_never_exceeds_cap():
    for M in (1, 7, 100, 5000, 10 ** 6, 10 ** 8):
        for Kd in (16, 128, 4096):
            for B in (1, 4, 16):
                p = g.plan_for("bf16", M, Kd, B, num_sms=152)
                assert 1 <= p["grid"] <= max(M, 152 * 32)


def test_w4_host_checks():
    w4 = g.lib().gemv_w4
    assert w4(None, None, None, None, None, 0, 256, 2, None) == 0            # M == 0: no-op
    assert w4(P, P + 64, P + 4096, None, P + 8192, 4, 100, 1, None) == 1     # K % 128 != 0
    assert w4(P, None, P + 4096, None, P + 8192, 4, 256, 1, None) == 1       # scales required
    assert w4(P, P + 64, P + 4096, None, P + 8192, 4, 256, 17, None) == 2    # B > 16
    assert w4(P, P + 66, P + 4096, None, P + 8192, 4, 256, 1, None) == 1     # scales not 4-byte aligned
    # y over the group scales (4 rows x 2 groups x 4 bytes at P + 8192)
    assert w4(P, P + 8192, P + 4096, None, P + 8200, 4, 256, 1, None) == 1
    # a row scale only for the int types
    assert g.lib().gemv_ex(2, P, P + 64, P + 4096, None, None, P + 8192, 4, 256, 1, 0, None) == 1


def test_plan_w4():
    K = g.KERNELS
    p = g.plan_for("w4", 8192, 8192, 1)   # one vector: the ring (x fp32, 16 slots, group-scale ring)
    assert p["kernel"] == K["batched"] and p["nb"] == 1 and p["smem_bytes"] == 8192 * 4 + 128 * 1024 + 32 * 1024
    p = g.plan_for("w4", 65536, 8192, 1)  # 65536 rows and more: not the ring
    assert p["kernel"] == K["warp_per_row"]
    for B, slices in ((2, 1), (4, 1), (9, 2), (16, 2)):  # the batched ring kernel
        p = g.plan_for("w4", 8192, 8192, B)
        assert p["kernel"] == K["batched"] and p["splits"] == slices, (B, p)
    # 32 weights per 16-byte chunk: K = 256 is 8 chunks -> 8 lanes per row
    p = g.plan_for("w4", 1000, 256, 1)
    assert p["kernel"] == K["rows_per_warp"] and p["lanes_per_row"] == 8
    assert g.plan_for("w4", 100, 4096, 1, aligned16=False)["kernel"] == K["scalar"]
    assert g.plan_for("w4", 8, 1 << 20, 1)["kernel"] == K["split_k"]


def test_plan_tensor_cores():
    K = g.KERNELS
    # 17..256 vectors of fp16/bf16: the tcgen05 kernel, N = B rounded up to 16
    p = g.plan_for("bf16", 4096, 4096, 32)
    assert p["kernel"] == K["tc"] and p["nb"] == 32 and p["threads"] == 128 and p["grid"] == 32
    # N <= 64: stages of two 64-column atoms (128 + N rows x 256 bytes); 32 row tiles
    # cover less than half the SMs: two CTAs per SM, as many stages as fit in 100 KB
    # (at most 8), + 1024 bytes to align them
    assert p["smem_bytes"] == 2 * (128 + 32) * 256 + 1024
    # split-K so that all CTAs run in one wave: 8 slices of 4 k-tiles of 128, one
    # cluster per row tile, summed in the kernel (no workspace)
    assert p["splits"] == 8 and p["unroll"] == 4 and p["workspace_bytes"] == 0
    assert p["grid"] * p["splits"] <= 2 * 152
    # tiles covering half the SMs or more (but not all), up to 64 vectors: the deep
    # ring (200 KB, one CTA per SM)
    p = g.plan_for("bf16", 14336, 4096, 32)
    assert p["grid"] == 112 and p["splits"] == 1 and p["smem_bytes"] == 5 * (128 + 32) * 256 + 1024
    p = g.plan_for("bf16", 14336, 4096, 128)  # 128 vectors: two CTAs per SM, 2 K slices
    assert p["splits"] == 2 and p["smem_bytes"] == 3 * (128 + 128) * 128 + 1024
    p = g.plan_for("f16", 4096, 4096, 17)
    assert p["kernel"] == K["tc"] and p["nb"] == 32
    # at least as many row tiles as SMs (up to two per SM): two CTAs per SM, a 100 KB ring
    p = g.plan_for("bf16", 38912, 4096, 256)
    assert p["kernel"] == K["tc"] and p["nb"] == 256 and p["splits"] == 1 and p["workspace_bytes"] == 0
    assert p["smem_bytes"] == 2 * (128 + 256) * 128 + 1024 and p["threads"] == 128
    # more: the persistent form, one CTA per SM, a deep ring
    p = g.plan_for("bf16", 128256, 4096, 256)
    assert p["threads"] == 192 and p["grid"] == 152 and p["smem_bytes"] == 4 * (128 + 256) * 128 + 1024
    p = g.plan_for("bf16", 28672, 4096, 32)
    assert p["smem_bytes"] == 2 * (128 + 32) * 256 + 1024 and p["grid"] == 224 and p["splits"] == 1
    # no empty slice: splits * k-tiles per slice covers K exactly once; at most 8
    # slices (one cluster of CTAs per row tile)
    for M, Kd in ((300, 1000), (1, 64), (5000, 4104), (128, 16384)):
        p = g.plan_for("bf16", M, Kd, 40)
        kt = -(-Kd // 128)  # N = 48: 128-column k-tiles
        assert (p["splits"] - 1) * p["unroll"] < kt <= p["splits"] * p["unroll"], (M, Kd, p)
        assert 1 <= p["splits"] <= 8 and p["workspace_bytes"] == 0, (M, Kd, p)
    p = g.plan_for("bf16", 4096, 4096, 48)  # 9 slices would fill the wave; a cluster holds 8
    assert p["splits"] == 8 and p["unroll"] == 4
    # 64 or more vectors on few row tiles: deep rings, one CTA per SM, SMs / tiles slices
    p = g.plan_for("f16", 4096, 4096, 256)
    assert p["splits"] == 4 and p["smem_bytes"] == 4 * (128 + 256) * 128 + 1024
    for dt in ("f32", "w8"):
        with pytest.raises(g.GemvError):
            g.plan_for(dt, 100, 64, 17)
    with pytest.raises(g.GemvError):
        g.plan_for("bf16", 100, 64, 257)
    with pytest.raises(g.GemvError):       # more than 16 vectors needs 16-byte rows
        g.plan_for("bf16", 100, 60, 17)


def test_launch_overlap_modes():
    # host-only setting of the calling thread: modes 0..2, anything else refused
    L = g.lib()
    for m in (1, 2, 0):
        assert L.gemv_set_launch_overlap(m) == 0
    assert L.gemv_set_launch_overlap(3) == g.ERR_INVALID_VALUE
    assert L.gemv_set_launch_overlap(-1) == g.ERR_INVALID_VALUE
    g.set_launch_overlap("launch")  # the default


def test_plan_tc_persistent():
    # more 128-row tiles than two CTAs per SM hold (and no K split): the persistent form,
    # 192 threads, one CTA per SM, k-tiles per tile in unroll, a deep ring
    for M, persist in ((128256, True), (39040, True), (38912, False), (14336, False)):
        p = g.plan_for("bf16", M, 4096, 64, num_sms=152)
        assert p["kernel_name"] == "tc" and p["splits"] == 1, (M, p)
        if persist:
            assert p["threads"] == 192 and p["grid"] == 152 and p["unroll"] == 32 and p["smem_bytes"] > 150 * 1024, p
        else:
            assert p["threads"] == 128 and p["grid"] == -(-M // 128), p
    assert g.plan_for("f16", 128256, 0, 64, num_sms=152)["threads"] == 128  # K = 0: the plain kernel


def test_plan_dispatcher_audit_cases():
    """Shapes where a forced kernel beat the dispatcher's choice by more than 5 % on a
    GB300, and the rules that now pick the faster kernel (CUDA-event means, cold L2)."""
    K = g.KERNELS
    # fp32, 2 vectors, fewer than 32 rows per SM of >= 2048 chunks: block per row
    for M, Kd in ((1024, 16384), (2048, 12288), (4096, 14336), (1024, 8192)):
        assert g.plan_for("f32", M, Kd, 2)["kernel"] == K["block_per_row"], (M, Kd)
    assert g.plan_for("f32", 8192, 14336, 2)["kernel"] == K["batched"]  # the ring leads here
    assert g.plan_for("f32", 1024, 16384, 4)["kernel"] == K["batched"]  # 4 vectors: batched
    assert g.plan_for("f32", 4096, 4096, 2)["kernel"] == K["xsplit"]    # short rows: K split
    # fp16/bf16, 1 vector, 1..11 rows per SM of 8192..16384 elements (1..15 from 12288):
    # the K-split kernel
    for dt, M, Kd in (("bf16", 1024, 16384), ("bf16", 256, 16384), ("f16", 1024, 16384), ("bf16", 1536, 16384),
                      ("bf16", 1024, 8192), ("bf16", 2048, 14336)):
        assert g.plan_for(dt, M, Kd, 1)["kernel"] == K["xsplit"], (dt, M, Kd)
    assert g.plan_for("bf16", 4096, 16384, 1)["kernel"] == K["stream"]  # from 16 rows per SM
    assert g.plan_for("bf16", 4096, 14336, 1)["kernel"] == K["stream"]
    assert g.plan_for("bf16", 1024, 4096, 1)["kernel"] != K["xsplit"]   # short rows keep theirs
    # fp16/bf16, 4 vectors, up to 2048 rows: the mixed-precision ring
    for dt, M, Kd in (("bf16", 1024, 16384), ("bf16", 2048, 16384), ("bf16", 2048, 8192), ("f16", 1024, 16384)):
        p = g.plan_for(dt, M, Kd, 4)
        assert p["kernel"] == K["batched"] and p["variant"] == g.BATCHED_RING_MIXED, (dt, M, Kd, p)
    p = g.plan_for("bf16", 4096, 14336, 4)
    assert p["kernel"] == K["batched"] and p["variant"] == g.BATCHED_ROWPAIR
    # 3..4 fp32 vectors up to one row pair per warp: the ring (fp32 4096x4096 B = 4
    # 16.6 us against 19.5 in the row pairs, 2048x4096 12.9 against 16.6)
    for M, B in ((1024, 4), (2048, 4), (4096, 4), (4096, 3)):
        p = g.plan_for("f32", M, 4096, B)
        assert p["kernel"] == K["batched"] and p["variant"] == g.BATCHED_RING, (M, B, p)
    assert g.plan_for("f32", 4096, 4096, 8)["variant"] == g.BATCHED_ROWPAIR  # 8 vectors keep them
    # beyond one row pair per warp: the ring for 4 vectors of fp16/bf16 and 2 or 8 of
    # int8 (bf16 8192x8192 B = 4 30.5 against 32.6, 6144x4096 16.1 against 18.5; int8
    # 6144x4096 B = 2 12.3 against 14.4, 9216x4096 B = 8 24.6 against 26.6) ...
    for dt, M, Kd, B in (("bf16", 8192, 8192, 4), ("bf16", 6144, 4096, 4), ("f16", 6144, 4096, 4),
                         ("bf16", 9216, 4096, 3), ("w8", 6144, 4096, 2), ("w8", 9216, 4096, 8), ("w8", 8192, 8192, 8)):
        p = g.plan_for(dt, M, Kd, B)
        assert p["kernel"] == K["batched"] and p["variant"] == g.BATCHED_RING, (dt, M, Kd, B, p)
    # ... while 4 vectors of int8 and 8 of fp16/bf16 keep the row pairs up to one ring
    # row group per warp (int8 8192x8192 B = 4 26.4 against 27.3, bf16 8192x8192 B = 8
    # 36.9 against 40.9), as do all of these up to one row pair per warp
    for dt, M, Kd, B in (("w8", 8192, 8192, 4), ("bf16", 8192, 8192, 8), ("w8", 4096, 4096, 4),
                         ("bf16", 4096, 4096, 4), ("w8", 4096, 8192, 2), ("bf16", 4096, 4096, 8)):
        p = g.plan_for(dt, M, Kd, B)
        assert p["kernel"] == K["batched"] and p["variant"] == g.BATCHED_ROWPAIR, (dt, M, Kd, B, p)

