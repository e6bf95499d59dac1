"""The dispatcher on random shapes (host only): every plan it returns is one the
launch code accepts and the kernels can run.

Checked for each (dtype, M, K, B, alignment, SM count):
* the status: success for every size the entry points accept, UNSUPPORTED beyond
  the batch limits;
* the launch shape: threads, grid, dynamic shared memory within one CTA's limit;
* per kernel family, the invariants its launcher and kernel rely on: K slices with
  no empty slice and a workspace of slices x B x M fp32 partial sums, the batched
  variants' rows per warp and ring sizes, the tensor-core stage arithmetic, the
  streaming kernel's single vector.
"""
from __future__ import annotations

import pytest

import decode_linear_layers_gb300 as g

hypothesis = pytest.importorskip("hypothesis")
st = hypothesis.strategies

K_ = g.KERNELS
SMEM_MAX = 227 * 1024
VEC = {"f32": 4, "f16": 8, "bf16": 8, "w8": 16, "w4": 32}
SX = {"f32": 4, "f16": 2, "bf16": 2, "w8": 2, "w4": 2}


def _cdiv(a, b):
    return -(-a // b)


@hypothesis.settings(max_examples=3000, deadline=None, derandomize=True)
@hypothesis.given(
    dtype=st.sampled_from(["f32", "f16", "bf16", "w8", "w4"]),
    M=st.one_of(st.integers(1, 300), st.integers(300, 20000), st.integers(20000, 200000)),
    kmul=st.one_of(st.integers(0, 40), st.integers(40, 6000)),
    kpad=st.one_of(st.just(0), st.just(0), st.integers(1, 15)),
    B=st.one_of(st.integers(1, 4), st.integers(1, 16), st.integers(17, 300)),
    aligned=st.booleans(),
    sms=st.sampled_from([152, 148, 132, 8]),
)
def test_plan_invariants(dtype, M, kmul, kpad, B, aligned, sms):
    vec = VEC[dtype]
    K = kmul * vec + (0 if dtype == "w4" else kpad)
    if dtype == "w4":
        K = (K // 128) * 128  # int4 takes K in whole groups of 128
    half16 = dtype in ("f16", "bf16")
    try:
        p = g.plan_for(dtype, M, K, B, aligned16=aligned, num_sms=sms)
    except g.GemvError as e:
        # only the batch limits (and 17..256 vectors needing 16-byte rows) refuse
        assert e.status == g.ERR_UNSUPPORTED, (dtype, M, K, B, e.status)
        assert B > 16 and (not half16 or B > 256 or not aligned or K % vec)
        return
    assert B <= 16 or (half16 and B <= 256), (dtype, B)
    kern = p["kernel"]
    assert kern in K_.values() and kern != 0
    assert p["threads"] in (128, 192, 256, 512)
    assert p["grid"] >= 1 and p["splits"] >= 1
    assert 0 <= p["smem_bytes"] <= SMEM_MAX, p
    nch = K // vec
    if kern == K_["split_k"]:
        per = _cdiv(nch, p["splits"])
        assert (p["splits"] - 1) * per < nch  # no empty slice
        assert p["workspace_bytes"] == p["splits"] * B * M * 4
    elif kern == K_["batched"]:
        assert B >= 2 or dtype in ("w8", "w4"), p
        v = p["variant"]
        assert v in (g.BATCHED_ROWPAIR, g.BATCHED_RING, g.BATCHED_RING_MIXED)
        # one CTA per SM in all, unless x needs more K slices than the device has SMs
        assert p["threads"] == 512 and p["grid"] * p["splits"] <= max(sms, p["splits"])
        if v == g.BATCHED_ROWPAIR:
            assert dtype != "w4" and p["splits"] == 1 and p["smem_bytes"] == p["nb"] * K * SX[dtype]
        else:
            if v == g.BATCHED_RING_MIXED:
                assert half16 and p["rows_per_warp"] == 2 and p["x_staging"] == 1
            slots = 16 if p["nb"] == 1 else 8  # ring slots per thread
            assert p["rows_per_warp"] * p["unroll"] == slots
            assert p["rows_per_warp"] * p["nb"] <= 32
            cps = _cdiv(nch, p["splits"])
            assert (p["splits"] - 1) * cps < nch
            xe = 4 if p["x_staging"] == 2 or dtype == "f32" else 2
            extra = slots * 2 * 1024 if dtype == "w4" else 0  # a 4-byte group scale per slot
            assert p["smem_bytes"] == p["nb"] * cps * vec * xe + slots * 8 * 1024 + extra
            assert p["workspace_bytes"] == (p["splits"] * B * M * 4 if p["splits"] > 1 else 0)
    elif kern == K_["tc"]:
        assert half16 and aligned and K % vec == 0
        nb = p["nb"]
        assert nb % 16 == 0 and 16 <= nb <= 256 and nb >= B
        tiles = _cdiv(M, 128)
        persist = tiles > 2 * sms and K > 0
        ka = 2 if nb <= 64 or persist else 1  # (the persistent form: 128-column stages for every N)
        stage = (128 + nb) * 64 * 2 * ka
        stages = (p["smem_bytes"] - 1024) // stage
        assert 2 <= stages <= 16 and p["smem_bytes"] == stages * stage + 1024
        ktiles = _cdiv(K, 64 * ka) if K > 0 else 1
        if persist:
            # the persistent form: one 192-thread CTA per SM over its tiles, no K split
            assert p["threads"] == 192 and p["grid"] == sms and p["splits"] == 1 and p["unroll"] == ktiles
        else:
            assert p["threads"] == 128 and p["grid"] == tiles
        assert p["splits"] * p["unroll"] >= ktiles and (p["splits"] - 1) * p["unroll"] < ktiles
        # the slices of a row tile are one cluster (at most 8 CTAs), reduced in the kernel
        assert 1 <= p["splits"] <= 8 and p["workspace_bytes"] == 0
    elif kern == K_["stream"]:
        assert B == 1 and p["threads"] == 512
    elif kern == K_["xsplit"]:
        assert (dtype == "f32" and B in (1, 2, 4)) or (half16 and B in (1, 2))
        # x of all vectors in registers: J chunks per thread x NB vectors x VEC values
        assert p["unroll"] in (1, 2, 4) and p["unroll"] * p["nb"] * vec <= 64
        assert p["smem_bytes"] == 128 * 1024 and p["grid"] == min(M, sms)
    elif kern == K_["scalar"]:
        assert p["lanes_per_row"] in (4, 32)
    else:
        assert kern in (K_["rows_per_warp"], K_["warp_per_row"], K_["block_per_row"])
        if kern != K_["block_per_row"]:
            assert p["lanes_per_row"] in (1, 2, 4, 8, 16, 32)
