"""Byte and flop accounting of the benchmark against the numbers the pages print."""
import json
import os
from fractions import Fraction

import workloads as W

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "roofline_pages.json")))
E = {e["id"]: e for e in GOLD["entries"]}


def rel(a, b):
    return abs(a - b) / abs(b)


def test_sgemv_notes_problem_bytes():
    e = E["sgemv_notes_problem_bytes"]
    sa, sx, sy, _ = W.ELEM_BYTES[e["dtype"]]
    q = W.qmin_bytes(e["dtype"], e["M"], e["K"], e["B"])
    assert q - e["K"] * sx - e["M"] * sy == e["a_bytes"]
    assert q == 528896


def test_lesson_fp32_intensity():
    e = E["lesson_ai_fp32"]
    for M, N in e["shapes"]:
        ai = Fraction(W.flops(M, N, 1), W.qmin_bytes("f32", M, N, 1))
        assert ai == Fraction(2 * M * N, 4 * M * N + 4 * N + 4 * M)
        assert ai < Fraction(1, 2)
    # the limit as M, N grow
    big = Fraction(W.flops(1 << 20, 1 << 20, 1), W.qmin_bytes("f32", 1 << 20, 1 << 20, 1))
    assert abs(float(big) - e["ai_limit"]) < 1e-5


def test_lesson_h100_bound():
    e = E["lesson_h100_bound"]
    assert rel(0.5 * e["hbm_tbs"], e["tflops"]) < e["rel_tol"]


def test_npu_post_decode():
    e = E["npu_post_decode_fp16"]
    f = W.flops(e["M"], e["K"], e["B"])
    q = W.qmin_bytes(e["dtype"], e["M"], e["K"], e["B"])
    assert rel(f / 1e6, e["mflops"]) < e["rel_tol"]
    assert rel(e["M"] * e["K"] * 2 / 1e6, e["weight_mb"]) < e["rel_tol"]
    assert rel(f / q, e["ai"]) < e["rel_tol"]


def test_npu_post_prefill():
    e = E["npu_post_prefill_fp16"]
    M, K, B = e["M"], e["K"], e["B"]
    f = W.flops(M, K, B)
    q = W.qmin_bytes(e["dtype"], M, K, B)
    assert rel(f / 1e9, e["gflops"]) < e["rel_tol_small"]
    assert rel(B * K * 2 / 1e6, e["act_mb"]) < e["rel_tol_small"]
    assert rel(B * M * 2 / 1e6, e["out_mb"]) < e["rel_tol_small"]
    assert rel(q / 1e6, e["total_mb"]) < e["rel_tol_total"]
    assert rel(f / q, e["ai"]) < e["rel_tol_ai"]


def test_glossary_flop_ratio():
    e = E["glossary_decode_vs_batch16"]
    assert W.flops(e["M"], e["K"], e["B_big"]) == e["flop_ratio"] * W.flops(e["M"], e["K"], e["B_small"])


def test_config_qmin_values():
    # Q_min per config (M*K*s_A + B*K*s_x + B*M*s_y)
    want = {
        "f32_1024x128_b1": 528896,
        "f32_16384x16_b1_bias": 1114176,
        "f32_16384x32_b1_bias": 2162816,
        "f32_16384x4096_b1_bias": 268517376,
        "f16_4096x4096_b1": 33570816,
        "f16_4096x4096_b16": 33816576,
        "bf16_14336x4096_b1": 117477376,
        "bf16_4096x14336_b1": 117477376,
        "bf16_128256x4096_b1": 1050937856,
        "w8_8192x8192_b1_bias": 67141632,
        "w8_8192x8192_b4_bias": 67239936,
    }
    assert {w.name: w.qmin_bytes for w in W.CONFIGS} == want


def test_inputs_are_seeded_and_shaped():
    w = W.small("w8", 37, 53, 3, True, seed=5)
    a = W.make_inputs(w)
    b = W.make_inputs(w)
    for k in ("A", "x", "bias", "scale"):
        assert a[k].shape == b[k].shape
        assert bool((a[k] == b[k]).all())
    assert a["A"].shape == (37, 53) and a["x"].shape == (3, 53)
    assert int(a["A"].min()) >= -127 and int(a["A"].max()) <= 127
    s = a["scale"].numpy()
    assert s.min() >= 1e-3 and s.max() <= 1e-2


def test_traffic_record_matches_kernel_sources():
    # profiles/traffic.txt carries the ncu DRAM traffic of the benchmark's step kernel
    # for the kernel code and launch configuration it was captured from; the record
    # must be for them as committed (else the benchmark reports traffic as unknown), and
    # the captured bytes must be the workload's Q_min within a few percent (no re-reads)
    import bench

    name = W.HEADLINE[0]
    t = bench.read_traffic(name)
    assert t is not None, "profiles/traffic.txt was captured from other kernel code"
    q = W.BY_NAME[name].qmin_bytes
    assert 0.99 * q <= t <= 1.03 * q, (t, q)


def test_code_hash_ignores_comments_only():
    import bench

    a = "int f(int x) { return x + 1; }  // one\n/* two */"
    b = "int f(int x) {\n  /* changed */ return x + 1;\n}"
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(a.replace("x + 1", "x + 2"))
