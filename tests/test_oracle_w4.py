"""The oracle's int4 path against its pins (no GPU), and planted mistakes.

Every pin in ``oracle_pins_w4`` must hold for the oracle; every plausible mistake
planted in a CPU copy of the int4 definition (nibble order, sign, scale index,
group size, dropped bias, a dropped group, bf16 x read as fp16) must break one.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from tests import oracle_pins as P
from tests import oracle_pins_w4 as P4


def oracle_impl(A, S, G, x, bias):
    y, _ = oracle.gemv("w4", A, x, bias, S, group=G)
    return y


@pytest.mark.parametrize("pin", P4.ALL_PINS_W4, ids=lambda f: f.__name__)
def test_oracle_w4_pin(pin):
    pin(oracle_impl)


def test_oracle_w4_threads():
    rng = np.random.default_rng(3)
    A, S, x, bb = P4.rand_inputs(rng, 300, 256, 128, 3, True)
    y1, a1 = oracle.gemv("w4", A, x, bb, S, nthreads=1)
    y8, a8 = oracle.gemv("w4", A, x, bb, S, nthreads=8)
    assert np.array_equal(y1, y8) and np.array_equal(a1, a8)


def test_decode_w4_all_bytes():
    b = np.arange(256, dtype=np.uint8)
    got = oracle.decode("w4", b)
    lo = np.where((b & 15) >= 8, (b & 15).astype(int) - 16, b & 15)
    hi = np.where((b >> 4) >= 8, (b >> 4).astype(int) - 16, b >> 4)
    want = np.empty(512)
    want[0::2], want[1::2] = lo, hi
    assert np.array_equal(got, want)


def test_w4_argument_errors():
    A = np.zeros((2, 64), dtype=np.uint8)
    x = P4.bf16_bits(np.zeros((1, 128)))
    with pytest.raises(ValueError):
        oracle.gemv("w4", A, x, None, np.ones((2, 3), dtype=np.float32), group=40)   # group does not divide K
    with pytest.raises(ValueError):
        oracle.gemv("w4", A, x, None, np.ones((2, 2), dtype=np.float32), group=128)  # scales of the wrong shape
    with pytest.raises(TypeError):
        oracle.gemv("w4", A.astype(np.int8), x, None, np.ones((2, 1), dtype=np.float32))


def test_w4_absdot():
    rng = np.random.default_rng(4)
    A, S, x, _ = P4.rand_inputs(rng, 5, 64, 32, 2, False)
    _, ad = oracle.gemv("w4", A, x, None, S, group=32)
    q = P4.nibbles(A)
    deq = q * np.repeat(S.astype(np.float64), 32, axis=1)
    want = np.abs(P.dec_bf16(x)) @ np.abs(deq).T
    assert np.allclose(ad, want, rtol=1e-14, atol=0)


# ------------------------------------------------------------ planted mistakes
def _base(A, S, G, x, bias, *, order="lo", signed=True, sidx="div", gsize=None, bias_mode="add",
          drop_group=False, xdec=P.dec_bf16):
    A = np.asarray(A, dtype=np.uint8).astype(np.int64)
    lo, hi = A & 15, A >> 4
    if order != "lo":
        lo, hi = hi, lo
    q = np.empty((A.shape[0], 2 * A.shape[1]), dtype=np.int64)
    q[:, 0::2], q[:, 1::2] = lo, hi
    if signed:
        q = np.where(q >= 8, q - 16, q)
    M, K = q.shape
    ng = K // G
    gg = G if gsize is None else gsize
    xd = xdec(x)
    y = np.zeros((xd.shape[0], M))
    for b in range(xd.shape[0]):
        for m in range(M):
            s = 0.0
            for k in range(K):
                if drop_group and k >= K - G:
                    continue
                if sidx == "div":
                    sc = S[m, min(k // gg, ng - 1)]
                elif sidx == "mod":
                    sc = S[m, k % ng]
                else:  # "row"
                    sc = S[m, 0]
                s += float(sc) * float(q[m, k]) * float(xd[b, k])
            bm = 0.0 if bias is None else float(P.dec_bf16(bias)[m])
            y[b, m] = s + (bm if bias_mode == "add" else 0.0)
    return y


MUTANTS = {
    "nibble_order": lambda *a: _base(*a, order="hi"),
    "unsigned_nibble": lambda *a: _base(*a, signed=False),
    "scale_per_row_only": lambda *a: _base(*a, sidx="row"),
    "scale_index_mod": lambda *a: _base(*a, sidx="mod"),
    "group_half_size": lambda *a: _base(*a, gsize=max(1, a[2] // 2)),
    "dropped_bias": lambda *a: _base(*a, bias_mode="drop"),
    "dropped_last_group": lambda *a: _base(*a, drop_group=True),
    "x_read_as_f16": lambda *a: _base(*a, xdec=P.dec_f16),
}


def test_correct_copy_passes_pins():
    for pin in P4.ALL_PINS_W4:
        pin(_base)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    failed = []
    for pin in P4.ALL_PINS_W4:
        try:
            with np.errstate(all="ignore"):
                pin(MUTANTS[name])
        except (AssertionError, IndexError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin catches the planted mistake {name}"
