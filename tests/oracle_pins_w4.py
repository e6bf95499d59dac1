"""Pins for the oracle's int4 path (weight-only int4 with per-group scales).

The format (the NPU MatMul post, section 5.2, leaves it open; this is the reading
the library implements): symmetric two's complement int4 in [-8, 7], two per byte,
element k of a row in byte k/2, low nibble for even k; one fp32 scale per `group`
consecutive elements of a row, scales stored M x K/group; x and bias bf16.

    y[b][m] = sum_k s[m][k/group] * q[m][k] * x[b][k] + bias[m]

Each pin is a function of `impl(A, S, group, x, bias) -> y (B x M float64)` and
checks it against something other than the oracle: exact rationals over an
independent nibble decoder, closed forms, and the (independently pinned) int8
oracle on scales that make the two formats agree exactly.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

import oracle
from tests import oracle_pins as P

U64 = 2.0 ** -53


def nibbles(A: np.ndarray) -> np.ndarray:
    """Independent int4 decoder: (M, K/2) bytes -> (M, K) int64, low nibble first."""
    A = np.asarray(A, dtype=np.uint8).astype(np.int64)
    lo = ((A & 15) ^ 8) - 8
    hi = ((A >> 4) ^ 8) - 8
    out = np.empty((A.shape[0], 2 * A.shape[1]), dtype=np.int64)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


def pack(q: np.ndarray) -> np.ndarray:
    """(M, K) ints in [-8, 7] -> (M, K/2) bytes, low nibble first."""
    q = np.asarray(q, dtype=np.int64)
    assert q.min() >= -8 and q.max() <= 7
    u = q & 15
    return (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)


def exact(A, S, G, x, bias):
    q = nibbles(A)
    xd = P.dec_bf16(x)
    bd = None if bias is None else P.dec_bf16(bias)
    M, K = q.shape
    B = xd.shape[0]
    y = [[None] * M for _ in range(B)]
    mag = np.zeros((B, M))
    for b in range(B):
        for m in range(M):
            acc = Fraction(0)
            tot = 0.0
            for k in range(K):
                p = Fraction(float(S[m, k // G])) * int(q[m, k]) * Fraction(float(xd[b, k]))
                acc += p
                tot += abs(float(p))
            y[b][m] = acc + (Fraction(float(bd[m])) if bd is not None else 0)
            mag[b, m] = tot + (abs(float(bd[m])) if bd is not None else 0.0)
    return y, mag


def bf16_bits(v) -> np.ndarray:
    return (np.asarray(v, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def rand_inputs(rng, M, K, G, B, bias):
    A = rng.integers(0, 256, size=(M, K // 2)).astype(np.uint8)
    S = (rng.uniform(1e-3, 1e-1, size=(M, K // G)) * rng.choice([-1, 1], size=(M, K // G))).astype(np.float32)
    x = bf16_bits(rng.standard_normal((B, K)))
    bb = bf16_bits(rng.standard_normal(M)) if bias else None
    return A, S, x, bb


def pin_w4_bruteforce(impl, seed=10):
    """Exact rationals on tiny random inputs: fp64 result within gamma_{K+2}."""
    rng = np.random.default_rng(seed)
    for (M, K, G, B) in ((1, 2, 2, 1), (3, 8, 4, 2), (2, 16, 16, 1), (4, 16, 2, 2), (2, 12, 6, 3)):
        for bias in (False, True):
            A, S, x, bb = rand_inputs(rng, M, K, G, B, bias)
            y = impl(A, S, G, x, bb)
            ye, mag = exact(A, S, G, x, bb)
            g = (K + 3) * U64 / (1 - (K + 3) * U64)
            for b in range(B):
                for m in range(M):
                    err = abs(Fraction(float(y[b, m])) - ye[b][m])
                    assert float(err) <= g * mag[b, m] + 1e-300, (M, K, G, B, bias, b, m)


def pin_w4_one_hot(impl, seed=11):
    """x = e_k picks s[m][k/G] * q[m][k] exactly: nibble order, sign and group index."""
    rng = np.random.default_rng(seed)
    M, K, G = 5, 16, 4
    A, S, _, _ = rand_inputs(rng, M, K, G, 1, False)
    q = nibbles(A)
    for k in range(K):
        x = np.zeros((1, K), dtype=np.float32)
        x[0, k] = 1.0
        y = impl(A, S, G, bf16_bits(x), None)
        want = S[:, k // G].astype(np.float64) * q[:, k]
        assert np.array_equal(y[0], want), (k, y[0], want)


def pin_w4_equals_int8_on_row_scales(impl, seed=12):
    """Power-of-two scales, equal across a row's groups: the int4 result equals the
    int8 oracle on the same integers with that per-row scale, bit for bit."""
    rng = np.random.default_rng(seed)
    M, K, G, B = 6, 32, 8, 2
    q = rng.integers(-8, 8, size=(M, K))
    srow = (2.0 ** rng.integers(-6, 2, size=M)).astype(np.float32)
    S = np.repeat(srow[:, None], K // G, axis=1).astype(np.float32)
    x = bf16_bits(rng.standard_normal((B, K)))
    bb = bf16_bits(rng.standard_normal(M))
    y = impl(pack(q), S, G, x, bb)
    y8, _ = oracle.gemv("w8", q.astype(np.int8), x, bb, srow)
    assert np.array_equal(y, y8)


def pin_w4_group_locality(impl, seed=13):
    """Doubling scale[m][g] moves y[m] by exactly s * sum_{k in g} q x (integer data),
    and no other output."""
    rng = np.random.default_rng(seed)
    M, K, G = 4, 24, 8
    q = rng.integers(-8, 8, size=(M, K))
    x = rng.integers(-4, 5, size=(1, K)).astype(np.float32)
    S = (2.0 ** rng.integers(-3, 3, size=(M, K // G))).astype(np.float32)
    A, xb = pack(q), bf16_bits(x)
    y0 = impl(A, S, G, xb, None)
    for m in range(M):
        for g in range(K // G):
            S2 = S.copy()
            S2[m, g] *= 2
            y1 = impl(A, S2, G, xb, None)
            d = float(S[m, g]) * float(np.dot(q[m, g * G:(g + 1) * G], x[0, g * G:(g + 1) * G]))
            want = y0.copy()
            want[0, m] += d
            assert np.array_equal(y1, want), (m, g)


def pin_w4_extremes(impl):
    """All -8 and all 7 with x = 1, scale 0.5: y = 0.5 * q * K exactly (+ bias)."""
    M, K, G = 3, 256, 128
    x = bf16_bits(np.ones((1, K)))
    S = np.full((M, K // G), 0.5, dtype=np.float32)
    for byte, qv in ((0x88, -8), (0x77, 7)):
        A = np.full((M, K // 2), byte, dtype=np.uint8)
        assert np.array_equal(impl(A, S, G, x, None)[0], np.full(M, 0.5 * qv * K))
        bb = bf16_bits(np.array([1.0, -2.0, 0.25]))
        assert np.array_equal(impl(A, S, G, x, bb)[0], 0.5 * qv * K + np.array([1.0, -2.0, 0.25]))


def pin_w4_bias_null(impl, seed=14):
    """bias = None equals an all-zero bias, bit for bit."""
    rng = np.random.default_rng(seed)
    A, S, x, _ = rand_inputs(rng, 3, 16, 8, 2, False)
    assert np.array_equal(impl(A, S, 8, x, None), impl(A, S, 8, x, bf16_bits(np.zeros(3))))


ALL_PINS_W4 = [pin_w4_bruteforce, pin_w4_one_hot, pin_w4_equals_int8_on_row_scales,
               pin_w4_group_locality, pin_w4_extremes, pin_w4_bias_null]
