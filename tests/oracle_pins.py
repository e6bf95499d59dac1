"""Pins for the GEMV oracle: checks fixed by the pages and by mathematics.

Each pin takes an implementation ``impl(dtype, A, x, bias, scale) -> y`` (y float64,
shape (B, M); A, x, bias in storage form as the oracle takes them) and raises
AssertionError when the implementation disagrees with what the definition fixes.
The reference values here never come from the oracle itself: they come from exact
rational arithmetic over independently decoded inputs (numpy's float16 and a
float32 bit view for bf16), from closed forms, or from algebraic identities.

Definition pinned: y[b][m] = s_m * sum_k A[m][k] * x[b][k] + bias[m]
("16-sgemv" notes, problem definition; "GEMV and row-level parallelism" lesson,
section 1 and its reference kernel's bias epilogue, which allows bias == NULL;
per-row int8 weight scale from the NPU MatMul post, section 1.2).
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

U64 = 2.0 ** -53


# ---------------------------------------------------------------- independent decoders
def dec_f16(bits: np.ndarray) -> np.ndarray:
    """fp16 bit patterns -> float64 through numpy's own float16 type."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def dec_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64: a bf16 is the top half of a float32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def enc_f16(v) -> np.ndarray:
    return np.asarray(v, dtype=np.float64).astype(np.float16).view(np.uint16)


def enc_bf16_exact(v) -> np.ndarray:
    """Encode values that are exactly representable in bf16 (asserted)."""
    f = np.asarray(v, dtype=np.float32)
    bits = f.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (bits >> 16).astype(np.uint16)


def decode_any(kind: str, a) -> np.ndarray:
    a = np.asarray(a)
    if kind == "f32":
        return a.astype(np.float64)
    if kind == "f16":
        return dec_f16(a)
    if kind == "bf16":
        return dec_bf16(a)
    return a.astype(np.float64)  # int8


def xkind(dtype: str) -> str:
    return "bf16" if dtype == "w8" else dtype


def encode(kind: str, v) -> np.ndarray:
    """Encode exactly representable values into storage form (asserts exactness)."""
    v = np.asarray(v, dtype=np.float64)
    if kind == "f32":
        out = v.astype(np.float32)
        assert np.array_equal(out.astype(np.float64), v)
        return out
    if kind == "f16":
        out = enc_f16(v)
        assert np.array_equal(dec_f16(out), v)
        return out
    if kind == "bf16":
        return enc_bf16_exact(v)
    out = v.astype(np.int8)
    assert np.array_equal(out.astype(np.float64), v)
    return out


def exact(dtype, A, x, bias, scale):
    """Exact rational y and sum |terms| over independently decoded stored values."""
    Ad = decode_any(dtype, A)
    xd = decode_any(xkind(dtype), x)
    bd = None if bias is None else decode_any(xkind(dtype), bias)
    M, K = Ad.shape
    B = xd.shape[0]
    y = [[None] * M for _ in range(B)]
    mag = np.zeros((B, M))
    for b in range(B):
        for m in range(M):
            s = Fraction(float(scale[m])) if dtype == "w8" else Fraction(1)
            acc = Fraction(0)
            tot = 0.0
            for k in range(K):
                p = Fraction(float(Ad[m, k])) * Fraction(float(xd[b, k]))
                acc += p
                tot += abs(float(p))
            v = s * acc + (Fraction(float(bd[m])) if bd is not None else 0)
            y[b][m] = v
            mag[b, m] = abs(float(s)) * tot + (abs(float(bd[m])) if bd is not None else 0.0)
    return y, mag


# ---------------------------------------------------------------- random tiny inputs
def tiny_inputs(rng, dtype, M, K, B, bias, integers=False):
    """Random storage arrays; integers=True gives small integers (exact everywhere)."""
    xk = xkind(dtype)
    if dtype == "w8":
        A = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
    elif integers:
        A = encode(dtype, rng.integers(-8, 9, size=(M, K)).astype(np.float64))
    elif dtype == "f32":
        A = rng.standard_normal((M, K)).astype(np.float32)
    elif dtype == "f16":
        A = enc_f16(rng.standard_normal((M, K)))
    else:
        A = (rng.standard_normal((M, K)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    if integers:
        x = encode(xk, rng.integers(-8, 9, size=(B, K)).astype(np.float64))
        bb = encode(xk, rng.integers(-8, 9, size=M).astype(np.float64)) if bias else None
        scale = np.ones(M, dtype=np.float32) if dtype == "w8" else None
    else:
        def rnd(shape):
            v = rng.standard_normal(shape)
            if xk == "f32":
                return v.astype(np.float32)
            if xk == "f16":
                return enc_f16(v)
            return (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        x = rnd((B, K))
        bb = rnd((M,)) if bias else None
        scale = rng.uniform(1e-3, 1e-2, size=M).astype(np.float32) if dtype == "w8" else None
    return A, x, bb, scale


DTYPES = ("f32", "f16", "bf16", "w8")


# ---------------------------------------------------------------- the pins
def pin_bruteforce(impl, seed=0):
    """Exact rationals on tiny random inputs: fp64 result within gamma_{K+2}."""
    rng = np.random.default_rng(seed)
    for dtype in DTYPES:
        for (M, K, B) in ((1, 1, 1), (3, 5, 2), (5, 3, 3), (4, 8, 1), (2, 7, 2)):
            for bias in (False, True):
                A, x, bb, sc = tiny_inputs(rng, dtype, M, K, B, bias)
                y = impl(dtype, A, x, bb, sc)
                ye, mag = exact(dtype, A, x, bb, sc)
                g = (K + 3) * U64 / (1 - (K + 3) * U64)
                for b in range(B):
                    for m in range(M):
                        err = abs(Fraction(float(y[b, m])) - ye[b][m])
                        assert float(err) <= g * mag[b, m] + 1e-300, \
                            (dtype, M, K, B, bias, b, m, float(y[b, m]), float(ye[b][m]))


def pin_small_integers_exact(impl, seed=1):
    """Small-integer inputs: every partial sum is an exact double, so y is exact."""
    rng = np.random.default_rng(seed)
    for dtype in DTYPES:
        for (M, K, B) in ((3, 4, 2), (6, 9, 3), (1, 16, 1)):
            for bias in (False, True):
                A, x, bb, sc = tiny_inputs(rng, dtype, M, K, B, bias, integers=True)
                y = impl(dtype, A, x, bb, sc)
                ye, _ = exact(dtype, A, x, bb, sc)
                want = np.array([[float(v) for v in row] for row in ye])
                assert np.array_equal(y, want), (dtype, M, K, B, bias)


def pin_identity_permutation(impl, seed=2):
    """A = I gives y = x (+ bias); A = P gives y = P x, exactly."""
    rng = np.random.default_rng(seed)
    for dtype in DTYPES:
        n = 7
        xk = xkind(dtype)
        one = 1.0
        for perm in (np.arange(n), rng.permutation(n)):
            P = np.zeros((n, n))
            P[np.arange(n), perm] = one
            A = encode(dtype, P)
            _, x, bb, _ = tiny_inputs(rng, dtype, n, n, 2, True)
            sc = np.ones(n, dtype=np.float32) if dtype == "w8" else None
            xd = decode_any(xk, x)
            y = impl(dtype, A, x, None, sc)
            assert np.array_equal(y, xd[:, perm]), (dtype, "no bias")
            y = impl(dtype, A, x, bb, sc)
            assert np.array_equal(y, xd[:, perm] + decode_any(xk, bb)[None, :]), (dtype, "bias")


def pin_one_hot(impl, seed=3):
    """x = e_j picks column j of A (times the row scale), exactly."""
    rng = np.random.default_rng(seed)
    for dtype in DTYPES:
        M, K = 5, 6
        A, _, _, sc = tiny_inputs(rng, dtype, M, K, 1, False)
        xk = xkind(dtype)
        Ad = decode_any(dtype, A)
        for j in range(K):
            e = np.zeros((1, K))
            e[0, j] = 1.0
            y = impl(dtype, A, encode(xk, e), None, sc)
            col = Ad[:, j] * (sc.astype(np.float64) if dtype == "w8" else 1.0)
            assert np.array_equal(y[0], col), (dtype, j)


def pin_linearity(impl, seed=4):
    """y(a*x1 + c*x2) = a*y(x1) + c*y(x2): exact on small integers."""
    rng = np.random.default_rng(seed)
    for dtype in DTYPES:
        M, K = 6, 10
        A, x1, _, sc = tiny_inputs(rng, dtype, M, K, 2, False, integers=True)
        _, x2, _, _ = tiny_inputs(rng, dtype, M, K, 2, False, integers=True)
        xk = xkind(dtype)
        a, c = 3.0, -2.0
        x3 = encode(xk, a * decode_any(xk, x1) + c * decode_any(xk, x2))
        y1, y2, y3 = (impl(dtype, A, xx, None, sc) for xx in (x1, x2, x3))
        assert np.array_equal(y3, a * y1 + c * y2), dtype
        # and the batch rows are independent: row b of a batched call equals a B=1 call
        for b in range(2):
            yb = impl(dtype, A, x3[b:b + 1], None, sc)
            assert np.array_equal(yb[0], y3[b]), (dtype, b)


def pin_bias_null(impl, seed=5):
    """bias == NULL is the same as an all-zero bias, bit for bit."""
    rng = np.random.default_rng(seed)
    for dtype in DTYPES:
        A, x, _, sc = tiny_inputs(rng, dtype, 9, 13, 3, False)
        z = encode(xkind(dtype), np.zeros(9))
        assert np.array_equal(impl(dtype, A, x, None, sc), impl(dtype, A, x, z, sc)), dtype


def pin_all_ones(impl):
    """A = 1, x = 1 gives y = K (times s_m); with bias b_m = m, y = K + m."""
    for dtype in DTYPES:
        for K in (1, 16, 32, 128, 300):
            M = 4
            A = encode(dtype, np.ones((M, K)))
            x = encode(xkind(dtype), np.ones((2, K)))
            sc = np.full(M, 0.5, dtype=np.float32) if dtype == "w8" else None
            s = 0.5 if dtype == "w8" else 1.0
            y = impl(dtype, A, x, None, sc)
            assert np.all(y == s * K), (dtype, K)
            bb = encode(xkind(dtype), np.arange(M, dtype=np.float64))
            y = impl(dtype, A, x, bb, sc)
            assert np.array_equal(y, s * K + np.arange(M)[None, :].repeat(2, 0)), (dtype, K)


def pin_rank_one(impl, seed=6):
    """A = u v^T gives y = u (v . x), exactly for small integers."""
    rng = np.random.default_rng(seed)
    for dtype in DTYPES:
        M, K = 5, 12
        u = rng.integers(-11, 12, size=M).astype(np.float64)
        v = rng.integers(-11, 12, size=K).astype(np.float64)
        A = encode(dtype, np.outer(u, v))
        xv = rng.integers(-8, 9, size=(3, K)).astype(np.float64)
        x = encode(xkind(dtype), xv)
        sc = np.ones(M, dtype=np.float32) if dtype == "w8" else None
        y = impl(dtype, A, x, None, sc)
        assert np.array_equal(y, (xv @ v)[:, None] * u[None, :]), dtype


def pin_rectangular_orientation(impl):
    """Row m of A meets x: A[m][k] = m + 1 on a 3 x 1024 matrix (the lesson's
    worked-example shape, 3 rows of 1024 columns) with x = 1 gives y[m] = 1024 (m + 1),
    and with bias[m] = m, y[m] = 1024 (m + 1) + m.  A transposed reading of A would
    index outside a 3-row matrix or give different sums."""
    for dtype in DTYPES:
        M, K = 3, 1024
        A = encode(dtype, np.repeat(np.arange(1, M + 1, dtype=np.float64)[:, None], K, 1))
        x = encode(xkind(dtype), np.ones((1, K)))
        sc = np.ones(M, dtype=np.float32) if dtype == "w8" else None
        bb = encode(xkind(dtype), np.arange(M, dtype=np.float64))
        y = impl(dtype, A, x, bb, sc)
        assert np.array_equal(y[0], 1024.0 * np.arange(1, M + 1) + np.arange(M)), dtype
        # a distinct x per column pins the k index: x[k] = k gives sum_k (m+1) k
        if dtype in ("f32",):
            xk = encode("f32", np.arange(K, dtype=np.float64)[None, :])
            y = impl(dtype, A, xk, None, sc)
            assert np.array_equal(y[0], (np.arange(1, M + 1) * (K * (K - 1) // 2)).astype(np.float64))


def pin_w8_scale_per_row(impl, seed=7):
    """int8 weights with a per-row scale: y[m] = s_m * (integer dot product); the
    scale follows the output row, not the column."""
    rng = np.random.default_rng(seed)
    M, K = 4, 9
    q = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
    xv = rng.integers(-8, 9, size=(2, K)).astype(np.float64)
    x = encode("bf16", xv)
    sc = np.array([1.0, 2.0, 0.25, -4.0], dtype=np.float32)
    y = impl("w8", q, x, None, sc)
    dots = xv @ q.astype(np.float64).T          # (B, M) integers, exact
    assert np.array_equal(y, dots * sc.astype(np.float64)[None, :])


def pin_empty_and_k0(impl):
    """K = 0 is the empty sum: y = bias (or 0)."""
    for dtype in DTYPES:
        M = 3
        A = np.zeros((M, 0), dtype={"f32": np.float32, "w8": np.int8}.get(dtype, np.uint16))
        xk = xkind(dtype)
        x = np.zeros((2, 0), dtype=np.float32 if xk == "f32" else np.uint16)
        sc = np.ones(M, dtype=np.float32) if dtype == "w8" else None
        y = impl(dtype, A, x, None, sc)
        assert y.shape == (2, M) and np.all(y == 0), dtype
        bb = encode(xk, np.array([1.0, -2.0, 0.5]))
        y = impl(dtype, A, x, bb, sc)
        assert np.array_equal(y, np.array([[1.0, -2.0, 0.5]] * 2)), dtype


def pin_special_values(impl):
    """IEEE propagation: a NaN in x poisons every row; inf * 0 is NaN; inf passes."""
    for dtype in ("f32", "f16", "bf16"):
        M, K = 3, 4
        A = encode(dtype, np.array([[1, 0, 0, 0], [0, 1, 0, 0], [0, 0, 0, 1.0]]))
        xv = np.array([[np.inf, 2.0, 3.0, 4.0]])
        if dtype == "f32":
            x = xv.astype(np.float32)
        elif dtype == "f16":
            x = enc_f16(xv)
        else:
            x = enc_bf16_exact(xv)
        y = impl(dtype, A, x, None, None)
        assert np.isnan(y[0, 1]) and np.isnan(y[0, 2]), dtype   # inf * 0 in the sum
        assert y[0, 0] == np.inf, dtype
        xn = x.copy()
        xn[0, 3] = np.float32(np.nan) if dtype == "f32" else np.uint16(0x7FC0 if dtype == "bf16" else 0x7E00)
        y = impl(dtype, A, xn, None, None)
        assert np.all(np.isnan(y)), dtype


ALL_PINS = [
    pin_bruteforce,
    pin_small_integers_exact,
    pin_identity_permutation,
    pin_one_hot,
    pin_linearity,
    pin_bias_null,
    pin_all_ones,
    pin_rank_one,
    pin_rectangular_orientation,
    pin_w8_scale_per_row,
    pin_empty_and_k0,
    pin_special_values,
]
