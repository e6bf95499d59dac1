"""The CPU oracle against its pins (no GPU).

Every pin in ``oracle_pins`` must hold for the oracle; and every plausible
mistake planted in a CPU copy of the definition (a dropped term, a transposed
operand, a wrong index or sign, a wrong decoder, fp32 accumulation) must break at
least one pin, which shows the pins can tell a right oracle from a wrong one.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from tests import oracle_pins as P


def oracle_impl(dtype, A, x, bias, scale):
    y, _ = oracle.gemv(dtype, A, x, bias, scale)
    return y


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle_impl)


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin_threads(pin):
    # the row-parallel build must give the same numbers as the one-thread run
    pin(lambda *a: oracle.gemv(*a, nthreads=4)[0])


def test_decode_f16_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.decode("f16", bits)
    want = P.dec_f16(bits)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_decode_bf16_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.decode("bf16", bits)
    want = P.dec_bf16(bits)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_decode_int8_and_f32():
    q = np.arange(-128, 128, dtype=np.int8)
    assert np.array_equal(oracle.decode("w8", q), np.arange(-128, 128, dtype=np.float64))
    f = np.array([0.0, -0.0, 1.5, -3.25e-39, np.float32(3.4e38)], dtype=np.float32)
    assert np.array_equal(oracle.decode("f32", f), f.astype(np.float64))


def test_absdot_is_sum_of_magnitudes():
    A = np.array([[1.0, -2.0, 3.0], [-1.0, 0.5, 0.0]], dtype=np.float32)
    x = np.array([[2.0, 1.0, -1.0]], dtype=np.float32)
    y, ad = oracle.gemv("f32", A, x)
    assert np.array_equal(y, [[2 - 2 - 3, -2 + 0.5 + 0]])
    assert np.array_equal(ad, [[2 + 2 + 3, 2 + 0.5 + 0]])
    q = np.array([[1, -2], [3, 4]], dtype=np.int8)
    xb = P.enc_bf16_exact([[1.0, 1.0]])
    y, ad = oracle.gemv("w8", q, xb, scale=np.array([2.0, -0.5], dtype=np.float32))
    assert np.array_equal(y, [[-2.0, -3.5]])
    assert np.array_equal(ad, [[6.0, 3.5]])


def test_argument_errors():
    A = np.zeros((2, 3), dtype=np.float32)
    with pytest.raises(ValueError):
        oracle.gemv("f32", A, np.zeros((1, 4), dtype=np.float32))
    with pytest.raises(ValueError):
        oracle.gemv("w8", np.zeros((2, 3), dtype=np.int8), np.zeros((1, 3), dtype=np.uint16))
    with pytest.raises(TypeError):
        oracle.gemv("f16", A, np.zeros((1, 3), dtype=np.uint16))


# ------------------------------------------------------------ planted mistakes
def _base(dtype, A, x, bias, scale, *, dec=P.decode_any, acc=np.float64,
          bias_mode="add", scale_mode="row", k_hi=None, xrow0=False, transpose=False,
          nansum=False):
    Ad = dec(dtype, A)
    xd = dec(P.xkind(dtype), x)
    if transpose:
        Ad = Ad.T
    M, K = Ad.shape
    B = xd.shape[0]
    kk = K if k_hi is None else max(0, K + k_hi)
    y = np.zeros((B, M))
    for b in range(B):
        xb = xd[0] if xrow0 else xd[b]
        for m in range(M):
            terms = (Ad[m, :kk] * xb[:kk]).astype(acc)
            s = acc(0)
            if nansum:
                s = np.nansum(terms)
            else:
                for t in terms:
                    s = acc(s + t)
            if dtype == "w8":
                sc = float(scale[m]) if scale_mode == "row" else float(scale[0])
            else:
                sc = 1.0
            bm = 0.0 if bias is None else float(dec(P.xkind(dtype), bias)[m])
            if bias_mode == "add":
                v = sc * float(s) + bm
            elif bias_mode == "drop":
                v = sc * float(s)
            elif bias_mode == "inside":
                v = sc * (float(s) + bm)
            else:  # "sub"
                v = sc * float(s) - bm
            y[b, m] = v
    return y


def _dec_f16_wrong_bias(kind, a):
    v = P.decode_any(kind, a)
    return v * 0.5 if kind == "f16" else v


def _dec_bf16_as_f16(kind, a):
    return P.dec_f16(a) if kind == "bf16" else P.decode_any(kind, a)


def _dec_int8_unsigned(kind, a):
    if kind == "w8":
        return np.asarray(a).view(np.uint8).astype(np.float64)
    return P.decode_any(kind, a)


MUTANTS = {
    "transposed_A": lambda *a: _base(*a, transpose=True),
    "dropped_bias": lambda *a: _base(*a, bias_mode="drop"),
    "bias_inside_scale": lambda *a: _base(*a, bias_mode="inside"),
    "bias_sign": lambda *a: _base(*a, bias_mode="sub"),
    "scale_not_per_row": lambda *a: _base(*a, scale_mode="first"),
    "dropped_last_k": lambda *a: _base(*a, k_hi=-1),
    "x_row_index": lambda *a: _base(*a, xrow0=True),
    "f16_exponent_bias": lambda *a: _base(*a, dec=_dec_f16_wrong_bias),
    "bf16_read_as_f16": lambda *a: _base(*a, dec=_dec_bf16_as_f16),
    "int8_read_unsigned": lambda *a: _base(*a, dec=_dec_int8_unsigned),
    "fp32_accumulate": lambda *a: _base(*a, acc=np.float32),
    "nan_dropped": lambda *a: _base(*a, nansum=True),
}


def test_correct_copy_passes_pins():
    # the unmutated CPU copy satisfies every pin, so a mutant's failure is its own
    for pin in P.ALL_PINS:
        pin(_base)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    impl = MUTANTS[name]
    failed = []
    for pin in P.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(impl)
        except (AssertionError, IndexError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin catches the planted mistake {name}"


# ------------------------------------------------------------ fused epilogues
# SiLU, the residual add and SwiGLU are pinned against an independent logistic
# function (scipy.special.expit), exact identities and closed forms.
def test_silu_closed_forms():
    import math
    from scipy.special import expit
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(math.log(3.0)) == pytest.approx(0.75 * math.log(3.0), rel=1e-15)
    for v in (-30.0, -3.5, -1.0, -1e-3, 1e-3, 0.5, 2.0, 7.25, 40.0):
        assert oracle.silu(v) - oracle.silu(-v) == pytest.approx(v, rel=1e-14, abs=1e-300)
        assert oracle.silu(v) == pytest.approx(v * expit(v), rel=1e-14)
    assert oracle.silu(100.0) == 100.0
    assert abs(oracle.silu(-100.0)) < 1e-40


def test_gemv_ex_is_gemv_then_elementwise():
    from scipy.special import expit
    rng = np.random.default_rng(20)
    for dtype in P.DTYPES:
        M, K, B = 7, 11, 3
        A, x, bb, sc = P.tiny_inputs(rng, dtype, M, K, B, True)
        y0, ad0 = oracle.gemv(dtype, A, x, bb, sc)
        y, pre, ad = oracle.gemv_ex(dtype, A, x, bb, sc, act=0)
        assert np.array_equal(y, y0) and np.array_equal(pre, y0) and np.array_equal(ad, ad0)
        y, pre, _ = oracle.gemv_ex(dtype, A, x, bb, sc, act=1)
        assert np.array_equal(pre, y0)
        np.testing.assert_allclose(y, y0 * expit(y0), rtol=1e-14, atol=1e-300)
        # residual in y's storage type: small integers make the sum exact
        xk = P.xkind(dtype)
        rv = rng.integers(-9, 10, size=(B, M)).astype(np.float64)
        r = P.encode(xk, rv)
        y, _, _ = oracle.gemv_ex(dtype, A, x, bb, sc, residual=r, act=0)
        assert np.array_equal(y, y0 + rv)


def test_swiglu_on_permutations():
    """A = [P; Q] with permutation matrices: gate = P x, up = Q x, exactly; the
    first I rows are the gate (swapping the halves gives silu(Q x) * P x)."""
    from scipy.special import expit
    rng = np.random.default_rng(21)
    for dtype in P.DTYPES:
        I = 6
        p1, p2 = rng.permutation(I), rng.permutation(I)
        Pm, Qm = np.zeros((I, I)), np.zeros((I, I))
        Pm[np.arange(I), p1] = 1.0
        Qm[np.arange(I), p2] = 1.0
        A = P.encode(dtype, np.vstack([Pm, Qm]))
        _, x, _, _ = P.tiny_inputs(rng, dtype, I, I, 2, False)
        sc = np.ones(2 * I, dtype=np.float32) if dtype == "w8" else None
        xd = P.decode_any(P.xkind(dtype), x)
        y, g, u, adg, adu = oracle.swiglu(dtype, A, x, scale=sc)
        assert np.array_equal(g, xd[:, p1]) and np.array_equal(u, xd[:, p2])
        np.testing.assert_allclose(y, xd[:, p1] * expit(xd[:, p1]) * xd[:, p2], rtol=1e-14, atol=1e-300)
        assert np.array_equal(adg, np.abs(xd[:, p1])) and np.array_equal(adu, np.abs(xd[:, p2]))
        A2 = P.encode(dtype, np.vstack([Qm, Pm]))
        y2, *_ = oracle.swiglu(dtype, A2, x, scale=sc)
        np.testing.assert_allclose(y2, xd[:, p2] * expit(xd[:, p2]) * xd[:, p1], rtol=1e-14, atol=1e-300)


def test_swiglu_bias_and_scale_follow_rows():
    # bias/scale entries 0..I-1 belong to the gate rows, I..2I-1 to the up rows
    I, K = 3, 4
    A = P.encode("w8", np.ones((2 * I, K)))
    x = P.enc_bf16_exact([[1.0, 1.0, 1.0, 1.0]])
    sc = np.array([1, 2, 3, 0.5, 0.25, 2], dtype=np.float32)
    bb = P.enc_bf16_exact([0, 1, 2, 3, 4, 5])
    y, g, u, _, _ = oracle.swiglu("w8", A, x, bias=bb, scale=sc)
    assert np.array_equal(g[0], [4 * 1 + 0, 4 * 2 + 1, 4 * 3 + 2])
    assert np.array_equal(u[0], [4 * 0.5 + 3, 4 * 0.25 + 4, 4 * 2 + 5])
