"""The FP8 cache write's division by the KV head scale, checked on the CPU.

The e4m3 code of a new K/V value is that of the IEEE float32 quotient
x / scale ("FlashAttention と FlashInfer" 境界と失敗: per-head quantization
scales). The scatter kernel does not divide: from the correctly rounded
reciprocal y = RN(1/s) it forms q0 = RN(x y), the remainder r = RN(q0 * -s + x)
and q = RN(r y + q0) (Markstein's correction step, P. Markstein, "Computation
of elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
Dev. 34(1), 1990), keeping q0 where q0 = 0 or |q0| >= 512, for scales of
magnitude 2^-32 .. 2^32 (other scales divide). These tests replay those steps
in float32 with an exactly rounded FMA and compare, for every bf16 and every
f16 value and a spread of scales, the quotient bit for bit wherever it can
decide a code, and the e4m3 code everywhere.
"""
import numpy as np
import pytest
import torch

import oracle

F32, F64 = np.float32, np.float64


def fma32(a, b, c):
    """float32 RN(a * b + c), element-wise, from float64: a * b is exact in
    float64; the sum is rounded to odd in float64 (TwoSum gives the exact
    error) and then to float32, which equals one rounding of the exact value
    because float64 carries more than float32's 24 + 2 bits."""
    p = a.astype(F64) * b.astype(F64)
    c = c.astype(F64)
    s = p + c
    bb = s - p
    err = (p - (s - bb)) + (c - bb)
    even = (s.view(np.int64) & 1) == 0
    bump = (err != 0) & even & np.isfinite(s)
    s = np.where(bump, np.nextafter(s, np.where(err > 0, np.inf, -np.inf)), s)
    with np.errstate(over="ignore"):
        return s.astype(F32)


def fast_quotient(x, s):
    """The kernel's steps for x / s (x float32 array, s float32 scalar)."""
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        y = F32(F32(1.0) / s)                       # RN(1/s)
        q0 = x * y                                  # RN(x y)
        r = fma32(q0, np.full_like(x, -s), x)
        corrected = fma32(r, np.full_like(x, y), q0)
        keep = (q0 == 0) | ~(np.abs(q0) < 512)
        return np.where(keep, q0, corrected), q0


def every_value(dtype):
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    return bits.view(dtype).to(torch.float32).numpy()


def codes(v):
    """e4m3 bytes of float32 values (division by 1 is exact)."""
    t = torch.from_numpy(np.ascontiguousarray(v)).reshape(1, -1)
    return oracle.quantize_e4m3(t, [1.0]).numpy().reshape(-1)


def _scales():
    g = np.random.default_rng(91)
    s = [2.0 ** -32, 2.0 ** 32, np.nextafter(F32(2.0 ** -32), F32(1)),
         np.nextafter(F32(2.0 ** 32), F32(0)), 1.0, 0.5, 3.0, 1 / 3, 1 / 7, 0.1, 0.0123,
         3.7 / 448, 1.5 / 448, 12.0 / 448, 2 - 2.0 ** -23, 1 + 2.0 ** -23,
         (2 - 2.0 ** -23) * 2.0 ** -9, 1.0000001e-3, 255.0, 448.0, 1 / 448, -0.37]
    s += list(2.0 ** g.uniform(-32, 32, 60)) + list(g.uniform(0.001, 0.05, 30))
    return [F32(v) for v in s]


SCALES = _scales()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_fast_quotient_is_the_float32_quotient(dtype):
    x = every_value(dtype)
    for s in SCALES:
        with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
            ref = x / s                                     # IEEE float32 division
        q, q0 = fast_quotient(x, s)
        assert np.array_equal(codes(q), codes(ref)), f"scale {s!r}: e4m3 codes differ"
        # Bit for bit wherever the quotient is finite, at least 2^-11 in
        # magnitude and below the saturation shortcut.
        decide = np.isfinite(ref) & (np.abs(ref) >= 2.0 ** -11) & (np.abs(q0) < 512)
        assert np.array_equal(q[decide].view(np.int32), ref[decide].view(np.int32)), \
            f"scale {s!r}: quotient bits differ"


def test_uncorrected_product_is_not_enough():
    """Without the correction step the codes differ for some values and
    scales: the test above has teeth."""
    x = every_value(torch.bfloat16)
    bad_codes = bad_bits = 0
    for s in SCALES:
        with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
            ref = x / s
        _, q0 = fast_quotient(x, s)
        bad_codes += int((codes(q0) != codes(ref)).sum())
        fin = np.isfinite(ref)
        bad_bits += int((q0[fin].view(np.int32) != ref[fin].view(np.int32)).sum())
    assert bad_codes > 0 and bad_bits > 0


def test_fma32_is_exactly_rounded():
    """The emulated FMA against exact rational arithmetic on random operands
    chosen to cancel (the remainder's case) and on random ones."""
    from fractions import Fraction
    g = np.random.default_rng(92)
    a = g.standard_normal(3000).astype(F32)
    b = g.standard_normal(3000).astype(F32)
    c = np.concatenate([-(a[:1500] * b[:1500]), g.standard_normal(1500).astype(F32)])
    got = fma32(a, b, c)
    for i in range(len(a)):
        exact = Fraction(float(a[i])) * Fraction(float(b[i])) + Fraction(float(c[i]))
        # Round the exact value to float32: nearest of the two neighbours,
        # ties to even.
        f = F32(float(exact))
        lo, hi = (f, np.nextafter(f, F32(np.inf))) if Fraction(float(f)) <= exact else \
            (np.nextafter(f, F32(-np.inf)), f)
        dlo, dhi = exact - Fraction(float(lo)), Fraction(float(hi)) - exact
        want = lo if dlo < dhi or (dlo == dhi and (lo.view(np.int32) & 1) == 0) else hi
        assert got[i] == want or (got[i] == 0 and want == 0), (a[i], b[i], c[i])
