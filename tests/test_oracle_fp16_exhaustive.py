"""Exhaustive pin of the oracle's binary32 -> binary16 conversion against
numpy's cast.  Every binary32 pattern whose exponent field lies in
[101, 143] is checked -- that covers every input that rounds to a non-zero
finite binary16 value, the underflow boundary (half the smallest subnormal,
2^-25) and the overflow boundary (65520).  Below and above that range every
input rounds to zero or to infinity; those are checked on a stride.  The
per-block FP16 scale of the bitscom README ("Implemented Features") is
produced by this conversion.  NaN inputs are outside the codec's domain."""
import numpy as np


def _check(orc, u):
    x = u.view(np.float32)
    x = x[~np.isnan(x)]
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = orc.f32_to_f16_bits(x)
    if not np.array_equal(got, ref):
        i = int(np.nonzero(got != ref)[0][0])
        raise AssertionError(f"pattern {int(x.view(np.uint32)[i]):#x}: {got[i]:#x} != {ref[i]:#x}")


def test_f32_to_f16_exhaustive_finite_range(orc):
    chunk = 1 << 23
    for e in range(101, 144):
        u = np.arange(e << 23, (e + 1) << 23, dtype=np.uint32)
        _check(orc, u)
    _check(orc, np.array([0, 1, 0x7F800000], dtype=np.uint32))
    assert chunk == 1 << 23


def test_f32_to_f16_outside_range_strided(orc):
    lo = np.arange(0, 101 << 23, 4099, dtype=np.uint32)
    hi = np.arange(144 << 23, 0x7F800001, 4099, dtype=np.uint32)
    _check(orc, lo)
    _check(orc, hi)


def test_f32_to_f16_negative_strided(orc):
    u = np.arange(0x80000000, 0xFF800001, 61, dtype=np.uint64).astype(np.uint32)
    _check(orc, u)
