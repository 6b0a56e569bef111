"""The selection kernel's digit window, restated on the CPU (no GPU needed).

The kernel clamps each score between the smallest and the largest float of
a 256-digit window of order keys (a NaN lands on the low end) and takes the
top digit less the window's base as the score's bin.  Its shared histogram
has 256 bins, so every score must land in [0, 255] for every base the kernel
can pick, and, for bases the kernel does not treat as missed (base >= 8), the
bin must be the exact top digit clamped into the window.  This restates the
kernel's arithmetic (order key, window ends, clamp) in numpy and checks both
for every base, with random bit patterns and the special values (zeros of
both signs, infinities, NaNs, subnormals, the largest finite values), under
either answer min() may give for (+0, -0).
"""
import numpy as np
import pytest

WBINS = 256


def order_key(bits):
    b = bits.astype(np.uint64)
    neg = (b >> 31) & 1
    return np.where(neg == 1, (~b) & 0xFFFFFFFF, b | 0x80000000).astype(np.uint64)


def key_float(k):
    k = int(k) & 0xFFFFFFFF
    bits = (k & 0x7FFFFFFF) if (k & 0x80000000) else (~k) & 0xFFFFFFFF
    return np.array([bits], dtype=np.uint32).view(np.float32)[0]


def window_ends(base):
    lo = key_float(max(base << 20, 0x00800000))
    hik = min((((base + WBINS) << 20) - 1) & 0xFFFFFFFF, 0xFF800000)
    hi = key_float(0x7FFFFFFE if hik == 0x7FFFFFFF else hik)
    return lo, hi


SPECIAL = np.array([0x7F800000, 0xFF800000, 0x7FC00000, 0xFFC00000, 0x7F800001, 0xFF800001, 0x80000000, 0,
                    1, 0x80000001, 0x7F7FFFFF, 0xFF7FFFFF, 0x00800000, 0x80800000, 0x82000000, 0x3F800000],
                   dtype=np.uint32)


@pytest.mark.parametrize("zero_pick", ["minus", "plus"])
def test_every_base_bins_in_range_and_exact(zero_pick):
    rng = np.random.default_rng(7)
    vals = np.concatenate([rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32), SPECIAL])
    x = vals.view(np.float32)
    with np.errstate(invalid="ignore"):
        y0 = x + np.float32(0.0)                   # -0 -> +0
        nan = np.isnan(y0)
        exact = (order_key(np.where(x == 0, np.uint32(0), vals)) >> 20).astype(np.int64)
    exact = np.where(nan, 0, exact)                # NaN: key 0
    for base in range(0, 4096 - WBINS + 1):
        lo, hi = window_ends(base)
        assert not np.isnan(lo) and not np.isnan(hi)
        assert not (hi == 0 and np.signbit(hi))    # the top end is never -0
        y = np.where(nan, lo, np.maximum(y0, lo))  # fmaxf(NaN, lo) = lo
        m = np.minimum(y, hi)
        if zero_pick == "plus":                    # min(+0, -0) answered +0
            m = np.where((y == 0) & (hi == 0), np.float32(0.0), m)
        b = (order_key(m.view(np.uint32)) >> 20).astype(np.int64) - base
        assert b.min() >= 0 and b.max() <= WBINS - 1, base
        if base >= 8:
            assert np.array_equal(b, np.clip(exact - base, 0, WBINS - 1)), base
