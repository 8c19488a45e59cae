"""E4M3 (OCP 8-bit floating point, E4M3 encoding) values and nearest-even rounding, written
from the format's definition for the tests of the two-term activation split: sign bit,
4 exponent bits with bias 7, 3 mantissa bits; exponent 0 holds the subnormals m/8 * 2^-6;
S.1111.111 is NaN and there are no infinities (largest finite 448)."""
import numpy as np


def values() -> np.ndarray:
    v = np.empty(256)
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 0xF, c & 7
        if e == 15 and m == 7:
            v[c] = np.nan
        elif e == 0:
            v[c] = s * (m / 8.0) * 2.0 ** -6
        else:
            v[c] = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return v


VALUES = values()
POS = VALUES[:127]  # codes 0..126: the non-negative finite values, ascending


def rne(u: np.ndarray) -> np.ndarray:
    """The E4M3 value nearest to u, ties to the even code (|u| <= 448)."""
    a = np.abs(u)
    assert np.all(a <= 448.0)
    i = np.clip(np.searchsorted(POS, a), 1, 126)
    lo, hi = POS[i - 1], POS[i]
    dlo, dhi = a - lo, hi - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (i % 2 == 0))
    return np.sign(u) * np.where(pick_hi, hi, lo)


def split(x: np.ndarray):
    """The two-term split of a block of values (its largest magnitude sets both scales):
    s_hi = max(b - 7, 0) with b the biased fp32 exponent of the block maximum,
    s_lo = max(s_hi - 5, 0), u = x * 2^(127 - s_hi), hi = E4M3(u), lo = E4M3((u - hi) *
    2^(s_hi - s_lo)).  Returns (s_hi, s_lo, hi, lo) with hi and lo as values."""
    amax = float(np.max(np.abs(x)))
    b = int((np.float32(amax).view(np.uint32) >> 23) & 0xFF)
    s_hi = max(b - 7, 0)
    s_lo = max(s_hi - 5, 0)
    u = x * 2.0 ** (127 - s_hi)
    hi = rne(u)
    lo = rne((u - hi) * 2.0 ** (s_hi - s_lo))
    return s_hi, s_lo, hi, lo
