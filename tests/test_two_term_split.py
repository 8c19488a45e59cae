"""The two-term E4M3 split that carries bf16 activations into the block-scaled tensor cores
(MOE_PATH_PREFILL_FP8X2; its definition is in include/moe.h under moe_ffn), checked on the
CPU against the exactness it claims, over every bf16 magnitude up to the block maximum:

  exact (hi * 2^(s_hi - 127) + lo * 2^(s_lo - 127) == v) for every |v| >= 2^-14 * amax,
  within 2^-21 * amax below that, with no term saturating.

The E4M3 rounding comes from the format's definition (tests/e4m3.py), not from the GPU.  The
GPU's own split is held to the same definition bit for bit in tests/test_gpu_fp8x2.py."""
import numpy as np
import pytest

import e4m3


def _bf16_magnitudes(top: float) -> np.ndarray:
    """Every positive bf16 value (subnormals included) up to `top`."""
    bits = np.arange(1, 0x7F80, dtype=np.uint32) << 16
    v = bits.view(np.float32).astype(np.float64)
    return v[v <= top]


def _scales(amax: float):
    b = int((np.float32(amax).view(np.uint32) >> 23) & 0xFF)
    s_hi = max(b - 7, 0)
    return s_hi, max(s_hi - 5, 0)


@pytest.mark.parametrize("e_max", [-110, -40, -1, 0, 7, 60, 120])
@pytest.mark.parametrize("sig", [1.0, 1.0078125, 1.5, 1.9921875])
def test_split_exact_within_2_to_14_of_the_block_maximum(e_max, sig):
    amax = sig * 2.0 ** e_max  # a bf16 value: sig has at most 8 significant bits
    s_hi, s_lo = _scales(amax)
    assert s_hi >= 5
    v = _bf16_magnitudes(amax)
    v = np.concatenate([v, -v])
    # u in fp32, as the definition computes it (elements some 2^133 below amax underflow there)
    u = (v.astype(np.float32) * np.float32(2.0 ** (127 - s_hi))).astype(np.float64)
    assert np.abs(u).max() < 256.0  # no saturation of the high term (E4M3 max 448)
    hi = e4m3.rne(u)
    # the remainder is exact in fp32 (the same as in fp64)
    r32 = (u.astype(np.float32) - hi.astype(np.float32)).astype(np.float64)
    np.testing.assert_array_equal(r32, u - hi)
    w = (u - hi) * 2.0 ** (s_hi - s_lo)
    assert np.abs(w).max() <= 256.0  # nor of the low term
    lo = e4m3.rne(w)
    recon = hi * 2.0 ** (s_hi - 127) + lo * 2.0 ** (s_lo - 127)
    near = np.abs(v) >= amax * 2.0 ** -14
    np.testing.assert_array_equal(recon[near], v[near])
    assert np.all(np.abs(recon - v) <= amax * 2.0 ** -21)
    # the bound is not loose by much: some element between 2^-18 and 2^-14 of amax is rounded
    band = (np.abs(v) < amax * 2.0 ** -14) & (np.abs(v) >= amax * 2.0 ** -18)
    assert np.any(recon[band] != v[band])


def test_split_of_blocks_with_tiny_maxima_stays_within_the_grid():
    """Block maxima below 2^-120 clamp the scale bytes at 0; the terms then sit on the grid
    2^-136 and the split is still within half a grid step."""
    for bits in (0x0001, 0x0040, 0x007F, 0x0080, 0x0300, 0x0380):
        amax = float(np.array([bits << 16], np.uint32).view(np.float32)[0])
        s_hi, s_lo = _scales(amax)
        v = _bf16_magnitudes(amax)
        u = (v.astype(np.float32) * np.float32(2.0 ** (127 - s_hi))).astype(np.float64)
        hi = e4m3.rne(u)
        lo = e4m3.rne((u - hi) * 2.0 ** (s_hi - s_lo))
        recon = hi * 2.0 ** (s_hi - 127) + lo * 2.0 ** (s_lo - 127)
        assert np.all(np.abs(recon - v) <= 2.0 ** (s_lo - 127 - 10)), hex(bits)


def test_split_helper_matches_the_header_definition_on_a_block():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(32) * 3.0).astype(np.float32)
    x = ((x.view(np.uint32) + 0x7FFF + ((x.view(np.uint32) >> 16) & 1)) >> 16 << 16).view(np.float32)
    x = x.astype(np.float64)
    s_hi, s_lo, hi, lo = e4m3.split(x)
    assert (s_hi, s_lo) == _scales(float(np.abs(x).max()))
    np.testing.assert_array_equal(hi * 2.0 ** (s_hi - 127) + lo * 2.0 ** (s_lo - 127), x)


def test_e4m3_table_pins():
    """Closed-form pins of the E4M3 table: largest finite 448, smallest subnormal 2^-9,
    smallest normal 2^-6, 126 distinct positive finite values, NaN at S.1111.111."""
    v = e4m3.VALUES
    assert v[0x7E] == 448.0 and np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert v[0x01] == 2.0 ** -9 and v[0x08] == 2.0 ** -6 and v[0x80] == 0.0
    assert len(set(v[1:127])) == 126 and np.all(np.diff(v[:127]) > 0)
    np.testing.assert_array_equal(v[0x80:0xFF], -v[0x00:0x7F])
    # nearest even: 1.0625 is halfway between 1.0 (code 0x38) and 1.125 (0x39) -> 1.0
    assert e4m3.rne(np.array([1.0625, 1.1875, -3.25]))[0] == 1.0
    assert e4m3.rne(np.array([1.1875]))[0] == 1.25  # halfway 1.125 | 1.25 -> even code 0x3A
    assert e4m3.rne(np.array([-3.25]))[0] == -3.25
