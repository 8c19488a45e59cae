"""Pins for the oracle's MXFP4-activation mode (CPU only).

The pages fuse the activation with an MXFP4 quantisation that feeds an MXFP4
x MXFP4 GEMM (OpenRelay, "Gemma 4 31B from B200 to MI355X", section
"optimisation 4" and section "how far from the ceiling").  The quantisation
rule is the OCP Microscaling v1.0 conversion (the pages print none); the pins
below check the oracle against that rule written another way (tests'
bruteforce module), its defining inequalities, error bounds, idempotence, a
closed form and a float64 brute force of the whole layer on tiny shapes.
"""
import numpy as np
import pytest

import bruteforce as bf

GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _probe_values():
    vals = []
    for a, b in zip(GRID, GRID[1:]):
        mid = (a + b) / 2
        vals += [a, mid, np.nextafter(mid, -1.0), np.nextafter(mid, 9.0), (a + mid) / 2]
    vals += [6.0, 6.5, 7.0, 7.999, 100.0, 1e-30, 0.0]
    rng = np.random.default_rng(3)
    vals += list(rng.uniform(0, 8, 500))
    out = []
    for v in vals:
        out += [float(np.float32(v)), -float(np.float32(v))]
    return out


def test_e2m1_round_matches_binade_rounding(oracle_mod):
    for v in _probe_values():
        assert oracle_mod.e2m1_round(v) == bf.e2m1_round_binade(v), v


def test_e2m1_round_is_identity_on_the_grid(oracle_mod):
    for c in range(16):
        assert oracle_mod.e2m1_round(bf.e2m1_closed_form(c)) == c, c


def test_e2m1_round_ties_go_to_even_codes(oracle_mod):
    # midpoints between neighbours: the result's mantissa bit (code bit 0) is 0
    for a, b in zip(GRID, GRID[1:]):
        c = oracle_mod.e2m1_round((a + b) / 2)
        assert c & 1 == 0 and bf.e2m1_closed_form(c) in (a, b), (a, b, c)


def _blocks(rng, nblk, spread=20):
    """Random blocks of 32 with per-block magnitudes over many binades, some
    exact zeros and exact powers of two."""
    v = rng.standard_normal((nblk, 32)) * 2.0 ** rng.integers(-spread, spread, (nblk, 1))
    v[0] = 0.0
    v[1, :] = 0.0
    v[1, 7] = 2.0 ** -5           # amax exactly a power of two
    v[2, :] = 1.5 * 2.0 ** 3      # amax / X = 6 exactly
    v[3, 0] = -(2.0 ** 4)         # negative power of two as amax
    v[4, :] = -1e-3               # negative values that may round to -0
    return v.astype(np.float32)


def test_quantize_matches_independent_rule(oracle_mod):
    rng = np.random.default_rng(7)
    v = _blocks(rng, 64).reshape(8, 256)
    codes, scales = oracle_mod.quantize_mxfp4(v)
    c2, s2 = bf.quantize_mxfp4(v)
    np.testing.assert_array_equal(scales, s2)
    np.testing.assert_array_equal(codes, c2)


def test_quantize_scale_inequality_and_error_bound(oracle_mod):
    rng = np.random.default_rng(11)
    v = _blocks(rng, 400).reshape(100, 128)
    codes, scales = oracle_mod.quantize_mxfp4(v)
    dq = bf.decode_mxfp4(codes, scales)
    vb = v.astype(np.float64).reshape(100, 4, 32)
    dqb = dq.reshape(100, 4, 32)
    for r in range(100):
        for b in range(4):
            amax = np.abs(vb[r, b]).max()
            s = int(scales[r, b])
            if amax == 0:
                assert s == 0 and not dqb[r, b].any()
                continue
            X = 2.0 ** (s - 127)
            assert 4 * X <= amax < 8 * X, (r, b)
            # elements within range: at most half a grid step off; saturated: below 2X
            a = np.abs(vb[r, b]) / X
            step = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
            err = np.abs(dqb[r, b] - vb[r, b]) / X
            inr = a <= 6
            assert (err[inr] <= step[inr] / 2).all()
            assert (err[~inr] < 2).all()
            assert np.max(np.abs(dqb[r, b])) >= 4 * X     # the block maximum keeps its binade


def test_quantize_is_idempotent(oracle_mod):
    rng = np.random.default_rng(5)
    v = _blocks(rng, 128).reshape(16, 256)
    codes, scales = oracle_mod.quantize_mxfp4(v)
    dq = bf.decode_mxfp4(codes, scales).astype(np.float32)
    c2, s2 = oracle_mod.quantize_mxfp4(dq)
    np.testing.assert_array_equal(s2, scales)
    np.testing.assert_array_equal(c2, codes)


def test_quantize_rejects_non_finite(oracle_mod):
    v = np.zeros((1, 32), np.float32)
    v[0, 3] = np.nan
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.quantize_mxfp4(v)


def _bf16(a):
    return (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _tiny(synth_mod, **kw):
    w = synth_mod.scaled(synth_mod.WORKLOADS["tiny16"], **kw)
    return w, synth_mod.make_inputs(w)


@pytest.mark.parametrize("shape", [dict(T=5, H=64, I=64, E=4, K=2, with_shared=False),
                                   dict(T=4, H=128, I=96, E=5, K=3, with_shared=True),
                                   dict(T=16, H=256, I=128, E=8, K=2, with_shared=False)])
def test_ffn_mxfp4act_matches_float64_bruteforce(oracle_mod, synth_mod, shape):
    """Stage by stage against float64: x's encoding exactly; the SwiGLU output
    before quantisation to fp32 accuracy; h's encoding exactly (decided, like
    the oracle, on the oracle's own fp32 values); the output from float64
    products of the decoded h."""
    w, d = _tiny(synth_mod, **shape)
    ids, wt = oracle_mod.route(d["logits"], w.K, w.with_shared)
    out, acc, h = oracle_mod.ffn_mxfp4act(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt,
                                          want_f32=True, want_h=True)
    T, H = d["x"].shape
    I = d["w13"].shape[1] // 2
    Kt = ids.shape[1]
    xc, xs = bf.quantize_mxfp4(bf.bf16_bits_to_f64(d["x"]))
    xq = bf.decode_mxfp4(xc, xs)
    W13 = bf.decode_mxfp4(d["w13"], d["s13"])
    W2 = bf.decode_mxfp4(d["w2"], d["s2"])
    ref = np.zeros((T, H))
    for t in range(T):
        for j in range(Kt):
            e, r = ids[t, j], t * Kt + j
            g = W13[e, :I] @ xq[t]
            u = W13[e, I:] @ xq[t]
            a64 = g / (1 + np.exp(-g)) * u
            np.testing.assert_allclose(h["a"][r], a64, rtol=2e-4, atol=2e-5 * np.abs(a64).max())
            hc, hs = bf.quantize_mxfp4(h["a"][r])
            np.testing.assert_array_equal(h["codes"][r], hc)
            np.testing.assert_array_equal(h["scales"][r], hs)
            ref[t] += wt[t, j] * (W2[e] @ bf.decode_mxfp4(hc, hs))
    np.testing.assert_allclose(acc, ref, rtol=1e-4, atol=1e-5 * np.abs(ref).max())


def test_ffn_mxfp4act_closed_form_constant_codes(oracle_mod):
    """All weight codes 2 (value 1), scales 2^0, x already on the MXFP4 grid:
    g = u = S = sum(x), every a_n = silu(S) S, so every h block holds one value
    whose code is 6 (4 X) with X = 2^(floor(log2 a) - 2) unless a is zero;
    y_m = I * hq for every m."""
    H, I = 64, 64
    w13 = np.full((1, 2 * I, H // 2), 0x22, np.uint8)
    s13 = np.full((1, 2 * I, H // 32), 127, np.uint8)
    w2 = np.full((1, H, I // 2), 0x22, np.uint8)
    s2 = np.full((1, H, I // 32), 127, np.uint8)
    xs = np.zeros((1, H), np.float32)
    xs[0, [0, 5, 17, 40]] = [4.0, 2.0, -1.0, 6.0]     # on the grid with block scales 2^0
    ids = np.zeros((1, 1), np.int32)
    wt = np.ones((1, 1), np.float32)
    out, acc, h = oracle_mod.ffn_mxfp4act(_bf16(xs), w13, s13, w2, s2, ids, wt, want_f32=True,
                                          want_h=True)
    S = 11.0
    a = np.float32(oracle_mod.silu(np.float32(S)) * np.float32(S))
    assert np.all(h["a"] == a)
    X = 2.0 ** (np.floor(np.log2(a)) - 2)
    hq = bf.e2m1_closed_form(bf.e2m1_round_binade(a / X)) * X
    assert np.all(bf.decode_mxfp4(h["codes"], h["scales"]) == hq)
    assert np.all(acc == np.float32(I * hq))


def test_ffn_mxfp4act_w2_scale_increment_doubles_output(oracle_mod, synth_mod):
    w, d = _tiny(synth_mod)
    ids, wt = oracle_mod.route(d["logits"], w.K, w.with_shared)
    a = oracle_mod.ffn_mxfp4act(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt)
    b = oracle_mod.ffn_mxfp4act(d["x"], d["w13"], d["s13"], d["w2"], d["s2"] + 1, ids, wt)
    np.testing.assert_array_equal(bf.bf16_bits_to_f64(b), 2 * bf.bf16_bits_to_f64(a))


def test_quantize_x_scale_by_power_of_two(oracle_mod, synth_mod):
    """x times 4 moves every scale byte of x's encoding up by 2 and leaves its
    codes unchanged (a power-of-two factor commutes with the rounding)."""
    w, d = _tiny(synth_mod, T=6, H=64, I=64, E=4, K=2, with_shared=False)
    x1 = bf.bf16_bits_to_f64(d["x"]).astype(np.float32)
    xc1, xs1 = oracle_mod.quantize_mxfp4(x1)
    xc2, xs2 = oracle_mod.quantize_mxfp4(x1 * np.float32(4.0))
    np.testing.assert_array_equal(xc1, xc2)
    np.testing.assert_array_equal(xs2.astype(int), xs1.astype(int) + 2)


def test_ffn_mxfp4act_threads_and_token_subset(oracle_mod, synth_mod):
    w, d = _tiny(synth_mod)
    ids, wt = oracle_mod.route(d["logits"], w.K, w.with_shared)
    a = oracle_mod.ffn_mxfp4act(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt)
    b = oracle_mod.ffn_mxfp4act(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt,
                                n_threads=4)
    np.testing.assert_array_equal(a, b)
    sub = np.array([9, 2], np.int32)
    c = oracle_mod.ffn_mxfp4act(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt,
                                tokens=sub)
    np.testing.assert_array_equal(c, a[sub])
