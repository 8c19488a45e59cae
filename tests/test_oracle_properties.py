"""Randomised pins of the oracle (CPU only): routing, permutation, MXFP4
quantisation, the expert FFN and the MXFP4-activation layer against the
independent brute-force forms in bruteforce.py on
shapes and value mixes drawn by hypothesis -- exact ties, -inf logits, empty
batches, tile heights of 1 and tiles larger than the batch, zero blocks,
signed zeros, rounding midpoints and exponents across the E8M0 range."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import HealthCheck, given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

import bruteforce as bf  # noqa: E402

# derandomized: the same examples every run, so the suite is a stable gate
SETTINGS = settings(max_examples=150, deadline=None, derandomize=True, database=None,
                    suppress_health_check=[HealthCheck.too_slow])


@st.composite
def routing_cases(draw):
    T = draw(st.integers(0, 5))
    E = draw(st.integers(1, 70))
    K = draw(st.integers(1, E))
    rng = np.random.default_rng(draw(st.integers(0, 2**32 - 1)))
    kind = draw(st.sampled_from(["normal", "grid", "wide"]))
    if kind == "normal":
        logits = rng.standard_normal((T, E))
    elif kind == "grid":  # coarse grid: many exactly equal logits
        logits = np.round(rng.standard_normal((T, E)) * 2) / 2
    else:  # probabilities spanning many orders of magnitude
        logits = rng.standard_normal((T, E)) * 30
    logits = logits.astype(np.float32)
    neg_inf = rng.random((T, E)) < draw(st.sampled_from([0.0, 0.1, 0.6]))
    if T:  # at least one finite logit per token
        neg_inf[np.arange(T), rng.integers(0, E, T)] = False
    logits[neg_inf] = -np.inf
    return logits, K, draw(st.booleans()), draw(st.booleans())


@SETTINGS
@given(routing_cases())
def test_route_matches_bruteforce(oracle_mod, case):
    logits, K, shared, renormalize = case
    ids, w = oracle_mod.route(logits, K, shared, renormalize)
    ids_b, w_b = bf.route(logits, K, shared, renormalize)
    np.testing.assert_array_equal(ids, ids_b)
    np.testing.assert_allclose(w, w_b, rtol=2e-6, atol=2e-7)


@SETTINGS
@given(T=st.integers(0, 30), Kt=st.integers(1, 6), Et=st.integers(1, 40),
       tile_m=st.sampled_from([1, 2, 3, 8, 32, 256]), seed=st.integers(0, 2**32 - 1))
def test_permute_matches_bruteforce(oracle_mod, T, Kt, Et, tile_m, seed):
    rng = np.random.default_rng(seed)
    # skewed or uniform expert choice, repeats within a token allowed
    p = rng.dirichlet(np.full(Et, 0.3)) if seed % 2 else None
    ids = rng.choice(Et, size=(T, Kt), p=p).astype(np.int32)
    got = oracle_mod.permute(ids, Et, tile_m)
    exp = bf.permute(ids, Et, tile_m)
    for k in ("sorted_pairs", "offsets", "inv", "tile_expert"):
        np.testing.assert_array_equal(got[k], exp[k], err_msg=k)
    assert got["num_tiles"] == exp["num_tiles"]


@st.composite
def mx_blocks(draw):
    nb = draw(st.integers(1, 4))
    rng = np.random.default_rng(draw(st.integers(0, 2**32 - 1)))
    kind = draw(st.sampled_from(["normal", "grid", "midpoints", "wide", "sparse"]))
    e0 = draw(st.integers(-120, 120))
    if kind == "normal":
        v = rng.standard_normal(32 * nb) * 2.0**e0
    elif kind == "grid":  # exact E2M1 values times a power of two
        mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
        v = rng.choice(mags, 32 * nb) * rng.choice([-1.0, 1.0], 32 * nb) * 2.0**e0
    elif kind == "midpoints":  # halfway between neighbouring E2M1 values: the tie rule decides
        mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0])
        v = rng.choice(mids, 32 * nb) * rng.choice([-1.0, 1.0], 32 * nb) * 2.0**e0
    elif kind == "wide":  # magnitudes spread over 2^-30 .. 2^30 of each other
        v = rng.standard_normal(32 * nb) * 2.0 ** rng.integers(-30, 31, 32 * nb) * 2.0 ** (e0 // 4)
    else:  # mostly zeros of either sign
        v = np.where(rng.random(32 * nb) < 0.9, rng.choice([0.0, -0.0], 32 * nb),
                     rng.standard_normal(32 * nb))
    v = v.astype(np.float32)
    assert np.isfinite(v).all()
    return v


@SETTINGS
@given(mx_blocks())
def test_quantize_mxfp4_matches_bruteforce(oracle_mod, v):
    codes, scales = oracle_mod.quantize_mxfp4(v)
    codes_b, scales_b = bf.quantize_mxfp4(v)
    np.testing.assert_array_equal(scales, scales_b)
    np.testing.assert_array_equal(codes, codes_b)


@SETTINGS
@given(st.floats(min_value=-40.0, max_value=40.0, allow_nan=False, width=64))
def test_e2m1_round_matches_binade_rounding(oracle_mod, x):
    assert oracle_mod.e2m1_round(x) == bf.e2m1_round_binade(x)


@st.composite
def ffn_cases(draw):
    T = draw(st.integers(1, 4))
    H = draw(st.sampled_from([32, 64, 96, 128]))
    I = draw(st.sampled_from([32, 64, 96]))
    E = draw(st.integers(1, 6))
    K = draw(st.integers(1, E))
    shared = draw(st.booleans())
    rng = np.random.default_rng(draw(st.integers(0, 2**32 - 1)))
    lo = draw(st.integers(100, 130))
    Et = E + int(shared)
    w13 = rng.integers(0, 256, (Et, 2 * I, H // 2), dtype=np.uint8)
    s13 = rng.integers(lo, lo + 6, (Et, 2 * I, H // 32), dtype=np.uint8)
    w2 = rng.integers(0, 256, (Et, H, I // 2), dtype=np.uint8)
    s2 = rng.integers(lo, lo + 6, (Et, H, I // 32), dtype=np.uint8)
    xf = rng.standard_normal((T, H)).astype(np.float32)
    x = (xf.view(np.uint32) >> 16).astype(np.uint16)  # bf16 bits (truncated: any bf16 will do)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    return x, w13, s13, w2, s2, logits, K, shared


@SETTINGS
@given(ffn_cases())
def test_ffn_matches_double_bruteforce(oracle_mod, case):
    """The per-token fp32 loop against float64 products of the closed-form
    decode (h rounded to bf16 in both).  Only fp32 rounding separates them, but
    it can flip an h element's bf16 rounding, and one flipped ulp of a
    dominant h moves y by up to 2^-8 of its norm: the bounds below allow a few
    flips and still fail any wrong index, term or operand (O(1) errors)."""
    x, w13, s13, w2, s2, logits, K, shared = case
    ids, wt = oracle_mod.route(logits, K, shared)
    got = bf.bf16_bits_to_f64(oracle_mod.ffn(x, w13, s13, w2, s2, ids, wt))
    with np.errstate(over="ignore"):  # silu of a large negative g is -0 in both
        ref = bf.bf16_round(bf.ffn(x, w13, s13, w2, s2, ids, wt))
    rms = np.sqrt(np.mean(ref**2))
    assert (np.abs(got - ref) <= 5e-2 * (np.abs(ref) + rms)).all()
    assert np.linalg.norm(got - ref) <= 1e-2 * np.linalg.norm(ref)


@SETTINGS
@given(ffn_cases())
def test_ffn_mxfp4act_stage_by_stage(oracle_mod, case):
    """The MXFP4-activation layer on drawn shapes, stage by stage against
    float64: x's encoding exactly, the SwiGLU output a to fp32 accuracy, h's
    encoding exactly when decided on the oracle's own a (as the oracle does),
    and the output from float64 products of the decoded h."""
    x, w13, s13, w2, s2, logits, K, shared = case
    ids, wt = oracle_mod.route(logits, K, shared)
    out, acc, h = oracle_mod.ffn_mxfp4act(x, w13, s13, w2, s2, ids, wt, want_f32=True, want_h=True)
    T, H = x.shape
    I = w13.shape[1] // 2
    Kt = ids.shape[1]
    xc, xs = bf.quantize_mxfp4(bf.bf16_bits_to_f64(x))
    xq = bf.decode_mxfp4(xc, xs)
    W13 = bf.decode_mxfp4(w13, s13)
    W2 = bf.decode_mxfp4(w2, s2)
    ref = np.zeros((T, H))
    for t in range(T):
        for j in range(Kt):
            e, r = ids[t, j], t * Kt + j
            g = W13[e, :I] @ xq[t]
            u = W13[e, I:] @ xq[t]
            with np.errstate(over="ignore"):
                a64 = g / (1 + np.exp(-g)) * u
            scale = np.abs(a64).max()
            assert (np.abs(h["a"][r] - a64) <= 1e-3 * np.abs(a64) + 1e-4 * scale).all()
            hc, hs = bf.quantize_mxfp4(h["a"][r])
            np.testing.assert_array_equal(h["codes"][r], hc)
            np.testing.assert_array_equal(h["scales"][r], hs)
            ref[t] += wt[t, j] * (W2[e] @ bf.decode_mxfp4(hc, hs))
    np.testing.assert_allclose(acc, ref, rtol=1e-4, atol=1e-5 * np.abs(ref).max())
