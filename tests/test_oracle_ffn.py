"""Pins for the oracle's MXFP4 decode and expert FFN (CPU only).

MXFP4 weights dequantised inside the fused MoE kernel: VibeSys Qwen3.5-397B on
4x MI300A, sections "baseline" and "kernels and graph capture".  Shared expert
as one more routed expert: InferenceX MI355X Qwen3.5 blog, PR #20736; vLLM
MiniMax M3 on MI355X, section "shared expert fusion".
"""
import numpy as np
import pytest

import bruteforce as bf


def test_mxfp4_decode_exhaustive(oracle_mod):
    """All 16 codes x 256 scale bytes against the closed form."""
    for code in range(16):
        for s in range(256):
            got = np.float32(oracle_mod.mxfp4_value(code, s))
            with np.errstate(over="ignore"):
                exp = np.float32(bf.e2m1_closed_form(code) * bf.e8m0_closed_form(s))
            if np.isnan(exp):
                assert np.isnan(got), (code, s)
            else:
                assert got == exp, (code, s, got, exp)


def test_bf16_rounding_and_silu(oracle_mod):
    # ties to even, and a carry into the exponent
    assert oracle_mod.f32_to_bf16(np.float32(1.0 + 2.0 ** -8)) == 0x3F80  # tie -> even (down)
    assert oracle_mod.f32_to_bf16(np.float32(1.0 + 3 * 2.0 ** -8)) == 0x3F82  # tie -> even (up)
    assert oracle_mod.f32_to_bf16(np.float32(1.0 + 2.0 ** -8 + 2.0 ** -20)) == 0x3F81
    assert oracle_mod.f32_to_bf16(np.float32(-(2.0 - 2.0 ** -9))) == 0xC000   # rounds up into the exponent
    assert oracle_mod.f32_to_bf16(np.float32(np.inf)) == 0x7F80
    for g in (-30.0, -1.5, 0.0, 0.25, 3.0, 20.0):
        assert abs(oracle_mod.silu(g) - g / (1 + np.exp(-g))) <= 1e-6 * max(1.0, abs(g))


def _tiny(synth_mod, **kw):
    w = synth_mod.scaled(synth_mod.WORKLOADS["tiny16"], **kw)
    d = synth_mod.make_inputs(w)
    return w, d


def _tol_check(got_bits, exp64):
    """The oracle (fp32 sums) against the float64 brute force rounded to bf16:
    the only allowed differences are rare 1-2 ulp flips from fp32 rounding."""
    got = bf.bf16_bits_to_f64(got_bits)
    r = bf.bf16_round(exp64)
    ulp = np.abs(r) * 2.0 ** -7 + 1e-30
    assert (np.abs(got - r) <= 2 * ulp).all()
    assert (got != r).mean() <= 0.01
    assert np.linalg.norm(got - r) <= 2e-4 * np.linalg.norm(r)


@pytest.mark.parametrize("shape", [dict(T=6, H=64, I=32, E=4, K=2, with_shared=False),
                                   dict(T=5, H=96, I=64, E=6, K=3, with_shared=True),
                                   dict(T=16, H=256, I=128, E=8, K=2, with_shared=False)])
def test_ffn_matches_double_bruteforce(oracle_mod, synth_mod, shape):
    w, d = _tiny(synth_mod, **shape)
    ids, wt = oracle_mod.route(d["logits"], w.K, w.with_shared)
    got = oracle_mod.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt)
    exp = bf.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt)
    _tol_check(got, exp)


def _one_expert_weights(H, I, scale=127):
    w13 = np.zeros((1, 2 * I, H // 2), np.uint8)
    s13 = np.full((1, 2 * I, H // 32), scale, np.uint8)
    w2 = np.zeros((1, H, I // 2), np.uint8)
    s2 = np.full((1, H, I // 32), scale, np.uint8)
    return w13, s13, w2, s2


def _set_code(codes, row, k, code):
    b = codes[row, k // 2]
    codes[row, k // 2] = (b & 0xF0) | code if k % 2 == 0 else (b & 0x0F) | (code << 4)


def test_ffn_closed_form_constant_codes(oracle_mod):
    """All codes 2 (value 1) with scale 2^0: g = u = sum(x); h = bf16(silu(S) S);
    y_m = I * h for every m; with weight 1, out = bf16(I * h)."""
    H, I = 64, 32
    w13, s13, w2, s2 = _one_expert_weights(H, I)
    w13[:] = 0x22
    w2[:] = 0x22
    xs = np.zeros((1, H), np.float32)
    xs[0, [0, 5, 17, 63]] = [1.0, 0.5, 2.0, -1.25]  # S = 2.25 exactly
    x = (xs.view(np.uint32) >> 16).astype(np.uint16)
    ids = np.zeros((1, 1), np.int32)
    wt = np.ones((1, 1), np.float32)
    out, acc = oracle_mod.ffn(x, w13, s13, w2, s2, ids, wt, want_f32=True)
    S = 2.25
    h = bf.bf16_round(S / (1 + np.exp(-S)) * S)
    assert np.all(acc == np.float32(I * h))
    assert np.all(bf.bf16_bits_to_f64(out) == bf.bf16_round(I * h))


def test_ffn_closed_form_one_hot(oracle_mod):
    """One nonzero code per row picks one element of x: pins the nibble order,
    the scale group index, gate-before-up rows and the W2 row/column roles."""
    H, I = 128, 64
    w13, s13, w2, s2 = _one_expert_weights(H, I)
    rng = np.random.default_rng(5)
    xs = rng.standard_normal((1, H)).astype(np.float32)
    x = (xs.view(np.uint32) >> 16).astype(np.uint16)
    x64 = bf.bf16_bits_to_f64(x)[0]
    kg = rng.integers(0, H, I)
    ku = rng.integers(0, H, I)
    cg = rng.integers(1, 16, I)
    for n in range(I):
        _set_code(w13[0], n, kg[n], cg[n])
        _set_code(w13[0], I + n, ku[n], 4)              # value 2
        s13[0, n, kg[n] // 32] = 126                     # 2^-1 on the gate's group
    nd = rng.integers(0, I, H)
    for m in range(H):
        _set_code(w2[0], m, nd[m], 3)                    # value 1.5
        s2[0, m, nd[m] // 32] = 129                      # 2^2
    ids = np.zeros((1, 1), np.int32)
    wt = np.full((1, 1), 0.5, np.float32)
    _, acc = oracle_mod.ffn(x, w13, s13, w2, s2, ids, wt, want_f32=True)
    g = np.array([bf.e2m1_closed_form(int(cg[n])) * 0.5 * x64[kg[n]] for n in range(I)])
    u = 2.0 * x64[ku]
    h = np.array([bf.bf16_round(np.float32(oracle_mod.silu(np.float32(g[n])) * np.float32(u[n])))
                  for n in range(I)])
    y = 1.5 * 4.0 * h[nd]
    np.testing.assert_array_equal(acc[0], (0.5 * y).astype(np.float32))


def test_ffn_grouped_equals_per_token(oracle_mod, synth_mod):
    w, d = _tiny(synth_mod, T=24, H=64, I=32, E=5, K=3, with_shared=True)
    ids, wt = oracle_mod.route(d["logits"], w.K, w.with_shared)
    per_tok = oracle_mod.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt)
    for tile_m in (1, 8, 32):
        perm = oracle_mod.permute(ids, w.Et, tile_m)
        grouped = oracle_mod.ffn_grouped(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], wt, perm)
        np.testing.assert_array_equal(grouped, per_tok)


def test_shared_as_expert_equals_routed_plus_dense(oracle_mod, synth_mod):
    w, d = _tiny(synth_mod, T=12, H=64, I=32, E=6, K=2, with_shared=True)
    ids, wt = oracle_mod.route(d["logits"], w.K, True)
    full, _ = oracle_mod.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt,
                             want_f32=True)
    _, routed = oracle_mod.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"],
                               np.ascontiguousarray(ids[:, :2]), np.ascontiguousarray(wt[:, :2]),
                               want_f32=True)
    E = w.E
    _, dense = oracle_mod.ffn(d["x"], d["w13"][E:E + 1].copy(), d["s13"][E:E + 1].copy(),
                              d["w2"][E:E + 1].copy(), d["s2"][E:E + 1].copy(),
                              np.zeros((w.T, 1), np.int32), np.ones((w.T, 1), np.float32),
                              want_f32=True)
    comb = (routed + dense).astype(np.float32)
    bits = (comb.view(np.uint32).astype(np.uint64) + 0x7FFF + ((comb.view(np.uint32) >> 16) & 1))
    np.testing.assert_array_equal(full, (bits >> 16).astype(np.uint16))


def test_w2_scale_increment_doubles_output(oracle_mod, synth_mod):
    w, d = _tiny(synth_mod)
    ids, wt = oracle_mod.route(d["logits"], w.K, w.with_shared)
    a = oracle_mod.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt)
    b = oracle_mod.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"] + 1, ids, wt)
    np.testing.assert_array_equal(bf.bf16_bits_to_f64(b), 2 * bf.bf16_bits_to_f64(a))


def test_token_permutation_equivariance(oracle_mod, synth_mod):
    w, d = _tiny(synth_mod)
    ids, wt = oracle_mod.route(d["logits"], w.K, w.with_shared)
    a = oracle_mod.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt)
    p = np.random.default_rng(0).permutation(w.T)
    b = oracle_mod.ffn(np.ascontiguousarray(d["x"][p]), d["w13"], d["s13"], d["w2"], d["s2"],
                       np.ascontiguousarray(ids[p]), np.ascontiguousarray(wt[p]))
    np.testing.assert_array_equal(b, a[p])
    # the token subset path returns the same rows
    sub = np.array([3, 0, 15], np.int32)
    c = oracle_mod.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt, tokens=sub)
    np.testing.assert_array_equal(c, a[sub])


def test_threads_do_not_change_results(oracle_mod, synth_mod):
    w, d = _tiny(synth_mod)
    ids, wt = oracle_mod.route(d["logits"], w.K, w.with_shared)
    a = oracle_mod.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt, n_threads=1)
    b = oracle_mod.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt, n_threads=4)
    np.testing.assert_array_equal(a, b)
