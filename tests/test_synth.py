"""The seeded input generator: SplitMix64 counter streams (CPU only)."""
import numpy as np

M64 = (1 << 64) - 1
G = 0x9E3779B97F4A7C15


def _mix(z):
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def test_splitmix_counter_stream(synth_mod):
    seed, stream = 7, 3
    base = _mix((seed * G + stream + 1) & M64)
    exp = [_mix((base + (i + 1) * G) & M64) for i in range(10)]
    np.testing.assert_array_equal(synth_mod.u64(seed, stream, 10), np.array(exp, np.uint64))


def test_deterministic_and_sliceable(synth_mod):
    w = synth_mod.WORKLOADS["tiny16"]
    a, b = synth_mod.make_inputs(w), synth_mod.make_inputs(w)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])
    big = synth_mod.normal_f32(3, 0, (64,))
    np.testing.assert_array_equal(big[:10], synth_mod.normal_f32(3, 0, (10,)))


def test_distributions(synth_mod):
    w = synth_mod.scaled(synth_mod.WORKLOADS["decode64"], E=16, H=512, I=256)
    d = synth_mod.make_inputs(w)
    assert d["w13"].shape == (w.Et, 2 * w.I, w.H // 2) and d["s2"].shape == (w.Et, w.H, w.I // 32)
    assert d["s13"].min() == 127 - 8 and d["s13"].max() == 127 - 4
    nib = np.concatenate([d["w13"].ravel() & 15, d["w13"].ravel() >> 4])
    counts = np.bincount(nib, minlength=16) / nib.size
    assert np.abs(counts - 1 / 16).max() < 0.002
    x = synth_mod.bf16_bits_to_f32(d["x"])
    assert abs(float(x.mean())) < 0.05 and abs(float(x.std()) - 1) < 0.05
    lg = d["logits"]
    assert lg.dtype == np.float32 and abs(float(lg.std()) - 1) < 0.05


def test_skewed_prefill_calibration(synth_mod, oracle_mod):
    """The calibrated Zipf coefficient gives the hottest routed expert about
    10x the mean load; the literal coefficient 2 leaves most experts empty."""
    w = synth_mod.WORKLOADS["skewed_prefill8192_cal"]
    ids, _ = oracle_mod.route(synth_mod.make_logits(w), w.K, True)
    c = np.bincount(ids[:, :w.K].ravel(), minlength=w.E)
    assert 9.0 <= c.max() / c.mean() <= 11.0
    w = synth_mod.WORKLOADS["skewed_prefill8192"]
    ids, _ = oracle_mod.route(synth_mod.make_logits(w), w.K, True)
    c = np.bincount(ids[:, :w.K].ravel(), minlength=w.E)
    assert c.max() == w.T and (c == 0).sum() > 400
