"""GPU parity of MOE_PATH_PREFILL_FP8X2: the block-scaled GEMMs fed the MXFP4
weights as stored and each bf16 activation as two E4M3 terms.

The two-term split is checked value by value against the definition in
include/moe.h (scale bytes bit for bit; each term the nearest-even E4M3 value,
found by search over the 256 codes of the OCP FP8 E4M3 format; exact
reconstruction where the definition promises it).  The layer is held to the
oracle at the parity bar: every output element on small shapes, every token of
the 288- and 1536-token workloads, tile-edge tokens at 8192 plus a cross-check
of every token against the prefill path.
"""
import numpy as np
import pytest

import e4m3
import gpu_common as gc

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from mxfp4_mixture_experts_softmax_gb300 import libmoe  # noqa: E402
from mxfp4_mixture_experts_softmax_gb300 import synth  # noqa: E402

import oracle  # noqa: E402

THREADS = synth.cpu_threads()
P = libmoe.MOE_PATH_PREFILL_FP8X2


E4M3 = e4m3.VALUES
_rne_e4m3 = e4m3.rne


def _bf16_rows(rng, rows, cols):
    """bf16 bit patterns: N(0,1); N(0,1) x 2^k with k in [-40, 20] per element;
    zeros and signed zeros; bf16 subnormals; 8-significant-bit values at the
    top of their binade; a block holding one large value and tiny others."""
    def to_bf16(f):
        b = np.asarray(f, np.float32).view(np.uint32)
        return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)

    out = np.empty((rows, cols), np.uint16)
    kinds = rows // 6 + 1
    r = 0
    for kind in range(6):
        for _ in range(kinds):
            if r == rows:
                break
            if kind == 0:
                out[r] = to_bf16(rng.standard_normal(cols))
            elif kind == 1:
                out[r] = to_bf16(rng.standard_normal(cols) * 2.0 ** rng.integers(-40, 21, cols))
            elif kind == 2:
                out[r] = np.where(rng.random(cols) < 0.5, 0x0000, 0x8000)
                out[r, ::7] = to_bf16(rng.standard_normal(cols // 7 + 1) * 1e-3)[: len(out[r, ::7])]
            elif kind == 3:
                out[r] = rng.integers(1, 0x80, cols).astype(np.uint16) | (
                    rng.integers(0, 2, cols).astype(np.uint16) << 15)
            elif kind == 4:
                e = rng.integers(100, 160, cols).astype(np.uint16)
                out[r] = (e << 7) | 0x7F | (rng.integers(0, 2, cols).astype(np.uint16) << 15)
            else:
                out[r] = to_bf16(rng.standard_normal(cols) * 1e-6)
                out[r, ::32] = to_bf16(rng.standard_normal(cols // 32) * 1e3)
            r += 1
    return out


def test_split_matches_its_definition():
    rng = np.random.default_rng(5)
    rows, cols = 48, 1024
    bits = _bf16_rows(rng, rows, cols)
    x = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    q_hi, q_lo, s_hi, s_lo = libmoe.moe_split_e4m3x2(gc.to_dev(bits))
    torch.cuda.synchronize()
    q_hi, q_lo = q_hi.cpu().numpy(), q_lo.cpu().numpy()
    s_hi, s_lo = s_hi.cpu().numpy().astype(np.int64), s_lo.cpu().numpy().astype(np.int64)
    blocks = x.reshape(rows, cols // 32, 32)
    amax = np.abs(blocks).max(axis=2)
    b = (amax.astype(np.float32).view(np.uint32) >> 23).astype(np.int64) & 0xFF
    np.testing.assert_array_equal(s_hi, np.maximum(b - 7, 0))
    np.testing.assert_array_equal(s_lo, np.maximum(s_hi - 5, 0))
    sh = np.repeat(s_hi, 32, axis=1)
    sl = np.repeat(s_lo, 32, axis=1)
    u = x * 2.0 ** (127 - sh)
    hi = E4M3[q_hi]
    lo = E4M3[q_lo]
    assert np.isfinite(hi).all() and np.isfinite(lo).all()
    np.testing.assert_array_equal(hi, _rne_e4m3(u))
    np.testing.assert_array_equal(lo, _rne_e4m3((u - hi) * 2.0 ** (sh - sl)))
    recon = hi * 2.0 ** (sh - 127) + lo * 2.0 ** (sl - 127)
    am = np.repeat(amax, 32, axis=1)
    exact = (np.abs(x) >= am * 2.0 ** -14) & (sh >= 5)
    normal_rows = rows // 6 + 1  # the N(0,1) rows come first: nearly every element exact
    assert exact[:normal_rows].mean() > 0.99
    np.testing.assert_array_equal(recon[exact], x[exact])
    assert np.all(np.abs(recon - x)[sh >= 5] <= (am * 2.0 ** -21)[sh >= 5])


def _layer_inputs(w):
    d = synth.make_inputs(w)
    ids, wt = oracle.route(d["logits"], w.K, w.with_shared)
    return d, ids, wt


def _run(d, ids, wt, Et, tile_m, path=P, dev_w=None):
    dev_w = dev_w or gc.upload_weights(d)
    perm = libmoe.moe_permute(gc.to_dev(ids), Et, tile_m)
    out = libmoe.moe_ffn(gc.to_dev(d["x"]), dev_w["w13"], dev_w["s13"], dev_w["w2"], dev_w["s2"],
                         gc.to_dev(wt), perm, path=path)
    torch.cuda.synchronize()
    assert libmoe.moe_device_error() == 0
    return gc.bf16_dev_to_f64(out)


SMALL = {
    "h512_i512": dict(T=37, H=512, I=512, E=16, K=4, with_shared=True, seed=21),
    "h1024_i512": dict(T=130, H=1024, I=512, E=9, K=3, with_shared=True, seed=22),
    "h512_i1024": dict(T=300, H=512, I=1024, E=40, K=6, with_shared=False, seed=23),
    "one_token": dict(T=1, H=512, I=512, E=3, K=2, with_shared=True, seed=24),
}


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("tile_m", [32, 64, 96, 128])
def test_small_full_output(name, tile_m):
    w = synth.scaled(synth.WORKLOADS["tiny16"], **SMALL[name])
    d, ids, wt = _layer_inputs(w)
    ref = gc.bits_to_f64(oracle.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt,
                                    n_threads=THREADS))
    stats = gc.ffn_parity(_run(d, ids, wt, w.Et, tile_m), ref, f"{name}/{tile_m}")
    print(name, tile_m, stats)


@pytest.mark.parametrize("seed", range(8))
def test_random_shapes(seed):
    rng = np.random.default_rng(3000 + seed)
    H = int(rng.choice([512, 1024, 1536]))
    I = int(rng.choice([512, 1024]))
    E = int(rng.integers(1, 41))
    K = int(rng.integers(1, min(E, 12) + 1))
    T = int(rng.integers(1, 300))
    tile_m = int(rng.choice([32, 64, 96, 128]))
    w = synth.scaled(synth.WORKLOADS["tiny16"], T=T, H=H, I=I, E=E, K=K,
                     with_shared=bool(rng.integers(0, 2)), seed=70 + seed)
    d, ids, wt = _layer_inputs(w)
    ref = gc.bits_to_f64(oracle.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt,
                                    n_threads=THREADS))
    gc.ffn_parity(_run(d, ids, wt, w.Et, tile_m), ref, f"seed {seed}: T={T} H={H} I={I} E={E} K={K}")


@pytest.mark.parametrize("tile_m", [32, 96])
def test_split_steps(tile_m):
    """moe_ffn_gate_up, moe_ffn_down (y by pair) and moe_combine on this path
    meet the bar, and agree with moe_ffn (y staged as scaled f16 by position)
    to the staging bound."""
    w = synth.scaled(synth.WORKLOADS["tiny16"], **SMALL["h1024_i512"])
    d, ids, wt = _layer_inputs(w)
    dw = gc.upload_weights(d)
    perm = libmoe.moe_permute(gc.to_dev(ids), w.Et, tile_m)
    ws = libmoe.alloc_workspace(w.T, w.H, w.I, w.Et, ids.shape[1], tile_m)
    x_d, wt_d = gc.to_dev(d["x"]), gc.to_dev(wt)
    libmoe.moe_ffn_gate_up(x_d, dw["w13"], dw["s13"], perm, ws, P)
    libmoe.moe_ffn_down(dw["w2"], dw["s2"], wt_d, perm, ws, w.T, P)
    _, y = libmoe.ffn_views(ws, w.T, w.H, w.I, w.Et, ids.shape[1], tile_m)
    split = torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    libmoe.moe_combine(y, w.T, w.H, ids.shape[1], split)
    torch.cuda.synchronize()
    assert libmoe.moe_device_error() == 0
    whole = _run(d, ids, wt, w.Et, tile_m, dev_w=dw)
    ref = gc.bits_to_f64(oracle.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt,
                                    n_threads=THREADS))
    a = gc.bf16_dev_to_f64(split)
    gc.ffn_parity(a, ref, "split steps")
    gc.staged_close(whole, a, "moe_ffn vs split steps")


FULL = {  # workload -> (tile_m, tokens compared: None = all)
    "mtp_verify288": (32, None),
    "prefill1536": (64, None),
    "skewed_prefill8192": (128, 256),
    "skewed_prefill8192_cal": (128, 256),
}


@pytest.mark.parametrize("name", list(FULL))
def test_full_size(name):
    """Full size in the bench's launch configuration against the oracle; at
    8192 tokens also every token against the prefill path at the bar."""
    w = synth.WORKLOADS[name]
    tile_m, n_tok = FULL[name]
    d, ids, wt = _layer_inputs(w)
    tokens = (np.arange(w.T, dtype=np.int32) if n_tok is None
              else gc.edge_tokens(ids, tile_m, n_tok, 97))
    ref = gc.bits_to_f64(oracle.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt,
                                    tokens=tokens, n_threads=THREADS))
    dev_w = gc.upload_weights(d)
    logits, x = gc.to_dev(d["logits"]), gc.to_dev(d["x"])
    out = gc.bf16_dev_to_f64(libmoe.moe_layer(logits, x, dev_w["w13"], dev_w["s13"], dev_w["w2"],
                                              dev_w["s2"], w.K, w.with_shared, tile_m=tile_m, path=P))
    torch.cuda.synchronize()
    assert libmoe.moe_device_error() == 0
    print(name, "fp8x2", tokens.size, "tokens", gc.ffn_parity(out[tokens], ref, name))
    if n_tok is not None:
        other = gc.bf16_dev_to_f64(libmoe.moe_layer(
            logits, x, dev_w["w13"], dev_w["s13"], dev_w["w2"], dev_w["s2"], w.K, w.with_shared,
            tile_m=tile_m, path=libmoe.MOE_PATH_PREFILL))
        torch.cuda.synchronize()
        print(name, "fp8x2 vs prefill", gc.ffn_parity(out, other, f"{name} fp8x2 vs prefill"))
    del dev_w
    torch.cuda.empty_cache()
