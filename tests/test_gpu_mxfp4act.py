"""GPU parity of the MXFP4-activation layer (moe_quantize_mxfp4,
moe_ffn_mxfp4act and its two steps) against the CPU oracle's second mode.

x's MXFP4 encoding depends only on bf16 inputs and is compared bit for bit.
h's encoding is decided on fp32 SwiGLU values whose accumulation order
differs between the tensor cores and the oracle's sequential sums, so an
element may land on the neighbouring E2M1 code when the oracle's value lies
within rounding distance of a decision boundary (or a block maximum sits at a
power of two, where the scale itself is decided).  The tests allow a mismatch
only at such elements, check the output on every token whose h matched with
the standard bar, and check the down step on every token by feeding it the
oracle's own h.
"""
import numpy as np
import pytest

import bruteforce as bf
import gpu_common as gc

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from mxfp4_mixture_experts_softmax_gb300 import libmoe  # noqa: E402
from mxfp4_mixture_experts_softmax_gb300 import synth  # noqa: E402

import oracle  # noqa: E402

THREADS = synth.cpu_threads()
E2M1_MIDPOINTS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
# distance (in units of the block scale) from a decision boundary below which
# either neighbouring code is accepted; fp32 sums of 4096 exact products in
# another order differ by far less
BOUNDARY_TOL = 2e-3


def _dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.uint8)).cuda()


def _ambiguous(a: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Elements whose encoding is decided within rounding distance: |a| / X
    near an E2M1 midpoint, or the whole block when its largest magnitude is
    near a power of two (the scale decision)."""
    P, I = a.shape
    X = np.repeat(2.0 ** (scales.astype(np.float64) - 127), 32, axis=1)
    r = np.abs(a.astype(np.float64)) / X
    near = np.min(np.abs(r[..., None] - E2M1_MIDPOINTS), axis=-1) <= BOUNDARY_TOL
    amax = np.abs(a.astype(np.float64)).reshape(P, I // 32, 32).max(-1)
    with np.errstate(divide="ignore"):
        lg = np.log2(np.where(amax > 0, amax, 1.0))
    blk = np.abs(lg - np.round(lg)) <= 1e-5
    return near | np.repeat(blk, 32, axis=1)


def _perm_dev(ids, Et, tile_m):
    return libmoe.moe_permute(gc.to_dev(ids), Et, tile_m)


def _h_by_pair(ws, perm, T, H, I, Et, Kt, tile_m, pairs):
    """GPU h (decoded float64) for the given pair indices, from the workspace."""
    codes, scales = libmoe.mxfp4act_h_views(ws, T, H, I, Et, Kt, tile_m)
    inv = perm["inv_pairs"].cpu().numpy()
    pos = inv[pairs]
    c = codes.cpu().numpy()[pos]
    s = scales.cpu().numpy()[pos]
    return bf.decode_mxfp4(c, s), c, s


def _compare_h(gpu_hd, ref, rows):
    """gpu_hd [n, I] against the oracle's h rows; returns mismatch mask."""
    ref_hd = bf.decode_mxfp4(ref["codes"][rows], ref["scales"][rows])
    mism = gpu_hd != ref_hd
    amb = _ambiguous(ref["a"][rows], ref["scales"][rows])
    bad = mism & ~amb
    assert not bad.any(), f"{int(bad.sum())} h elements differ away from any decision boundary"
    assert mism.mean() <= 1e-3, f"too many boundary flips: {mism.mean():.2e}"
    return mism


# --------------------------------------------------------------- quantiser

@pytest.mark.parametrize("rows,cols", [(37, 256), (1, 4096), (300, 96), (64, 4096)])
def test_quantize_mxfp4_bitexact(rows, cols):
    rng = np.random.default_rng(rows * 7 + cols)
    v = rng.standard_normal((rows, cols)) * 2.0 ** rng.integers(-30, 30, (rows, 1))
    v = v.astype(np.float32)
    v[0, :32] = 0.0                      # all-zero block
    v[0, 32:64] = -1e-3                  # negative values, some rounding to -0
    v[0, 37] = 2.0 ** -3                 # amax exactly a power of two
    if rows > 1:
        v[1, :32] = 2.0 ** -133          # subnormal (also in bf16): scale byte 0, codes 0
        v[1, 32:64] = 3.0 * 2.0 ** 100   # large
    x = (v.view(np.uint32) >> 16).astype(np.uint16)   # bf16 (truncated: exact representable values)
    xf = gc.bits_to_f64(x).astype(np.float32)
    rc, rs = oracle.quantize_mxfp4(xf)
    gc_, gs_ = libmoe.moe_quantize_mxfp4(gc.to_dev(x))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(gs_.cpu().numpy(), rs)
    np.testing.assert_array_equal(gc_.cpu().numpy(), rc)


# -------------------------------------------------------------------- ffn

SMALL = {
    "tiny16": dict(),
    "ragged37": dict(T=37, H=512, I=256, E=16, K=4, with_shared=True, seed=11),
    "wide_k": dict(T=9, H=1024, I=512, E=12, K=5, with_shared=False, seed=13),
    "many_tiles": dict(T=300, H=256, I=256, E=6, K=3, with_shared=True, seed=14),
}


def _case(name):
    w = synth.scaled(synth.WORKLOADS["tiny16"], **SMALL[name])
    d = synth.make_inputs(w)
    ids, wt = oracle.route(d["logits"], w.K, w.with_shared)
    return w, d, ids, wt


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("tile_m", [32, 64, 128, 256])
def test_ffn_mxfp4act_small(name, tile_m):
    w, d, ids, wt = _case(name)
    T, H = d["x"].shape
    Et, I, Kt = w.Et, w.I, ids.shape[1]
    out_ref, ref = oracle.ffn_mxfp4act(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt,
                                       want_h=True, n_threads=THREADS)
    ref_out = gc.bits_to_f64(out_ref)
    dw = gc.upload_weights(d)
    perm = _perm_dev(ids, Et, tile_m)
    ws = libmoe.alloc_workspace_mxfp4act(T, H, I, Et, Kt, tile_m)
    x_d, wt_d = gc.to_dev(d["x"]), gc.to_dev(wt)
    libmoe.moe_ffn_mxfp4act_gate_up(x_d, dw["w13"], dw["s13"], perm, ws)
    torch.cuda.synchronize()
    pairs = np.arange(T * Kt)
    gpu_hd, _, _ = _h_by_pair(ws, perm, T, H, I, Et, Kt, tile_m, pairs)
    mism = _compare_h(gpu_hd, ref, pairs)
    # padding positions of the used tiles encode zeros
    sp = perm["sorted_pairs"].cpu().numpy()
    nt = int(perm["num_tiles"].cpu().numpy()[0])
    codes, scales = libmoe.mxfp4act_h_views(ws, T, H, I, Et, Kt, tile_m)
    pad = np.nonzero(sp[:nt * tile_m] < 0)[0]
    assert not codes.cpu().numpy()[pad].any() and not scales.cpu().numpy()[pad].any()
    # down + combine on the GPU's h: every token whose h matched meets the bar
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    libmoe.moe_ffn_mxfp4act_down(dw["w2"], dw["s2"], wt_d, perm, ws, T, out)
    torch.cuda.synchronize()
    got = gc.bf16_dev_to_f64(out)
    bad_tok = mism.reshape(T, Kt, I).any(axis=(1, 2))
    assert bad_tok.sum() <= max(1, T // 50)
    good = ~bad_tok
    gc.ffn_parity(got[good], ref_out[good], f"{name} tile_m={tile_m}")
    # the whole call runs exactly these steps
    full = libmoe.moe_ffn_mxfp4act(x_d, dw["w13"], dw["s13"], dw["w2"], dw["s2"], wt_d, perm)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(gc.bf16_dev_to_f64(full), got)
    # the down step on the oracle's h: every token meets the bar
    inv = perm["inv_pairs"].cpu().numpy()
    c_all = codes.cpu().numpy().copy()
    s_all = scales.cpu().numpy().copy()
    c_all[inv] = ref["codes"]
    s_all[inv] = ref["scales"]
    codes.copy_(torch.from_numpy(c_all))
    scales.copy_(torch.from_numpy(s_all))
    libmoe.moe_ffn_mxfp4act_down(dw["w2"], dw["s2"], wt_d, perm, ws, T, out)
    torch.cuda.synchronize()
    gc.ffn_parity(gc.bf16_dev_to_f64(out), ref_out, f"{name} tile_m={tile_m} oracle h")
    assert libmoe.moe_device_error() == 0


def test_ffn_mxfp4act_w2_scale_increment_doubles_exactly():
    w, d, ids, wt = _case("ragged37")
    dw = gc.upload_weights(d)
    perm = _perm_dev(ids, w.Et, 32)
    x_d, wt_d = gc.to_dev(d["x"]), gc.to_dev(wt)
    a = libmoe.moe_ffn_mxfp4act(x_d, dw["w13"], dw["s13"], dw["w2"], dw["s2"], wt_d, perm)
    b = libmoe.moe_ffn_mxfp4act(x_d, dw["w13"], dw["s13"], dw["w2"], _dev_u8(d["s2"] + 1), wt_d,
                                perm)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(gc.bf16_dev_to_f64(b), 2 * gc.bf16_dev_to_f64(a))


def test_ffn_mxfp4act_token_permutation_equivariance():
    """Reordering tokens reorders the output rows; h is decided per pair, so
    the results are identical, not just close."""
    w, d, ids, wt = _case("ragged37")
    dw = gc.upload_weights(d)
    p = np.random.default_rng(3).permutation(w.T)

    def run(x, i, wts):
        perm = _perm_dev(i, w.Et, 64)
        o = libmoe.moe_ffn_mxfp4act(gc.to_dev(x), dw["w13"], dw["s13"], dw["w2"], dw["s2"],
                                    gc.to_dev(wts), perm)
        torch.cuda.synchronize()
        return gc.bf16_dev_to_f64(o)

    a = run(d["x"], ids, wt)
    b = run(np.ascontiguousarray(d["x"][p]), np.ascontiguousarray(ids[p]),
            np.ascontiguousarray(wt[p]))
    np.testing.assert_array_equal(b, a[p])


def test_ffn_mxfp4act_rejections_and_empty_batch():
    w, d, ids, wt = _case("tiny16")
    dw = gc.upload_weights(d)
    x_d, wt_d = gc.to_dev(d["x"]), gc.to_dev(wt)
    for tile_m in (8, 16):
        perm = _perm_dev(ids, w.Et, tile_m)
        with pytest.raises(libmoe.MoeError) as e:
            libmoe.moe_ffn_mxfp4act(x_d, dw["w13"], dw["s13"], dw["w2"], dw["s2"], wt_d, perm)
        assert e.value.status == libmoe.MOE_ERR_UNSUPPORTED_SHAPE
    w2_ = synth.scaled(synth.WORKLOADS["tiny16"], H=160, I=96)
    d2 = synth.make_inputs(w2_)
    ids2, wt2 = oracle.route(d2["logits"], w2_.K, w2_.with_shared)
    dw2 = gc.upload_weights(d2)
    perm2 = _perm_dev(ids2, w2_.Et, 32)
    with pytest.raises(libmoe.MoeError) as e:
        libmoe.moe_ffn_mxfp4act(gc.to_dev(d2["x"]), dw2["w13"], dw2["s13"], dw2["w2"], dw2["s2"],
                                gc.to_dev(wt2), perm2)
    assert e.value.status == libmoe.MOE_ERR_UNSUPPORTED_SHAPE
    with pytest.raises(libmoe.MoeError) as e:
        libmoe.moe_quantize_mxfp4(gc.to_dev(np.zeros((2, 48), np.uint16)))
    assert e.value.status == libmoe.MOE_ERR_UNSUPPORTED_SHAPE
    # T = 0: nothing to do
    x0 = torch.empty((0, w.H), dtype=torch.bfloat16, device="cuda")
    perm0 = libmoe.moe_permute(torch.empty((0, ids.shape[1]), dtype=torch.int32, device="cuda"),
                               w.Et, 32)
    out0 = libmoe.moe_ffn_mxfp4act(x0, dw["w13"], dw["s13"], dw["w2"], dw["s2"],
                                   torch.empty((0, ids.shape[1]), dtype=torch.float32,
                                               device="cuda"), perm0)
    assert out0.shape == (0, w.H)


FULL = {"decode64": (32, None), "prefill1536": (64, 64), "skewed_prefill8192": (128, 64),
        "skewed_prefill8192_cal": (128, 64)}


@pytest.mark.parametrize("name", list(FULL))
def test_ffn_mxfp4act_full_size(name):
    """Full-size workloads in the bench's launch configuration, sampled
    tokens against the oracle (h per pair, then the output rows)."""
    w = synth.WORKLOADS[name]
    tile_m, n_tok = FULL[name]
    d = synth.make_inputs(w)
    ids, wt = oracle.route(d["logits"], w.K, w.with_shared)
    T, H = d["x"].shape
    I, Et, Kt = w.I, w.Et, ids.shape[1]
    tokens = (np.arange(T, dtype=np.int32) if n_tok is None
              else gc.edge_tokens(ids, tile_m, n_tok, 97))
    out_ref, ref = oracle.ffn_mxfp4act(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt,
                                       tokens=tokens, want_h=True, n_threads=THREADS)
    dw = gc.upload_weights(d)
    perm = _perm_dev(ids, Et, tile_m)
    ws = libmoe.alloc_workspace_mxfp4act(T, H, I, Et, Kt, tile_m)
    out = libmoe.moe_ffn_mxfp4act(gc.to_dev(d["x"]), dw["w13"], dw["s13"], dw["w2"], dw["s2"],
                                  gc.to_dev(wt), perm, workspace=ws)
    torch.cuda.synchronize()
    assert libmoe.moe_device_error() == 0
    pairs = (tokens[:, None] * Kt + np.arange(Kt)[None, :]).reshape(-1)
    gpu_hd, _, _ = _h_by_pair(ws, perm, T, H, I, Et, Kt, tile_m, pairs)
    mism = _compare_h(gpu_hd, ref, np.arange(pairs.size))
    bad_tok = mism.reshape(tokens.size, Kt, I).any(axis=(1, 2))
    assert bad_tok.sum() <= max(1, tokens.size // 32)
    got = gc.bf16_dev_to_f64(out)[tokens]
    stats = gc.ffn_parity(got[~bad_tok], gc.bits_to_f64(out_ref)[~bad_tok], name)
    print(name, "mxfp4act", stats, "h flips", int(mism.sum()))
    del dw, ws
    torch.cuda.empty_cache()
