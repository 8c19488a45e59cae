"""GPU parity: libmoe (through its C ABI) against the CPU oracle.

Routing ids and the permutation bit for bit; moe_ffn within the stated
floating-point bar (gpu_common.ffn_parity).  Small shapes compare every
output element; the full-size workloads compare every token of the 64-, 288-
and 1536-token workloads and, at 8192 tokens, a sample chosen at the tiles'
edges plus a cross-check of the two GEMM paths on every token, in the launch
configuration the bench times.
"""
import numpy as np
import pytest

import gpu_common as gc

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # the suite is only collected for a GPU run
    pytest.skip("needs a CUDA device", allow_module_level=True)

from mxfp4_mixture_experts_softmax_gb300 import libmoe  # noqa: E402  (loads libmoe, no fallback)
from mxfp4_mixture_experts_softmax_gb300 import synth  # noqa: E402

import oracle  # noqa: E402

THREADS = synth.cpu_threads()
ALL = list(synth.WORKLOADS)


def _route_check(logits, K, shared, renorm=True):
    ids_r, w_r = oracle.route(logits, K, shared, renorm)
    ids_g, w_g = libmoe.moe_route(gc.to_dev(logits), K, shared, renorm)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ids_g.cpu().numpy(), ids_r)
    np.testing.assert_allclose(w_g.cpu().numpy(), w_r, rtol=0, atol=gc.ROUTE_W_ATOL)
    return ids_r, w_r


@pytest.mark.parametrize("name", ALL)
def test_route_workloads(name):
    w = synth.WORKLOADS[name]
    ids, wt = _route_check(synth.make_logits(w), w.K, w.with_shared)
    np.testing.assert_allclose(wt[:, :w.K].sum(1), 1.0, atol=1e-6)


@pytest.mark.parametrize("T,E,K", [(5, 1, 1), (33, 8, 2), (17, 33, 32), (9, 100, 7), (64, 512, 10),
                                   (7, 1024, 32), (3, 64, 32)])
def test_route_shapes(T, E, K):
    rng = np.random.default_rng(T * 131 + E)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    _route_check(logits, K, True)
    _route_check(logits, K, False, renorm=False)


def test_route_ties_zeros_and_neg_inf():
    rng = np.random.default_rng(7)
    T, E = 40, 512
    logits = (np.round(rng.standard_normal((T, E)) * 2) / 2).astype(np.float32)  # many ties
    logits[0] = 0.0
    logits[1, ::2] = -0.0
    logits[2] = -np.inf
    logits[2, 400] = 3.0
    logits[2, 7] = 3.0
    _route_check(logits, 10, True)


@pytest.mark.parametrize("T,E,K,shared,tile_m", [(1, 8, 2, False, 8), (16, 8, 2, False, 8),
                                                 (32, 512, 10, True, 8), (32, 1024, 32, True, 128),
                                                 (33, 512, 10, True, 32), (37, 16, 4, True, 16),
                                                 (64, 512, 10, True, 8), (288, 512, 10, True, 64),
                                                 (0, 64, 4, True, 8)])
def test_route_permute_equals_route_then_permute(T, E, K, shared, tile_m):
    """The fused call (one launch up to MOE_ROUTE_PERMUTE_FUSED_MAX_T tokens) is bit-identical to
    moe_route + moe_permute and to the oracle, with and without per-token shared weights."""
    rng = np.random.default_rng(T * 7 + E)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    sw = (1.0 / (1.0 + np.exp(-rng.standard_normal(T)))).astype(np.float32) if shared else None
    ids_r, w_r = oracle.route(logits, K, shared, True, shared_w=sw)
    Et = E + (1 if shared else 0)
    p_r = oracle.permute(ids_r, Et, tile_m)
    ld = gc.to_dev(logits)
    sw_d = gc.to_dev(sw) if sw is not None else None
    ids_f, w_f, perm_f = libmoe.moe_route_permute(ld, K, tile_m, shared, True, shared_w=sw_d)
    ids_s, w_s = libmoe.moe_route(ld, K, shared, True, shared_w=sw_d)
    perm_s = libmoe.moe_permute(ids_s, Et, tile_m)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ids_f.cpu().numpy(), ids_r)
    np.testing.assert_array_equal(ids_f.cpu().numpy(), ids_s.cpu().numpy())
    np.testing.assert_array_equal(w_f.cpu().numpy(), w_s.cpu().numpy())
    np.testing.assert_allclose(w_f.cpu().numpy(), w_r, rtol=0, atol=gc.ROUTE_W_ATOL)
    if shared:
        np.testing.assert_array_equal(w_f.cpu().numpy()[:, K], sw)
    for key in ("sorted_pairs", "expert_offsets", "inv_pairs", "tile_expert", "num_tiles"):
        np.testing.assert_array_equal(perm_f[key].cpu().numpy(), perm_s[key].cpu().numpy(), key)
    np.testing.assert_array_equal(perm_f["sorted_pairs"].cpu().numpy(), p_r["sorted_pairs"])
    np.testing.assert_array_equal(perm_f["expert_offsets"].cpu().numpy(), p_r["offsets"])


def test_route_shared_weight_rejected_without_shared_slot():
    logits = torch.zeros((4, 16), dtype=torch.float32, device="cuda")
    sw = torch.ones(4, dtype=torch.float32, device="cuda")
    with pytest.raises(libmoe.MoeError):
        libmoe.moe_route(logits, 2, False, True, shared_w=sw)


@pytest.mark.parametrize("name", ALL)
@pytest.mark.parametrize("tile_m", [8, 32, 128])
def test_permute_workloads(name, tile_m):
    w = synth.WORKLOADS[name]
    ids, _ = oracle.route(synth.make_logits(w), w.K, w.with_shared)
    _permute_check(ids, w.Et, tile_m)


def _permute_check(ids, Et, tile_m):
    ref = oracle.permute(ids, Et, tile_m)
    got = libmoe.moe_permute(gc.to_dev(ids.astype(np.int32)), Et, tile_m)
    torch.cuda.synchronize()
    for k_ref, k_got in (("sorted_pairs", "sorted_pairs"), ("offsets", "expert_offsets"),
                         ("inv", "inv_pairs"), ("tile_expert", "tile_expert")):
        np.testing.assert_array_equal(got[k_got].cpu().numpy(), ref[k_ref], err_msg=k_ref)
    assert int(got["num_tiles"].cpu()[0]) == ref["num_tiles"]


@pytest.mark.parametrize("case", ["one_expert", "all_experts_max", "empty", "tile1", "tile256",
                                  "single_token"])
def test_permute_edges(case):
    rng = np.random.default_rng(3)
    if case == "one_expert":
        ids, Et, tm = np.full((500, 1), 2, np.int32), 5, 32
    elif case == "all_experts_max":
        ids = np.stack([rng.permutation(1025)[:33] for _ in range(40)]).astype(np.int32)
        Et, tm = 1025, 16
    elif case == "empty":
        ids, Et, tm = np.zeros((0, 11), np.int32), 513, 8
    elif case == "tile1":
        ids, Et, tm = rng.integers(0, 9, (100, 1)).astype(np.int32), 9, 1
    elif case == "tile256":
        ids = np.stack([rng.permutation(40)[:5] for _ in range(300)]).astype(np.int32)
        Et, tm = 40, 256
    else:
        ids, Et, tm = np.array([[3, 0, 8]], np.int32), 9, 8
    _permute_check(ids, Et, tm)


def _permute_dev(ids, Et, tile_m, multi):
    import os
    old = os.environ.get("MOE_PERMUTE_MULTI")
    os.environ["MOE_PERMUTE_MULTI"] = multi
    try:
        got = libmoe.moe_permute(gc.to_dev(ids.astype(np.int32)), Et, tile_m)
        torch.cuda.synchronize()
    finally:
        if old is None:
            del os.environ["MOE_PERMUTE_MULTI"]
        else:
            os.environ["MOE_PERMUTE_MULTI"] = old
    return {k: got[k].cpu().numpy() for k in ("sorted_pairs", "expert_offsets", "inv_pairs",
                                              "tile_expert", "num_tiles")}


@pytest.mark.parametrize("case", ["workload8192", "workload1536", "one_expert", "experts1025",
                                  "tile1", "tile256", "bad_ids", "few_pairs_many_blocks"])
def test_permute_multi_block_equals_single_block(case):
    """The multi-block sort (large batches) and the single-block kernel give
    the same bytes, including ids outside [0, Et) (skipped, inv = -1); where
    every id is valid both equal the oracle."""
    rng = np.random.default_rng(5)
    if case.startswith("workload"):
        w = synth.WORKLOADS["skewed_prefill8192" if case == "workload8192" else "prefill1536"]
        ids, _ = oracle.route(synth.make_logits(w), w.K, w.with_shared)
        Et, tm = w.Et, 128
    elif case == "one_expert":
        ids, Et, tm = np.full((20000, 1), 3, np.int32), 7, 64
    elif case == "experts1025":
        ids = np.stack([rng.permutation(1025)[:20] for _ in range(1000)]).astype(np.int32)
        Et, tm = 1025, 16
    elif case == "tile1":
        ids, Et, tm = rng.integers(0, 9, (9000, 2)).astype(np.int32), 9, 1
    elif case == "tile256":
        ids = np.stack([rng.permutation(60)[:6] for _ in range(3000)]).astype(np.int32)
        Et, tm = 60, 256
    elif case == "bad_ids":
        ids = rng.integers(0, 40, (3000, 5)).astype(np.int32)
        ids[rng.random(ids.shape) < 0.01] = -1
        ids[rng.random(ids.shape) < 0.01] = 40
        Et, tm = 40, 32
    else:  # slices of fewer pairs than blocks * 32: empty warp sub-slices
        ids, Et, tm = rng.integers(0, 2, (8192, 1)).astype(np.int32), 2, 8
    single = _permute_dev(ids, Et, tm, "0")
    multi = _permute_dev(ids, Et, tm, "1")
    for k in single:
        np.testing.assert_array_equal(multi[k], single[k], err_msg=k)
    if case != "bad_ids":
        _permute_check(ids, Et, tm)
    else:
        bad = (ids.reshape(-1) < 0) | (ids.reshape(-1) >= Et)
        assert (multi["inv_pairs"][bad] == -1).all() and (multi["inv_pairs"][~bad] >= 0).all()


# ------------------------------------------------------------------- ffn

def _layer_inputs(w):
    d = synth.make_inputs(w)
    ids, wt = oracle.route(d["logits"], w.K, w.with_shared)
    return d, ids, wt


def _gpu_ffn(d, ids, wt, Et, tile_m, path=libmoe.MOE_PATH_AUTO, dev_w=None):
    dev_w = dev_w or gc.upload_weights(d)
    ids_d = gc.to_dev(ids)
    perm = libmoe.moe_permute(ids_d, Et, tile_m)
    out = libmoe.moe_ffn(gc.to_dev(d["x"]), dev_w["w13"], dev_w["s13"], dev_w["w2"], dev_w["s2"],
                         gc.to_dev(wt), perm, path=path)
    torch.cuda.synchronize()
    return gc.bf16_dev_to_f64(out)


SMALL = {
    "tiny16": dict(),
    "ragged37": dict(T=37, H=512, I=256, E=16, K=4, with_shared=True, seed=11),
    "k_tail": dict(T=21, H=160, I=96, E=6, K=3, with_shared=True, seed=12),
    "wide_k": dict(T=9, H=1024, I=512, E=12, K=5, with_shared=False, seed=13),
}


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("tile_m", [8, 16, 32, 64])
def test_ffn_small_full_output(name, tile_m):
    w = synth.scaled(synth.WORKLOADS["tiny16"], **SMALL[name])
    d, ids, wt = _layer_inputs(w)
    ref = gc.bits_to_f64(oracle.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt,
                                    n_threads=THREADS))
    got = _gpu_ffn(d, ids, wt, w.Et, tile_m, libmoe.MOE_PATH_DECODE)
    gc.ffn_parity(got, ref, f"{name} tile_m={tile_m}")


def test_ffn_tile_m_does_not_change_results():
    w = synth.scaled(synth.WORKLOADS["tiny16"], **SMALL["ragged37"])
    d, ids, wt = _layer_inputs(w)
    outs = [_gpu_ffn(d, ids, wt, w.Et, tm, libmoe.MOE_PATH_DECODE) for tm in (8, 16, 32, 64)]
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])


def test_ffn_scale_bytes_above_128():
    """Large E8M0 scales take the second power-of-two multiply."""
    w = synth.scaled(synth.WORKLOADS["tiny16"], T=12, H=128, I=64, E=4, K=2, seed=21)
    d, ids, wt = _layer_inputs(w)
    rng = np.random.default_rng(0)
    d["s13"] = rng.integers(118, 136, d["s13"].shape).astype(np.uint8)
    d["s2"] = rng.integers(100, 120, d["s2"].shape).astype(np.uint8)
    ref = gc.bits_to_f64(oracle.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt))
    gc.ffn_parity(_gpu_ffn(d, ids, wt, w.Et, 8, libmoe.MOE_PATH_DECODE), ref, "big scales")


@pytest.mark.parametrize("path,tile_m", [(libmoe.MOE_PATH_DECODE, 8), (libmoe.MOE_PATH_PREFILL, 32)])
def test_ffn_activation_dynamic_range(path, tile_m):
    """Token rows scaled by 2^-30 .. 2^30, an all-zero row and a row with one
    element 2^40 above the rest: each output row meets the bar on its own
    scale (the decode path re-encodes rows as f16 with a per-row factor)."""
    w = synth.scaled(synth.WORKLOADS["tiny16"], **SMALL["ragged37"])
    d, ids, wt = _layer_inputs(w)
    xf = gc.bits_to_f64(d["x"])
    exps = np.resize(np.array([-30, -12, 0, 9, 30]), w.T)
    xf *= np.exp2(exps)[:, None]
    xf[3] = 0.0
    xf[7, 5] = 2.0 ** 40
    d["x"] = (xf.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)  # exact: powers of two
    assert np.array_equal(gc.bits_to_f64(d["x"]), xf)
    ref = gc.bits_to_f64(oracle.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt,
                                    n_threads=THREADS))
    got = _gpu_ffn(d, ids, wt, w.Et, tile_m, path)
    assert (got[3] == 0).all() and (ref[3] == 0).all()
    for t in range(w.T):
        gc.ffn_parity(got[t], ref[t], f"row {t} (x scaled 2^{exps[t]})")


def test_ffn_w2_scale_increment_doubles_exactly():
    w = synth.scaled(synth.WORKLOADS["tiny16"], **SMALL["ragged37"])
    d, ids, wt = _layer_inputs(w)
    a = _gpu_ffn(d, ids, wt, w.Et, 16, libmoe.MOE_PATH_DECODE)
    d2 = dict(d, s2=d["s2"] + 1)
    b = _gpu_ffn(d2, ids, wt, w.Et, 16, libmoe.MOE_PATH_DECODE)
    np.testing.assert_array_equal(b, 2 * a)


def test_ffn_token_permutation_equivariance():
    w = synth.scaled(synth.WORKLOADS["tiny16"], **SMALL["ragged37"])
    d, ids, wt = _layer_inputs(w)
    a = _gpu_ffn(d, ids, wt, w.Et, 8, libmoe.MOE_PATH_DECODE)
    p = np.random.default_rng(1).permutation(w.T)
    d2 = dict(d, x=np.ascontiguousarray(d["x"][p]))
    b = _gpu_ffn(d2, np.ascontiguousarray(ids[p]), np.ascontiguousarray(wt[p]), w.Et, 8,
                 libmoe.MOE_PATH_DECODE)
    np.testing.assert_array_equal(b, a[p])


def test_shared_as_expert_equals_routed_plus_dense():
    w = synth.scaled(synth.WORKLOADS["tiny16"], **SMALL["ragged37"])
    d, ids, wt = _layer_inputs(w)
    full = _gpu_ffn(d, ids, wt, w.Et, 8, libmoe.MOE_PATH_DECODE)
    K = w.K
    routed = _gpu_ffn(d, np.ascontiguousarray(ids[:, :K]), np.ascontiguousarray(wt[:, :K]), w.Et,
                      8, libmoe.MOE_PATH_DECODE)
    E = w.E
    dense_w = {k: np.ascontiguousarray(d[k][E:E + 1]) for k in ("w13", "s13", "w2", "s2")}
    dense = _gpu_ffn(dict(d, **dense_w), np.zeros((w.T, 1), np.int32),
                     np.ones((w.T, 1), np.float32), 1, 8, libmoe.MOE_PATH_DECODE)
    # full = bf16(acc_routed + y_shared); routed and dense are each rounded to
    # bf16 on their own, so allow the three roundings (1/2 ulp each, 2^-8 rel)
    s = routed + dense
    bound = 2.0 ** -8 * (np.abs(routed) + np.abs(dense) + np.abs(full)) + 1e-30
    assert (np.abs(full - s) <= bound).all()
    assert np.linalg.norm(full - s) <= 5e-3 * np.linalg.norm(full)


def test_ffn_empty_batch():
    w = synth.scaled(synth.WORKLOADS["tiny16"], T=0)
    d = synth.make_weights(w)
    dev_w = gc.upload_weights(d)
    ids = torch.zeros((0, w.Kt), dtype=torch.int32, device="cuda")
    perm = libmoe.moe_permute(ids, w.Et, 8)
    out = libmoe.moe_ffn(torch.zeros((0, w.H), dtype=torch.bfloat16, device="cuda"), dev_w["w13"],
                         dev_w["s13"], dev_w["w2"], dev_w["s2"],
                         torch.zeros((0, w.Kt), dtype=torch.float32, device="cuda"), perm)
    torch.cuda.synchronize()
    assert out.shape == (0, w.H)
    assert int(perm["num_tiles"].cpu()[0]) == 0


# ------------------------------------------------- full-size workloads

FULL = {  # workload -> (tile_m, tokens compared: None = all), on the decode path
    "decode64": (8, None),
    "mtp_verify288": (8, None),
    "prefill1536": (8, 96),
    "skewed_prefill8192": (8, 64),
    "skewed_prefill8192_cal": (8, 64),
}


def _tokens_for(w, ids, tile_m, n_tok, seed):
    if n_tok is None:
        return np.arange(w.T, dtype=np.int32)
    return gc.edge_tokens(ids, tile_m, n_tok, seed)


@pytest.mark.parametrize("name", list(FULL))
def test_ffn_full_size(name):
    w = synth.WORKLOADS[name]
    tile_m, n_tok = FULL[name]
    d, ids, wt = _layer_inputs(w)
    tokens = _tokens_for(w, ids, tile_m, n_tok, 99)
    ref = gc.bits_to_f64(oracle.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt,
                                    tokens=tokens, n_threads=THREADS))
    dev_w = gc.upload_weights(d)
    # the whole layer: route -> permute -> ffn on the device
    out = libmoe.moe_layer(gc.to_dev(d["logits"]), gc.to_dev(d["x"]), dev_w["w13"], dev_w["s13"],
                           dev_w["w2"], dev_w["s2"], w.K, w.with_shared, tile_m=tile_m,
                           path=libmoe.MOE_PATH_DECODE)
    torch.cuda.synchronize()
    assert libmoe.moe_device_error() == 0
    got = gc.bf16_dev_to_f64(out)[tokens]
    stats = gc.ffn_parity(got, ref, name)
    print(name, tokens.size, "tokens", stats)
    del dev_w
    torch.cuda.empty_cache()


@pytest.mark.parametrize("path,tile_m", [(libmoe.MOE_PATH_DECODE, 8), (libmoe.MOE_PATH_PREFILL, 128)])
def test_gemm_events_bracket_the_gemm_kernel(path, tile_m):
    """The profiling hook records its events around the GEMM kernel alone: the
    interval is positive and shorter than the whole call's; switched off, the
    events are not recorded again and the result is unchanged."""
    w = synth.scaled(synth.WORKLOADS["tiny16"], T=300, H=512, I=256, E=16, K=4, with_shared=True,
                     seed=17)
    d, ids, wt = _layer_inputs(w)
    dw = gc.upload_weights(d)
    x, wt_d = gc.to_dev(d["x"]), gc.to_dev(wt)
    perm = libmoe.moe_permute(gc.to_dev(ids), w.Et, tile_m)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    ev[0].record()
    libmoe.moe_set_gemm_events(ev[1], ev[2])
    try:
        out = libmoe.moe_ffn_gate_up(x, dw["w13"], dw["s13"], perm,
                                     libmoe.alloc_workspace(w.T, w.H, w.I, w.Et, w.Kt, tile_m), path)
    finally:
        libmoe.moe_set_gemm_events(None, None)
    ev[3].record()
    torch.cuda.synchronize()
    gemm_ms, call_ms = ev[1].elapsed_time(ev[2]), ev[0].elapsed_time(ev[3])
    assert 0.0 < gemm_ms < call_ms
    before = ev[2].elapsed_time(ev[3])
    ref = libmoe.moe_ffn(x, dw["w13"], dw["s13"], dw["w2"], dw["s2"], wt_d, perm, path=path)
    torch.cuda.synchronize()
    assert ev[2].elapsed_time(ev[3]) == before  # not re-recorded once switched off
    gc.ffn_parity(gc.bf16_dev_to_f64(ref), gc.bits_to_f64(
        oracle.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt)), "after the hook")


def test_layer_graph_capture_replays_identically():
    w = synth.scaled(synth.WORKLOADS["tiny16"], **SMALL["ragged37"])
    d = synth.make_inputs(w)
    dev_w = gc.upload_weights(d)
    logits, x = gc.to_dev(d["logits"]), gc.to_dev(d["x"])
    bufs = libmoe.alloc_layer(w.T, w.E, w.K, w.with_shared, w.H, w.I, w.Et, 8)
    eager = libmoe.moe_layer(logits, x, dev_w["w13"], dev_w["s13"], dev_w["w2"], dev_w["s2"], w.K,
                             w.with_shared, tile_m=8, bufs=bufs).clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            libmoe.moe_layer(logits, x, dev_w["w13"], dev_w["s13"], dev_w["w2"], dev_w["s2"], w.K,
                             w.with_shared, tile_m=8, bufs=bufs)
    torch.cuda.current_stream().wait_stream(s)
    bufs["out"].zero_()
    g.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(gc.bf16_dev_to_f64(bufs["out"]), gc.bf16_dev_to_f64(eager))


@pytest.mark.parametrize("path,tile_m", [(libmoe.MOE_PATH_DECODE, 8),
                                         (libmoe.MOE_PATH_DECODE, 64),
                                         (libmoe.MOE_PATH_PREFILL, 64)])
def test_split_steps_equal_moe_ffn(path, tile_m):
    """gate_up, down and combine as separate calls reproduce moe_ffn: bit for
    bit on the decode path; on the prefill path moe_ffn's combine reads y
    staged as scaled f16, so the two agree to the staging bound and both
    meet the bar against the oracle."""
    w = synth.scaled(synth.WORKLOADS["tiny16"], **SMALL["ragged37"])
    d, ids, wt = _layer_inputs(w)
    dev_w = gc.upload_weights(d)
    x, topk_w = gc.to_dev(d["x"]), gc.to_dev(wt)
    perm = libmoe.moe_permute(gc.to_dev(ids), w.Et, tile_m)
    whole = libmoe.moe_ffn(x, dev_w["w13"], dev_w["s13"], dev_w["w2"], dev_w["s2"], topk_w, perm,
                           path=path).clone()
    ws = libmoe.alloc_workspace(w.T, w.H, w.I, w.Et, w.Kt, tile_m)
    ws.fill_(0xFF)  # every byte the steps read must be written by an earlier step
    libmoe.moe_ffn_gate_up(x, dev_w["w13"], dev_w["s13"], perm, ws, path)
    libmoe.moe_ffn_down(dev_w["w2"], dev_w["s2"], topk_w, perm, ws, w.T, path)
    _, y = libmoe.ffn_views(ws, w.T, w.H, w.I, w.Et, w.Kt, tile_m)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    libmoe.moe_combine(y, w.T, w.H, w.Kt, out)
    torch.cuda.synchronize()
    a, b = gc.bf16_dev_to_f64(out), gc.bf16_dev_to_f64(whole)
    assert np.isfinite(a).all()
    if path == libmoe.MOE_PATH_DECODE:
        np.testing.assert_array_equal(a, b)
    else:
        gc.staged_close(a, b, "split steps vs moe_ffn")
        ref = gc.bits_to_f64(oracle.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt,
                                        n_threads=THREADS))
        gc.ffn_parity(a, ref, "split steps")
        gc.ffn_parity(b, ref, "moe_ffn")


# ------------------------------------------------------ prefill (tcgen05)

@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("tile_m", [32, 64, 128, 256])
def test_prefill_small_full_output(name, tile_m):
    w = synth.scaled(synth.WORKLOADS["tiny16"], **SMALL[name])
    d, ids, wt = _layer_inputs(w)
    ref = gc.bits_to_f64(oracle.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt,
                                    n_threads=THREADS))
    got = _gpu_ffn(d, ids, wt, w.Et, tile_m, libmoe.MOE_PATH_PREFILL)
    assert libmoe.moe_device_error() == 0
    gc.ffn_parity(got, ref, f"prefill {name} tile_m={tile_m}")


def test_prefill_scale_bytes_above_128():
    w = synth.scaled(synth.WORKLOADS["tiny16"], T=12, H=128, I=64, E=4, K=2, seed=21)
    d, ids, wt = _layer_inputs(w)
    rng = np.random.default_rng(0)
    d["s13"] = rng.integers(118, 136, d["s13"].shape).astype(np.uint8)
    d["s2"] = rng.integers(100, 120, d["s2"].shape).astype(np.uint8)
    ref = gc.bits_to_f64(oracle.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt))
    gc.ffn_parity(_gpu_ffn(d, ids, wt, w.Et, 32, libmoe.MOE_PATH_PREFILL), ref, "big scales")


@pytest.mark.parametrize("path,tile_m", [(libmoe.MOE_PATH_DECODE, 8), (libmoe.MOE_PATH_PREFILL, 32)])
def test_ffn_scales_spread_within_rows(path, tile_m):
    """Scale bytes spread over 2^-60..2^20 inside each weight row, and rows
    whose largest scale is tiny or huge (the prefill path stores each row
    relative to its largest scale; groups more than 2^36 below it round)."""
    w = synth.scaled(synth.WORKLOADS["tiny16"], T=20, H=512, I=128, E=4, K=2, seed=23)
    d, ids, wt = _layer_inputs(w)
    rng = np.random.default_rng(5)
    d["s13"] = rng.integers(67, 148, d["s13"].shape).astype(np.uint8)
    d["s13"][:, 0, :] = rng.integers(60, 70, d["s13"].shape[2])     # a row of tiny scales
    d["s13"][:, 1, :] = rng.integers(140, 150, d["s13"].shape[2])   # a row of large ones
    d["s2"] = rng.integers(90, 140, d["s2"].shape).astype(np.uint8)
    ref = gc.bits_to_f64(oracle.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt))
    assert np.isfinite(ref).all()
    gc.ffn_parity(_gpu_ffn(d, ids, wt, w.Et, tile_m, path), ref, "spread scales")


def test_prefill_tile_m_and_permutation_invariance():
    w = synth.scaled(synth.WORKLOADS["tiny16"], **SMALL["ragged37"])
    d, ids, wt = _layer_inputs(w)
    outs = [_gpu_ffn(d, ids, wt, w.Et, tm, libmoe.MOE_PATH_PREFILL) for tm in (32, 64, 128, 256)]
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])
    p = np.random.default_rng(1).permutation(w.T)
    b = _gpu_ffn(dict(d, x=np.ascontiguousarray(d["x"][p])), np.ascontiguousarray(ids[p]),
                 np.ascontiguousarray(wt[p]), w.Et, 32, libmoe.MOE_PATH_PREFILL)
    np.testing.assert_array_equal(b, outs[0][p])
    d2 = dict(d, s2=d["s2"] + 1)
    np.testing.assert_array_equal(_gpu_ffn(d2, ids, wt, w.Et, 32, libmoe.MOE_PATH_PREFILL),
                                  2 * outs[0])


@pytest.mark.parametrize("path,tile_m", [(libmoe.MOE_PATH_DECODE, 8), (libmoe.MOE_PATH_PREFILL, 32),
                                         (libmoe.MOE_PATH_PREFILL, 128)])
def test_many_slots_per_token(path, tile_m):
    """Top-16 plus the shared expert (17 slots, an odd count above the
    combines' groups of loads) over 40 experts: every output element meets
    the bar on the decode path, the single-CTA prefill kernel and the CTA
    pairs."""
    w = synth.scaled(synth.WORKLOADS["tiny16"], T=40, H=256, I=128, E=40, K=16, with_shared=True,
                     seed=17)
    d, ids, wt = _layer_inputs(w)
    assert ids.shape[1] == 17
    ref = gc.bits_to_f64(oracle.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt,
                                    n_threads=THREADS))
    got = _gpu_ffn(d, ids, wt, w.Et, tile_m, path)
    gc.ffn_parity(got, ref, f"17 slots path={path} tile_m={tile_m}")
    assert libmoe.moe_device_error() == 0


def _random_case(seed):
    """A seeded random layer shape and launch configuration: widths multiples
    of 32 (H of 128 for an even number of 128-row blocks only some of the
    time, so the CTA-pair launcher also falls back to the single-CTA kernel),
    1-40 experts, top-1 to top-12, with or without the shared expert, and a
    tile height and path the shape allows."""
    rng = np.random.default_rng(1000 + seed)
    H = int(rng.choice([128, 256, 384, 512, 640, 1024]))
    I = int(rng.choice([64, 96, 128, 192, 256, 384]))
    E = int(rng.integers(1, 41))
    K = int(rng.integers(1, min(E, 12) + 1))
    T = int(rng.integers(1, 260))
    shared = bool(rng.integers(0, 2))
    path, tile_m = [(libmoe.MOE_PATH_DECODE, 8), (libmoe.MOE_PATH_DECODE, 16),
                    (libmoe.MOE_PATH_DECODE, 64), (libmoe.MOE_PATH_PREFILL, 32),
                    (libmoe.MOE_PATH_PREFILL, 64), (libmoe.MOE_PATH_PREFILL, 128),
                    (libmoe.MOE_PATH_PREFILL, 256)][int(rng.integers(0, 7))]
    w = synth.scaled(synth.WORKLOADS["tiny16"], T=T, H=H, I=I, E=E, K=K, with_shared=shared,
                     seed=50 + seed)
    return w, path, tile_m


@pytest.mark.parametrize("seed", range(12))
def test_random_shapes_every_path(seed):
    """Seeded random shapes and launch configurations, every output element
    against the oracle at the bar."""
    w, path, tile_m = _random_case(seed)
    d, ids, wt = _layer_inputs(w)
    ref = gc.bits_to_f64(oracle.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt,
                                    n_threads=THREADS))
    got = _gpu_ffn(d, ids, wt, w.Et, tile_m, path)
    gc.ffn_parity(got, ref, f"seed {seed}: T={w.T} H={w.H} I={w.I} E={w.E} K={w.K} "
                            f"shared={w.with_shared} path={path} tile_m={tile_m}")
    assert libmoe.moe_device_error() == 0


PREFILL_FULL = {  # workload -> (tile_m as the bench runs it, tokens compared: None = all)
    "mtp_verify288": (32, None),
    "prefill1536": (64, None),
    "skewed_prefill8192": (128, 256),
    "skewed_prefill8192_cal": (128, 256),
}


@pytest.mark.parametrize("name", list(PREFILL_FULL))
def test_prefill_full_size(name):
    """The prefill path at full size in the bench's launch configuration:
    every token of the 288- and 1536-token workloads; on the 8192-token
    ones 256 tokens that include the first and last row of each hot
    expert's last partial tile and of the first and last work items."""
    w = synth.WORKLOADS[name]
    tile_m, n_tok = PREFILL_FULL[name]
    d, ids, wt = _layer_inputs(w)
    tokens = _tokens_for(w, ids, tile_m, n_tok, 98)
    ref = gc.bits_to_f64(oracle.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt,
                                    tokens=tokens, n_threads=THREADS))
    dev_w = gc.upload_weights(d)
    out = libmoe.moe_layer(gc.to_dev(d["logits"]), gc.to_dev(d["x"]), dev_w["w13"], dev_w["s13"],
                           dev_w["w2"], dev_w["s2"], w.K, w.with_shared, tile_m=tile_m,
                           path=libmoe.MOE_PATH_PREFILL)
    torch.cuda.synchronize()
    assert libmoe.moe_device_error() == 0
    stats = gc.ffn_parity(gc.bf16_dev_to_f64(out)[tokens], ref, name)
    print(name, "prefill", tokens.size, "tokens", stats)
    del dev_w
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["skewed_prefill8192", "skewed_prefill8192_cal"])
def test_decode_and_prefill_paths_agree_on_every_token(name):
    """All 8192 tokens: the prefill path (128-row tiles, tcgen05) against the
    decode path (8-row tiles, warp MMA) -- two independent kernel families
    held to the parity bar against each other, so a broken tile that the
    oracle's token sample misses still shows."""
    w = synth.WORKLOADS[name]
    d, ids, wt = _layer_inputs(w)
    dev_w = gc.upload_weights(d)
    logits, x = gc.to_dev(d["logits"]), gc.to_dev(d["x"])
    outs = {}
    for path, tile_m in ((libmoe.MOE_PATH_DECODE, 8), (libmoe.MOE_PATH_PREFILL, 128)):
        outs[path] = gc.bf16_dev_to_f64(libmoe.moe_layer(
            logits, x, dev_w["w13"], dev_w["s13"], dev_w["w2"], dev_w["s2"], w.K, w.with_shared,
            tile_m=tile_m, path=path))
    torch.cuda.synchronize()
    assert libmoe.moe_device_error() == 0
    stats = gc.ffn_parity(outs[libmoe.MOE_PATH_PREFILL], outs[libmoe.MOE_PATH_DECODE],
                          f"{name} prefill vs decode")
    print(name, "prefill vs decode", stats)
    del dev_w
    torch.cuda.empty_cache()


@pytest.mark.parametrize("path,tile_m,name", [(libmoe.MOE_PATH_PREFILL, 32, "ragged37"),
                                              (libmoe.MOE_PATH_PREFILL, 64, "k_tail"),
                                              (libmoe.MOE_PATH_PREFILL, 128, "wide_k"),
                                              (libmoe.MOE_PATH_DECODE, 8, "ragged37")])
def test_down_combine_equals_down_then_combine(path, tile_m, name):
    """moe_ffn_down_combine gives the bytes of moe_ffn_down followed by
    moe_combine (y by pair) on the decode path; on the prefill path (y staged
    as scaled f16 rows by position) it agrees with them to the staging bound;
    both meet the bar."""
    w = synth.scaled(synth.WORKLOADS["tiny16"], **SMALL[name])
    d, ids, wt = _layer_inputs(w)
    dw = gc.upload_weights(d)
    perm = libmoe.moe_permute(gc.to_dev(ids), w.Et, tile_m)
    ws = libmoe.alloc_workspace(w.T, w.H, w.I, w.Et, ids.shape[1], tile_m)
    x_d, wt_d = gc.to_dev(d["x"]), gc.to_dev(wt)
    libmoe.moe_ffn_gate_up(x_d, dw["w13"], dw["s13"], perm, ws, path)
    a = torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    libmoe.moe_ffn_down(dw["w2"], dw["s2"], wt_d, perm, ws, w.T, path)
    _, y = libmoe.ffn_views(ws, w.T, w.H, w.I, w.Et, ids.shape[1], tile_m)
    libmoe.moe_combine(y, w.T, w.H, ids.shape[1], a)
    b = torch.empty_like(a)
    libmoe.moe_ffn_down_combine(dw["w2"], dw["s2"], wt_d, perm, ws, w.T, b, path)
    torch.cuda.synchronize()
    if path == libmoe.MOE_PATH_DECODE:
        np.testing.assert_array_equal(gc.bf16_dev_to_f64(b), gc.bf16_dev_to_f64(a))
    else:
        gc.staged_close(gc.bf16_dev_to_f64(a), gc.bf16_dev_to_f64(b), f"down_combine {name}")
    ref = gc.bits_to_f64(oracle.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt,
                                    n_threads=THREADS))
    gc.ffn_parity(gc.bf16_dev_to_f64(a), ref, f"down then combine {name}")
    gc.ffn_parity(gc.bf16_dev_to_f64(b), ref, f"down_combine {name}")
    assert libmoe.moe_device_error() == 0


# ------------------------------------------- shared expert of another width

def _dense_shared_case(I_s, seed=31, T=37, with_gate=True):
    w = synth.scaled(synth.WORKLOADS["tiny16"], T=T, H=512, I=128, E=16, K=4, with_shared=False,
                     seed=seed)
    d, ids, wt = _layer_inputs(w)
    ws = synth.scaled(synth.WORKLOADS["tiny16"], T=T, H=512, I=I_s, E=1, K=1, with_shared=False,
                      seed=seed + 1)
    dsh = synth.make_weights(ws)
    rng = np.random.default_rng(seed)
    sw = (1.0 / (1.0 + np.exp(-rng.standard_normal(T)))).astype(np.float32) if with_gate else None
    return w, d, ids, wt, dsh, sw


@pytest.mark.parametrize("I_s,gate", [(96, True), (192, False), (128, True)])
def test_dense_shared_expert_against_oracle(I_s, gate):
    """Routed slots (fp32, ascending) then the dense shared expert, rounded once to bf16."""
    w, d, ids, wt, dsh, sw = _dense_shared_case(I_s, with_gate=gate)
    _, f_routed = oracle.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt, want_f32=True)
    sw_col = (sw if sw is not None else np.ones(w.T, np.float32)).reshape(-1, 1)
    _, f_shared = oracle.ffn(d["x"], dsh["w13"], dsh["s13"], dsh["w2"], dsh["s2"],
                             np.zeros((w.T, 1), np.int32), sw_col, want_f32=True)
    total = (f_routed.astype(np.float32) + f_shared.astype(np.float32)).astype(np.float32)
    ref = gc.bits_to_f64(np.vectorize(oracle.f32_to_bf16, otypes=[np.uint16])(total))
    dev_w, dev_s = gc.upload_weights(d), gc.upload_weights(dsh)
    perm = libmoe.moe_permute(gc.to_dev(ids), w.Et, 8)
    out = libmoe.moe_ffn_dense_shared(gc.to_dev(d["x"]), dev_w["w13"], dev_w["s13"], dev_w["w2"],
                                      dev_w["s2"], gc.to_dev(wt), perm, dev_s["w13"], dev_s["s13"],
                                      dev_s["w2"], dev_s["s2"],
                                      shared_w=gc.to_dev(sw) if sw is not None else None)
    torch.cuda.synchronize()
    gc.ffn_parity(gc.bf16_dev_to_f64(out), ref, f"dense shared Is={I_s}")


def test_dense_shared_equal_width_equals_fused_shared_slot():
    """With Is = I and the shared expert's weights, the separate dense path gives the fused
    layer's bytes exactly (the shared term is added last in both)."""
    w, d, ids, wt, dsh, sw = _dense_shared_case(128, seed=41)
    # the fused layer: the shared expert as expert E in slot K with weight sw
    fused_w = {k: np.concatenate([d[k], dsh[k]], axis=0) for k in ("w13", "s13", "w2", "s2")}
    ids_f = np.concatenate([ids, np.full((w.T, 1), w.E, np.int32)], axis=1)
    wt_f = np.concatenate([wt, sw.reshape(-1, 1)], axis=1)
    dev_f = gc.upload_weights(fused_w)
    perm_f = libmoe.moe_permute(gc.to_dev(ids_f), w.E + 1, 8)
    fused = libmoe.moe_ffn(gc.to_dev(d["x"]), dev_f["w13"], dev_f["s13"], dev_f["w2"], dev_f["s2"],
                           gc.to_dev(wt_f), perm_f, path=libmoe.MOE_PATH_DECODE)
    dev_w, dev_s = gc.upload_weights(d), gc.upload_weights(dsh)
    perm = libmoe.moe_permute(gc.to_dev(ids), w.Et, 8)
    dense = libmoe.moe_ffn_dense_shared(gc.to_dev(d["x"]), dev_w["w13"], dev_w["s13"],
                                        dev_w["w2"], dev_w["s2"], gc.to_dev(wt), perm,
                                        dev_s["w13"], dev_s["s13"], dev_s["w2"], dev_s["s2"],
                                        shared_w=gc.to_dev(sw))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(gc.bf16_dev_to_f64(dense), gc.bf16_dev_to_f64(fused))
