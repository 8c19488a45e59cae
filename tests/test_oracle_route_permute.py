"""Pins for the oracle's routing and permutation (CPU only).

Routing: softmax-scored top-K selection (InferenceX MI355X Qwen3.5 blog,
optimisations section, PR #21421 fused_topk at E=512, K=10) with the shared
expert appended as slot K (same blog, PR #20736).  Permutation: tokens grouped
by expert in tile-aligned buckets (VibeSys Qwen3.5-397B on 4x MI300A, section
"cheaper prefill and collectives", 32-row MoE tiles).
"""
import numpy as np
import pytest

import bruteforce as bf


def _rng(seed):
    return np.random.default_rng(seed)


@pytest.mark.parametrize("T,E,K,shared", [(7, 8, 2, False), (5, 64, 10, True), (3, 512, 10, True),
                                          (2, 33, 33, False), (1, 1, 1, True)])
def test_route_matches_full_sort_bruteforce(oracle_mod, T, E, K, shared):
    logits = _rng(T * E + K).standard_normal((T, E)).astype(np.float32)
    ids, w = oracle_mod.route(logits, K, shared)
    ids_b, w_b = bf.route(logits, K, shared)
    np.testing.assert_array_equal(ids, ids_b)
    np.testing.assert_allclose(w, w_b, rtol=2e-6, atol=2e-7)


def test_route_ties_pick_lower_index(oracle_mod):
    # values on a coarse grid so that many logits are exactly equal
    logits = np.round(_rng(1).standard_normal((32, 64)) * 2) / 2
    logits = logits.astype(np.float32)
    ids, _ = oracle_mod.route(logits, 10, False)
    ids_b, _ = bf.route(logits, 10, False)
    np.testing.assert_array_equal(ids, ids_b)
    # explicit: all equal -> 0..K-1
    ids, w = oracle_mod.route(np.zeros((2, 16), np.float32), 4, False)
    np.testing.assert_array_equal(ids, [[0, 1, 2, 3]] * 2)
    np.testing.assert_allclose(w, 0.25, rtol=0, atol=1e-7)


def test_route_signed_zero_is_a_tie(oracle_mod):
    logits = np.array([[-0.0, 0.0, -1.0, 0.0]], np.float32)
    ids, _ = oracle_mod.route(logits, 2, False)
    np.testing.assert_array_equal(ids, [[0, 1]])


def test_route_neg_inf(oracle_mod):
    logits = np.full((1, 8), -np.inf, np.float32)
    logits[0, 5] = 1.0
    logits[0, 2] = 0.5
    ids, w = oracle_mod.route(logits, 4, True)
    # two finite values first, then -inf ties by lower index, shared last
    np.testing.assert_array_equal(ids, [[5, 2, 0, 1, 8]])
    assert w[0, 2] == 0.0 and w[0, 3] == 0.0 and w[0, 4] == 1.0
    np.testing.assert_allclose(w[0, :2].sum(), 1.0, atol=1e-7)


def test_route_full_k_is_softmax(oracle_mod):
    logits = _rng(3).standard_normal((4, 16)).astype(np.float32)
    ids, w = oracle_mod.route(logits, 16, False)
    p = np.exp(logits.astype(np.float64))
    p /= p.sum(1, keepdims=True)
    for t in range(4):
        np.testing.assert_allclose(w[t], p[t, ids[t]], rtol=2e-6)
        assert (np.diff(logits[t, ids[t]]) <= 0).all()


def test_route_invariants_and_no_renorm(oracle_mod):
    logits = _rng(4).standard_normal((64, 512)).astype(np.float32)
    ids, w = oracle_mod.route(logits, 10, True)
    assert (ids[:, 10] == 512).all() and (w[:, 10] == 1.0).all()
    for t in range(64):
        assert len(set(ids[t, :10].tolist())) == 10
        assert (np.diff(logits[t, ids[t, :10]]) <= 0).all()
    np.testing.assert_allclose(w[:, :10].sum(1), 1.0, atol=1e-6)
    ids2, w2 = oracle_mod.route(logits, 10, True, renormalize=False)
    np.testing.assert_array_equal(ids, ids2)
    ids_b, w_b = bf.route(logits, 10, True, renormalize=False)
    np.testing.assert_allclose(w2, w_b, rtol=2e-6, atol=1e-9)


def test_route_rejects_nan(oracle_mod):
    logits = np.zeros((2, 8), np.float32)
    logits[1, 3] = np.nan
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.route(logits, 2, False)


@pytest.mark.parametrize("T,Kt,Et,tile_m", [(16, 2, 8, 32), (64, 11, 513, 32), (5, 3, 4, 1),
                                            (40, 4, 7, 8), (0, 3, 5, 16), (9, 11, 513, 128)])
def test_permute_matches_bruteforce(oracle_mod, T, Kt, Et, tile_m):
    rng = _rng(T + Et)
    ids = np.stack([rng.permutation(Et)[:Kt] for _ in range(T)]) if T else np.zeros((0, Kt), int)
    ids = ids.astype(np.int32)
    got = oracle_mod.permute(ids, Et, tile_m)
    exp = bf.permute(ids, Et, tile_m)
    for k in ("sorted_pairs", "offsets", "inv", "tile_expert"):
        np.testing.assert_array_equal(got[k], exp[k], err_msg=k)
    assert got["num_tiles"] == exp["num_tiles"]


def test_permute_invariants_skewed(oracle_mod):
    rng = _rng(9)
    T, Kt, Et, tile_m = 300, 5, 20, 16
    # heavy skew: most pairs go to expert 3
    ids = np.where(rng.random((T, Kt)) < 0.7, 3, rng.integers(0, Et, (T, Kt))).astype(np.int32)
    got = oracle_mod.permute(ids, Et, tile_m)
    sp, off, inv = got["sorted_pairs"], got["offsets"], got["inv"]
    flat = ids.reshape(-1)
    valid = sp >= 0
    # bijection between pairs and non-pad slots
    assert np.array_equal(np.sort(sp[valid]), np.arange(flat.size))
    np.testing.assert_array_equal(sp[inv], np.arange(flat.size))
    # every bucket aligned to tile_m, holds its own expert's pairs in increasing order
    assert (off % tile_m == 0).all()
    for e in range(Et):
        seg = sp[off[e]:off[e + 1]]
        real = seg[seg >= 0]
        assert (flat[real] == e).all()
        assert (np.diff(real) > 0).all()
        assert (seg[real.size:] == -1).all()  # pads at the end of the bucket
    nt = got["num_tiles"]
    for i in range(nt):
        e = got["tile_expert"][i]
        assert off[e] <= i * tile_m < off[e + 1]
    assert (got["tile_expert"][nt:] == -1).all()


def test_permute_rejects_bad_ids(oracle_mod):
    ids = np.array([[0, 9]], np.int32)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.permute(ids, 8, 4)


def test_route_shared_weight_per_token(oracle_mod):
    """A caller-supplied shared-slot weight (e.g. a sigmoid gate per token) lands in slot K
    unchanged and leaves the routed slots as they are with the default weight 1."""
    rng = np.random.default_rng(17)
    T, E, K = 23, 64, 6
    logits = rng.standard_normal((T, E)).astype(np.float32)
    gate = rng.standard_normal(T).astype(np.float32)
    sw = (1.0 / (1.0 + np.exp(-gate.astype(np.float64)))).astype(np.float32)
    ids0, w0 = oracle_mod.route(logits, K, True)
    ids1, w1 = oracle_mod.route(logits, K, True, shared_w=sw)
    np.testing.assert_array_equal(ids1, ids0)
    np.testing.assert_array_equal(w1[:, :K], w0[:, :K])
    assert (w0[:, K] == 1.0).all()
    np.testing.assert_array_equal(w1[:, K], sw)
    np.testing.assert_array_equal(ids1[:, K], np.full(T, E))
    with pytest.raises(ValueError):
        oracle_mod.route(logits, K, True, shared_w=sw[:-1])
