"""Failure paths on the GPU, driven without faulting or hanging it.

* A bounded mbarrier wait that runs out (a barrier nothing arrives at, limit
  2 ms) raises the device error flag, the kernel returns and the context stays
  usable: the next layer call matches the oracle.
* Inputs that moe_permute would never produce -- a tile whose expert is out
  of range, a pair index past T*Kt, a tile count above the buffers -- are
  caught by the kernels' own index checks (they skip that work instead of
  reading or writing out of bounds) and reported as error bit 2.
"""
import numpy as np
import pytest

import gpu_common as gc

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from mxfp4_mixture_experts_softmax_gb300 import libmoe  # noqa: E402
from mxfp4_mixture_experts_softmax_gb300 import synth  # noqa: E402

import oracle  # noqa: E402

CASE = dict(T=37, H=512, I=256, E=16, K=4, with_shared=True, seed=11)


def _case():
    w = synth.scaled(synth.WORKLOADS["tiny16"], **CASE)
    d = synth.make_inputs(w)
    ids, wt = oracle.route(d["logits"], w.K, w.with_shared)
    ref = gc.bits_to_f64(oracle.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt))
    return w, d, ids, wt, ref


def _run(w, d, ids, wt, tile_m, path, corrupt=None):
    dev_w = gc.upload_weights(d)
    perm = libmoe.moe_permute(gc.to_dev(ids), w.Et, tile_m)
    if corrupt is not None:
        corrupt(perm)
    out = libmoe.moe_ffn(gc.to_dev(d["x"]), dev_w["w13"], dev_w["s13"], dev_w["w2"], dev_w["s2"],
                         gc.to_dev(wt), perm, path=path)
    torch.cuda.synchronize()
    return gc.bf16_dev_to_f64(out)


def test_wait_timeout_raises_flag_and_context_survives():
    assert libmoe.moe_device_error(clear=True) in (0, 1, 2, 3)  # start clean
    assert libmoe.moe_device_error(clear=False) == 0
    libmoe.moe_selftest_wait_timeout(2000)
    torch.cuda.synchronize()
    assert libmoe.moe_device_error(clear=True) == 1
    assert libmoe.moe_device_error(clear=False) == 0
    w, d, ids, wt, ref = _case()
    gc.ffn_parity(_run(w, d, ids, wt, 8, libmoe.MOE_PATH_DECODE), ref, "after the timeout")
    assert libmoe.moe_device_error(clear=True) == 0


def test_split_wait_outcomes_stop_both_warps():
    """One warp's wait runs out while the other's completes: both act on the
    failed outcome (neither is left at the named barrier that follows), the
    kernel returns, the flag is raised and the context stays usable."""
    assert libmoe.moe_device_error(clear=True) in (0, 1, 2, 3)
    outcome = libmoe.moe_selftest_wait_split(2000)
    torch.cuda.synchronize()
    assert outcome.cpu().tolist() == [0, 0]
    assert libmoe.moe_device_error(clear=True) == 1
    w, d, ids, wt, ref = _case()
    gc.ffn_parity(_run(w, d, ids, wt, 32, libmoe.MOE_PATH_PREFILL), ref, "after the split wait")
    assert libmoe.moe_device_error(clear=True) == 0


def test_selftest_rejects_bad_limits():
    for bad in (0, -5, 2_000_000):
        with pytest.raises(libmoe.MoeError):
            libmoe.moe_selftest_wait_timeout(bad)
        with pytest.raises(libmoe.MoeError):
            libmoe.moe_selftest_wait_split(bad)


def _bad_expert(perm):
    perm["tile_expert"][0] = 10_000


def _bad_pair(perm):
    perm["sorted_pairs"][1] = 1 << 30


def _bad_tile_count(perm):
    perm["num_tiles"][0] = perm["tile_expert"].numel() + 5


@pytest.mark.parametrize("corrupt", [_bad_expert, _bad_pair, _bad_tile_count])
@pytest.mark.parametrize("path,tile_m", [(libmoe.MOE_PATH_DECODE, 8), (libmoe.MOE_PATH_PREFILL, 32)])
def test_out_of_range_indices_are_flagged_not_followed(corrupt, path, tile_m):
    w, d, ids, wt, ref = _case()
    assert libmoe.moe_device_error(clear=True) in (0, 1, 2, 3)
    _run(w, d, ids, wt, tile_m, path, corrupt)  # outputs of the skipped work are unspecified
    assert libmoe.moe_device_error(clear=True) & 2
    # the context and the library are intact: a valid call matches the oracle
    gc.ffn_parity(_run(w, d, ids, wt, tile_m, path), ref, "after the index error")
    assert libmoe.moe_device_error(clear=True) == 0


@pytest.mark.parametrize("corrupt", [_bad_expert, _bad_pair, _bad_tile_count])
@pytest.mark.parametrize("tile_m", [32, 128])
def test_fp8x2_out_of_range_indices_are_flagged_not_followed(corrupt, tile_m):
    """The two-term path (one CTA per weight block at 32-row tiles, CTA pairs at 128): the
    split, both GEMMs and the position weights skip out-of-range work and flag it."""
    w = synth.scaled(synth.WORKLOADS["tiny16"], **dict(CASE, I=512))
    d = synth.make_inputs(w)
    ids, wt = oracle.route(d["logits"], w.K, w.with_shared)
    ref = gc.bits_to_f64(oracle.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt))
    P = libmoe.MOE_PATH_PREFILL_FP8X2
    assert libmoe.moe_device_error(clear=True) in (0, 1, 2, 3)
    _run(w, d, ids, wt, tile_m, P, corrupt)  # outputs of the skipped work are unspecified
    assert libmoe.moe_device_error(clear=True) & 2
    gc.ffn_parity(_run(w, d, ids, wt, tile_m, P), ref, "after the index error")
    assert libmoe.moe_device_error(clear=True) == 0


@pytest.mark.parametrize("corrupt", [_bad_expert, _bad_pair, _bad_tile_count])
@pytest.mark.parametrize("tile_m", [32, 64])
def test_mxfp4act_out_of_range_indices_are_flagged_not_followed(corrupt, tile_m):
    """The MXFP4-activation path (gather, both GEMMs with their scale warps,
    the position weights, the blocked combine) under the same corruptions: the
    index checks flag them, nothing faults, and the next valid call gives the
    bytes of the valid call before it."""
    w, d, ids, wt, _ = _case()
    dev_w = gc.upload_weights(d)
    x_d, wt_d = gc.to_dev(d["x"]), gc.to_dev(wt)

    def run(corrupt_fn=None):
        perm = libmoe.moe_permute(gc.to_dev(ids), w.Et, tile_m)
        if corrupt_fn is not None:
            corrupt_fn(perm)
        out = libmoe.moe_ffn_mxfp4act(x_d, dev_w["w13"], dev_w["s13"], dev_w["w2"], dev_w["s2"],
                                      wt_d, perm)
        torch.cuda.synchronize()
        return gc.bf16_dev_to_f64(out)

    assert libmoe.moe_device_error(clear=True) in (0, 1, 2, 3)
    before = run()
    assert libmoe.moe_device_error(clear=True) == 0
    run(corrupt)  # outputs of the skipped work are unspecified
    assert libmoe.moe_device_error(clear=True) & 2
    np.testing.assert_array_equal(run(), before)
    assert libmoe.moe_device_error(clear=True) == 0
