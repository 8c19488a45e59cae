"""moe_ffn_noalloc: the FFN for callers that cannot allocate device memory.

It runs the same kernels as moe_ffn with the workspace in the library's fixed
device array.  The GPU test calls it twice in a row through the C ABI (the
second call reuses the array the first one left behind) and compares each
result with moe_ffn on a caller-allocated workspace (identical bytes) and
with the oracle.  This file is collected last so that a failure here does not
hide the other tests.
"""
import ctypes

import numpy as np
import pytest

import gpu_common as gc


def test_noalloc_rejects_sizes_beyond_the_scratch():
    from mxfp4_mixture_experts_softmax_gb300 import libmoe as m
    lib = m.load()
    fake, nul = ctypes.c_void_p(0x1000), ctypes.c_void_p(0)
    # 8192 tokens x 11 slots of a 4096/1024 layer need ~1.6 GB of scratch
    rc = lib.moe_ffn_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                             8192, 4096, 1024, 513, 11, 8, fake, nul)
    assert rc == m.MOE_ERR_UNSUPPORTED_SHAPE
    assert m.moe_ffn_workspace_size(8192, 4096, 1024, 513, 11, 8) > m.MOE_NOALLOC_SCRATCH_BYTES
    assert m.moe_ffn_workspace_size(64, 4096, 1024, 513, 11, 8) <= m.MOE_NOALLOC_SCRATCH_BYTES


@pytest.mark.gpu
def test_noalloc_matches_moe_ffn_on_two_calls_in_a_row():
    """Three layers back to back, within the fixed scratch: two on the decode
    path (8-row tiles) and one on the prefill path (64-row tiles, ~59 rows
    per expert, so the gathered rows, the row factors and the blocked y
    regions of the scratch are used).  The same kernels run on the same
    inputs, so each result must have moe_ffn's bytes exactly, and it must
    meet the parity bar against the oracle."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import oracle
    from mxfp4_mixture_experts_softmax_gb300 import libmoe, synth

    cases = [
        (synth.scaled(synth.WORKLOADS["tiny16"], T=37, H=512, I=256, E=16, K=4,
                      with_shared=True, seed=31), 8, libmoe.MOE_PATH_DECODE),
        (synth.scaled(synth.WORKLOADS["tiny16"], T=200, H=512, I=256, E=16, K=4,
                      with_shared=True, seed=33), 64, libmoe.MOE_PATH_PREFILL),
        (synth.scaled(synth.WORKLOADS["tiny16"], T=200, H=512, I=512, E=16, K=4,
                      with_shared=True, seed=35), 64, libmoe.MOE_PATH_PREFILL_FP8X2),
        (synth.WORKLOADS["decode64"], 8, libmoe.MOE_PATH_DECODE),
    ]
    for w, tile_m, want_path in cases:
        assert libmoe.moe_ffn_auto_path_shape(w.T, w.H, w.I, w.Et, w.Kt, tile_m) == want_path
        d = synth.make_inputs(w)
        ids, wt = oracle.route(d["logits"], w.K, w.with_shared)
        dev_w = gc.upload_weights(d)
        x, wt_d = gc.to_dev(d["x"]), gc.to_dev(wt)
        perm = libmoe.moe_permute(gc.to_dev(ids), w.Et, tile_m)
        assert libmoe.moe_ffn_workspace_size(w.T, w.H, w.I, w.Et, w.Kt, tile_m) \
            <= libmoe.MOE_NOALLOC_SCRATCH_BYTES
        ref = libmoe.moe_ffn(x, dev_w["w13"], dev_w["s13"], dev_w["w2"], dev_w["s2"], wt_d, perm)
        got = libmoe.moe_ffn_noalloc(x, dev_w["w13"], dev_w["s13"], dev_w["w2"], dev_w["s2"],
                                     wt_d, perm)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), f"noalloc {w.name}"
        tokens = np.arange(min(w.T, 48), dtype=np.int32)
        want = gc.bits_to_f64(oracle.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt,
                                         tokens=tokens))
        gc.ffn_parity(gc.bf16_dev_to_f64(got)[tokens], want, f"noalloc {w.name} vs oracle")
        assert libmoe.moe_device_error() == 0
        del dev_w
        torch.cuda.empty_cache()
