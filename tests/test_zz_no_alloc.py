"""moe_ffn_noalloc: the FFN for callers that cannot allocate device memory.

It runs the same kernels as moe_ffn with the workspace in the library's fixed
device array.  The GPU test calls it twice in a row through the C ABI (the
second call reuses the array the first one left behind) and compares each
result with moe_ffn on a caller-allocated workspace.  This file is collected
last so that a failure here does not hide the other tests.
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
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import oracle
    from mxfp4_mixture_experts_softmax_gb300 import libmoe, synth

    cases = [  # two different layers back to back, both within the fixed scratch
        (synth.scaled(synth.WORKLOADS["tiny16"], T=37, H=512, I=256, E=16, K=4,
                      with_shared=True, seed=31), 8),
        (synth.WORKLOADS["decode64"], 8),
    ]
    for w, tile_m in cases:
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
        gc.ffn_parity(gc.bf16_dev_to_f64(got), gc.bf16_dev_to_f64(ref), f"noalloc {w.name}")
        del dev_w
        torch.cuda.empty_cache()
