"""Writes the golden fixtures of this directory from the CPU oracle alone.

The pages print no worked example of the layer, so these fixtures are not
values from the pages: they record the oracle's results on the seeded tiny
workload (16 tokens, H=256, I=128, 8 experts, top-2) so that a later change
to the oracle's arithmetic shows up as a diff.  Run from the repository root:

    python tests/golden/make_golden.py
"""
from __future__ import annotations

import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from mxfp4_mixture_experts_softmax_gb300 import synth  # noqa: E402


def sha(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def fixture() -> dict:
    w = synth.WORKLOADS["tiny16"]
    d = synth.make_inputs(w)
    ids, wt = oracle.route(d["logits"], w.K, w.with_shared)
    perm = oracle.permute(ids, w.Et, 8)
    out = oracle.ffn(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt)
    out_mx = oracle.ffn_mxfp4act(d["x"], d["w13"], d["s13"], d["w2"], d["s2"], ids, wt)
    return {
        "workload": "tiny16 (seed 0): T=16, H=256, I=128, E=8, K=2, no shared expert",
        "writer": "tests/golden/make_golden.py (oracle only)",
        "route_ids": ids.tolist(),
        "route_weights_hex": [[float(v).hex() for v in row] for row in wt],
        "permute_tile8_sorted_pairs": perm["sorted_pairs"].tolist(),
        "permute_tile8_offsets": perm["offsets"].tolist(),
        "ffn_out_bf16_token0_first16": [int(v) for v in out[0, :16]],
        "ffn_out_bf16_sha256": sha(out),
        "ffn_mxfp4act_out_bf16_token0_first16": [int(v) for v in out_mx[0, :16]],
        "ffn_mxfp4act_out_bf16_sha256": sha(out_mx),
    }


if __name__ == "__main__":
    oracle.build()
    synth.build()
    with open(os.path.join(HERE, "oracle_tiny16.json"), "w") as f:
        json.dump(fixture(), f, indent=1)
        f.write("\n")
