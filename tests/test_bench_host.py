"""bench.py's host-side arithmetic on CPU: algorithmic work per step, the
launch count it claims, the roofline entry and the ncu-summary lookup.

The work figures are checked against the closed forms of the layer: per
routed pair 2 * (2I * H + H * I) flops, and per touched expert the packed
MXFP4 bytes of W13 and W2 (codes + one E8M0 byte per 32 elements)."""
import os
import re

import numpy as np
import pytest

import bench
from mxfp4_mixture_experts_softmax_gb300 import libmoe, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _ids(w, oracle_mod):
    ids, _ = oracle_mod.route(synth.make_logits(w), w.K, w.with_shared, w.renormalize)
    return ids


def test_weight_bytes_per_expert_closed_form():
    w = synth.WORKLOADS["decode64"]
    # W13: 2048 rows x (2048 code bytes + 128 scale bytes); W2: 4096 rows x (512 + 32)
    assert synth.weight_bytes_per_expert(w) == 2048 * 2176 + 4096 * 544 == 6_684_672


@pytest.mark.parametrize("name", ["tiny16", "decode64"])
def test_layer_work_matches_the_closed_forms(name, synth_mod, oracle_mod):
    w = synth.WORKLOADS[name]
    ids = _ids(w, oracle_mod)
    work = bench.layer_work(w, ids)
    H, I, T, P = w.H, w.I, w.T, w.pairs
    touched = len(set(ids.ravel().tolist()))
    assert work["touched"] == touched
    if name == "decode64":
        assert work["flops"] == P * 25_165_824
    assert work["flops"] == 2 * P * 3 * I * H
    assert work["gate_up_flops"] == 2 * P * 2 * I * H
    w13 = 2 * I * (H // 2 + H // 32)
    w2 = H * (I // 2 + I // 32)
    assert work["gate_up_bytes"] == touched * w13 + 2 * T * H + 2 * P * I
    # algorithmic only: no per-pair fp32 outputs written and read back
    assert work["down_bytes"] == touched * w2 + 2 * P * I + 2 * T * H
    assert work["layer_bytes"] == touched * (w13 + w2) + 4 * T * H + 4 * P * I + 4 * T * w.E


def test_layer_work_mxfp4_moves_encoded_rows(synth_mod, oracle_mod):
    w = synth.WORKLOADS["decode64"]
    ids = _ids(w, oracle_mod)
    bf = bench.layer_work(w, ids, act="bf16")
    mx = bench.layer_work(w, ids, act="mxfp4")
    assert mx["flops"] == bf["flops"] and mx["touched"] == bf["touched"]
    # h crosses HBM as 0.53 bytes per value instead of 2 (written once, read once)
    hq = w.I // 2 + w.I // 32
    assert bf["layer_bytes"] - mx["layer_bytes"] == 4 * w.pairs * w.I - 2 * w.pairs * hq


def test_per_config_covers_every_full_size_workload():
    full = [n for n, w in synth.WORKLOADS.items() if w.H == 4096]
    assert sorted(bench.PER_CONFIG) == sorted(full)
    assert bench.DEFAULT_WORKLOAD in bench.PER_CONFIG
    for n in bench.PER_CONFIG:  # the bf16 tile height gives the path the pages' regime names
        w = synth.WORKLOADS[n]
        tm = bench.default_tile_m(w, "bf16")
        regime = libmoe.moe_ffn_auto_path(w.T, w.Kt, w.Et, tm)
        assert regime == (libmoe.MOE_PATH_DECODE if w.T <= 288 else libmoe.MOE_PATH_PREFILL), n
        # the large-M regime runs the two-term path at these widths (H, I multiples of 512)
        path = libmoe.moe_ffn_auto_path_shape(w.T, w.H, w.I, w.Et, w.Kt, tm)
        assert path == (libmoe.MOE_PATH_DECODE if w.T <= 288 else libmoe.MOE_PATH_PREFILL_FP8X2), n


def test_launch_counts_per_path():
    W = synth.WORKLOADS
    # fused route + permute (one launch) up to the header's token limit
    assert bench.launches_per_step(W["tiny16"], "decode") == 1 + 5
    # decode64: route, single-block permute, x -> f16, gate_up, h -> f16, down, combine
    assert bench.launches_per_step(W["decode64"], "decode") == 7
    assert bench.launches_per_step(W["decode64"], "mxfp4act") == 8
    # 16,896 and 90,112 pairs: the four-launch multi-block sort
    assert bench.launches_per_step(W["prefill1536"], "prefill") == 11
    assert bench.launches_per_step(W["skewed_prefill8192"], "prefill") == 11
    # split of x into tile order, gate_up | position weights, down, combine
    assert bench.launches_per_step(W["skewed_prefill8192"], "prefill_fp8x2") == 10
    assert bench.launches_per_step(W["skewed_prefill8192"], "mxfp4act") == 11


def test_fused_token_limit_matches_the_header():
    txt = open(os.path.join(ROOT, "include", "moe.h")).read()
    m = re.search(r"#define\s+MOE_ROUTE_PERMUTE_FUSED_MAX_T\s+(\d+)", txt)
    assert m and int(m.group(1)) == libmoe.MOE_ROUTE_PERMUTE_FUSED_MAX_T


def test_roofline_entry_picks_the_binding_bound(monkeypatch):
    monkeypatch.setattr(bench, "measured_peaks", lambda: None)
    # 1 GB and 1 GFLOP in 0.5 ms: HBM-bound (0.147 ms at 6.8 TB/s vs 0.5 us at 1.9 PF)
    e = bench.roofline_entry("k", 1e9, 1e9, 0.5e-3, None, None)
    assert e["bound"] == "hbm" and e["unit"] == "GB/s"
    assert e["achieved"] == pytest.approx(2000.0)
    assert e["frac"] == pytest.approx(2000.0 / bench.FALLBACK_HBM_GBS)
    assert e["peak_source"].startswith("fallback")
    # 1 MB and 1 TFLOP in 1 ms: tensor-bound
    e = bench.roofline_entry("k", 1e6, 1e12, 1e-3, None, None)
    assert e["bound"] == "tensor" and e["unit"] == "TFLOP/s"
    assert e["frac"] == pytest.approx(1000.0 / bench.FALLBACK_BF16_TFLOPS)
    # MXFP4 operands: the peak is the bf16 peak times the nominal FP4/BF16 ratio
    e = bench.roofline_entry("k", 1e6, 1e12, 1e-3, None, None, fp4=True)
    assert e["peak"] == pytest.approx(bench.FALLBACK_BF16_TFLOPS * 6.0)
    assert e["peak_source"].startswith("derived")


def test_measured_peaks_take_precedence(monkeypatch):
    monkeypatch.setattr(bench, "measured_peaks",
                        lambda: {"gb300": {"hbm_gbs": 7000.0, "bf16_tflops": 2000.0}})
    assert bench.hbm_peak() == (7000.0, "measured (MEASURED_PEAKS.json hbm_gbs)")
    assert bench.tensor_peak()[0] == 2000.0


def test_traffic_lookup_is_keyed_to_the_kernel_source(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("// kernel v1\n")
    import hashlib
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "k.md").write_text(
        f"traffic_bytes_per_launch kernel=decode_gate_up workload=decode64 src_sha256={sha} bytes=1234\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_from_profiles("decode_gate_up", "decode64", str(src)) == (
        1234, os.path.join("profiles", "k.md"))
    assert bench.traffic_from_profiles("decode_gate_up", "prefill1536", str(src)) == (None, None)
    src.write_text("// kernel v2\n")  # the kernel changed since the counters were taken
    assert bench.traffic_from_profiles("decode_gate_up", "decode64", str(src)) == (None, None)


def test_weak_scaling_value_counts_all_ranks():
    # 64 tokens per rank-step, 30 steps, 4 ranks, slowest rank 15 ms
    assert bench.weak_scaling_value(64, 30, 4, 15.0) == pytest.approx(64 * 30 * 4 / 0.015)


def test_reference_arm_prints_the_contract_line():
    """--impl reference times the CPU oracle and prints one JSON line with the
    same metric, unit and workload keys as the GPU arm."""
    import json
    import subprocess
    import sys
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny16",
                        "--steps", "2", "--warmup", "1"], cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["higher_is_better"] is True and d["steps"] == 2 and d["warmup"] == 1
    assert d["value"] > 0 and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"] == bench.workload_config(synth.WORKLOADS["tiny16"], "bf16", 1)
