"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in a copy of oracle/moe_oracle.c (a swapped
nibble order, a wrong index, a dropped rounding, a changed tie rule, ...),
builds it with the oracle's own compiler flags, and runs the oracle's pin
tests against that build (MOE_ORACLE_LIB).  Every planted mistake must make
at least one pin fail, and the unmodified copy must pass them all.  The
regression fixture under tests/golden/ is left out: it was written by the
oracle itself, so only the independent pins (closed forms, brute force,
invariants) count here."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.c")
PIN_FILES = ["tests/test_oracle_ffn.py", "tests/test_oracle_route_permute.py",
             "tests/test_oracle_mxfp4_act.py"]

# (name, text in moe_oracle.c, replacement); the text must occur exactly once
MUTANTS = [
    ("nibble_order",
     "int code = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);",
     "int code = (k % 2 == 0) ? (byte >> 4) : (byte & 0xF);"),
    ("e2m1_table_entry",
     "{0.0f,  0.5f,  1.0f,  1.5f,  2.0f,  3.0f,  4.0f,  6.0f,",
     "{0.0f,  0.5f,  1.0f,  1.5f,  2.0f,  2.5f,  4.0f,  6.0f,"),
    ("e8m0_bias",
     "return ldexpf(1.0f, s - 127);",
     "return ldexpf(1.0f, s - 126);"),
    ("scale_group_order",
     "float scale = moe_ref_e8m0(scales_row[g]);",
     "float scale = moe_ref_e8m0(scales_row[len / 32 - 1 - g]);"),
    ("gate_up_swapped",
     "h[n] = moe_ref_bf16_to_f32(moe_ref_f32_to_bf16(moe_ref_silu(g) * u));",
     "h[n] = moe_ref_bf16_to_f32(moe_ref_f32_to_bf16(moe_ref_silu(u) * g));"),
    ("h_not_rounded_to_bf16",
     "h[n] = moe_ref_bf16_to_f32(moe_ref_f32_to_bf16(moe_ref_silu(g) * u));",
     "h[n] = moe_ref_silu(g) * u;"),
    ("w2_rows_reversed",
     "ref_decode_row(w2 + (size_t)m * (I / 2), s2 + (size_t)m * (I / 32), I, wd);\n"
     "        float acc = 0.0f;\n"
     "        for (int n = 0; n < I; ++n) acc += wd[n] * h[n];",
     "ref_decode_row(w2 + (size_t)(H - 1 - m) * (I / 2), s2 + (size_t)(H - 1 - m) * (I / 32), I, wd);\n"
     "        float acc = 0.0f;\n"
     "        for (int n = 0; n < I; ++n) acc += wd[n] * h[n];"),
    ("last_slot_dropped",
     "for (int j = 0; j < Kt; ++j) {\n"
     "            int e = topk_ids[(size_t)t * Kt + j];\n"
     "            float wj = topk_w[(size_t)t * Kt + j];\n"
     "            ref_expert_forward(",
     "for (int j = 0; j < Kt - 1; ++j) {\n"
     "            int e = topk_ids[(size_t)t * Kt + j];\n"
     "            float wj = topk_w[(size_t)t * Kt + j];\n"
     "            ref_expert_forward("),
    ("ties_to_upper_index",
     "if (best < 0 || l[e] > l[best]) best = e;",
     "if (best < 0 || l[e] >= l[best]) best = e;"),
    ("not_renormalised",
     "w[k] = renormalize ? p[ids[k]] / s : p[ids[k]];",
     "w[k] = p[ids[k]];"),
    ("softmax_not_normalised",
     "for (int e = 0; e < E; ++e) p[e] = p[e] / z;",
     "for (int e = 0; e < E; ++e) p[e] = p[e] / (z + 1.0f);"),
    ("permutation_unstable",
     "for (int64_t q = 0; q < P; ++q) {\n"
     "        int e = topk_ids[q];\n"
     "        int64_t pos = offsets[e] + cursor[e];",
     "for (int64_t q = P - 1; q >= 0; --q) {\n"
     "        int e = topk_ids[q];\n"
     "        int64_t pos = offsets[e] + cursor[e];"),
    ("no_tile_padding",
     "acc += (count[e] + tile_m - 1) / tile_m * tile_m;",
     "acc += count[e];"),
    ("e2m1_ties_away_from_zero",
     "if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) != 0)) {",
     "if (d <= best_d) {"),
    ("mx_shared_exponent_off_by_one",
     "e = ex - 1 - 2;",
     "e = ex - 1 - 1;"),
    ("mx_negative_zero_dropped",
     "return best | (signbit(v) ? 8 : 0);",
     "return best | (signbit(v) && best != 0 ? 8 : 0);"),
    ("selects_smallest_logits",
     "if (best < 0 || l[e] > l[best]) best = e;",
     "if (best < 0 || l[e] < l[best]) best = e;"),
    ("shared_weight_ignored",
     "w[K] = shared_w ? shared_w[t] : 1.0f;",
     "w[K] = 1.0f;"),
    ("tile_map_off_by_one",
     "int64_t row = i * tile_m;",
     "int64_t row = i > 0 ? i * tile_m - 1 : 0;"),
    ("inverse_map_shifted",
     "inv[q] = (int32_t)pos;",
     "inv[q] = (int32_t)(pos + 1);"),
    ("padding_not_minus_one",
     "for (int64_t i = 0; i < cap; ++i) sorted_pairs[i] = -1;",
     "for (int64_t i = 0; i < cap; ++i) sorted_pairs[i] = 0;"),
    ("silu_sign",
     "float moe_ref_silu(float g) { return g / (1.0f + expf(-g)); }",
     "float moe_ref_silu(float g) { return g / (1.0f + expf(g)); }"),
    ("routing_weight_not_applied",
     "s2 + e * s2_e, H, I, h, y);\n"
     "            for (int m = 0; m < H; ++m) acc[m] += wj * y[m];",
     "s2 + e * s2_e, H, I, h, y);\n"
     "            for (int m = 0; m < H; ++m) acc[m] += y[m];"),
    ("bf16_ties_away_from_zero",
     "if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1u;",
     "if (rest >= 0x8000u) keep += 1u;"),
    ("mx_swiglu_rounded_before_quantisation",
     "a[n] = moe_ref_silu(g) * u;",
     "a[n] = moe_ref_bf16_to_f32(moe_ref_f32_to_bf16(moe_ref_silu(g) * u));"),
]


def _build(tmp_path, text):
    import oracle
    src = tmp_path / "moe_oracle.c"
    src.write_text(text)
    lib = tmp_path / "libmoe_oracle.so"
    subprocess.check_call(["gcc", *oracle.GCC_FLAGS, str(src), "-o", str(lib), "-lm"])
    return str(lib)


def _run_pins(lib):
    env = dict(os.environ, MOE_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", *PIN_FILES, "-x", "-q", "-p", "no:cacheprovider",
                        "-m", "not gpu"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:]


def test_unmodified_copy_passes_the_pins(tmp_path):
    rc, out = _run_pins(_build(tmp_path, open(SRC).read()))
    assert rc == 0, out


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(name, old, new, tmp_path):
    text = open(SRC).read()
    assert text.count(old) == 1, f"{name}: the text to change is not unique in moe_oracle.c"
    rc, out = _run_pins(_build(tmp_path, text.replace(old, new)))
    assert rc == 1 and " failed" in out, f"{name} was not caught:\n{out}"
