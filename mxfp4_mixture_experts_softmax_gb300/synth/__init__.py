"""Seeded synthetic workloads for the MXFP4 MoE layer.

This module only draws inputs: router logits, bf16 activations and packed
MXFP4 expert weights.  It holds none of the layer's arithmetic, so both the
CUDA path and the CPU oracle can consume its bytes without sharing code.

Workload shapes follow the serving scenarios the source pages discuss:
  * Qwen3.5-397B-A17B: 512 routed MXFP4 experts, softmax top-10
    (VibeSys Qwen3.5-397B on 4x MI300A, section "Goal"; InferenceX MI355X
    Qwen3.5 blog, section "optimisations", PR #21421 fused_topk at E=512/K=10),
  * the shared expert folded in as routed expert K+1
    (InferenceX MI355X Qwen3.5 blog, PR #20736),
  * MTP verification with 2 draft tokens, 1,536-token prefill chunks
    (VibeSys Qwen3.5-397B, section "prefill, caching and speculation").
Hidden 4096 / intermediate 1024 and the value distributions are the plain
synthetic stand-ins for the model's layer (no trained weights are used).

Random streams (SplitMix64, counter based, see synth.c):
  0 router logits, 1 activations, 2 W13 codes, 3 W13 scales,
  4 W2 codes, 5 W2 scales.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

STREAM_LOGITS, STREAM_X, STREAM_W13, STREAM_S13, STREAM_W2, STREAM_S2 = range(6)


def build(force: bool = False) -> str:
    """Compile synth.c into libsynth.so next to it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            u64, i64, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
            lib.synth_u64.argtypes = [u64, u64, i64, vp]
            lib.synth_bytes.argtypes = [u64, u64, i64, vp]
            lib.synth_int_bytes.argtypes = [u64, u64, i64, ctypes.c_int, ctypes.c_int, vp]
            lib.synth_normal_f32.argtypes = [u64, u64, i64, vp]
            lib.synth_normal_bf16.argtypes = [u64, u64, i64, vp]
            for f in (lib.synth_u64, lib.synth_bytes, lib.synth_int_bytes,
                      lib.synth_normal_f32, lib.synth_normal_bf16):
                f.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def u64(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, np.uint64)
    _load().synth_u64(seed, stream, n, _ptr(out))
    return out


def uniform_bytes(seed: int, stream: int, shape) -> np.ndarray:
    out = np.empty(shape, np.uint8)
    _load().synth_bytes(seed, stream, out.size, _ptr(out))
    return out


def int_bytes(seed: int, stream: int, shape, lo: int, hi: int) -> np.ndarray:
    out = np.empty(shape, np.uint8)
    _load().synth_int_bytes(seed, stream, out.size, lo, hi, _ptr(out))
    return out


def normal_f32(seed: int, stream: int, shape) -> np.ndarray:
    out = np.empty(shape, np.float32)
    _load().synth_normal_f32(seed, stream, out.size, _ptr(out))
    return out


def normal_bf16(seed: int, stream: int, shape) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0,1) draws rounded to nearest even."""
    out = np.empty(shape, np.uint16)
    _load().synth_normal_bf16(seed, stream, out.size, _ptr(out))
    return out


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int                 # tokens
    H: int                 # hidden size (K of gate_up, N of down)
    I: int                 # expert intermediate size
    E: int                 # routed experts
    K: int                 # routed experts per token
    with_shared: bool      # shared expert folded in as expert E, slot K
    seed: int
    scale_exp_lo: int      # E8M0 scales uniform over 2^lo .. 2^hi
    scale_exp_hi: int
    zipf_alpha: float = 0.0  # logits += alpha * ln(rank^-1.1), rank = e + 1
    renormalize: bool = True

    @property
    def Et(self) -> int:
        return self.E + (1 if self.with_shared else 0)

    @property
    def Kt(self) -> int:
        return self.K + (1 if self.with_shared else 0)

    @property
    def pairs(self) -> int:
        return self.T * self.Kt

    def describe(self) -> dict:
        d = dataclasses.asdict(self)
        d["Et"], d["Kt"] = self.Et, self.Kt
        return d


_Q = dict(H=4096, I=1024, E=512, K=10, with_shared=True, scale_exp_lo=-8, scale_exp_hi=-4)

# Calibrated Zipf coefficient for the skewed prefill: with alpha = 0.22 the
# hottest expert receives about 10x the mean routed load on seed 4 (checked by
# the oracle tests).  The literal coefficient 2 concentrates almost all load on
# a handful of experts; both are kept.
ZIPF_ALPHA_CALIBRATED = 0.22

WORKLOADS = {
    "tiny16": Workload("tiny16", T=16, H=256, I=128, E=8, K=2, with_shared=False, seed=0,
                       scale_exp_lo=-6, scale_exp_hi=-2),
    "decode64": Workload("decode64", T=64, seed=1, **_Q),
    "mtp_verify288": Workload("mtp_verify288", T=288, seed=2, **_Q),
    "prefill1536": Workload("prefill1536", T=1536, seed=3, **_Q),
    "skewed_prefill8192": Workload("skewed_prefill8192", T=8192, seed=4, zipf_alpha=2.0, **_Q),
    "skewed_prefill8192_cal": Workload("skewed_prefill8192_cal", T=8192, seed=4,
                                       zipf_alpha=ZIPF_ALPHA_CALIBRATED, **_Q),
}


def scaled(w: Workload, **kw) -> Workload:
    """Same distributions at other sizes (for small parity cases)."""
    return dataclasses.replace(w, **kw)


def make_logits(w: Workload) -> np.ndarray:
    logits = normal_f32(w.seed, STREAM_LOGITS, (w.T, w.E))
    if w.zipf_alpha != 0.0:
        rank = np.arange(1, w.E + 1, dtype=np.float64)
        bias = (w.zipf_alpha * (-1.1) * np.log(rank)).astype(np.float32)
        logits = (logits + bias[None, :]).astype(np.float32)
    return logits


def make_x(w: Workload) -> np.ndarray:
    return normal_bf16(w.seed, STREAM_X, (w.T, w.H))


def make_weights(w: Workload) -> dict:
    """Packed MXFP4 expert weights, all Et experts (the shared one is index E).

    W13 [Et, 2I, H/2] codes + [Et, 2I, H/32] E8M0 scales (gate rows, then up rows);
    W2  [Et, H, I/2]  codes + [Et, H, I/32]  scales.  Two E2M1 codes per byte.
    """
    lo, hi = 127 + w.scale_exp_lo, 127 + w.scale_exp_hi
    return dict(
        w13=uniform_bytes(w.seed, STREAM_W13, (w.Et, 2 * w.I, w.H // 2)),
        s13=int_bytes(w.seed, STREAM_S13, (w.Et, 2 * w.I, w.H // 32), lo, hi),
        w2=uniform_bytes(w.seed, STREAM_W2, (w.Et, w.H, w.I // 2)),
        s2=int_bytes(w.seed, STREAM_S2, (w.Et, w.H, w.I // 32), lo, hi),
    )


def make_inputs(w: Workload) -> dict:
    d = dict(logits=make_logits(w), x=make_x(w))
    d.update(make_weights(w))
    return d


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    return (a.astype(np.uint32) << 16).view(np.float32)


def weight_bytes_per_expert(w: Workload) -> int:
    return 2 * w.I * (w.H // 2 + w.H // 32) + w.H * (w.I // 2 + w.I // 32)


def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


__all__ = ["Workload", "WORKLOADS", "make_inputs", "make_logits", "make_x", "make_weights",
           "scaled", "bf16_bits_to_f32", "weight_bytes_per_expert", "build"]
