"""CPU oracle for the MXFP4 MoE layer (test infrastructure only).

Only the tests, the smoke check and the bench's CPU-baseline leg may import
this package.  The product path (the CUDA library and its binding) never does.

The arithmetic lives in moe_oracle.c (plain C, fp32, per-token loop); this
module compiles it with gcc (-ffp-contract=off, so no fused multiply-add
changes the rounding between x86 and Arm hosts) and wraps it with ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")
# A prebuilt oracle library to load instead of building this one: the
# mutation test points it at copies of moe_oracle.c with planted mistakes to
# show that the pins catch them.
_LIB_OVERRIDE = os.environ.get("MOE_ORACLE_LIB")
_lock = threading.Lock()
_lib = None

GCC_FLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-fopenmp"]


def build(force: bool = False) -> str:
    if _LIB_OVERRIDE:
        return _LIB_OVERRIDE
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *GCC_FLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, ci = ctypes.c_void_p, ctypes.c_int
            lib.moe_ref_route.argtypes = [vp, vp, ci, ci, ci, ci, ci, vp, vp]
            lib.moe_ref_route.restype = ci
            lib.moe_ref_permute.argtypes = [vp, ci, ci, ci, ci, vp, vp, vp, vp, vp]
            lib.moe_ref_permute.restype = ci
            lib.moe_ref_capacity.argtypes = [ci, ci, ci, ci]
            lib.moe_ref_capacity.restype = ctypes.c_int64
            lib.moe_ref_ffn.argtypes = [vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, vp, ci,
                                        vp, vp, ci]
            lib.moe_ref_ffn.restype = ci
            lib.moe_ref_ffn_grouped.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci,
                                                ci, vp]
            lib.moe_ref_ffn_grouped.restype = ci
            lib.moe_ref_mxfp4_value.argtypes = [ci, ci]
            lib.moe_ref_mxfp4_value.restype = ctypes.c_double
            lib.moe_ref_silu.argtypes = [ctypes.c_float]
            lib.moe_ref_silu.restype = ctypes.c_float
            lib.moe_ref_f32_to_bf16.argtypes = [ctypes.c_float]
            lib.moe_ref_f32_to_bf16.restype = ctypes.c_uint16
            lib.moe_ref_e2m1_round.argtypes = [ctypes.c_double]
            lib.moe_ref_e2m1_round.restype = ci
            lib.moe_ref_quantize_mxfp4.argtypes = [vp, ci, vp, vp]
            lib.moe_ref_quantize_mxfp4.restype = ci
            lib.moe_ref_ffn_mxfp4act.argtypes = [vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci,
                                                 vp, ci, vp, vp, vp, vp, vp, ci]
            lib.moe_ref_ffn_mxfp4act.restype = ci
            lib.moe_ref_max_threads.argtypes = []
            lib.moe_ref_max_threads.restype = ci
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "oracle wants C-contiguous numpy"
    return a.ctypes.data


def _check(rc, what):
    if rc != 0:
        raise OracleError(f"{what} failed with status {rc}")


def route(logits: np.ndarray, K: int, with_shared: bool, renormalize: bool = True,
          shared_w: np.ndarray | None = None):
    """fp32 logits [T, E] -> (ids int32 [T, Kt], weights fp32 [T, Kt]).  shared_w (fp32 [T],
    optional) is the shared slot's weight per token; 1.0 when absent."""
    logits = np.ascontiguousarray(logits, np.float32)
    T, E = logits.shape
    Kt = K + (1 if with_shared else 0)
    ids = np.empty((T, Kt), np.int32)
    w = np.empty((T, Kt), np.float32)
    sw = None if shared_w is None else np.ascontiguousarray(shared_w, np.float32)
    if sw is not None and sw.shape != (T,):
        raise ValueError("shared_w must be [T]")
    _check(_load().moe_ref_route(_p(logits), None if sw is None else _p(sw), T, E, K,
                                 int(with_shared), int(renormalize), _p(ids), _p(w)), "route")
    return ids, w


def capacity(T: int, Kt: int, Et: int, tile_m: int) -> int:
    return int(_load().moe_ref_capacity(T, Kt, Et, tile_m))


def permute(ids: np.ndarray, Et: int, tile_m: int):
    """Stable counting sort of pairs by expert with tile-aligned buckets.

    Returns dict(sorted_pairs [cap], offsets [Et+1], inv [T*Kt],
    tile_expert [cap // tile_m], num_tiles int)."""
    ids = np.ascontiguousarray(ids, np.int32)
    T, Kt = ids.shape
    cap = capacity(T, Kt, Et, tile_m)
    out = dict(sorted_pairs=np.empty(cap, np.int32), offsets=np.empty(Et + 1, np.int32),
               inv=np.empty(T * Kt, np.int32), tile_expert=np.empty(cap // tile_m, np.int32))
    nt = np.zeros(1, np.int32)
    _check(_load().moe_ref_permute(_p(ids), T, Kt, Et, tile_m, _p(out["sorted_pairs"]),
                                   _p(out["offsets"]), _p(out["inv"]), _p(out["tile_expert"]),
                                   _p(nt)), "permute")
    out["num_tiles"] = int(nt[0])
    return out


def ffn(x, w13, s13, w2, s2, ids, w, tokens=None, want_f32=False, n_threads=1):
    """Per-token loop oracle.  x: bf16 bits uint16 [T, H]; returns bf16 bits
    [n, H] for the requested tokens (all when tokens is None) and optionally
    the fp32 accumulator before rounding."""
    x = np.ascontiguousarray(x, np.uint16)
    T, H = x.shape
    Et, twoI, _ = w13.shape
    I = twoI // 2
    ids = np.ascontiguousarray(ids, np.int32)
    w = np.ascontiguousarray(w, np.float32)
    Kt = ids.shape[1]
    tok = None if tokens is None else np.ascontiguousarray(tokens, np.int32)
    n = T if tok is None else tok.size
    out = np.empty((n, H), np.uint16)
    of = np.empty((n, H), np.float32) if want_f32 else None
    for a in (w13, s13, w2, s2):
        assert a.dtype == np.uint8 and a.flags["C_CONTIGUOUS"]
    _check(_load().moe_ref_ffn(_p(x), _p(w13), _p(s13), _p(w2), _p(s2), _p(ids), _p(w), T, H, I,
                               Et, Kt, _p(tok), n, _p(out), _p(of), int(n_threads)), "ffn")
    return (out, of) if want_f32 else out


def ffn_grouped(x, w13, s13, w2, s2, w, perm):
    x = np.ascontiguousarray(x, np.uint16)
    T, H = x.shape
    Et, twoI, _ = w13.shape
    w = np.ascontiguousarray(w, np.float32)
    Kt = w.shape[1]
    out = np.empty((T, H), np.uint16)
    _check(_load().moe_ref_ffn_grouped(_p(x), _p(w13), _p(s13), _p(w2), _p(s2), _p(w),
                                       _p(perm["sorted_pairs"]), _p(perm["offsets"]), T, H,
                                       twoI // 2, Et, Kt, _p(out)), "ffn_grouped")
    return out


def mxfp4_value(code: int, scale: int) -> float:
    return float(_load().moe_ref_mxfp4_value(code, scale))


def silu(g: float) -> float:
    return float(_load().moe_ref_silu(g))


def f32_to_bf16(f: float) -> int:
    return int(_load().moe_ref_f32_to_bf16(f))


def max_threads() -> int:
    return int(_load().moe_ref_max_threads())


def e2m1_round(v: float) -> int:
    """E2M1 code of v rounded to nearest (ties to the even code, saturating at 6, sign kept)."""
    return int(_load().moe_ref_e2m1_round(float(v)))


def quantize_mxfp4(v: np.ndarray):
    """MXFP4 quantisation along the last axis (length a multiple of 32):
    fp32 [..., n] -> (codes uint8 [..., n/2], scales uint8 [..., n/32])."""
    v = np.ascontiguousarray(v, np.float32)
    n = v.shape[-1]
    if n % 32:
        raise ValueError("last axis must be a multiple of 32")
    rows = v.reshape(-1, n)
    codes = np.empty((rows.shape[0], n // 2), np.uint8)
    scales = np.empty((rows.shape[0], n // 32), np.uint8)
    lib = _load()
    for r in range(rows.shape[0]):
        _check(lib.moe_ref_quantize_mxfp4(_p(rows[r]), n, _p(codes[r]), _p(scales[r])),
               "quantize_mxfp4")
    return codes.reshape(*v.shape[:-1], n // 2), scales.reshape(*v.shape[:-1], n // 32)


def ffn_mxfp4act(x, w13, s13, w2, s2, ids, w, tokens=None, want_f32=False, want_h=False,
                 n_threads=1):
    """Per-token loop oracle of the layer with MXFP4-quantised activations (x
    and the SwiGLU output).  Returns out (bf16 bits [n, H]); with want_f32 also
    the fp32 accumulator; with want_h also dict(a fp32 [n*Kt, I] = SwiGLU output
    before quantisation, codes uint8 [n*Kt, I/2], scales uint8 [n*Kt, I/32]),
    row i*Kt + j for requested token i and slot j."""
    x = np.ascontiguousarray(x, np.uint16)
    T, H = x.shape
    Et, twoI, _ = w13.shape
    I = twoI // 2
    ids = np.ascontiguousarray(ids, np.int32)
    w = np.ascontiguousarray(w, np.float32)
    Kt = ids.shape[1]
    tok = None if tokens is None else np.ascontiguousarray(tokens, np.int32)
    n = T if tok is None else tok.size
    out = np.empty((n, H), np.uint16)
    of = np.empty((n, H), np.float32) if want_f32 else None
    h = None
    if want_h:
        h = dict(a=np.empty((n * Kt, I), np.float32), codes=np.empty((n * Kt, I // 2), np.uint8),
                 scales=np.empty((n * Kt, I // 32), np.uint8))
    for arr in (w13, s13, w2, s2):
        assert arr.dtype == np.uint8 and arr.flags["C_CONTIGUOUS"]
    _check(_load().moe_ref_ffn_mxfp4act(
        _p(x), _p(w13), _p(s13), _p(w2), _p(s2), _p(ids), _p(w), T, H, I, Et, Kt, _p(tok), n,
        _p(out), _p(of), None if h is None else _p(h["a"]), None if h is None else _p(h["codes"]),
        None if h is None else _p(h["scales"]), int(n_threads)), "ffn_mxfp4act")
    res = [out]
    if want_f32:
        res.append(of)
    if want_h:
        res.append(h)
    return res[0] if len(res) == 1 else tuple(res)
