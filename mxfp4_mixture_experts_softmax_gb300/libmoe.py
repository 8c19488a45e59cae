"""Thin Python binding of the libmoe C ABI (include/moe.h), same entry-point names.

Argument marshalling only: every step runs in libmoe's CUDA kernels.  Torch
is used for device memory and the current stream.  If the shared library is
missing it is compiled with nvcc; if that is impossible the import fails --
there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build_lib

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED_SHAPE = 2
MOE_ERR_WORKSPACE_TOO_SMALL = 3
MOE_ERR_CUDA = 4
MOE_ERR_INTERNAL = 5

MOE_PATH_AUTO = 0
MOE_PATH_DECODE = 1
MOE_PATH_PREFILL = 2
MOE_PATH_PREFILL_FP8X2 = 3

EXPORTS = ("moe_status_string", "moe_version", "moe_route", "moe_route_ex", "moe_permute_capacity",
           "moe_permute_max_tiles", "moe_permute", "moe_route_permute", "moe_ffn_workspace_size",
           "moe_ffn",
           "moe_ffn_path", "moe_ffn_auto_path", "moe_ffn_gate_up", "moe_ffn_down", "moe_combine",
           "moe_ffn_y_offset", "moe_device_error", "moe_ffn_noalloc", "moe_combine_ex",
           "moe_ffn_dense_shared_workspace_size", "moe_ffn_dense_shared",
           "moe_selftest_wait_timeout", "moe_selftest_wait_split", "moe_set_gemm_events",
           "moe_quantize_mxfp4", "moe_ffn_mxfp4act_workspace_size",
           "moe_ffn_mxfp4act", "moe_ffn_mxfp4act_gate_up", "moe_ffn_mxfp4act_down",
           "moe_ffn_mxfp4act_h_offsets", "moe_ffn_down_combine", "moe_split_e4m3x2", "moe_ffn_auto_path_shape")

# bytes of the fixed device scratch behind moe_ffn_noalloc (include/moe.h)
MOE_NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024
# batches up to this many tokens route and permute in one launch (include/moe.h)
MOE_ROUTE_PERMUTE_FUSED_MAX_T = 32

_lock = threading.Lock()
_lib = None


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


def lib_path() -> str:
    return build_lib.LIB


def load(build: bool = True):
    """Load libmoe.so (building it first if needed) and declare the signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = build_lib.build() if build else build_lib.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libmoe is not built ({path}); run __graft_entry__.build()")
        L = ctypes.CDLL(path)
        vp, ci, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.moe_status_string.argtypes = [ci]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_version.argtypes = []
        L.moe_version.restype = ci
        L.moe_route.argtypes = [vp, ci, ci, ci, ci, ci, vp, vp, vp]
        L.moe_route.restype = ci
        L.moe_route_ex.argtypes = [vp, vp, ci, ci, ci, ci, ci, vp, vp, vp]
        L.moe_route_ex.restype = ci
        L.moe_route_permute.argtypes = [vp, vp, ci, ci, ci, ci, ci, ci, vp, vp, vp, vp, vp, vp, vp,
                                        vp]
        L.moe_route_permute.restype = ci
        L.moe_permute_capacity.argtypes = [ci, ci, ci, ci]
        L.moe_permute_capacity.restype = sz
        L.moe_permute_max_tiles.argtypes = [ci, ci, ci, ci]
        L.moe_permute_max_tiles.restype = sz
        L.moe_permute.argtypes = [vp, ci, ci, ci, ci, vp, vp, vp, vp, vp, vp]
        L.moe_permute.restype = ci
        L.moe_ffn_workspace_size.argtypes = [ci, ci, ci, ci, ci, ci]
        L.moe_ffn_workspace_size.restype = sz
        ffn_args = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, vp, vp, sz]
        L.moe_ffn.argtypes = ffn_args + [vp]
        L.moe_ffn.restype = ci
        L.moe_ffn_path.argtypes = ffn_args + [ci, vp]
        L.moe_ffn_path.restype = ci
        L.moe_ffn_auto_path.argtypes = [ci, ci, ci, ci]
        L.moe_ffn_auto_path.restype = ci
        L.moe_ffn_auto_path_shape.argtypes = [ci, ci, ci, ci, ci, ci]
        L.moe_ffn_auto_path_shape.restype = ci
        L.moe_ffn_gate_up.argtypes = [vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, vp, sz, ci, vp]
        L.moe_ffn_gate_up.restype = ci
        L.moe_ffn_down.argtypes = [vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, vp, sz, ci, vp]
        L.moe_ffn_down.restype = ci
        L.moe_combine.argtypes = [vp, ci, ci, ci, vp, vp]
        L.moe_combine.restype = ci
        L.moe_ffn_y_offset.argtypes = [ci, ci, ci, ci, ci]
        L.moe_ffn_y_offset.restype = sz
        L.moe_ffn_noalloc.argtypes = ffn_args[:-2] + [vp]
        L.moe_ffn_noalloc.restype = ci
        L.moe_combine_ex.argtypes = [vp, vp, ci, ci, ci, vp, vp]
        L.moe_combine_ex.restype = ci
        L.moe_ffn_dense_shared_workspace_size.argtypes = [ci, ci, ci, ci, ci, ci, ci]
        L.moe_ffn_dense_shared_workspace_size.restype = sz
        L.moe_ffn_dense_shared.argtypes = (ffn_args[:17] + [vp, vp, vp, vp, ci, vp, vp, vp, sz, vp])
        L.moe_ffn_dense_shared.restype = ci
        L.moe_selftest_wait_timeout.argtypes = [ci, vp]
        L.moe_selftest_wait_timeout.restype = ci
        L.moe_selftest_wait_split.argtypes = [ci, vp, vp]
        L.moe_selftest_wait_split.restype = ci
        L.moe_set_gemm_events.argtypes = [vp, vp]
        L.moe_set_gemm_events.restype = ci
        L.moe_ffn_down_combine.argtypes = [vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, vp, vp,
                                           sz, ci, vp]
        L.moe_ffn_down_combine.restype = ci
        L.moe_quantize_mxfp4.argtypes = [vp, ci, ci, vp, vp, vp]
        L.moe_quantize_mxfp4.restype = ci
        L.moe_split_e4m3x2.argtypes = [vp, ci, ci, vp, vp, vp, vp, vp]
        L.moe_split_e4m3x2.restype = ci
        L.moe_ffn_mxfp4act_workspace_size.argtypes = [ci, ci, ci, ci, ci, ci]
        L.moe_ffn_mxfp4act_workspace_size.restype = sz
        L.moe_ffn_mxfp4act.argtypes = ffn_args + [vp]
        L.moe_ffn_mxfp4act.restype = ci
        L.moe_ffn_mxfp4act_gate_up.argtypes = [vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, vp, sz,
                                               vp]
        L.moe_ffn_mxfp4act_gate_up.restype = ci
        L.moe_ffn_mxfp4act_down.argtypes = [vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, vp,
                                            vp, sz, vp]
        L.moe_ffn_mxfp4act_down.restype = ci
        L.moe_ffn_mxfp4act_h_offsets.argtypes = [ci, ci, ci, ci, ci, ci, vp, vp]
        L.moe_ffn_mxfp4act_h_offsets.restype = ci
        L.moe_device_error.argtypes = [vp, ci]
        L.moe_device_error.restype = ci
        _lib = L
        return L


def status_string(status: int) -> str:
    return load().moe_status_string(status).decode()


def _check(status: int, what: str):
    if status != MOE_OK:
        raise MoeError(status, what)


def _ptr(t):
    if t is None:
        return None
    return t.data_ptr() if t.numel() > 0 else None


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t, dtype_name: str):
    import torch
    assert t.is_cuda and t.is_contiguous(), f"{dtype_name} must be a contiguous CUDA tensor"
    return t


def _route_outputs(logits, K, with_shared, topk_ids, topk_w, shared_w):
    import torch
    _dev(logits, "logits")
    assert logits.dtype == torch.float32
    T, E = logits.shape
    Kt = K + (1 if with_shared else 0)
    if topk_ids is None:
        topk_ids = torch.empty((T, Kt), dtype=torch.int32, device=logits.device)
    if topk_w is None:
        topk_w = torch.empty((T, Kt), dtype=torch.float32, device=logits.device)
    if shared_w is not None:
        _dev(shared_w, "shared_w")
        assert shared_w.dtype == torch.float32 and shared_w.shape == (T,)
    return T, E, Kt, topk_ids, topk_w


def moe_route(logits, K: int, with_shared: bool = True, renormalize: bool = True,
              topk_ids=None, topk_w=None, stream=None, shared_w=None):
    """fp32 logits [T, E] -> (int32 ids [T, Kt], fp32 weights [T, Kt]).  shared_w (fp32 [T],
    optional): per-token weight of the shared slot (moe_route_ex)."""
    T, E, Kt, topk_ids, topk_w = _route_outputs(logits, K, with_shared, topk_ids, topk_w, shared_w)
    if shared_w is None:
        _check(load().moe_route(_ptr(logits), T, E, K, int(with_shared), int(renormalize),
                                _ptr(topk_ids), _ptr(topk_w), _stream(stream)), "moe_route")
    else:
        _check(load().moe_route_ex(_ptr(logits), _ptr(shared_w), T, E, K, int(with_shared),
                                   int(renormalize), _ptr(topk_ids), _ptr(topk_w),
                                   _stream(stream)), "moe_route_ex")
    return topk_ids, topk_w


def moe_route_permute(logits, K: int, tile_m: int, with_shared: bool = True,
                      renormalize: bool = True, topk_ids=None, topk_w=None,
                      perm: dict | None = None, shared_w=None, stream=None):
    """moe_route_ex + moe_permute in one call (one launch for small batches):
    returns (ids, weights, perm dict as from moe_permute)."""
    T, E, Kt, topk_ids, topk_w = _route_outputs(logits, K, with_shared, topk_ids, topk_w, shared_w)
    Et = E + (1 if with_shared else 0)
    if perm is None:
        perm = alloc_permute(T, Kt, Et, tile_m, logits.device)
    _check(load().moe_route_permute(_ptr(logits), _ptr(shared_w), T, E, K, int(with_shared),
                                    int(renormalize), tile_m, _ptr(topk_ids), _ptr(topk_w),
                                    _ptr(perm["sorted_pairs"]), _ptr(perm["expert_offsets"]),
                                    _ptr(perm["inv_pairs"]), _ptr(perm["tile_expert"]),
                                    _ptr(perm["num_tiles"]), _stream(stream)), "moe_route_permute")
    return topk_ids, topk_w, perm


def moe_permute_capacity(T: int, Kt: int, Et: int, tile_m: int) -> int:
    return int(load().moe_permute_capacity(T, Kt, Et, tile_m))


def moe_permute_max_tiles(T: int, Kt: int, Et: int, tile_m: int) -> int:
    return int(load().moe_permute_max_tiles(T, Kt, Et, tile_m))


def alloc_permute(T: int, Kt: int, Et: int, tile_m: int, device="cuda") -> dict:
    import torch
    cap = moe_permute_capacity(T, Kt, Et, tile_m)
    mt = moe_permute_max_tiles(T, Kt, Et, tile_m)
    i32 = dict(dtype=torch.int32, device=device)
    return dict(sorted_pairs=torch.empty(max(cap, 1), **i32)[:cap],
                expert_offsets=torch.empty(Et + 1, **i32),
                inv_pairs=torch.empty(max(T * Kt, 1), **i32)[:T * Kt],
                tile_expert=torch.empty(max(mt, 1), **i32)[:mt],
                num_tiles=torch.empty(1, **i32), T=T, Kt=Kt, Et=Et, tile_m=tile_m)


def moe_permute(topk_ids, Et: int, tile_m: int, out: dict | None = None, stream=None) -> dict:
    """int32 ids [T, Kt] -> dict of sorted_pairs, expert_offsets, inv_pairs,
    tile_expert, num_tiles (device tensors) plus the sizes."""
    T, Kt = topk_ids.shape
    _dev(topk_ids, "topk_ids")
    if out is None:
        out = alloc_permute(T, Kt, Et, tile_m, topk_ids.device)
    _check(load().moe_permute(_ptr(topk_ids), T, Kt, Et, tile_m, _ptr(out["sorted_pairs"]),
                              _ptr(out["expert_offsets"]), _ptr(out["inv_pairs"]),
                              _ptr(out["tile_expert"]), _ptr(out["num_tiles"]), _stream(stream)),
           "moe_permute")
    return out


def moe_ffn_workspace_size(T: int, H: int, I: int, Et: int, Kt: int, tile_m: int) -> int:
    return int(load().moe_ffn_workspace_size(T, H, I, Et, Kt, tile_m))


def moe_ffn_auto_path(T: int, Kt: int, Et: int, tile_m: int) -> int:
    return int(load().moe_ffn_auto_path(T, Kt, Et, tile_m))


def moe_ffn_auto_path_shape(T: int, H: int, I: int, Et: int, Kt: int, tile_m: int) -> int:
    return int(load().moe_ffn_auto_path_shape(T, H, I, Et, Kt, tile_m))


def alloc_workspace(T: int, H: int, I: int, Et: int, Kt: int, tile_m: int, device="cuda"):
    import torch
    n = moe_ffn_workspace_size(T, H, I, Et, Kt, tile_m)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def moe_ffn(x, w13, s13, w2, s2, topk_w, perm: dict, out=None, workspace=None,
            path: int = MOE_PATH_AUTO, stream=None):
    """bf16 x [T, H] -> bf16 out [T, H] through the grouped MXFP4 expert MLPs."""
    import torch
    T, H = x.shape
    Et, twoI, _ = w13.shape
    I = twoI // 2
    Kt, tile_m = perm["Kt"], perm["tile_m"]
    for t in (x, w13, s13, w2, s2, topk_w):
        _dev(t, "ffn input")
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = alloc_workspace(T, H, I, Et, Kt, tile_m, x.device)
    _check(load().moe_ffn_path(_ptr(x), _ptr(w13), _ptr(s13), _ptr(w2), _ptr(s2), _ptr(topk_w),
                               _ptr(perm["sorted_pairs"]), _ptr(perm["expert_offsets"]),
                               _ptr(perm["inv_pairs"]), _ptr(perm["tile_expert"]),
                               _ptr(perm["num_tiles"]), T, H, I, Et, Kt, tile_m, _ptr(out),
                               _ptr(workspace), workspace.numel(), int(path), _stream(stream)),
           "moe_ffn")
    return out


def moe_device_error(clear: bool = True) -> int:
    """The device error bits: 1 = a bounded wait inside a kernel gave up, 2 = an index out of
    range was met and that work skipped (include/moe.h)."""
    flag = ctypes.c_int(0)
    _check(load().moe_device_error(ctypes.byref(flag), int(clear)), "moe_device_error")
    return flag.value


def moe_selftest_wait_timeout(limit_us: int = 2000, stream=None):
    """Diagnostic: a bounded wait that runs out (include/moe.h)."""
    _check(load().moe_selftest_wait_timeout(int(limit_us), _stream(stream)),
           "moe_selftest_wait_timeout")


def moe_set_gemm_events(before=None, after=None):
    """Profiling hook (include/moe.h): record the torch.cuda.Event pair around
    the grouped GEMM kernel of each following FFN call; None, None switches it
    off.  The events are created here if they have not been recorded yet."""
    import torch
    handles = []
    for ev in (before, after):
        if ev is None:
            handles.append(None)
            continue
        if ev.cuda_event == 0:  # torch creates an event lazily, on its first record
            ev.record(torch.cuda.current_stream())
        handles.append(ctypes.c_void_p(ev.cuda_event))
    _check(load().moe_set_gemm_events(*handles), "moe_set_gemm_events")


def moe_selftest_wait_split(limit_us: int = 2000, stream=None):
    """Diagnostic: two warps whose bounded waits end differently must stop
    together (include/moe.h).  Returns the device tensor of the two warps'
    outcomes (int32 [2]; 0 = stopped)."""
    import torch
    out = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    _check(load().moe_selftest_wait_split(int(limit_us), _ptr(out), _stream(stream)),
           "moe_selftest_wait_split")
    return out


def moe_ffn_noalloc(x, w13, s13, w2, s2, topk_w, perm: dict, out=None, stream=None):
    """moe_ffn without a workspace argument: the scratch is the library's fixed
    device array (for callers that cannot allocate device memory).  Calls on
    one device share that array: do not overlap them on the GPU."""
    import torch
    T, H = x.shape
    Et, twoI, _ = w13.shape
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _check(load().moe_ffn_noalloc(_ptr(x), _ptr(w13), _ptr(s13), _ptr(w2), _ptr(s2), _ptr(topk_w),
                                  _ptr(perm["sorted_pairs"]), _ptr(perm["expert_offsets"]),
                                  _ptr(perm["inv_pairs"]), _ptr(perm["tile_expert"]),
                                  _ptr(perm["num_tiles"]), T, H, twoI // 2, Et, perm["Kt"],
                                  perm["tile_m"], _ptr(out), _stream(stream)), "moe_ffn_noalloc")
    return out


def moe_ffn_y_offset(T: int, I: int, Et: int, Kt: int, tile_m: int) -> int:
    return int(load().moe_ffn_y_offset(T, I, Et, Kt, tile_m))


def ffn_views(workspace, T: int, H: int, I: int, Et: int, Kt: int, tile_m: int):
    """(h [cap, I] 16-bit, y fp32 [T*Kt, H]) views of a moe_ffn workspace (after the gate_up
    step h holds scaled f16 rows: see moe_ffn_gate_up in include/moe.h)."""
    import torch
    cap = moe_permute_capacity(T, Kt, Et, tile_m)
    off = moe_ffn_y_offset(T, I, Et, Kt, tile_m)
    h = workspace[:cap * I * 2].view(torch.bfloat16).view(cap, I)
    y = workspace[off:off + T * Kt * H * 4].view(torch.float32).view(T * Kt, H)
    return h, y


def moe_ffn_gate_up(x, w13, s13, perm: dict, workspace, path: int = MOE_PATH_AUTO, stream=None):
    """gate_up + SwiGLU into the workspace's h (see ffn_views)."""
    T, H = x.shape
    Et, twoI, _ = w13.shape
    _check(load().moe_ffn_gate_up(_ptr(x), _ptr(w13), _ptr(s13), _ptr(perm["sorted_pairs"]),
                                  _ptr(perm["tile_expert"]), _ptr(perm["num_tiles"]), T, H,
                                  twoI // 2, Et, perm["Kt"], perm["tile_m"], _ptr(workspace),
                                  workspace.numel(), int(path), _stream(stream)), "moe_ffn_gate_up")
    return workspace


def moe_ffn_down(w2, s2, topk_w, perm: dict, workspace, T: int, path: int = MOE_PATH_AUTO,
                 stream=None):
    """down x routing weight from the workspace's h into its y (see ffn_views)."""
    Et, H, halfI = w2.shape
    _check(load().moe_ffn_down(_ptr(w2), _ptr(s2), _ptr(topk_w), _ptr(perm["sorted_pairs"]),
                               _ptr(perm["tile_expert"]), _ptr(perm["num_tiles"]), T, H, 2 * halfI,
                               Et, perm["Kt"], perm["tile_m"], _ptr(workspace), workspace.numel(),
                               int(path), _stream(stream)), "moe_ffn_down")
    return workspace


def moe_ffn_down_combine(w2, s2, topk_w, perm: dict, workspace, T: int, out,
                         path: int = MOE_PATH_AUTO, stream=None):
    """down x routing weight and the combine into out (include/moe.h)."""
    Et, H, halfI = w2.shape
    _check(load().moe_ffn_down_combine(
        _ptr(w2), _ptr(s2), _ptr(topk_w), _ptr(perm["sorted_pairs"]), _ptr(perm["inv_pairs"]),
        _ptr(perm["tile_expert"]), _ptr(perm["num_tiles"]), T, H, 2 * halfI, Et, perm["Kt"],
        perm["tile_m"], _ptr(out), _ptr(workspace), workspace.numel(), int(path),
        _stream(stream)), "moe_ffn_down_combine")
    return out


def moe_combine(y, T: int, H: int, Kt: int, out, stream=None):
    _check(load().moe_combine(_ptr(y), T, H, Kt, _ptr(out), _stream(stream)), "moe_combine")
    return out


def moe_layer(logits, x, w13, s13, w2, s2, K: int, with_shared: bool = True,
              renormalize: bool = True, tile_m: int = 8, path: int = MOE_PATH_AUTO,
              bufs: dict | None = None, stream=None):
    """The whole layer: route -> permute -> ffn, all on one stream.  `bufs`
    (from alloc_layer) reuses preallocated device buffers."""
    T, E = logits.shape
    Et = w13.shape[0]
    if bufs is None:
        bufs = alloc_layer(T, E, K, with_shared, x.shape[1], w13.shape[1] // 2, Et, tile_m,
                           x.device)
    if Et != E + (1 if with_shared else 0):
        raise ValueError("weights must hold E experts plus the shared one when with_shared")
    ids, w, perm = moe_route_permute(logits, K, tile_m, with_shared, renormalize, bufs["topk_ids"],
                                     bufs["topk_w"], bufs["perm"], stream=stream)
    return moe_ffn(x, w13, s13, w2, s2, w, perm, bufs["out"], bufs["workspace"], path, stream)


def alloc_layer(T, E, K, with_shared, H, I, Et, tile_m, device="cuda") -> dict:
    import torch
    Kt = K + (1 if with_shared else 0)
    return dict(topk_ids=torch.empty((T, Kt), dtype=torch.int32, device=device),
                topk_w=torch.empty((T, Kt), dtype=torch.float32, device=device),
                perm=alloc_permute(T, Kt, Et, tile_m, device),
                workspace=alloc_workspace(T, H, I, Et, Kt, tile_m, device),
                out=torch.empty((T, H), dtype=torch.bfloat16, device=device))


def moe_ffn_dense_shared(x, w13, s13, w2, s2, topk_w, perm: dict, w13s, s13s, w2s, s2s,
                         shared_w=None, out=None, workspace=None, stream=None):
    """Routed layer + a shared expert of another width run as a dense MLP over all tokens
    (include/moe.h, moe_ffn_dense_shared)."""
    import torch
    T, H = x.shape
    Et, twoI, _ = w13.shape
    Is = w13s.shape[1] // 2
    Kt, tm = perm["Kt"], perm["tile_m"]
    n = int(load().moe_ffn_dense_shared_workspace_size(T, H, twoI // 2, Et, Kt, Is, tm))
    if workspace is None:
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _check(load().moe_ffn_dense_shared(
        _ptr(x), _ptr(w13), _ptr(s13), _ptr(w2), _ptr(s2), _ptr(topk_w),
        _ptr(perm["sorted_pairs"]), _ptr(perm["expert_offsets"]), _ptr(perm["inv_pairs"]),
        _ptr(perm["tile_expert"]), _ptr(perm["num_tiles"]), T, H, twoI // 2, Et, Kt, tm,
        _ptr(w13s), _ptr(s13s), _ptr(w2s), _ptr(s2s), Is, _ptr(shared_w), _ptr(out),
        _ptr(workspace), workspace.numel(), _stream(stream)), "moe_ffn_dense_shared")
    return out


# ------------------------------------------------ MXFP4-quantised activations

def moe_split_e4m3x2(x, stream=None):
    """bf16 [rows, cols] -> (q_hi, q_lo uint8 [rows, cols], s_hi, s_lo uint8
    [rows, cols/32]): the two-term E4M3 encoding of MOE_PATH_PREFILL_FP8X2
    (include/moe.h)."""
    import torch
    _dev(x, "x")
    rows, cols = x.shape
    q_hi = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    q_lo = torch.empty_like(q_hi)
    s_hi = torch.empty((rows, cols // 32), dtype=torch.uint8, device=x.device)
    s_lo = torch.empty_like(s_hi)
    _check(load().moe_split_e4m3x2(_ptr(x), rows, cols, _ptr(q_hi), _ptr(q_lo), _ptr(s_hi), _ptr(s_lo),
                                   _stream(stream)), "moe_split_e4m3x2")
    return q_hi, q_lo, s_hi, s_lo


def moe_quantize_mxfp4(x, codes=None, scales=None, stream=None):
    """bf16 [rows, cols] -> (codes uint8 [rows, cols/2], scales uint8 [rows, cols/32]),
    OCP MX rounding (include/moe.h)."""
    import torch
    _dev(x, "x")
    rows, cols = x.shape
    if codes is None:
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((rows, cols // 32), dtype=torch.uint8, device=x.device)
    _check(load().moe_quantize_mxfp4(_ptr(x), rows, cols, _ptr(codes), _ptr(scales),
                                     _stream(stream)), "moe_quantize_mxfp4")
    return codes, scales


def moe_ffn_mxfp4act_workspace_size(T: int, H: int, I: int, Et: int, Kt: int, tile_m: int) -> int:
    return int(load().moe_ffn_mxfp4act_workspace_size(T, H, I, Et, Kt, tile_m))


def alloc_workspace_mxfp4act(T: int, H: int, I: int, Et: int, Kt: int, tile_m: int,
                             device="cuda"):
    import torch
    n = moe_ffn_mxfp4act_workspace_size(T, H, I, Et, Kt, tile_m)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def moe_ffn_mxfp4act(x, w13, s13, w2, s2, topk_w, perm: dict, out=None, workspace=None,
                     stream=None):
    """The expert FFN with MXFP4-quantised activations (both GEMMs block-scaled MXFP4 x MXFP4)."""
    import torch
    T, H = x.shape
    Et, twoI, _ = w13.shape
    Kt, tile_m = perm["Kt"], perm["tile_m"]
    for t in (x, w13, s13, w2, s2, topk_w):
        _dev(t, "ffn input")
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = alloc_workspace_mxfp4act(T, H, twoI // 2, Et, Kt, tile_m, x.device)
    _check(load().moe_ffn_mxfp4act(_ptr(x), _ptr(w13), _ptr(s13), _ptr(w2), _ptr(s2), _ptr(topk_w),
                                   _ptr(perm["sorted_pairs"]), _ptr(perm["expert_offsets"]),
                                   _ptr(perm["inv_pairs"]), _ptr(perm["tile_expert"]),
                                   _ptr(perm["num_tiles"]), T, H, twoI // 2, Et, Kt, tile_m,
                                   _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_ffn_mxfp4act")
    return out


def moe_ffn_mxfp4act_gate_up(x, w13, s13, perm: dict, workspace, stream=None):
    T, H = x.shape
    Et, twoI, _ = w13.shape
    _check(load().moe_ffn_mxfp4act_gate_up(
        _ptr(x), _ptr(w13), _ptr(s13), _ptr(perm["sorted_pairs"]), _ptr(perm["tile_expert"]),
        _ptr(perm["num_tiles"]), T, H, twoI // 2, Et, perm["Kt"], perm["tile_m"], _ptr(workspace),
        workspace.numel(), _stream(stream)), "moe_ffn_mxfp4act_gate_up")
    return workspace


def moe_ffn_mxfp4act_down(w2, s2, topk_w, perm: dict, workspace, T: int, out, stream=None):
    Et, H, halfI = w2.shape
    _check(load().moe_ffn_mxfp4act_down(
        _ptr(w2), _ptr(s2), _ptr(topk_w), _ptr(perm["sorted_pairs"]), _ptr(perm["inv_pairs"]),
        _ptr(perm["tile_expert"]),
        _ptr(perm["num_tiles"]), T, H, 2 * halfI, Et, perm["Kt"], perm["tile_m"], _ptr(out),
        _ptr(workspace), workspace.numel(), _stream(stream)), "moe_ffn_mxfp4act_down")
    return out


def mxfp4act_h_views(workspace, T: int, H: int, I: int, Et: int, Kt: int, tile_m: int):
    """(h codes uint8 [cap, I/2], h scales uint8 [cap, I/32]) views of a moe_ffn_mxfp4act
    workspace, rows by sorted position."""
    co, so = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(load().moe_ffn_mxfp4act_h_offsets(T, H, I, Et, Kt, tile_m, ctypes.byref(co),
                                             ctypes.byref(so)), "moe_ffn_mxfp4act_h_offsets")
    cap = moe_permute_capacity(T, Kt, Et, tile_m)
    codes = workspace[co.value:co.value + cap * (I // 2)].view(cap, I // 2)
    scales = workspace[so.value:so.value + cap * (I // 32)].view(cap, I // 32)
    return codes, scales
