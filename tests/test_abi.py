"""The C-ABI library loads and exports every entry point include/moe.h
declares; host-side argument checks reject bad calls before any launch.
CPU only: no call here reaches a CUDA kernel."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from mxfp4_mixture_experts_softmax_gb300 import libmoe
    return libmoe.load()


def test_header_declares_the_binding_names():
    from mxfp4_mixture_experts_softmax_gb300 import libmoe
    assert set(_declared()) == set(libmoe.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings_and_sizes(lib):
    from mxfp4_mixture_experts_softmax_gb300 import libmoe as m
    for s in range(6):
        assert m.status_string(s).startswith("MOE_")
    assert m.status_string(99).startswith("MOE_ERR_UNKNOWN")
    assert m.moe_permute_capacity(64, 11, 513, 8) == 64 * 11 + 513 * 7
    assert m.moe_permute_max_tiles(64, 11, 513, 8) == (64 * 11 + 513 * 7) // 8
    assert m.moe_permute_capacity(-1, 11, 513, 8) == 0
    cap = 64 * 11 + 513 * 7
    ws = m.moe_ffn_workspace_size(64, 4096, 1024, 513, 11, 8)
    assert ws >= cap * 1024 * 2 + 64 * 11 * 4096 * 4
    assert m.moe_ffn_auto_path(64, 11, 513, 8) == m.MOE_PATH_DECODE
    # the large-M regime: the two-term path where widths and tile height allow it
    assert m.moe_ffn_auto_path_shape(1536, 4096, 1024, 513, 11, 64) == m.MOE_PATH_PREFILL_FP8X2
    assert m.moe_ffn_auto_path_shape(8192, 4096, 1024, 513, 11, 128) == m.MOE_PATH_PREFILL_FP8X2
    assert m.moe_ffn_auto_path_shape(8192, 4096, 1024, 513, 11, 256) == m.MOE_PATH_PREFILL
    assert m.moe_ffn_auto_path_shape(1536, 4096, 256, 513, 11, 64) == m.MOE_PATH_PREFILL
    assert m.moe_ffn_auto_path_shape(64, 4096, 1024, 513, 11, 8) == m.MOE_PATH_DECODE
    assert m.moe_ffn_auto_path_shape(64, 250, 1024, 513, 11, 8) == m.MOE_PATH_AUTO  # H % 32
    # 96-row tiles: only the two-term path has them
    assert m.moe_ffn_auto_path_shape(8192, 4096, 1024, 513, 11, 96) == m.MOE_PATH_PREFILL_FP8X2
    assert m.moe_ffn_auto_path_shape(8192, 4096, 256, 513, 11, 96) == m.MOE_PATH_AUTO


def test_host_validation_rejects_before_launch(lib):
    from mxfp4_mixture_experts_softmax_gb300 import libmoe as m
    nul = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: every call below fails validation
    # route: negative T, K > E, E too large, NULL pointers
    assert lib.moe_route(fake, -1, 8, 2, 0, 1, fake, fake, nul) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_route(fake, 4, 8, 9, 0, 1, fake, fake, nul) == m.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_route(fake, 4, 2048, 2, 0, 1, fake, fake, nul) == m.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_route(nul, 4, 8, 2, 0, 1, fake, fake, nul) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_route(nul, 0, 8, 2, 0, 1, nul, nul, nul) == m.MOE_OK  # T = 0: nothing to do
    # permute: bad sizes, NULL outputs
    assert lib.moe_permute(fake, 4, 2, 8, 0, fake, fake, fake, fake, fake, nul) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_permute(fake, 4, 40, 8, 8, fake, fake, fake, fake, fake, nul) == m.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_permute(fake, 4, 2, 8, 8, fake, nul, fake, fake, fake, nul) == m.MOE_ERR_INVALID_ARG
    # ffn: H not a multiple of 32, unsupported tile, tiny workspace, misaligned pointer
    def ffn(T=4, H=256, I=128, Et=8, Kt=2, tile_m=8, ws=1 << 30, x=fake, path=0):
        return lib.moe_ffn_path(x, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                T, H, I, Et, Kt, tile_m, fake, fake, ws, path, nul)
    assert ffn(H=250) == m.MOE_ERR_UNSUPPORTED_SHAPE
    assert ffn(tile_m=12, path=m.MOE_PATH_DECODE) == m.MOE_ERR_UNSUPPORTED_SHAPE
    assert ffn(ws=16) == m.MOE_ERR_WORKSPACE_TOO_SMALL
    assert ffn(x=ctypes.c_void_p(0x1008)) == m.MOE_ERR_INVALID_ARG
    assert ffn(path=7) == m.MOE_ERR_INVALID_ARG
    assert ffn(T=-2) == m.MOE_ERR_INVALID_ARG


def test_mxfp4act_host_validation_and_layout(lib):
    """The MXFP4-activation entries: shape and argument checks before any
    launch; workspace regions 256-byte aligned and large enough."""
    from mxfp4_mixture_experts_softmax_gb300 import libmoe as m
    nul = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(0x1000)

    def mx(T=4, H=256, I=128, Et=8, Kt=2, tile_m=32, ws=1 << 30, x=fake):
        return lib.moe_ffn_mxfp4act(x, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                    T, H, I, Et, Kt, tile_m, fake, fake, ws, nul)
    assert mx(H=160) == m.MOE_ERR_UNSUPPORTED_SHAPE       # H % 128
    assert mx(I=96) == m.MOE_ERR_UNSUPPORTED_SHAPE        # I % 128
    for tm in (8, 16, 48, 512):
        assert mx(tile_m=tm) == m.MOE_ERR_UNSUPPORTED_SHAPE
    assert mx(T=-1) == m.MOE_ERR_INVALID_ARG
    assert mx(ws=64) == m.MOE_ERR_WORKSPACE_TOO_SMALL
    assert mx(x=nul) == m.MOE_ERR_INVALID_ARG
    assert mx(x=ctypes.c_void_p(0x1004)) == m.MOE_ERR_INVALID_ARG  # not 16-byte aligned
    assert mx(T=0) == m.MOE_OK
    # quantiser: columns not a multiple of 32, negative rows, NULL pointers
    assert lib.moe_quantize_mxfp4(fake, 4, 48, fake, fake, nul) == m.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_quantize_mxfp4(fake, -1, 64, fake, fake, nul) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_mxfp4(nul, 4, 64, fake, fake, nul) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_mxfp4(nul, 0, 64, nul, nul, nul) == m.MOE_OK
    # workspace layout: h regions aligned, inside the workspace, sized for cap rows
    for T, tm in ((64, 32), (1536, 64), (8192, 128)):
        H, I, Et, Kt = 4096, 1024, 513, 11
        ws = m.moe_ffn_mxfp4act_workspace_size(T, H, I, Et, Kt, tm)
        cap = m.moe_permute_capacity(T, Kt, Et, tm)
        co, so = ctypes.c_size_t(), ctypes.c_size_t()
        assert lib.moe_ffn_mxfp4act_h_offsets(T, H, I, Et, Kt, tm, ctypes.byref(co),
                                              ctypes.byref(so)) == m.MOE_OK
        assert co.value % 256 == 0 and so.value % 256 == 0
        assert so.value >= co.value + cap * (I // 2)
        # the position weights, y (staged f16 rows by position [cap, H]) and its
        # shift bytes ([ceil(cap/32), H/8]) follow the scales
        assert ws >= so.value + cap * (I // 32) + cap * 4 + cap * H * 2 + (cap + 31) // 32 * (H // 8)
    assert lib.moe_ffn_mxfp4act_h_offsets(4, 256, 128, 8, 2, 32, None, None) == m.MOE_ERR_INVALID_ARG


def test_fp8x2_path_host_validation(lib):
    """MOE_PATH_PREFILL_FP8X2: widths multiples of 512 (whole 16-byte scale
    boxes), tile heights 32/64/128, weights 32-byte aligned; the split call's
    checks; all before any launch."""
    from mxfp4_mixture_experts_softmax_gb300 import libmoe as m
    nul = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(0x1000)
    P = m.MOE_PATH_PREFILL_FP8X2

    def ffn(T=64, H=512, I=512, Et=8, Kt=2, tile_m=64, ws=1 << 30, w=fake, path=P):
        return lib.moe_ffn_path(fake, w, fake, w, fake, fake, fake, fake, fake, fake, fake,
                                T, H, I, Et, Kt, tile_m, fake, fake, ws, path, nul)
    assert ffn(H=256) == m.MOE_ERR_UNSUPPORTED_SHAPE      # H % 512
    assert ffn(I=1536 + 256) == m.MOE_ERR_UNSUPPORTED_SHAPE  # I % 512
    for tm in (8, 16, 256):
        assert ffn(tile_m=tm) == m.MOE_ERR_UNSUPPORTED_SHAPE
    assert ffn(ws=64) == m.MOE_ERR_WORKSPACE_TOO_SMALL
    assert ffn(w=ctypes.c_void_p(0x1010)) == m.MOE_ERR_INVALID_ARG  # 16- but not 32-byte aligned
    assert ffn(T=0) == m.MOE_OK
    assert lib.moe_split_e4m3x2(fake, 4, 48, fake, fake, fake, fake, nul) == m.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_split_e4m3x2(fake, -1, 64, fake, fake, fake, fake, nul) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_split_e4m3x2(fake, 4, 64, fake, fake, nul, fake, nul) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_split_e4m3x2(nul, 0, 64, nul, nul, nul, nul, nul) == m.MOE_OK
    # the workspace holds h's two terms (2 tile_m rows per tile) in the h
    # area, x's in the tile-ordered copy's area and h's scale bytes at its end
    H, I, Et, Kt = 4096, 1024, 513, 11
    for T, tm in ((288, 32), (1536, 64), (8192, 128)):
        cap = m.moe_permute_capacity(T, Kt, Et, tm)
        tiles = m.moe_permute_max_tiles(T, Kt, Et, tm)
        assert tiles * 2 * tm * I <= m.moe_ffn_y_offset(T, I, Et, Kt, tm)
        assert m.moe_ffn_workspace_size(T, H, I, Et, Kt, tm) >= (
            m.moe_ffn_y_offset(T, I, Et, Kt, tm) + max(T * Kt * H * 4, cap * H * 2) + T * H * 2
            + cap * H * 2 + (T + 2 * cap) * 4 + tiles * 2 * tm * (I // 32))


def test_bf16_workspace_holds_staged_y_for_prefill_tiles(lib):
    """moe_ffn_down_combine's prefill path writes y as f16 rows over cap
    positions: the workspace reserves that much for prefill tile heights."""
    from mxfp4_mixture_experts_softmax_gb300 import libmoe as m
    H, I, Et, Kt = 4096, 1024, 513, 11
    for T, tm in ((1536, 64), (8192, 128)):
        cap = m.moe_permute_capacity(T, Kt, Et, tm)
        ws = m.moe_ffn_workspace_size(T, H, I, Et, Kt, tm)
        y_off = m.moe_ffn_y_offset(T, I, Et, Kt, tm)
        assert y_off % 256 == 0 and y_off >= cap * I * 2
        assert ws >= y_off + max(T * Kt * H * 4, cap * H * 2)


def test_gemm_events_hook_argument_rule(lib):
    """moe_set_gemm_events takes both events or neither (host-side check only)."""
    from mxfp4_mixture_experts_softmax_gb300 import libmoe as m
    nul, fake = ctypes.c_void_p(0), ctypes.c_void_p(0x1000)
    assert lib.moe_set_gemm_events(fake, nul) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_set_gemm_events(nul, fake) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_set_gemm_events(nul, nul) == m.MOE_OK
