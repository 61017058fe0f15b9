"""The C-ABI library without a GPU: it loads, exports every entry point the
header declares, its host-side logic (sizes, argument checks) answers, and the
exact block-scale division it relies on holds for every E4M3 divisor."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4_moe.h")


@pytest.fixture(scope="session")
def lib():
    import nvfp4_w4a4_moe_gb300 as m
    m.build()
    return m.load()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_path():
    names = declared_functions()
    for must in ("nvfp4_validate_scales", "nvfp4_quantize_experts", "nvfp4_moe_forward"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_version_and_error_string(lib):
    assert lib.nvfp4_version() >= 100
    assert isinstance(lib.nvfp4_last_error_string(), bytes)


def test_block_division_is_exact_for_every_e4m3_scale(lib):
    assert lib.nvfp4_selftest_block_division(0) == 0


def test_workspace_sizes(lib):
    import nvfp4_w4a4_moe_gb300 as m
    H, I, E, k = 2816, 704, 128, 8
    prev = 0
    for T in (0, 1, 8, 64, 512, 8192):
        n = m.moe_workspace_size(T, H, I, E, k)
        assert n >= prev and n % 256 == 0
        assert m.moe_host_workspace_size(T, H, I, E, k) >= n
        prev = n
    # the padded row capacity covers the worst case: every busy expert ends
    # on a partial 128-row tile
    R = 8192 * k
    assert m.intermediates_rows_cap(8192, E, k) >= R + E * 255  # room for rows padded to 256 per expert
    assert m.intermediates_rows_cap(1, E, k) == 8 * 256
    # the two scale sets in the tensor-core layout, then a 256-byte slot for the format word
    # both scale layouts, then the UE8M0 weight-row factors (FP32 per row of w13 and w2), then the format word
    factors = -(-(4 * E * (2 * I + H)) // 256) * 256
    assert m.prepared_weights_size(E, H, I) == E * 11 * 44 * 512 + E * 22 * 12 * 512 + factors + 256
    assert m.quantize_workspace_size(4096, 8, 128) > 0
    assert m.moe_workspace_size(-1, H, I, E, k) == 0


def test_argument_errors_need_no_gpu(lib):
    import nvfp4_w4a4_moe_gb300 as m
    P = ctypes.c_void_p
    # null weights struct
    rc = lib.nvfp4_moe_forward(None, None, None, 4, None, None, 8, None, None, 0, 0, None)
    assert rc == m.ERR_INVALID_ARG
    # unsupported shapes
    w = m._Weights(128, 2816 + 64, 704, *([P(256)] * 10))
    rc = lib.nvfp4_moe_forward(ctypes.byref(w), P(256), P(256), 1, P(256), P(256), 8, P(256), P(256), 1 << 30, 0, None)
    assert rc == m.ERR_UNSUPPORTED_SHAPE
    assert b"256" in lib.nvfp4_last_error_string()
    w = m._Weights(128, 2816, 700, *([P(256)] * 10))
    rc = lib.nvfp4_moe_forward(ctypes.byref(w), P(256), P(256), 1, P(256), P(256), 8, P(256), P(256), 1 << 30, 0, None)
    assert rc == m.ERR_UNSUPPORTED_SHAPE
    w = m._Weights(2000, 2816, 704, *([P(256)] * 10))
    rc = lib.nvfp4_moe_forward(ctypes.byref(w), P(256), P(256), 1, P(256), P(256), 8, P(256), P(256), 1 << 30, 0, None)
    assert rc == m.ERR_UNSUPPORTED_SHAPE
    # workspace too small
    w = m._Weights(128, 2816, 704, *([P(256)] * 10))
    rc = lib.nvfp4_moe_forward(ctypes.byref(w), P(256), P(256), 64, P(256), P(256), 8, P(256), P(256), 1024, 0, None)
    assert rc == m.ERR_WORKSPACE_TOO_SMALL
    # misaligned workspace
    rc = lib.nvfp4_moe_forward(ctypes.byref(w), P(256), P(256), 64, P(256), P(256), 8, P(256), P(264), 1 << 40, 0, None)
    assert rc == m.ERR_INVALID_ARG
    # quantiser: unknown scale layout, H not a multiple of 64
    rc = lib.nvfp4_quantize_experts(P(256), 4, 256, P(256), 2, 4, P(256), P(256), P(256), 7, P(256), P(256), P(256),
                                    1 << 20, None)
    assert rc == m.ERR_INVALID_ARG
    rc = lib.nvfp4_quantize_experts(P(256), 4, 100, P(256), 2, 4, P(256), P(256), P(256), 0, P(256), P(256), P(256),
                                    1 << 20, None)
    assert rc == m.ERR_UNSUPPORTED_SHAPE
    # validate: null result pointers
    rc = lib.nvfp4_validate_scales(P(256), None, 4, P(256), None, None, None)
    assert rc == m.ERR_INVALID_ARG
    # router: k outside [1, min(32, E)], E outside [1, 1024], unknown dtype, null or misaligned logits
    for E, k, dt in ((128, 0, 0), (128, 33, 0), (4, 8, 0), (1025, 8, 0), (0, 1, 0), (128, 8, 2)):
        assert lib.nvfp4_router_topk(P(256), dt, 1, E, k, P(256), P(256), None) == m.ERR_INVALID_ARG, (E, k, dt)
    assert lib.nvfp4_router_topk(None, 0, 1, 128, 8, P(256), P(256), None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_router_topk(P(258), 0, 1, 128, 8, P(256), P(256), None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_router_topk(None, 0, 0, 128, 8, None, None, None) == m.OK  # T = 0 launches nothing


def test_w4a16_and_format_argument_errors_need_no_gpu(lib):
    import nvfp4_w4a4_moe_gb300 as m
    P = ctypes.c_void_p
    H, I, E, k = 2816, 704, 128, 8
    # sizes: the prepared scales are as many bytes as the weights' scales, rearranged
    assert m.load().nvfp4_w4a16_prepared_size(E, H, I) == E * 2 * I * (H // 16) + E * H * (I // 16)
    assert m.load().nvfp4_w4a16_prepared_size(E, H, 700) == 0
    n = m.moe_w4a16_workspace_size(64, H, I, E, k)
    assert n % 256 == 0 and n >= 64 * k * H * 2  # holds at least the gathered BF16 rows
    assert m.moe_w4a16_workspace_size(-1, H, I, E, k) == 0
    # forward: null weights, unsupported shape, workspace too small, misaligned output
    assert lib.nvfp4_moe_forward_w4a16(None, P(256), P(256), 4, P(256), P(256), k, P(256), P(256), 1 << 30, 0,
                                       None) == m.ERR_INVALID_ARG
    w = m._Weights(E, H, 700, *([P(256)] * 10))
    assert lib.nvfp4_moe_forward_w4a16(ctypes.byref(w), P(256), P(256), 4, P(256), P(256), k, P(256), P(256),
                                       1 << 30, 0, None) == m.ERR_UNSUPPORTED_SHAPE
    w = m._Weights(E, H, I, *([P(256)] * 10))
    assert lib.nvfp4_moe_forward_w4a16(ctypes.byref(w), P(256), P(256), 64, P(256), P(256), k, P(256), P(256),
                                       1024, 0, None) == m.ERR_WORKSPACE_TOO_SMALL
    assert lib.nvfp4_moe_forward_w4a16(ctypes.byref(w), P(256), P(256), 64, P(256), P(256), k, P(264), P(256),
                                       1 << 40, 0, None) == m.ERR_INVALID_ARG
    # input scales may be null on this path; weight scales may not
    w = m._Weights(E, H, I, P(256), P(256), P(256), None, None, P(256), P(256), P(256), None, None)
    assert lib.nvfp4_moe_forward_w4a16(ctypes.byref(w), P(256), P(256), 0, P(256), P(256), k, P(256), P(256),
                                       1 << 30, 0, None) == m.OK  # T = 0 launches nothing
    w = m._Weights(E, H, I, P(256), P(256), None, None, None, P(256), P(256), P(256), None, None)
    assert lib.nvfp4_moe_forward_w4a16(ctypes.byref(w), P(256), P(256), 0, P(256), P(256), k, P(256), P(256),
                                       1 << 30, 0, None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_prepare_weights_w4a16(None, P(256), 1 << 30, None) == m.ERR_INVALID_ARG
    # weight quantiser: unknown scale format
    assert lib.nvfp4_quantize_weights_format(P(256), 1, 64, 64, 3, P(256), P(256), P(256), P(256), 1 << 20,
                                             None) == m.ERR_INVALID_ARG
    # activation quantiser: a layout with an unknown bit
    assert lib.nvfp4_quantize_experts(P(256), 4, 256, P(256), 2, 4, P(256), P(256), P(256), 2 | m.SF_UE8M0,
                                      P(256), P(256), P(256), 1 << 20, None) == m.ERR_INVALID_ARG
    # weight preparation: unknown scale format; the W4A16 path refuses the UE8M0 variant
    assert lib.nvfp4_prepare_weights_format(None, P(256), 1 << 30, 3, None) == m.ERR_INVALID_ARG
    assert b"format" in lib.nvfp4_last_error_string()
    w = m._Weights(E, H, I, *([P(256)] * 10))
    assert lib.nvfp4_moe_forward_w4a16(ctypes.byref(w), P(256), P(256), 0, P(256), P(256), k, P(256), P(256),
                                       1 << 30, m.UE8M0_SCALES, None) == m.ERR_INVALID_ARG
    assert b"UE8M0" in lib.nvfp4_last_error_string()
    # the device-wait self-test: bad workspace or limit
    assert lib.nvfp4_selftest_device_wait(None, 256, 1000, None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_selftest_device_wait(P(264), 256, 1000, None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_selftest_device_wait(P(256), 128, 1000, None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_selftest_device_wait(P(256), 256, 0, None) == m.ERR_INVALID_ARG
    assert lib.nvfp4_selftest_device_wait(P(256), 256, 2000000, None) == m.ERR_INVALID_ARG


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    import nvfp4_w4a4_moe_gb300 as m
    monkeypatch.setattr(m, "_lib", None)
    monkeypatch.setattr(m, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(m.Nvfp4Error):
        m.load()


def test_static_scratch_refuses_shapes_like_the_workspace_entry_point(lib):
    """The entry point without a workspace applies the workspace entry point's
    shape checks first, so a shape that one refuses is refused by both with the
    same status.  Every case returns before any CUDA call (no GPU needed)."""
    import nvfp4_w4a4_moe_gb300 as m
    null = ctypes.c_void_p(0)
    cases = [  # (T, H, k, E)
        (4, 256, 2, 1025),     # E above 1024
        (4, 256, 33, 64),      # k above 32
        (4, 256, 5, 4),        # k above E
        (-1, 256, 2, 4),       # negative T
        (4, 100, 2, 4),        # H not a multiple of 64
        (2 ** 30, 256, 8, 128),  # T * k overflows an int
    ]
    for T, H, k, E in cases:
        rc_ws = lib.nvfp4_quantize_experts(null, T, H, null, k, E, null, null, null, 0, null, null, null,
                                           ctypes.c_size_t(0), null)
        rc_st = lib.nvfp4_quantize_experts_static_scratch(null, T, H, null, k, E, null, null, null, 0, null, null,
                                                          null)
        assert rc_ws == m.ERR_UNSUPPORTED_SHAPE, (T, H, k, E, rc_ws)
        assert rc_st == rc_ws, (T, H, k, E, rc_st)
    assert lib.nvfp4_quantize_workspace_size(2 ** 30, 8, 128) == 0
    assert lib.nvfp4_moe_workspace_size(2 ** 30, 2816, 704, 128, 8) == 0
