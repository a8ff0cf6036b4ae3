"""Host-side checks of the C ABI that need no GPU: the library builds, loads and
exports every function include/*.h declares, and argument validation rejects
bad calls before any CUDA call.

Every call below carries at least one defect that the host checks catch, so no
call ever reaches a kernel launch (the pointers are fake addresses and are
never dereferenced).
"""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_PARAM, ERR_OVERLAP, ERR_WORKSPACE = -1, -2, -3, -4, -5, -6
K, H = 20480, 5120


@pytest.fixture(scope="module")
def lib():
    from hyper_connection_residual_mhc_gb300 import build
    build.build()
    import hyper_connection_residual_mhc_gb300 as m
    return m.lib()


def declared_functions():
    names = set()
    for hdr in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(hdr).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(mhc_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("mhc_pre", "mhc_post", "mhc_combine_norm", "mhc_pre_workspace_bytes",
              "mhc_default_params", "mhc_strerror", "mhc_last_cuda_error"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_signatures_cover_the_header():
    import hyper_connection_residual_mhc_gb300 as m
    assert set(declared_functions()) <= set(m.SIGNATURES)


def test_strerror_and_defaults(lib):
    import hyper_connection_residual_mhc_gb300 as m
    for code in range(0, -9, -1):
        assert lib.mhc_strerror(code)
    p = m.default_params()
    assert p.sinkhorn_iters == 20 and p.post_mult == 2.0
    assert abs(p.rms_eps - 1e-6) < 1e-12 and abs(p.norm_eps - 1e-6) < 1e-12
    assert lib.mhc_pre_workspace_bytes(0) == 0
    # the larger of fn's operand image (16 ranks x 5 blocks x 192 x 64 bf16,
    # for mhc_pre's streamed build) and the fused call's hand-off: the pre
    # gates [rows, 4] then the comb logits [rows, 16], fp32, each 256-byte
    # rounded
    img = 16 * 5 * 192 * 64 * 2
    assert lib.mhc_pre_workspace_bytes(1) == img
    assert lib.mhc_pre_workspace_bytes(1000) == img
    assert lib.mhc_pre_workspace_bytes(24576) == img          # hand-off 1966080 too
    assert lib.mhc_pre_workspace_bytes(30001) == 480256 + 1920256


A = 1 << 32          # fake, 256-byte aligned device addresses, far apart
BIG = 1 << 34


def fake(i):
    return A + i * BIG


def call_post(lib, R=fake(0), y=fake(1), post=fake(2), comb=fake(3), rows=4, logical=4,
              out=fake(4)):
    return lib.mhc_post(R, y, post, comb, rows, logical, out, None)


def call_pre(lib, rows=4, logical=4, params=None, ws=fake(9), ws_bytes=None, **over):
    import hyper_connection_residual_mhc_gb300 as m
    a = dict(R=fake(0), fn=fake(1), scale=fake(2), base=fake(3), w=fake(4), xn=fake(5),
             post=fake(6), comb=fake(7), pre=None, mix=None)
    a.update(over)
    p = m.default_params() if params is None else params
    wsb = lib.mhc_pre_workspace_bytes(rows) if ws_bytes is None else ws_bytes
    return lib.mhc_pre(a["R"], a["fn"], a["scale"], a["base"], a["w"], rows, logical,
                       ctypes.byref(p), ws, wsb, a["xn"], a["post"], a["comb"], a["pre"],
                       a["mix"], None)


def test_post_validation(lib):
    assert call_post(lib, rows=-1) == ERR_SHAPE
    assert call_post(lib, rows=8, logical=4) == ERR_SHAPE
    assert call_post(lib, R=None) == ERR_NULL
    assert call_post(lib, out=None) == ERR_NULL
    assert call_post(lib, y=fake(1) + 8) == ERR_ALIGN
    assert call_post(lib, out=fake(0) + 4 * K * 2 - 16) == ERR_OVERLAP     # tail overlaps R
    assert call_post(lib, out=fake(1)) == ERR_OVERLAP


def test_post_zero_rows_is_a_no_op(lib):
    assert call_post(lib, rows=0, logical=0, R=None, out=None) == 0


def test_pre_validation(lib):
    import hyper_connection_residual_mhc_gb300 as m
    assert call_pre(lib, rows=-3) == ERR_SHAPE
    assert call_pre(lib, rows=5, logical=4) == ERR_SHAPE
    assert call_pre(lib, params=m.default_params(sinkhorn_iters=0)) == ERR_PARAM
    assert call_pre(lib, params=m.default_params(norm_eps=-1.0)) == ERR_PARAM
    assert call_pre(lib, params=m.default_params(rms_eps=float("nan"))) == ERR_PARAM
    assert call_pre(lib, fn=None) == ERR_NULL
    assert call_pre(lib, comb=fake(7) + 4) == ERR_ALIGN
    assert call_pre(lib, mix=fake(8) + 4) == ERR_ALIGN
    assert call_pre(lib, ws=None) == ERR_WORKSPACE
    assert call_pre(lib, ws_bytes=16) == ERR_WORKSPACE
    assert call_pre(lib, ws=fake(9) + 16) == ERR_WORKSPACE                # not 256-byte aligned
    assert call_pre(lib, ws=fake(5)) == ERR_OVERLAP                         # workspace on x_norm
    assert call_pre(lib, xn=fake(0)) == ERR_OVERLAP                         # x_norm on R
    assert call_pre(lib, post=fake(7)) == ERR_OVERLAP                       # post on comb


def call_noalloc(lib, rows=4, logical=4, params=None, **over):
    import hyper_connection_residual_mhc_gb300 as m
    a = dict(R=fake(0), fn=fake(1), scale=fake(2), base=fake(3), w=fake(4), xn=fake(5),
             post=fake(6), comb=fake(7), pre=None, mix=None)
    a.update(over)
    p = m.default_params() if params is None else params
    return lib.mhc_pre_noalloc(a["R"], a["fn"], a["scale"], a["base"], a["w"], rows, logical,
                               ctypes.byref(p), a["xn"], a["post"], a["comb"], a["pre"],
                               a["mix"], None)


def test_noalloc_validation_matches_mhc_pre(lib):
    # the same checks as mhc_pre, minus the workspace; the row limit is the
    # library-wide one
    import hyper_connection_residual_mhc_gb300 as m
    assert lib.mhc_pre_noalloc_max_rows() == 1 << 24
    big = (1 << 24) + 1
    assert call_noalloc(lib, rows=big, logical=big) == ERR_SHAPE
    assert call_pre(lib, rows=big, logical=big) == ERR_SHAPE
    assert call_noalloc(lib, rows=-3) == ERR_SHAPE
    assert call_noalloc(lib, rows=5, logical=4) == ERR_SHAPE
    assert call_noalloc(lib, params=m.default_params(sinkhorn_iters=0)) == ERR_PARAM
    assert call_noalloc(lib, fn=None) == ERR_NULL
    assert call_noalloc(lib, comb=fake(7) + 4) == ERR_ALIGN
    assert call_noalloc(lib, xn=fake(0)) == ERR_OVERLAP
    assert call_noalloc(lib, post=fake(7)) == ERR_OVERLAP
    assert call_noalloc(lib, rows=0, logical=0, R=None) == 0


def test_combine_norm_validation(lib):
    f = lib.mhc_combine_norm
    assert f(fake(0), fake(1), fake(2), ctypes.c_float(-1.0), 4, 4, fake(3), None) == ERR_PARAM
    assert f(fake(0), None, fake(2), ctypes.c_float(1e-6), 4, 4, fake(3), None) == ERR_NULL
    assert f(fake(0), fake(1), fake(2), ctypes.c_float(1e-6), 4, 2, fake(3), None) == ERR_SHAPE
    assert f(fake(0), fake(1), fake(2), ctypes.c_float(1e-6), 4, 4, fake(0), None) == ERR_OVERLAP


def call_head(lib, rows=4, logical=4, ws=fake(9), ws_bytes=None, norm_eps=1e-6, hc_eps=1e-6,
              **over):
    a = dict(R=fake(0), fn=fake(1), scale=fake(2), base=fake(3), y=fake(5), pre=None, mix=None)
    a.update(over)
    wsb = lib.mhc_pre_workspace_bytes(rows) if ws_bytes is None else ws_bytes
    return lib.mhc_hc_head(a["R"], a["fn"], a["scale"], a["base"], rows, logical,
                           ctypes.c_float(norm_eps), ctypes.c_float(hc_eps), ws, wsb, a["y"],
                           a["pre"], a["mix"], None)


def test_hc_head_validation(lib):
    assert call_head(lib, rows=-1) == ERR_SHAPE
    assert call_head(lib, rows=5, logical=4) == ERR_SHAPE
    assert call_head(lib, norm_eps=-1.0) == ERR_PARAM
    assert call_head(lib, hc_eps=float("inf")) == ERR_PARAM
    assert call_head(lib, rows=0, logical=0, R=None) == 0
    assert call_head(lib, base=None) == ERR_NULL
    assert call_head(lib, y=fake(5) + 2) == ERR_ALIGN
    assert call_head(lib, pre=fake(6) + 4) == ERR_ALIGN
    assert call_head(lib, ws=None) == ERR_WORKSPACE
    assert call_head(lib, ws_bytes=8) == ERR_WORKSPACE
    assert call_head(lib, y=fake(0)) == ERR_OVERLAP                       # y on R
    assert call_head(lib, ws=fake(5)) == ERR_OVERLAP                      # workspace on y
    assert call_head(lib, pre=fake(6), mix=fake(6)) == ERR_OVERLAP        # two outputs


def call_fpp(lib, rows=4, logical=4, ws=fake(20), ws_bytes=None, **over):
    import hyper_connection_residual_mhc_gb300 as m
    a = dict(R=fake(0), y=fake(1), post=fake(2), comb=fake(3), fn=fake(4), scale=fake(5),
             base=fake(6), w=fake(7), R_out=fake(8), xn=fake(9), post_out=fake(10),
             comb_out=fake(11), pre=None, mix=None)
    a.update(over)
    p = m.default_params()
    wsb = lib.mhc_fused_post_pre_workspace_bytes(rows) if ws_bytes is None else ws_bytes
    return lib.mhc_fused_post_pre(a["R"], a["y"], a["post"], a["comb"], a["fn"], a["scale"],
                                  a["base"], a["w"], rows, logical, ctypes.byref(p), ws, wsb,
                                  a["R_out"], a["xn"], a["post_out"], a["comb_out"], a["pre"],
                                  a["mix"], None)


def test_fused_post_pre_validation(lib):
    assert call_fpp(lib, rows=-1) == ERR_SHAPE
    assert call_fpp(lib, rows=0, logical=0, R=None) == 0
    assert call_fpp(lib, y=None) == ERR_NULL
    assert call_fpp(lib, comb_out=fake(11) + 4) == ERR_ALIGN
    assert call_fpp(lib, ws=None) == ERR_WORKSPACE
    assert call_fpp(lib, ws_bytes=lib.mhc_pre_workspace_bytes(4)) == ERR_WORKSPACE   # no fn image room
    assert (lib.mhc_fused_post_pre_workspace_bytes(4)
            == lib.mhc_pre_workspace_bytes(4) + 640 * 48 * 64)
    assert call_fpp(lib, post_out=fake(2)) == ERR_OVERLAP      # next post on this post
    assert call_fpp(lib, R_out=fake(0)) == ERR_OVERLAP         # in-place residual
    assert call_fpp(lib, xn=fake(8)) == ERR_OVERLAP            # two outputs
    assert call_fpp(lib, ws=fake(1)) == ERR_OVERLAP            # workspace on y


def test_prepared_weights_host_checks(lib):
    import hyper_connection_residual_mhc_gb300 as m
    h = ctypes.c_void_p(123)
    assert lib.mhc_prepare_weights(None, ctypes.byref(h), None) == ERR_NULL
    assert lib.mhc_prepare_weights(fake(1), None, None) == ERR_NULL
    assert lib.mhc_prepare_weights(fake(1) + 4, ctypes.byref(h), None) == ERR_ALIGN
    assert h.value is None                      # *out is cleared once fn and out are given
    assert lib.mhc_release_weights(None) == 0   # like free(NULL)
    p = m.default_params()
    assert lib.mhc_pre_prepared(fake(0), None, fake(2), fake(3), fake(4), 4, 4, ctypes.byref(p),
                                fake(9), lib.mhc_pre_workspace_bytes(4), fake(5), fake(6), fake(7),
                                None, None, None) == ERR_NULL
    assert b"allocation" in lib.mhc_strerror(-10)


def test_fused_prepared_null_handle(lib):
    import hyper_connection_residual_mhc_gb300 as m
    p = m.default_params()
    assert lib.mhc_fused_post_pre_prepared(
        fake(0), fake(1), fake(2), fake(3), None, fake(5), fake(6), fake(7), 4, 4,
        ctypes.byref(p), fake(9), lib.mhc_pre_workspace_bytes(4), fake(10), fake(11), fake(12),
        fake(13), None, None, None) == ERR_NULL


def test_mxfp8_host_checks(lib):
    import hyper_connection_residual_mhc_gb300 as m
    p = m.default_params()
    # pre: a NULL handle, then (through the shared checks) NULL codes
    assert lib.mhc_pre_mxfp8(fake(0), None, fake(2), fake(3), fake(4), 4, 4, ctypes.byref(p),
                             fake(9), lib.mhc_pre_workspace_bytes(4), fake(5), fake(10),
                             fake(11), fake(6), fake(7), None) == ERR_NULL
    q = lib.mhc_quantize_mxfp8
    assert q(fake(0), 4, 48, 4, fake(1), fake(2), None) == ERR_SHAPE          # cols % 32
    assert q(fake(0), 4, 0, 4, fake(1), fake(2), None) == ERR_SHAPE
    assert q(fake(0), 4, 1 << 17, 4, fake(1), fake(2), None) == ERR_SHAPE     # too wide
    assert q(fake(0), 4, 64, 2, fake(1), fake(2), None) == ERR_SHAPE          # logical < rows
    assert q(fake(0), 0, 64, 0, None, None, None) == 0                        # empty: no launch
    assert q(None, 4, 64, 4, fake(1), fake(2), None) == ERR_NULL
    assert q(fake(0), 4, 64, 4, fake(1) + 8, fake(2), None) == ERR_ALIGN
    assert q(fake(0), 4, 64, 4, fake(0) + 256, fake(2), None) == ERR_OVERLAP  # codes on x
    assert q(fake(0), 4, 64, 4, fake(1), fake(1) + 128, None) == ERR_OVERLAP  # scales on codes
    sw = lib.mhc_swizzle_scales_128x4
    assert lib.mhc_swizzle_scales_128x4_bytes(1, 160) == 128 * 160
    assert lib.mhc_swizzle_scales_128x4_bytes(129, 8) == 256 * 8
    assert lib.mhc_swizzle_scales_128x4_bytes(0, 8) == 0
    assert sw(fake(0), 4, 6, fake(1), None) == ERR_SHAPE                      # groups % 4
    assert sw(fake(0), -1, 8, fake(1), None) == ERR_SHAPE
    assert sw(fake(0), 0, 8, None, None) == 0
    assert sw(None, 4, 8, fake(1), None) == ERR_NULL
    assert sw(fake(0) + 4, 4, 8, fake(1), None) == ERR_ALIGN
    assert sw(fake(0), 4, 8, fake(0) + 16, None) == ERR_OVERLAP
