"""CPU oracle for the mHC hot path: ctypes wrapper around ``mhc_oracle.c``.

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
``cpu_baseline`` leg are the only callers.  The product path (the CUDA library
and its Python binding) never imports this package, and this package imports
nothing from the product.  Inputs and outputs are numpy arrays: bf16 tensors
travel as ``uint16`` bit patterns, everything else as float32/float64.

Every function here is a thin marshalling layer; the arithmetic lives in
``mhc_oracle.c`` and follows deepseek_v4.py (sglang),
DeepseekV4DecoderLayer.hc_pre / hc_post and hc_head_torch, as its header
states.  Pins: tests/test_oracle_pins.py checks every function below against
closed forms, invariants and brute force on tiny inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HC, H, K, MIX = 4, 5120, 20480, 24

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mhc_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libmhc_oracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_F = ctypes.POINTER(ctypes.c_float)
_U16 = ctypes.POINTER(ctypes.c_uint16)
_U8 = ctypes.POINTER(ctypes.c_uint8)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call([
            "gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", _SRC, "-o", tmp, "-lm",
        ])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, c_int = ctypes.c_int64, ctypes.c_int
            dbl = ctypes.c_double
            lib.oracle_double_to_bf16.argtypes = [dbl]
            lib.oracle_double_to_bf16.restype = ctypes.c_uint16
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = dbl
            lib.oracle_stats.argtypes = [_U16, i64, _F, dbl, _D, _D]
            lib.oracle_split_sinkhorn.argtypes = [_D, i64, _F, _F, dbl, dbl, dbl, c_int,
                                                  _D, _D, _D, _D]
            lib.oracle_combine_norm.argtypes = [_U16, i64, _D, _U16, dbl, c_int, _U16]
            lib.oracle_post.argtypes = [_U16, _U16, _F, _F, i64, _U16]
            lib.oracle_pre.argtypes = [_U16, i64, _F, _F, _F, _U16, dbl, dbl, dbl, dbl, dbl,
                                       c_int, _D, _D, _D, _D, _D, _U16]
            lib.oracle_hc_head.argtypes = [_U16, i64, _F, _F, _F, dbl, dbl, _D, _D, _U16]
            lib.oracle_mxfp8_quantize.argtypes = [_U16, i64, i64, _U8, _U8]
            lib.oracle_swizzle_128x4.argtypes = [_U8, i64, i64, _U8]
            for f in ("oracle_stats", "oracle_split_sinkhorn", "oracle_combine_norm",
                      "oracle_post", "oracle_pre", "oracle_hc_head", "oracle_mxfp8_quantize",
                      "oracle_swizzle_128x4"):
                getattr(lib, f).restype = None
            _lib = lib
    return _lib


def _p(a, ptype):
    return None if a is None else a.ctypes.data_as(ptype)


def _u16(a, shape_tail):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected uint16 bf16 bits, got {a.dtype}")
    if tuple(a.shape[1:]) != tuple(shape_tail):
        raise ValueError(f"expected [rows, {shape_tail}], got {a.shape}")
    return a


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


# ---------------------------------------------------------------------------
def to_bf16(x) -> np.ndarray:
    """Round float64 values to bf16 bits, nearest-even, in one step."""
    lib = _load()
    x = np.asarray(x, dtype=np.float64)
    f = np.vectorize(lib.oracle_double_to_bf16, otypes=[np.uint16])
    return f(x).astype(np.uint16) if x.size else np.zeros(x.shape, np.uint16)


def from_bf16(b) -> np.ndarray:
    """bf16 bits -> float64 (exact)."""
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def stats(R, fn, rms_eps):
    """a1: (mix [rows,24], rsqrt [rows]) in float64."""
    R = _u16(R, (HC, H))
    fn = _f32(fn).reshape(MIX, K)
    rows = R.shape[0]
    mix = np.zeros((rows, MIX), np.float64)
    rsq = np.zeros((rows,), np.float64)
    _load().oracle_stats(_p(R, _U16), rows, _p(fn, _F), float(rms_eps), _p(mix, _D), _p(rsq, _D))
    return mix, rsq


def split_sinkhorn(mix, scale, base, pre_eps, sink_eps, post_mult, iters):
    """a2 + a3: dict of logits [rows,24], pre [rows,4], post [rows,4], comb [rows,4,4]."""
    mix = _f64(mix).reshape(-1, MIX)
    rows = mix.shape[0]
    out = {k: np.zeros(s, np.float64) for k, s in
           (("logits", (rows, MIX)), ("pre", (rows, HC)), ("post", (rows, HC)),
            ("comb", (rows, HC, HC)))}
    _load().oracle_split_sinkhorn(
        _p(mix, _D), rows, _p(_f32(scale), _F), _p(_f32(base), _F), float(pre_eps),
        float(sink_eps), float(post_mult), int(iters), _p(out["logits"], _D),
        _p(out["pre"], _D), _p(out["post"], _D), _p(out["comb"], _D))
    return out


def combine_norm(R, pre, w, norm_eps, round_y=False):
    """a4: x_norm [rows, 5120] bf16 bits."""
    R = _u16(R, (HC, H))
    pre = _f64(pre).reshape(-1, HC)
    w = _u16(np.asarray(w, np.uint16).reshape(1, H), (H,))
    rows = R.shape[0]
    out = np.zeros((rows, H), np.uint16)
    _load().oracle_combine_norm(_p(R, _U16), rows, _p(pre, _D), _p(w, _U16), float(norm_eps),
                                int(bool(round_y)), _p(out, _U16))
    return out


def post(R, y, post_w, comb):
    """a5: R_out [rows, 4, 5120] bf16 bits; post_w [rows,4] and comb [rows,4,4] as fp32."""
    R = _u16(R, (HC, H))
    y = _u16(y, (H,))
    rows = R.shape[0]
    pw = _f32(post_w).reshape(rows, HC)
    cb = _f32(comb).reshape(rows, HC, HC)
    out = np.zeros((rows, HC, H), np.uint16)
    _load().oracle_post(_p(R, _U16), _p(y, _U16), _p(pw, _F), _p(cb, _F), rows, _p(out, _U16))
    return out


def pre(R, fn, scale, base, w, *, rms_eps=1e-6, hc_pre_eps=1e-6, hc_sinkhorn_eps=1e-6,
        norm_eps=1e-6, post_mult=2.0, iters=20, want_x_norm=True):
    """a1..a4 for every row of R: dict of mix, logits, pre, post, comb (float64) and
    x_norm (bf16 bits, if asked)."""
    R = _u16(R, (HC, H))
    rows = R.shape[0]
    out = {k: np.zeros(s, np.float64) for k, s in
           (("mix", (rows, MIX)), ("logits", (rows, MIX)), ("pre", (rows, HC)),
            ("post", (rows, HC)), ("comb", (rows, HC, HC)))}
    out["x_norm"] = np.zeros((rows, H), np.uint16) if want_x_norm else None
    w = np.asarray(w, np.uint16).reshape(H)
    _load().oracle_pre(
        _p(R, _U16), rows, _p(_f32(fn).reshape(MIX, K), _F), _p(_f32(scale), _F),
        _p(_f32(base), _F), _p(np.ascontiguousarray(w), _U16), float(rms_eps),
        float(hc_pre_eps), float(hc_sinkhorn_eps), float(norm_eps), float(post_mult),
        int(iters), _p(out["mix"], _D), _p(out["logits"], _D), _p(out["pre"], _D),
        _p(out["post"], _D), _p(out["comb"], _D), _p(out["x_norm"], _U16))
    return out


def hc_head(R, fn, scale, base, *, norm_eps=1e-6, hc_eps=1e-6):
    """The final stream collapse (deepseek_v4.py, hc_head_torch): dict of mix
    [rows,4], pre [rows,4] (float64) and y [rows,5120] (bf16 bits)."""
    R = _u16(R, (HC, H))
    rows = R.shape[0]
    out = {"mix": np.zeros((rows, HC), np.float64), "pre": np.zeros((rows, HC), np.float64),
           "y": np.zeros((rows, H), np.uint16)}
    _load().oracle_hc_head(
        _p(R, _U16), rows, _p(_f32(fn).reshape(HC, K), _F), _p(_f32(scale).reshape(1), _F),
        _p(_f32(base).reshape(HC), _F), float(norm_eps), float(hc_eps), _p(out["mix"], _D),
        _p(out["pre"], _D), _p(out["y"], _U16))
    return out


def fused_post_pre(R, y, post_w, comb, fn, scale, base, w, **pre_kw):
    """hc_post of one sublayer followed by hc_pre of the next on its result
    (deepseek_v4.py, the fused post->pre path between sublayers): the
    definition is the plain composition, R' rounded to bf16 in between.
    Returns (R' bf16 bits, the pre dict of R')."""
    R2 = post(R, y, post_w, comb)
    return R2, pre(R2, fn, scale, base, w, **pre_kw)


def mxfp8_quantize(x):
    """MXFP8 of bf16 rows (prefill_sp.py, _mxfp8_quantize: per row, per 32
    columns, linear scale layout): x [rows, cols] bf16 bits, cols a multiple
    of 32 -> (q [rows, cols] uint8 E4M3 codes, s [rows, cols/32] uint8 ue8m0
    scales)."""
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16 or x.ndim != 2 or x.shape[1] % 32:
        raise ValueError("expected [rows, cols] uint16 bf16 bits with cols % 32 == 0")
    rows, cols = x.shape
    q = np.zeros((rows, cols), np.uint8)
    s = np.zeros((rows, cols // 32), np.uint8)
    _load().oracle_mxfp8_quantize(_p(x, _U16), rows, cols, _p(q, _U8), _p(s, _U8))
    return q, s


def swizzle_128x4(s):
    """The 128x4 tiled layout of linear ue8m0 scales (prefill_sp.py,
    swizzle_128x4): s [rows, groups] uint8, groups a multiple of 4 -> a flat
    uint8 array of ceil(rows/128)*128*groups bytes (padding rows zero)."""
    s = np.ascontiguousarray(s, dtype=np.uint8)
    if s.ndim != 2 or s.shape[1] % 4:
        raise ValueError("expected [rows, groups] with groups % 4 == 0")
    rows, groups = s.shape
    out = np.zeros(((rows + 127) // 128 * 128 * groups,), np.uint8)
    _load().oracle_swizzle_128x4(_p(s, _U8), rows, groups, _p(out, _U8))
    return out
