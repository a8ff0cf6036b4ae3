"""Python binding of libmhc (GB300 / sm_103a hyper-connection kernels).

Argument marshalling only: every step of the hot path runs in libmhc's CUDA
kernels.  Functions carry the C entry points' names (include/mhc.h) and take
torch CUDA tensors; torch provides device memory and the current stream.
Outputs the caller does not pass are allocated with torch.empty.

If ``_build/libmhc.so`` is missing, every call raises: there is no fallback.
Build it with ``python -m hyper_connection_residual_mhc_gb300.build`` (or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
import threading

HC, H, K, MIX = 4, 5120, 20480, 24

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libmhc.so")

MHC_OK = 0


class MhcParams(ctypes.Structure):
    """Mirror of ``mhc_params`` (include/mhc.h)."""
    _fields_ = [("rms_eps", ctypes.c_float), ("hc_pre_eps", ctypes.c_float),
                ("hc_sinkhorn_eps", ctypes.c_float), ("norm_eps", ctypes.c_float),
                ("post_mult", ctypes.c_float), ("sinkhorn_iters", ctypes.c_int32)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class MhcError(RuntimeError):
    def __init__(self, fn, code, text):
        super().__init__(f"{fn} failed with {code}: {text}")
        self.code = code


_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64

# name -> (restype, argtypes); keep in step with include/mhc.h
SIGNATURES = {
    "mhc_default_params": (None, [ctypes.POINTER(MhcParams)]),
    "mhc_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "mhc_last_cuda_error": (ctypes.c_char_p, []),
    "mhc_pre_workspace_bytes": (ctypes.c_size_t, [_i64]),
    "mhc_kernel_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]),
    "mhc_kernel_status_detail": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32)]),
    "mhc_pre": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, ctypes.POINTER(MhcParams),
                               _vp, ctypes.c_size_t, _vp, _vp, _vp, _vp, _vp, _vp]),
    "mhc_pre_noalloc": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64,
                                       ctypes.POINTER(MhcParams), _vp, _vp, _vp, _vp, _vp, _vp]),
    "mhc_pre_noalloc_max_rows": (ctypes.c_int64, []),
    "mhc_post": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i64, _i64, _vp, _vp]),
    "mhc_combine_norm": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_float, _i64, _i64, _vp, _vp]),
    "mhc_fused_post_pre": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64,
                                          ctypes.POINTER(MhcParams), _vp, ctypes.c_size_t, _vp,
                                          _vp, _vp, _vp, _vp, _vp, _vp]),
    "mhc_fused_post_pre_workspace_bytes": (ctypes.c_size_t, [_i64]),
    "mhc_hc_head": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i64, _i64, ctypes.c_float,
                                   ctypes.c_float, _vp, ctypes.c_size_t, _vp, _vp, _vp, _vp]),
    "mhc_prepare_weights": (ctypes.c_int, [_vp, ctypes.POINTER(_vp), _vp]),
    "mhc_release_weights": (ctypes.c_int, [_vp]),
    "mhc_pre_prepared": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64,
                                        ctypes.POINTER(MhcParams), _vp, ctypes.c_size_t, _vp,
                                        _vp, _vp, _vp, _vp, _vp]),
    "mhc_fused_post_pre_prepared": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64,
                                                   _i64, ctypes.POINTER(MhcParams), _vp,
                                                   ctypes.c_size_t, _vp, _vp, _vp, _vp, _vp, _vp,
                                                   _vp]),
    "mhc_pre_mxfp8": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64,
                                     ctypes.POINTER(MhcParams), _vp, ctypes.c_size_t, _vp, _vp,
                                     _vp, _vp, _vp, _vp]),
    "mhc_fused_post_pre_mxfp8": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64,
                                                _i64, ctypes.POINTER(MhcParams), _vp,
                                                ctypes.c_size_t, _vp, _vp, _vp, _vp, _vp, _vp,
                                                _vp]),
    "mhc_quantize_mxfp8": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _vp, _vp]),
    "mhc_swizzle_scales_128x4_bytes": (ctypes.c_size_t, [_i64, _i64]),
    "mhc_swizzle_scales_128x4": (ctypes.c_int, [_vp, _i64, _i64, _vp, _vp]),
}


def lib():
    """The loaded libmhc (ctypes.CDLL).  Raises if the library was not built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libmhc is not built ({LIB_PATH} missing); run "
                    "`python -m hyper_connection_residual_mhc_gb300.build`")
            l = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(l, name)
                f.restype, f.argtypes = res, args
            _lib = l
    return _lib


def default_params(**overrides) -> MhcParams:
    p = MhcParams()
    lib().mhc_default_params(ctypes.byref(p))
    for k, v in overrides.items():
        setattr(p, k, v)
    return p


def _check(fn, code):
    if code != MHC_OK:
        l = lib()
        text = l.mhc_strerror(code).decode()
        if code == -7:
            text += f" ({l.mhc_last_cuda_error().decode()})"
        raise MhcError(fn, code, text)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _need(t, name, dtype, shape):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return t


def mhc_kernel_status(reset: bool = False) -> int:
    """Device status word (0 = no kernel gave up a bounded wait); synchronous."""
    w = ctypes.c_uint32(0)
    _check("mhc_kernel_status", lib().mhc_kernel_status(ctypes.byref(w), int(bool(reset))))
    return int(w.value)


def mhc_kernel_status_detail() -> dict:
    """{"expired": {site: (tile, rank)}, "gave_up": {site: (tile, rank)}} of the
    fused pre kernel's bounded waits (diagnosis)."""
    arr = (ctypes.c_uint32 * 64)()
    _check("mhc_kernel_status_detail", lib().mhc_kernel_status_detail(arr))
    st = mhc_kernel_status()
    return {"expired": {s: (arr[s] >> 8, arr[s] & 0xFF) for s in range(16) if (st >> s) & 1},
            "gave_up": {s: (arr[32 + s] >> 8, arr[32 + s] & 0xFF) for s in range(16)
                        if (st >> (16 + s)) & 1}}


def mhc_pre_workspace_bytes(rows: int) -> int:
    return int(lib().mhc_pre_workspace_bytes(int(rows)))


def mhc_fused_post_pre_workspace_bytes(rows: int) -> int:
    return int(lib().mhc_fused_post_pre_workspace_bytes(int(rows)))


def mhc_pre(R, fn, scale, base, norm_w, *, logical_rows=None, params=None, workspace=None,
            x_norm=None, post=None, comb=None, pre_out=None, mix_out=None, stream=None):
    """Stats, split/Sinkhorn, combine + RMSNorm (see mhc_pre in include/mhc.h).

    Returns ``(x_norm [rows,5120] bf16, post [rows,4] f32, comb [rows,4,4] f32)``.
    """
    import torch
    _need(fn, "fn", torch.float32, (MIX, K))
    return _pre_call("mhc_pre", _ptr(fn), R, scale, base, norm_w, logical_rows, params, workspace,
                     x_norm, post, comb, pre_out, mix_out, stream)


def _pre_call(name, fn_arg, R, scale, base, norm_w, logical_rows, params, workspace, x_norm,
              post, comb, pre_out, mix_out, stream):
    import torch
    rows = int(R.shape[0])
    _need(R, "R", torch.bfloat16, (rows, HC, H))
    _need(scale, "scale", torch.float32, (3,))
    _need(base, "base", torch.float32, (MIX,))
    _need(norm_w, "norm_w", torch.bfloat16, (H,))
    dev = R.device
    x_norm = torch.empty((rows, H), dtype=torch.bfloat16, device=dev) if x_norm is None else x_norm
    post = torch.empty((rows, HC), dtype=torch.float32, device=dev) if post is None else post
    comb = torch.empty((rows, HC, HC), dtype=torch.float32, device=dev) if comb is None else comb
    _need(x_norm, "x_norm", torch.bfloat16, (rows, H))
    _need(post, "post", torch.float32, (rows, HC))
    _need(comb, "comb", torch.float32, (rows, HC, HC))
    if pre_out is not None:
        _need(pre_out, "pre_out", torch.float32, (rows, HC))
    if mix_out is not None:
        _need(mix_out, "mix_out", torch.float32, (rows, MIX))
    need = mhc_pre_workspace_bytes(rows)
    if workspace is None and need:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    p = default_params() if params is None else params
    code = getattr(lib(), name)(
        _ptr(R), fn_arg, _ptr(scale), _ptr(base), _ptr(norm_w), rows,
        rows if logical_rows is None else int(logical_rows), ctypes.byref(p),
        _ptr(workspace), ws_bytes, _ptr(x_norm), _ptr(post), _ptr(comb), _ptr(pre_out),
        _ptr(mix_out), _stream(stream))
    _check(name, code)
    return x_norm, post, comb


class Weights:
    """A prepared-weights handle (mhc_prepare_weights in include/mhc.h); freed by
    release() or when the object is collected."""

    def __init__(self, handle):
        self._h = handle

    @property
    def handle(self):
        if self._h is None:
            raise ValueError("the prepared weights were released")
        return self._h

    def release(self):
        if self._h is not None:
            h, self._h = self._h, None
            _check("mhc_release_weights", lib().mhc_release_weights(h))

    def __del__(self):
        try:
            self.release()
        except Exception:
            pass


def mhc_prepare_weights(fn, *, stream=None) -> Weights:
    """fn [24, 20480] f32 -> a handle holding fn's copy and the one-pass kernels
    operand image (see mhc_prepare_weights in include/mhc.h)."""
    import torch
    _need(fn, "fn", torch.float32, (MIX, K))
    h = ctypes.c_void_p()
    _check("mhc_prepare_weights", lib().mhc_prepare_weights(_ptr(fn), ctypes.byref(h),
                                                            _stream(stream)))
    return Weights(h.value)


def mhc_pre_prepared(R, weights, scale, base, norm_w, *, logical_rows=None, params=None,
                     workspace=None, x_norm=None, post=None, comb=None, pre_out=None,
                     mix_out=None, stream=None):
    """mhc_pre with fn from a prepared-weights handle (bit-identical to mhc_pre)."""
    return _pre_call("mhc_pre_prepared", weights.handle, R, scale, base, norm_w, logical_rows,
                     params, workspace, x_norm, post, comb, pre_out, mix_out, stream)


def mhc_pre_mxfp8(R, weights, scale, base, norm_w, *, logical_rows=None, params=None,
                  workspace=None, x_norm=None, x_q=None, x_s=None, post=None, comb=None,
                  stream=None):
    """mhc_pre_prepared that also writes x_norm's MXFP8 (see mhc_pre_mxfp8 in
    include/mhc.h). Returns ``(x_norm [rows,5120] bf16, x_q [rows,5120] uint8
    E4M3 codes, x_s [rows,160] uint8 ue8m0 scales, post, comb)``."""
    import torch
    rows = int(R.shape[0])
    _need(R, "R", torch.bfloat16, (rows, HC, H))
    _need(scale, "scale", torch.float32, (3,))
    _need(base, "base", torch.float32, (MIX,))
    _need(norm_w, "norm_w", torch.bfloat16, (H,))
    dev = R.device
    x_norm = torch.empty((rows, H), dtype=torch.bfloat16, device=dev) if x_norm is None else x_norm
    x_q = torch.empty((rows, H), dtype=torch.uint8, device=dev) if x_q is None else x_q
    x_s = torch.empty((rows, H // 32), dtype=torch.uint8, device=dev) if x_s is None else x_s
    post = torch.empty((rows, HC), dtype=torch.float32, device=dev) if post is None else post
    comb = torch.empty((rows, HC, HC), dtype=torch.float32, device=dev) if comb is None else comb
    _need(x_norm, "x_norm", torch.bfloat16, (rows, H))
    _need(x_q, "x_q", torch.uint8, (rows, H))
    _need(x_s, "x_s", torch.uint8, (rows, H // 32))
    _need(post, "post", torch.float32, (rows, HC))
    _need(comb, "comb", torch.float32, (rows, HC, HC))
    need = mhc_pre_workspace_bytes(rows)
    if workspace is None and need:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    p = default_params() if params is None else params
    code = lib().mhc_pre_mxfp8(
        _ptr(R), weights.handle, _ptr(scale), _ptr(base), _ptr(norm_w), rows,
        rows if logical_rows is None else int(logical_rows), ctypes.byref(p), _ptr(workspace),
        ws_bytes, _ptr(x_norm), _ptr(x_q), _ptr(x_s), _ptr(post), _ptr(comb), _stream(stream))
    _check("mhc_pre_mxfp8", code)
    return x_norm, x_q, x_s, post, comb


def mhc_quantize_mxfp8(x, *, logical_rows=None, q=None, s=None, stream=None):
    """MXFP8 of bf16 rows x [rows, cols] (see mhc_quantize_mxfp8 in
    include/mhc.h). Returns ``(q [rows, cols] uint8, s [rows, cols/32] uint8)``."""
    import torch
    rows, cols = int(x.shape[0]), int(x.shape[1])
    _need(x, "x", torch.bfloat16, (rows, cols))
    q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device) if q is None else q
    s = torch.empty((rows, cols // 32), dtype=torch.uint8, device=x.device) if s is None else s
    _need(q, "q", torch.uint8, (rows, cols))
    _need(s, "s", torch.uint8, (rows, cols // 32))
    code = lib().mhc_quantize_mxfp8(_ptr(x), rows, cols,
                                    rows if logical_rows is None else int(logical_rows),
                                    _ptr(q), _ptr(s), _stream(stream))
    _check("mhc_quantize_mxfp8", code)
    return q, s


def mhc_swizzle_scales_128x4(s, *, out=None, stream=None):
    """Linear ue8m0 scales s [rows, groups] -> the 128x4 tiled layout, a flat
    uint8 tensor (see mhc_swizzle_scales_128x4 in include/mhc.h)."""
    import torch
    rows, groups = int(s.shape[0]), int(s.shape[1])
    _need(s, "s", torch.uint8, (rows, groups))
    n = int(lib().mhc_swizzle_scales_128x4_bytes(rows, groups))
    out = torch.empty((n,), dtype=torch.uint8, device=s.device) if out is None else out
    _need(out, "out", torch.uint8, (n,))
    code = lib().mhc_swizzle_scales_128x4(_ptr(s), rows, groups, _ptr(out), _stream(stream))
    _check("mhc_swizzle_scales_128x4", code)
    return out


def mhc_pre_noalloc_max_rows() -> int:
    return int(lib().mhc_pre_noalloc_max_rows())


def mhc_pre_noalloc(R, fn, scale, base, norm_w, x_norm, post, comb, *, logical_rows=None,
                    params=None, pre_out=None, mix_out=None, stream=None):
    """mhc_pre for callers that cannot provide device scratch (see mhc_pre_noalloc
    in include/mhc.h).  Allocates nothing: every output is passed in, and the
    kernels take no scratch.  mhc_pre's launches and bits below 2048 logical
    rows; from 2048 on, the one-pass build that keeps fn resident (mhc_pre's
    values to within fp32 summation order)."""
    import torch
    rows = int(R.shape[0])
    _need(R, "R", torch.bfloat16, (rows, HC, H))
    _need(fn, "fn", torch.float32, (MIX, K))
    _need(scale, "scale", torch.float32, (3,))
    _need(base, "base", torch.float32, (MIX,))
    _need(norm_w, "norm_w", torch.bfloat16, (H,))
    _need(x_norm, "x_norm", torch.bfloat16, (rows, H))
    _need(post, "post", torch.float32, (rows, HC))
    _need(comb, "comb", torch.float32, (rows, HC, HC))
    if pre_out is not None:
        _need(pre_out, "pre_out", torch.float32, (rows, HC))
    if mix_out is not None:
        _need(mix_out, "mix_out", torch.float32, (rows, MIX))
    p = default_params() if params is None else params
    code = lib().mhc_pre_noalloc(
        _ptr(R), _ptr(fn), _ptr(scale), _ptr(base), _ptr(norm_w), rows,
        rows if logical_rows is None else int(logical_rows), ctypes.byref(p), _ptr(x_norm),
        _ptr(post), _ptr(comb), _ptr(pre_out), _ptr(mix_out), _stream(stream))
    _check("mhc_pre_noalloc", code)
    return x_norm, post, comb


def mhc_post(R, y, post, comb, *, logical_rows=None, out=None, stream=None):
    """New residual after a sublayer (see mhc_post in include/mhc.h)."""
    import torch
    rows = int(R.shape[0])
    _need(R, "R", torch.bfloat16, (rows, HC, H))
    _need(y, "y", torch.bfloat16, (rows, H))
    _need(post, "post", torch.float32, (rows, HC))
    _need(comb, "comb", torch.float32, (rows, HC, HC))
    out = torch.empty_like(R) if out is None else out
    _need(out, "out", torch.bfloat16, (rows, HC, H))
    code = lib().mhc_post(_ptr(R), _ptr(y), _ptr(post), _ptr(comb), rows,
                          rows if logical_rows is None else int(logical_rows), _ptr(out),
                          _stream(stream))
    _check("mhc_post", code)
    return out


def mhc_combine_norm(R, pre, norm_w, norm_eps=1e-6, *, logical_rows=None, out=None, stream=None):
    """Combine + RMSNorm with a given pre gate (see mhc_combine_norm in include/mhc.h)."""
    import torch
    rows = int(R.shape[0])
    _need(R, "R", torch.bfloat16, (rows, HC, H))
    _need(pre, "pre", torch.float32, (rows, HC))
    _need(norm_w, "norm_w", torch.bfloat16, (H,))
    out = torch.empty((rows, H), dtype=torch.bfloat16, device=R.device) if out is None else out
    _need(out, "out", torch.bfloat16, (rows, H))
    code = lib().mhc_combine_norm(_ptr(R), _ptr(pre), _ptr(norm_w), float(norm_eps), rows,
                                  rows if logical_rows is None else int(logical_rows),
                                  _ptr(out), _stream(stream))
    _check("mhc_combine_norm", code)
    return out


def mhc_hc_head(R, fn, scale, base, *, norm_eps=1e-6, hc_eps=1e-6, logical_rows=None,
                workspace=None, out=None, pre_out=None, mix_out=None, stream=None):
    """Final collapse of the 4 streams (see mhc_hc_head in include/mhc.h).

    Returns ``y [rows, 5120] bf16``."""
    import torch
    rows = int(R.shape[0])
    _need(R, "R", torch.bfloat16, (rows, HC, H))
    _need(fn, "fn", torch.float32, (HC, K))
    _need(scale, "scale", torch.float32, (1,))
    _need(base, "base", torch.float32, (HC,))
    dev = R.device
    out = torch.empty((rows, H), dtype=torch.bfloat16, device=dev) if out is None else out
    _need(out, "out", torch.bfloat16, (rows, H))
    if pre_out is not None:
        _need(pre_out, "pre_out", torch.float32, (rows, HC))
    if mix_out is not None:
        _need(mix_out, "mix_out", torch.float32, (rows, HC))
    need = mhc_pre_workspace_bytes(rows)
    if workspace is None and need:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    code = lib().mhc_hc_head(
        _ptr(R), _ptr(fn), _ptr(scale), _ptr(base), rows,
        rows if logical_rows is None else int(logical_rows), float(norm_eps), float(hc_eps),
        _ptr(workspace), ws_bytes, _ptr(out), _ptr(pre_out), _ptr(mix_out), _stream(stream))
    _check("mhc_hc_head", code)
    return out


def mhc_fused_post_pre(R, y, post, comb, fn, scale, base, norm_w, *, logical_rows=None,
                       params=None, workspace=None, R_out=None, x_norm=None, post_out=None,
                       comb_out=None, pre_out=None, mix_out=None, stream=None):
    """hc_post then the next hc_pre on its result (see mhc_fused_post_pre in
    include/mhc.h).  Returns ``(R_out, x_norm, post_out, comb_out)``."""
    import torch
    _need(fn, "fn", torch.float32, (MIX, K))
    return _fused_call("mhc_fused_post_pre", _ptr(fn), mhc_fused_post_pre_workspace_bytes, R, y,
                       post, comb, scale, base, norm_w, logical_rows, params, workspace, R_out,
                       x_norm, post_out, comb_out, pre_out, mix_out, stream)


def mhc_fused_post_pre_prepared(R, y, post, comb, weights, scale, base, norm_w, *,
                                logical_rows=None, params=None, workspace=None, R_out=None,
                                x_norm=None, post_out=None, comb_out=None, pre_out=None,
                                mix_out=None, stream=None):
    """mhc_fused_post_pre with the next sublayer's fn from a prepared-weights
    handle (bit-identical; the workspace needs no room for fn's image)."""
    return _fused_call("mhc_fused_post_pre_prepared", weights.handle, mhc_pre_workspace_bytes, R,
                       y, post, comb, scale, base, norm_w, logical_rows, params, workspace, R_out,
                       x_norm, post_out, comb_out, pre_out, mix_out, stream)


def _fused_call(name, fn_arg, ws_bytes_of, R, y, post, comb, scale, base, norm_w, logical_rows,
                params, workspace, R_out, x_norm, post_out, comb_out, pre_out, mix_out, stream):
    import torch
    rows = int(R.shape[0])
    _need(R, "R", torch.bfloat16, (rows, HC, H))
    _need(y, "y", torch.bfloat16, (rows, H))
    _need(post, "post", torch.float32, (rows, HC))
    _need(comb, "comb", torch.float32, (rows, HC, HC))
    _need(scale, "scale", torch.float32, (3,))
    _need(base, "base", torch.float32, (MIX,))
    _need(norm_w, "norm_w", torch.bfloat16, (H,))
    dev = R.device
    R_out = torch.empty_like(R) if R_out is None else R_out
    x_norm = torch.empty((rows, H), dtype=torch.bfloat16, device=dev) if x_norm is None else x_norm
    post_out = torch.empty((rows, HC), dtype=torch.float32, device=dev) if post_out is None else post_out
    comb_out = (torch.empty((rows, HC, HC), dtype=torch.float32, device=dev)
                if comb_out is None else comb_out)
    _need(R_out, "R_out", torch.bfloat16, (rows, HC, H))
    _need(x_norm, "x_norm", torch.bfloat16, (rows, H))
    _need(post_out, "post_out", torch.float32, (rows, HC))
    _need(comb_out, "comb_out", torch.float32, (rows, HC, HC))
    if pre_out is not None:
        _need(pre_out, "pre_out", torch.float32, (rows, HC))
    if mix_out is not None:
        _need(mix_out, "mix_out", torch.float32, (rows, MIX))
    need = ws_bytes_of(rows)
    if workspace is None and need:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    p = default_params() if params is None else params
    code = getattr(lib(), name)(
        _ptr(R), _ptr(y), _ptr(post), _ptr(comb), fn_arg, _ptr(scale), _ptr(base),
        _ptr(norm_w), rows, rows if logical_rows is None else int(logical_rows), ctypes.byref(p),
        _ptr(workspace), ws_bytes, _ptr(R_out), _ptr(x_norm), _ptr(post_out), _ptr(comb_out),
        _ptr(pre_out), _ptr(mix_out), _stream(stream))
    _check(name, code)
    return R_out, x_norm, post_out, comb_out


def mhc_fused_post_pre_mxfp8(R, y, post, comb, weights, scale, base, norm_w, *,
                             logical_rows=None, params=None, workspace=None, R_out=None,
                             x_norm=None, x_q=None, x_s=None, post_out=None, comb_out=None,
                             stream=None):
    """mhc_fused_post_pre_prepared that also writes the next x_norm's MXFP8 (see
    mhc_fused_post_pre_mxfp8 in include/mhc.h).  Returns ``(R_out, x_norm, x_q
    [rows,5120] uint8 E4M3 codes, x_s [rows,160] uint8 ue8m0 scales, post_out,
    comb_out)``."""
    import torch
    rows = int(R.shape[0])
    _need(R, "R", torch.bfloat16, (rows, HC, H))
    _need(y, "y", torch.bfloat16, (rows, H))
    _need(post, "post", torch.float32, (rows, HC))
    _need(comb, "comb", torch.float32, (rows, HC, HC))
    _need(scale, "scale", torch.float32, (3,))
    _need(base, "base", torch.float32, (MIX,))
    _need(norm_w, "norm_w", torch.bfloat16, (H,))
    dev = R.device
    R_out = torch.empty_like(R) if R_out is None else R_out
    x_norm = torch.empty((rows, H), dtype=torch.bfloat16, device=dev) if x_norm is None else x_norm
    x_q = torch.empty((rows, H), dtype=torch.uint8, device=dev) if x_q is None else x_q
    x_s = torch.empty((rows, H // 32), dtype=torch.uint8, device=dev) if x_s is None else x_s
    post_out = torch.empty((rows, HC), dtype=torch.float32, device=dev) if post_out is None else post_out
    comb_out = (torch.empty((rows, HC, HC), dtype=torch.float32, device=dev)
                if comb_out is None else comb_out)
    _need(R_out, "R_out", torch.bfloat16, (rows, HC, H))
    _need(x_norm, "x_norm", torch.bfloat16, (rows, H))
    _need(x_q, "x_q", torch.uint8, (rows, H))
    _need(x_s, "x_s", torch.uint8, (rows, H // 32))
    _need(post_out, "post_out", torch.float32, (rows, HC))
    _need(comb_out, "comb_out", torch.float32, (rows, HC, HC))
    need = mhc_pre_workspace_bytes(rows)
    if workspace is None and need:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    p = default_params() if params is None else params
    code = lib().mhc_fused_post_pre_mxfp8(
        _ptr(R), _ptr(y), _ptr(post), _ptr(comb), weights.handle, _ptr(scale), _ptr(base),
        _ptr(norm_w), rows, rows if logical_rows is None else int(logical_rows), ctypes.byref(p),
        _ptr(workspace), ws_bytes, _ptr(R_out), _ptr(x_norm), _ptr(x_q), _ptr(x_s),
        _ptr(post_out), _ptr(comb_out), _stream(stream))
    _check("mhc_fused_post_pre_mxfp8", code)
    return R_out, x_norm, x_q, x_s, post_out, comb_out
