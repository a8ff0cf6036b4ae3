"""Shared helpers of the parity tests: running the oracle over row blocks on all
host cores, and the element-wise tolerance checks.

Tolerances (GPU vs the fp64 oracle on identical inputs):
  mix      |d| <= 1e-4 * max(|ref|, rms of the row's 24 mixes)
  pre/post |d| <= 1e-6 absolute, or what the kernels' arithmetic allows:
           the tensor-core dots hold fn as bf16 hi + bf16 lo, whose residual
           is at most 2^-17 of each fn element; taken as independent uniform
           errors, a dot's error has sigma = 2^-17/sqrt(3) * ||x o fn_c||_2.
           Six sigma of that, times rsqrt, times |scale|, plus the fp32
           rounding of the logit (8 * 2^-24 of its largest term), times the
           gate's slope, is also accepted
  comb     |d| <= 1e-6 absolute
  bf16 outputs (x_norm, R_out): |d| <= 2 bf16 ulp of the reference value, or
           |d| <= 2e-2 on the scaled columns 0..63 of a stream, or
           |d| <= 2 bf16 ulp of the largest term of that element's sum
           (R_out: post_i*y and comb_ji*R_j; x_norm: pre_i*R_i*rsqrt*w).
The fp32 kernels round each bf16 output once from an fp32 value whose own
error is ~1e-7 relative to the largest term, so away from cancellation the
expected disagreement is <= 1 ulp.  Where the terms cancel (a result near 0
made of terms ~0.3), the fp32 error is a fixed fraction of the terms, not of
the result, and can exceed 2 ulp of the tiny result; the third clause is
that cancellation floor.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import synth

HC, H, K, MIX = 4, 5120, 20480, 24


def cores() -> int:
    return max(1, os.cpu_count() or 1)


def oracle_rows_parallel(func, *arrays, rows: int, block: int = 16, **kw):
    """Call oracle function ``func`` on row blocks of the row-indexed arrays in
    threads (the oracle is C; ctypes drops the GIL) and concatenate results."""
    spans = [(lo, min(rows, lo + block)) for lo in range(0, rows, block)]

    def one(span):
        lo, hi = span
        return func(*[a[lo:hi] for a in arrays], **kw)

    with ThreadPoolExecutor(max_workers=cores()) as ex:
        parts = list(ex.map(one, spans))
    if isinstance(parts[0], dict):
        return {k: (np.concatenate([p[k] for p in parts]) if parts[0][k] is not None else None)
                for k in parts[0]}
    if isinstance(parts[0], tuple):
        return tuple(np.concatenate([p[i] for p in parts]) for i in range(len(parts[0])))
    return np.concatenate(parts)


def unbf(b):
    return synth.bf16_bits_to_f32(b).astype(np.float64)


def bf16_ulp(x):
    """Spacing of bf16 values at |x| (normal range)."""
    a = np.maximum(np.abs(np.asarray(x, np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def _report(name, bad, diff, extra=""):
    """Raise on any element flagged bad.  Callers flag with ~(d <= tol) so that
    a NaN difference (a NaN output) counts as out of tolerance."""
    n = int(bad.sum())
    if n:
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{name}: {n} of {bad.size} elements out of tolerance "
                             f"(max |d| {np.max(diff):.3g}); first at {idx.tolist()} {extra}")


def check_mix(gpu, ref, name="mix"):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref * ref, axis=1, keepdims=True))
    tol = 1e-4 * np.maximum(np.abs(ref), rms)
    d = np.abs(gpu - ref)
    _report(name, ~(d <= tol), d)


def check_gates(gpu_pre, gpu_post, o, scale, R_bits, fn, post_mult=2.0, rms_eps=1e-6):
    """pre and post gates against the oracle dict `o` (mix, logits, pre, post)
    of the rows R_bits, whose stats used fn [24, 20480]."""
    mix = np.asarray(o["mix"], np.float64)
    logit = np.asarray(o["logits"], np.float64)
    scale = np.asarray(scale, np.float64).reshape(-1)
    g_of_c = np.where(np.arange(MIX) < 4, scale[0], np.where(np.arange(MIX) < 8, scale[1], scale[2]))
    base = logit - mix * g_of_c
    x = unbf(np.asarray(R_bits).reshape(len(mix), -1))
    rsq = 1.0 / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + rms_eps)
    f8 = np.asarray(fn, np.float64).reshape(MIX, -1)[:8]
    sig_dot = np.sqrt((x * x) @ (f8 * f8).T)                   # [rows, 8]
    dmix = 6.0 * 2.0 ** -17 / np.sqrt(3.0) * sig_dot * rsq
    for name, gpu, ref, lo, mult in (("pre", gpu_pre, o["pre"], 0, 1.0),
                                     ("post", gpu_post, o["post"], 4, post_mult)):
        l = logit[:, lo:lo + 4]
        sc = scale[0] if lo == 0 else scale[1]
        term = np.maximum(np.abs(mix[:, lo:lo + 4] * sc), np.abs(base[:, lo:lo + 4]))
        sg = 1.0 / (1.0 + np.exp(-l))
        dl = abs(sc) * dmix[:, lo:lo + 4] + 8 * 2.0 ** -24 * term
        d = np.abs(np.asarray(gpu, np.float64) - np.asarray(ref, np.float64))
        _report(name, ~(d <= np.maximum(1e-6, mult * sg * (1 - sg) * dl)), d)


def check_abs(gpu, ref, tol, name):
    d = np.abs(np.asarray(gpu, np.float64) - np.asarray(ref, np.float64))
    _report(name, ~(d <= tol), d)


def scaled_column_mask(shape_tail):
    """True on columns 0..63 of every stream (the x40 columns of the recipe)."""
    m = np.zeros(shape_tail, bool)
    m[..., :64] = True
    return m


def check_bf16(gpu_bits, ref_bits, name, term_mag=None):
    g = unbf(gpu_bits)
    r = unbf(ref_bits)
    d = np.abs(g - r)
    tol = 2.0 * bf16_ulp(r)
    if term_mag is not None:
        tol = np.maximum(tol, 2.0 * bf16_ulp(term_mag))
    scaled = np.broadcast_to(scaled_column_mask(ref_bits.shape[1:]), ref_bits.shape)
    ok = (d <= tol) | (scaled & (d <= 2e-2))
    _report(name, ~ok, d)


def post_term_magnitude(R_bits, y_bits, post, comb):
    """Largest |term| of each R_out element's sum: max(|post_i y|, |comb_ji R_j|)."""
    R = unbf(R_bits)
    y = unbf(y_bits)
    t = np.abs(np.asarray(post, np.float64))[:, :, None] * np.abs(y)[:, None, :]
    for j in range(HC):
        t = np.maximum(t, np.abs(np.asarray(comb, np.float64))[:, j, :, None] * np.abs(R[:, j, None, :]))
    return t


def combine_term_magnitude(R_bits, pre, w_bits, norm_eps):
    """Largest |term| of each x_norm element: max_i |pre_i R_i[h]| * rsqrt * |w[h]|,
    with rsqrt from the fp64 y (only scales the cancellation floor)."""
    R = unbf(R_bits)
    pre = np.asarray(pre, np.float64)
    y = np.einsum("mi,mih->mh", pre, R)
    rn = 1.0 / np.sqrt(np.mean(y * y, axis=1, keepdims=True) + norm_eps)
    t = np.max(np.abs(pre)[:, :, None] * np.abs(R), axis=1)
    return t * rn * np.abs(unbf(w_bits))[None, :]
