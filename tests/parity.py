"""Shared helpers of the parity tests: running the oracle over row blocks on all
host cores, and the element-wise tolerance checks.

Tolerances (GPU vs the fp64 oracle on identical inputs):
  mix      |d| <= 1e-4 * max(|ref|, rms of the row's 24 mixes)
  pre/post |d| <= 1e-6 absolute
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
    _report(name, d > tol, d)


def check_abs(gpu, ref, tol, name):
    d = np.abs(np.asarray(gpu, np.float64) - np.asarray(ref, np.float64))
    _report(name, d > tol, d)


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
