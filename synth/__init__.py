"""Seeded synthetic inputs for the mHC hot path.

This module is the one piece shared by the CUDA path's tests/benchmark and the
CPU oracle's tests.  It holds none of the method's arithmetic: it only draws
numbers.  The draws are defined here, independently of numpy's or torch's
generators, so that the same seed gives the same bits on every machine:

* SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014) used as a counter-based hash: draw n of stream
  (seed, tensor) is ``mix64(key + (n + 1) * 0x9E3779B97F4A7C15)``, where
  ``key = mix64(seed * 0x100000001B3 + tensor)``.
* Uniforms: the top or bottom 32 bits of a draw, ``(b + 0.5) / 2**32``.
* Normals: Box-Muller on the two 32-bit halves of one draw (element 2p gets
  the cosine branch, element 2p+1 the sine branch).

The workload recipe follows test_prefill_sp_gpu.py (recipes repo), the
``_residual``/``_hc_params``/``_norm`` helpers: R ~ N(0, 0.5^2) with the
first 64 columns of every stream scaled by 40; fn ~ N(0, 0.0225^2);
base ~ N(0, 3^2); scale ~ U(0.01, 0.06); norm weight 1 + 0.1 N(0, 1);
sublayer output y ~ N(0, 1).  Values are drawn in float64, scaled, rounded to
float32 and, for bf16 tensors, then to bf16 nearest-even.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

HC, H, K, MIX = 4, 5120, 20480, 24

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_LOW32 = np.uint64(0xFFFFFFFF)
_TWO_M32 = 1.0 / 4294967296.0

# tensor ids of the recipe
T_R, T_FN, T_BASE, T_SCALE, T_W, T_Y, T_Y2 = 1, 2, 3, 4, 5, 6, 7
T_HFN, T_HBASE, T_HSCALE = 8, 9, 10          # hc_head's parameters


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, tensor: int) -> np.uint64:
    v = np.array([(int(seed) * 0x100000001B3 + int(tensor)) & 0xFFFFFFFFFFFFFFFF], np.uint64)
    return _mix64(v)[0]


def draws(seed: int, tensor: int, start: int, n: int) -> np.ndarray:
    """Raw 64-bit draws start .. start+n-1 of stream (seed, tensor)."""
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(_key(seed, tensor) + idx * _GAMMA)


def uniform(seed: int, tensor: int, n: int, start: int = 0) -> np.ndarray:
    """n uniforms in (0, 1) as float64 (top 32 bits of each draw)."""
    z = draws(seed, tensor, start, n)
    return ((z >> np.uint64(32)).astype(np.float64) + 0.5) * _TWO_M32


def _normal_pairs(seed: int, tensor: int, p0: int, npairs: int) -> np.ndarray:
    z = draws(seed, tensor, p0, npairs)
    u1 = ((z >> np.uint64(32)).astype(np.float64) + 0.5) * _TWO_M32
    u2 = ((z & _LOW32).astype(np.float64) + 0.5) * _TWO_M32
    rad = np.sqrt(-2.0 * np.log(u1))
    ang = 2.0 * np.pi * u2
    out = np.empty(2 * npairs, np.float64)
    out[0::2] = rad * np.cos(ang)
    out[1::2] = rad * np.sin(ang)
    return out


def normal(seed: int, tensor: int, n: int, start: int = 0) -> np.ndarray:
    """Elements start .. start+n-1 of the standard-normal stream, float64.
    ``start`` must be even (elements come in Box-Muller pairs)."""
    if start % 2:
        raise ValueError("start must be even")
    npairs = (n + 1) // 2
    return _normal_pairs(seed, tensor, start // 2, npairs)[:n]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 bits, nearest-even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------------------
def _rows_parallel(fill, rows: int, width: int, dtype, chunk_rows: int):
    out = np.empty((rows, width), dtype)
    spans = [(r, min(rows, r + chunk_rows)) for r in range(0, rows, chunk_rows)]
    if len(spans) <= 1:
        for lo, hi in spans:
            fill(out, lo, hi)
    else:
        with ThreadPoolExecutor(max_workers=8) as ex:
            list(ex.map(lambda s: fill(out, *s), spans))
    return out


def residual(seed: int, rows: int, row0: int = 0) -> np.ndarray:
    """R rows row0 .. row0+rows-1 of the recipe, as bf16 bits [rows, 4, 5120]."""
    scale_cols = np.full(H, 0.5, np.float64)
    scale_cols[:64] *= 40.0
    scale_row = np.tile(scale_cols, HC)

    def fill(out, lo, hi):
        v = normal(seed, T_R, (hi - lo) * K, start=(row0 + lo) * K).reshape(hi - lo, K)
        out[lo:hi] = f32_to_bf16_bits((v * scale_row).astype(np.float32))

    return _rows_parallel(fill, rows, K, np.uint16, 256).reshape(rows, HC, H)


def sublayer_out(seed: int, rows: int, row0: int = 0, tensor: int = T_Y) -> np.ndarray:
    """y rows of the recipe, bf16 bits [rows, 5120]."""
    def fill(out, lo, hi):
        v = normal(seed, tensor, (hi - lo) * H, start=(row0 + lo) * H).reshape(hi - lo, H)
        out[lo:hi] = f32_to_bf16_bits(v.astype(np.float32))

    return _rows_parallel(fill, rows, H, np.uint16, 1024)


@dataclass
class Weights:
    fn: np.ndarray      # [24, 20480] float32
    base: np.ndarray    # [24] float32
    scale: np.ndarray   # [3] float32
    norm_w: np.ndarray  # [5120] bf16 bits


def weights(seed: int) -> Weights:
    fn = (0.0225 * normal(seed, T_FN, MIX * K)).astype(np.float32).reshape(MIX, K)
    base = (3.0 * normal(seed, T_BASE, MIX)).astype(np.float32)
    scale = (0.01 + 0.05 * uniform(seed, T_SCALE, 3)).astype(np.float32)
    w = f32_to_bf16_bits((1.0 + 0.1 * normal(seed, T_W, H)).astype(np.float32))
    return Weights(fn=fn, base=base, scale=scale, norm_w=w)


@dataclass
class HeadWeights:
    fn: np.ndarray      # [4, 20480] float32
    base: np.ndarray    # [4] float32
    scale: np.ndarray   # [1] float32


def head_weights(seed: int) -> HeadWeights:
    """hc_head's fn [4, 4H], base [4], scale [1] (deepseek_v4.py,
    make_hc_head_params), drawn like the layer's mixing parameters."""
    fn = (0.0225 * normal(seed, T_HFN, HC * K)).astype(np.float32).reshape(HC, K)
    base = (3.0 * normal(seed, T_HBASE, HC)).astype(np.float32)
    scale = (0.01 + 0.05 * uniform(seed, T_HSCALE, 1)).astype(np.float32)
    return HeadWeights(fn=fn, base=base, scale=scale)


@dataclass
class Workload:
    name: str
    rows: int
    seed: int


# The five workloads: sizes and seeds of the mHC hot-path configurations.
WORKLOADS = [
    Workload("M=128", 128, 0),
    Workload("M=1500", 1500, 1),
    Workload("M=2048", 2048, 2),
    Workload("M=4096", 4096, 3),
    Workload("M=16384", 16384, 4),
]
