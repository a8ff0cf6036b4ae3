"""Pins of the oracle's MXFP8 output (prefill_sp.py, _mxfp8_quantize and
swizzle_128x4), checked against facts the oracle's code does not restate:

- every code is the nearest E4M3 value to x / 2^e, found by brute force over
  a decode table built here from the format's definition (sign, 4-bit
  exponent with bias 7, 3-bit mantissa, subnormals at exponent 0, NaN at
  0x7F), ties going to the even code, magnitudes above 448 saturating;
- the block scale puts the block's largest magnitude in E4M3's top binade
  [256, 512) -- the property that fixes "floor(log2 amax) - 8" (an
  off-by-one lands it in [128, 256) or [512, 1024)) -- with worked values;
- E4M3-representable inputs survive a round trip exactly;
- the 128x4 scale layout holds each (row tile, group tile) in one 512-byte
  run, four groups of a row adjacent, rows m, m+32, m+64, m+96 adjacent,
  and zero padding rows.
"""
import numpy as np
import pytest

import oracle


def e4m3_table():
    """Values of the 256 codes (NaN for 0x7F and 0xFF), from the definition."""
    vals = np.zeros(256)
    for c in range(256):
        sgn = -1.0 if c & 0x80 else 1.0
        E, m = (c >> 3) & 15, c & 7
        if E == 15 and m == 7:
            vals[c] = np.nan
        elif E == 0:
            vals[c] = sgn * (m / 8.0) * 2.0 ** -6
        else:
            vals[c] = sgn * (1.0 + m / 8.0) * 2.0 ** (E - 7)
    return vals


TABLE = e4m3_table()


def nearest_code(t):
    """Brute force: the finite code nearest to t, ties to the even code,
    |t| > 448 saturating; the sign bit is t's sign."""
    mags = TABLE[:0x7F]                      # 0x00..0x7E, increasing
    out = np.zeros(t.shape, np.uint8)
    for idx, v in np.ndenumerate(t):
        a = min(abs(v), 448.0)
        d = np.abs(mags - a)
        best = np.flatnonzero(d == d.min())
        c = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        out[idx] = c | (0x80 if np.signbit(v) else 0)
    return out


def bf16_block(rng, rows, cols, scale_exp):
    """bf16 rows with a spread of block magnitudes (2^scale_exp per block)."""
    x = rng.standard_normal((rows, cols)) * np.repeat(2.0 ** scale_exp, 32, axis=1)
    return oracle.to_bf16(x)


def test_codes_are_the_nearest_e4m3_value():
    rng = np.random.default_rng(5)
    cols = 256
    exps = rng.integers(-20, 20, size=(6, cols // 32)).astype(float)
    x = bf16_block(rng, 6, cols, exps)
    q, s = oracle.mxfp8_quantize(x)
    e = s.astype(np.int64) - 127
    t = oracle.from_bf16(x) * np.repeat(2.0 ** (-e), 32, axis=1)
    assert np.array_equal(q, nearest_code(t))


def test_ties_go_to_even_and_saturation():
    # block exponent e = -8 (amax 1.75): t = 256 * x
    t_vals = [1.75,                    # 448 exactly: 0x7E
              1.8125,                  # 464: above 448, saturates to 0x7E
              1.0 + 1 / 16,            # 272: halfway 256 / 288 -> 256 (even, 0x78)
              1.0 + 3 / 16,            # 304: halfway 288 / 320 -> 320 (0x7A, even)
              2.0 ** -11 * 1.5,        # 1.5 * 2^-3 after scaling: an exact normal
              -(2.0 ** -17)]           # t = -2^-9: the smallest subnormal, negative
    x = np.zeros((1, 32))
    x[0, :len(t_vals)] = t_vals
    xb = oracle.to_bf16(x)
    assert np.array_equal(oracle.from_bf16(xb)[0, :len(t_vals)], t_vals)   # exact in bf16
    q, s = oracle.mxfp8_quantize(xb)
    assert s[0, 0] == 127 - 8
    assert q[0, 0] == 0x7E and q[0, 1] == 0x7E
    assert q[0, 2] == 0x78 and q[0, 3] == 0x7A
    # 1.5 * 2^-11 * 256 = 1.5 * 2^-3: exact normal (E = 4, m = 4)
    assert q[0, 4] == (4 << 3) | 4
    assert q[0, 5] == 0x81
    assert np.array_equal(q, nearest_code(oracle.from_bf16(xb) * 2.0 ** 8))


def test_subnormal_ties():
    # amax 1.0 -> e = -8; t = 2^-10 (half the smallest subnormal) ties to 0,
    # t = 3 * 2^-10 ties between 1 and 2 subnormal quanta -> 2 (even)
    x = np.zeros((1, 32))
    x[0, 0] = 1.0
    x[0, 1] = 2.0 ** -18
    x[0, 2] = 3 * 2.0 ** -18
    x[0, 3] = -(2.0 ** -18)
    q, s = oracle.mxfp8_quantize(oracle.to_bf16(x))
    assert s[0, 0] == 119
    assert q[0, 1] == 0x00 and q[0, 2] == 0x02 and q[0, 3] == 0x80


@pytest.mark.parametrize("amax,code", [(1.0, 119), (1.75, 119), (1.9921875, 119), (2.0, 120),
                                       (0.5, 118), (448.0, 127), (2.0 ** -119, 0),
                                       (2.0 ** -125, 0), (3.0e38, 246)])
def test_scale_worked_values(amax, code):
    x = np.zeros((1, 32))
    x[0, 7] = -amax
    xb = oracle.to_bf16(x)
    _, s = oracle.mxfp8_quantize(xb)
    assert s[0, 0] == code


def test_scale_puts_amax_in_the_top_binade():
    rng = np.random.default_rng(6)
    cols = 640
    exps = rng.integers(-60, 60, size=(8, cols // 32)).astype(float)
    x = bf16_block(rng, 8, cols, exps)
    q, s = oracle.mxfp8_quantize(x)
    e = s.astype(np.int64) - 127
    amax = np.abs(oracle.from_bf16(x)).reshape(8, -1, 32).max(axis=2)
    scaled = amax * 2.0 ** (-e)
    assert np.all((scaled >= 256) & (scaled < 512))
    dec = TABLE[q]
    assert np.all(np.isfinite(dec)) and np.abs(dec).max() <= 448


def test_zero_block_and_negative_zero():
    x = np.zeros((2, 64))
    x[1, 32] = 0.5
    x[1, 33] = -0.0
    q, s = oracle.mxfp8_quantize(oracle.to_bf16(x))
    assert np.all(s[0] == 0) and s[1, 0] == 0 and np.all(q[0] == 0) and np.all(q[1, :32] == 0)
    assert s[1, 1] == 127 + (-1 - 8)
    assert q[1, 33] == 0x80


def test_representable_values_round_trip():
    rng = np.random.default_rng(7)
    finite = np.array([c for c in range(256) if np.isfinite(TABLE[c])])
    codes = rng.choice(finite, size=(4, 96))
    codes[:, ::32] = 0x7E                    # a 448 in every block fixes e at the block's exponent
    e = rng.integers(-30, 30, size=(4, 3))
    x = TABLE[codes] * np.repeat(2.0 ** e, 32, axis=1)
    xb = oracle.to_bf16(x)
    assert np.array_equal(oracle.from_bf16(xb), x)      # E4M3 * 2^e fits bf16 here
    q, s = oracle.mxfp8_quantize(xb)
    assert np.array_equal(s.astype(np.int64) - 127, e)
    # +-0 keep their sign bit; everything else returns its own code
    assert np.array_equal(q, codes)


@pytest.mark.parametrize("rows,groups", [(1, 4), (128, 160), (300, 8), (1500, 160)])
def test_swizzle_layout_structure(rows, groups):
    m = np.repeat(np.arange(rows)[:, None], groups, axis=1)
    g = np.repeat(np.arange(groups)[None, :], rows, axis=0)
    pad = (rows + 127) // 128 * 128
    assert oracle.swizzle_128x4(np.ones((rows, groups), np.uint8)).size == pad * groups
    # rows and groups travel as separate byte planes (value + 1, so padding
    # stays recognisable as 0)
    rs = oracle.swizzle_128x4(((m % 255) + 1).astype(np.uint8)).astype(np.int64) - 1
    gs = oracle.swizzle_128x4((g + 1).astype(np.uint8)).astype(np.int64) - 1
    tiles = rs.reshape(-1, 512), gs.reshape(-1, 512)
    tg = groups // 4
    for t in range(pad // 128 * tg):
        tm, tgi = divmod(t, tg)
        r_t, g_t = tiles[0][t], tiles[1][t]
        real = g_t >= 0
        # the run holds this tile's groups only, each group's 4 columns adjacent
        assert set(np.unique(g_t[real])) <= set(range(4 * tgi, 4 * tgi + 4))
        quad = g_t.reshape(128, 4)
        assert np.all((quad[real.reshape(128, 4).all(1)] - 4 * tgi) == np.arange(4))
        # byte run k of 16 holds rows tm*128 + k + {0, 32, 64, 96}
        rows_here = r_t.reshape(32, 4, 4)[:, :, 0]
        for k in range(32):
            for a in range(4):
                want = tm * 128 + k + 32 * a
                got = rows_here[k, a]
                if want < rows:
                    assert got == want % 255
                else:
                    assert got == -1                   # padding row: zero scale
    # every real scale appears once
    assert (gs >= 0).sum() == rows * groups
