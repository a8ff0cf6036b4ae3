"""Pins of the oracle's hc_head and fused post->pre to facts other than its
own code (closed forms, exact small-integer arithmetic, invariants).

hc_head follows deepseek_v4.py (sglang), make_hc_head_params / hc_head_torch:
fn [4, 20480], base [4], scale [1]; rsqrt(mean x^2 + norm_eps);
pre = sigmoid(mix * scale + base) + hc_eps; y = sum_i pre_i x_i, cast once.
The fused post->pre (deepseek_v4.py, the mhc_fused_post_pre call between
sublayers) is the plain composition of hc_post and hc_pre.
"""
import math
from fractions import Fraction

import numpy as np

import synth

HC, H, K = 4, 5120, 20480


def bf(x):
    return synth.f32_to_bf16_bits(np.asarray(x, np.float32))


def unbf(b):
    return synth.bf16_bits_to_f32(b).astype(np.float64)


def _stream_constants(vals, rows=1):
    R = np.empty((rows, HC, H), np.float32)
    for i, v in enumerate(vals):
        R[:, i, :] = v
    return bf(R)


def test_gate_weights_each_stream_in_order(oracle_mod):
    # scale 0: pre_i = sigmoid(base_i) + eps.  base = (0, ln 3, -ln 3, 40) gives
    # gates (1/2, 3/4, 1/4, 1) and eps = 0; streams hold 2, 4, 8, 16, so
    # y = 1 + 3 + 2 + 16 = 22 exactly -- any swap of streams or gates, or a
    # dropped stream, moves it.
    R = _stream_constants([2.0, 4.0, 8.0, 16.0])
    fn = np.zeros((HC, K), np.float32)
    base = np.array([0.0, math.log(3.0), -math.log(3.0), 40.0], np.float32)
    o = oracle_mod.hc_head(R, fn, np.zeros(1, np.float32), base, norm_eps=1e-6, hc_eps=0.0)
    np.testing.assert_allclose(o["pre"][0], [0.5, 0.75, 0.25, 1.0], rtol=0, atol=1e-7)
    assert (unbf(o["y"]) == 22.0).all()


def test_hc_eps_is_added_after_the_sigmoid(oracle_mod):
    R = _stream_constants([1.0, 0.0, 0.0, 0.0])
    fn = np.zeros((HC, K), np.float32)
    o = oracle_mod.hc_head(R, fn, np.zeros(1, np.float32), np.zeros(4, np.float32),
                           norm_eps=1e-6, hc_eps=0.25)
    np.testing.assert_allclose(o["pre"][0], [0.75] * 4, rtol=0, atol=1e-15)
    assert (unbf(o["y"]) == 0.75).all()          # only stream 0 is non-zero


def test_rsqrt_uses_norm_eps_and_the_mean_over_all_streams(oracle_mod):
    # constant row c: rsqrt = 1/sqrt(c^2 + eps); a one-hot fn row at k gives
    # mix = x_k * rsqrt for each of the 4 mixes (one k in each stream).
    c, eps = 0.5, 0.25
    R = _stream_constants([c, c, c, c])
    fn = np.zeros((HC, K), np.float32)
    for i in range(HC):
        fn[i, i * H + 17 * (i + 1)] = 1.0
    o = oracle_mod.hc_head(R, fn, np.ones(1, np.float32), np.zeros(4, np.float32),
                           norm_eps=eps, hc_eps=0.0)
    want = c / math.sqrt(c * c + eps)
    np.testing.assert_allclose(o["mix"][0], [want] * 4, rtol=1e-15)
    np.testing.assert_allclose(o["pre"][0], [1 / (1 + math.exp(-want))] * 4, rtol=1e-15)
    # half the streams zero: the mean is over all 20480, so ss/K = c^2/2
    R2 = _stream_constants([c, c, 0.0, 0.0])
    o2 = oracle_mod.hc_head(R2, fn, np.ones(1, np.float32), np.zeros(4, np.float32),
                            norm_eps=eps, hc_eps=0.0)
    np.testing.assert_allclose(o2["mix"][0, :2], [c / math.sqrt(c * c / 2 + eps)] * 2, rtol=1e-15)
    assert o2["mix"][0, 2] == 0.0 and o2["mix"][0, 3] == 0.0


def test_mix_brute_force_exact_rationals(oracle_mod):
    # one small row of integers/8 and dyadic fn: the dot is exact in rationals
    rng = np.random.default_rng(3)
    x = rng.integers(-8, 9, size=K).astype(np.float64) / 8
    f = rng.integers(-4, 5, size=(HC, K)).astype(np.float64) / 64
    R = bf(x.reshape(1, HC, H))
    o = oracle_mod.hc_head(R, f.astype(np.float32), np.ones(1, np.float32),
                           np.zeros(4, np.float32), norm_eps=0.0, hc_eps=0.0)
    xs = [Fraction(v) for v in x]
    ss = sum(v * v for v in xs)
    rs = 1 / math.sqrt(float(ss / K))
    for c in range(HC):
        dot = sum(xv * Fraction(fv) for xv, fv in zip(xs, f[c]) if fv != 0)
        assert abs(o["mix"][0, c] - float(dot) * rs) <= 1e-12 * max(1.0, abs(float(dot) * rs))


def test_scale_by_two_doubles_the_output_exactly(oracle_mod):
    # with eps = 0, mix(2R) == mix(R) bit for bit (2 dot / (2 sqrt)); so the
    # gates repeat and y(2R) = 2 y(R) exactly (bf16 rounding commutes with 2x)
    W = synth.weights(2)
    R = synth.residual(2, 3)
    R2 = bf(unbf(R) * 2)
    fn4 = W.fn[:4]
    a = oracle_mod.hc_head(R, fn4, W.scale[:1], W.base[:4], norm_eps=0.0, hc_eps=1e-6)
    b = oracle_mod.hc_head(R2, fn4, W.scale[:1], W.base[:4], norm_eps=0.0, hc_eps=1e-6)
    np.testing.assert_array_equal(a["pre"], b["pre"])
    np.testing.assert_array_equal(unbf(b["y"]), 2 * unbf(a["y"]))


def test_gate_range(oracle_mod):
    W = synth.weights(1)
    R = synth.residual(1, 4)
    o = oracle_mod.hc_head(R, W.fn[:4], W.scale[:1], W.base[:4], hc_eps=1e-6)
    assert (o["pre"] > 1e-6).all() and (o["pre"] < 1 + 1e-6).all()


def test_head_gates_agree_with_the_pre_pass_gates(oracle_mod):
    # hc_head's pre gate is the pre pass's gate on the first 4 mixes (same
    # rsqrt, same sigmoid + eps) when fn, scale and base are shared
    W = synth.weights(4)
    R = synth.residual(4, 3)
    full = oracle_mod.pre(R, W.fn, W.scale, W.base, W.norm_w, rms_eps=1e-6, hc_pre_eps=1e-6)
    head = oracle_mod.hc_head(R, W.fn[:4], W.scale[:1], W.base[:4], norm_eps=1e-6, hc_eps=1e-6)
    np.testing.assert_allclose(head["mix"], full["mix"][:, :4], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(head["pre"], full["pre"], rtol=1e-13)


def test_fused_post_pre_is_post_then_pre(oracle_mod):
    # identity comb and zero post: R' == R, so the next pre sees R itself
    W = synth.weights(0)
    R = synth.residual(0, 2)
    y = synth.sublayer_out(0, 2)
    comb = np.tile(np.eye(HC, dtype=np.float32), (2, 1, 1))
    R2, nxt = oracle_mod.fused_post_pre(R, y, np.zeros((2, HC), np.float32), comb,
                                        W.fn, W.scale, W.base, W.norm_w)
    np.testing.assert_array_equal(R2, R)
    ref = oracle_mod.pre(R, W.fn, W.scale, W.base, W.norm_w)
    for k in ("mix", "pre", "post", "comb", "x_norm"):
        np.testing.assert_array_equal(nxt[k], ref[k])
