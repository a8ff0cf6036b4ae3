"""The GPU parity checker (tests/parity.py) on the CPU: it must reject what a
plausible kernel mistake produces and accept what legitimate rounding
differences produce.  Every "GPU result" here is made by the oracle on the
host, with the mistake (or the rounding difference) applied there."""
import numpy as np
import pytest

import synth
from tests import parity as P

HC, H = 4, 5120


@pytest.fixture(scope="module")
def case(oracle_mod):
    rows = 6
    R = synth.residual(3, rows)
    y = synth.sublayer_out(3, rows)
    W = synth.weights(3)
    o = oracle_mod.pre(R, W.fn, W.scale, W.base, W.norm_w)
    post32 = o["post"].astype(np.float32)
    comb32 = o["comb"].astype(np.float32)
    R2 = oracle_mod.post(R, y, post32, comb32)
    return dict(R=R, y=y, W=W, o=o, post32=post32, comb32=comb32, R2=R2)


def test_the_reference_itself_passes(case):
    o, W, R = case["o"], case["W"], case["R"]
    P.check_mix(o["mix"], o["mix"])
    P.check_gates(o["pre"], o["post"], o, W.scale, R, W.fn)
    tm = P.combine_term_magnitude(R, o["pre"], W.norm_w, 1e-6)
    P.check_bf16(o["x_norm"], o["x_norm"], "x_norm", term_mag=tm)


def test_gate_error_of_5e6_is_caught(case):
    o, W, R = case["o"], case["W"], case["R"]
    for key, col in (("pre", 2), ("post", 1)):
        g = {"pre": o["pre"].copy(), "post": o["post"].copy()}
        g[key][4, col] += 5e-6
        with pytest.raises(AssertionError):
            P.check_gates(g["pre"], g["post"], o, W.scale, R, W.fn)


def test_fp32_rounding_of_the_gates_passes(case):
    # the kernels return fp32 gates: rounding the fp64 reference to fp32 (and
    # one fp32 ulp more) stays inside the tolerance
    o, W, R = case["o"], case["W"], case["R"]
    pre = o["pre"].astype(np.float32)
    post = np.nextafter(o["post"].astype(np.float32), np.float32(3.0))
    P.check_gates(pre, post, o, W.scale, R, W.fn)


def test_stats_without_the_lo_half_of_fn_is_caught(case, oracle_mod):
    # a stats kernel that multiplied by bf16(fn) only (no lo correction)
    R, W, o = case["R"], case["W"], case["o"]
    fn_hi = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(W.fn.astype(np.float32)))
    mix_hi, _ = oracle_mod.stats(R, fn_hi, 1e-6)
    with pytest.raises(AssertionError):
        P.check_mix(mix_hi, o["mix"])


def test_unfused_combine_rounding_passes_and_a_dropped_weight_is_caught(case, oracle_mod):
    R, W, o = case["R"], case["W"], case["o"]
    tm = P.combine_term_magnitude(R, o["pre"], W.norm_w, 1e-6)
    unfused = oracle_mod.combine_norm(R, o["pre"], W.norm_w, 1e-6, round_y=True)
    P.check_bf16(unfused, o["x_norm"], "x_norm", term_mag=tm)
    no_w = oracle_mod.combine_norm(R, o["pre"], oracle_mod.to_bf16(np.ones(H)), 1e-6)
    with pytest.raises(AssertionError):
        P.check_bf16(no_w, o["x_norm"], "x_norm", term_mag=tm)


def test_post_mistakes_are_caught(case, oracle_mod):
    R, y, R2 = case["R"], case["y"], case["R2"]
    post32, comb32 = case["post32"], case["comb32"]
    tm = P.post_term_magnitude(R, y, post32, comb32)
    P.check_bf16(R2, R2, "R_out", term_mag=tm)
    # comb read as [i][j] instead of [j][i]
    wrong = oracle_mod.post(R, y, post32, np.ascontiguousarray(comb32.transpose(0, 2, 1)))
    with pytest.raises(AssertionError):
        P.check_bf16(wrong, R2, "R_out", term_mag=tm)
    # two rows' outputs swapped (a row-index slip)
    swapped = R2.copy()
    swapped[[1, 2]] = swapped[[2, 1]]
    with pytest.raises(AssertionError):
        P.check_bf16(swapped, R2, "R_out", term_mag=tm)
    # streams 0 and 3 of the output swapped
    streams = R2.copy()
    streams[:, [0, 3]] = streams[:, [3, 0]]
    with pytest.raises(AssertionError):
        P.check_bf16(streams, R2, "R_out", term_mag=tm)


def test_a_nan_output_is_caught_by_every_check(case):
    # a NaN compares false against any tolerance: every check must still fail
    o, W, R = case["o"], case["W"], case["R"]
    mix = o["mix"].copy()
    mix[1, 5] = np.nan
    with pytest.raises(AssertionError):
        P.check_mix(mix, o["mix"])
    for key in ("pre", "post"):
        g = {"pre": o["pre"].copy(), "post": o["post"].copy()}
        g[key][2, 3] = np.nan
        with pytest.raises(AssertionError):
            P.check_gates(g["pre"], g["post"], o, W.scale, R, W.fn)
    comb = o["comb"].copy()
    comb[0, 1, 2] = np.nan
    with pytest.raises(AssertionError):
        P.check_abs(comb, o["comb"], 1e-6, "comb")
    xn = o["x_norm"].copy()
    xn[3, 7] = 0x7FC0   # a bf16 quiet NaN
    with pytest.raises(AssertionError):
        P.check_bf16(xn, o["x_norm"], "x_norm")
