"""Pins of the CPU oracle to facts other than its own code.

Each test checks one oracle function against a closed form, an invariant, an
independent library (torch's bf16 cast), or exact arithmetic on a tiny input,
chosen so that a plausible slip (a dropped term, a wrong sign or index, a
transposed operand, a wrong denominator) fails at least one of them.

Definitions pinned (deepseek_v4.py, sglang): DeepseekV4DecoderLayer.hc_pre
(hc_pre_torch_impl and the combine after hc_split_sinkhorn), hc_post
(hc_post_torch_impl), and hc_head_torch for the sigmoid + eps gate.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import synth

HC, H, K, MIX = 4, 5120, 20480, 24


def bf(x):
    return synth.f32_to_bf16_bits(np.asarray(x, np.float32))


def unbf(b):
    return synth.bf16_bits_to_f32(b).astype(np.float64)


# --------------------------------------------------------------------------- rounding
def test_bf16_round_matches_torch_on_float32_values(oracle_mod):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    v = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(10.0) ** rng.integers(-30, 30, 4000),
        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 2.0 ** -133,
                  3 * 2.0 ** -134, 2.0 ** -126, 3.0e38, -3.0e38, 0.0], np.float32),
    ]).astype(np.float32)
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle_mod.to_bf16(v.astype(np.float64))
    np.testing.assert_array_equal(got, want)


def test_bf16_round_is_single_rounding_from_double(oracle_mod):
    # 1 + 2^-8 is a tie between bf16 1.0 and 1.0078125; a hair above it must
    # round up.  Going through float32 first would land on the tie and give 1.0.
    assert oracle_mod.to_bf16(np.array([1.0 + 2.0 ** -8 + 2.0 ** -40]))[0] == 0x3F81
    assert oracle_mod.to_bf16(np.array([1.0 + 2.0 ** -8]))[0] == 0x3F80          # tie -> even
    assert oracle_mod.to_bf16(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 0x3F82      # tie -> even
    assert oracle_mod.to_bf16(np.array([-(1.0 + 2.0 ** -8 - 2.0 ** -40)]))[0] == 0xBF80
    assert oracle_mod.to_bf16(np.array([2.0 ** -134]))[0] == 0x0000               # subnormal tie
    assert oracle_mod.to_bf16(np.array([2.0 ** -134 + 2.0 ** -160]))[0] == 0x0001
    assert oracle_mod.to_bf16(np.array([3.5e38]))[0] == 0x7F80                    # overflow


# --------------------------------------------------------------------------- a1 stats
def _random_rows(rows, seed=5, scale=0.5):
    rng = np.random.default_rng(seed)
    return bf(rng.standard_normal((rows, HC, H)) * scale)


def test_stats_constant_row_rsqrt_closed_form(oracle_mod):
    # x = c everywhere  =>  mean(x^2) = c^2  =>  rsqrt = 1/sqrt(c^2 + eps).
    # c^2 = 2^-20 is comparable to eps, so eps placement and the /20480 mean are visible.
    for c, eps in ((2.0 ** -10, 1e-6), (0.75, 1e-6), (-3.0, 0.5)):
        R = np.full((1, HC, H), bf(c), np.uint16)
        fn = np.zeros((MIX, K), np.float32)
        _, rsq = oracle_mod.stats(R, fn, eps)
        assert rsq[0] == pytest.approx(1.0 / math.sqrt(c * c + eps), rel=1e-14)


def test_stats_half_zero_row_uses_mean_over_all_4_streams(oracle_mod):
    # streams 0,1 = c, streams 2,3 = 0  =>  mean over 20480 = c^2/2.
    R = np.zeros((1, HC, H), np.uint16)
    R[0, :2, :] = bf(1.5)
    _, rsq = oracle_mod.stats(R, np.zeros((MIX, K), np.float32), 0.0)
    assert rsq[0] == pytest.approx(1.0 / math.sqrt(1.5 * 1.5 / 2), rel=1e-14)


def test_stats_one_hot_fn_picks_element_of_flattened_row(oracle_mod):
    # fn[c] = e_{k_c}  =>  mix[c] = x[k_c] * rsqrt, with k = i*5120 + h (stream-major).
    R = _random_rows(3)
    ks = [c * 853 + 17 for c in range(MIX)]       # spans all four streams
    ks[0], ks[1], ks[2] = 0, K - 1, 2 * H + 5
    fn = np.zeros((MIX, K), np.float32)
    for c, k in enumerate(ks):
        fn[c, k] = 1.0
    mix, rsq = oracle_mod.stats(R, fn, 1e-6)
    x = unbf(R).reshape(3, K)
    for c, k in enumerate(ks):
        np.testing.assert_allclose(mix[:, c], x[:, k] * rsq, rtol=1e-15)
        i, h = divmod(k, H)
        np.testing.assert_allclose(mix[:, c], unbf(R[:, i, h]) * rsq, rtol=1e-15)


def test_stats_exact_rational_brute_force_one_row(oracle_mod):
    # Exact dot products in rational arithmetic on a dyadic fn; only the final
    # sqrt is taken in float.  The oracle must agree to ~1e-13 relative.
    rng = np.random.default_rng(11)
    R = bf(rng.standard_normal((1, HC, H)) * 2.0)
    fn = (rng.integers(-64, 65, (2, K)) / 256.0).astype(np.float32)   # exact dyadics
    fn_full = np.zeros((MIX, K), np.float32)
    fn_full[3], fn_full[17] = fn[0], fn[1]
    mix, rsq = oracle_mod.stats(R, fn_full, 1e-6)
    xs = [Fraction(float(v)) for v in unbf(R).reshape(K)]
    ss = sum(v * v for v in xs)
    r = 1.0 / math.sqrt(float(ss / K + Fraction(1e-6)))
    assert rsq[0] == pytest.approx(r, rel=1e-15)
    for row, c in ((0, 3), (1, 17)):
        dot = sum(xv * Fraction(float(f)) for xv, f in zip(xs, fn[row]))
        assert mix[0, c] == pytest.approx(float(dot) * r, rel=1e-12, abs=1e-12)
    others = [c for c in range(MIX) if c not in (3, 17)]
    assert np.all(mix[0, others] == 0.0)


def test_stats_scale_and_sign_invariance(oracle_mod):
    # eps = 0: mix(2R) = mix(R) (rsqrt absorbs the scale), mix(-R) = -mix(R).
    R = _random_rows(2, seed=3)
    fn = np.random.default_rng(4).standard_normal((MIX, K)).astype(np.float32) * 0.02
    m1, _ = oracle_mod.stats(R, fn, 0.0)
    m2, _ = oracle_mod.stats(bf(unbf(R) * 2.0), fn, 0.0)
    m3, _ = oracle_mod.stats(R ^ np.uint16(0x8000), fn, 0.0)
    np.testing.assert_allclose(m2, m1, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(m3, -m1, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------- a2/a3 split + Sinkhorn
def _split(o, mix, scale=(0.0, 0.0, 0.0), base=None, pre_eps=1e-6, sink_eps=1e-6, post_mult=2.0,
           iters=20):
    mix = np.asarray(mix, np.float64).reshape(-1, MIX)
    base = np.zeros(MIX, np.float32) if base is None else np.asarray(base, np.float32)
    return o.split_sinkhorn(mix, np.asarray(scale, np.float32), base, pre_eps, sink_eps,
                            post_mult, iters)


def test_split_zero_logits(oracle_mod):
    out = _split(oracle_mod, np.ones((1, MIX)) * 7.0)     # scale = 0, base = 0
    np.testing.assert_allclose(out["pre"], 0.5 + 1e-6, rtol=0, atol=1e-15)
    np.testing.assert_allclose(out["post"], 1.0, rtol=0, atol=1e-15)
    np.testing.assert_allclose(out["comb"], 0.25, atol=1e-6)


def test_split_scale_groups_and_base(oracle_mod):
    mix = np.ones((1, MIX))
    base = np.arange(MIX, dtype=np.float32) * 0.125
    out = _split(oracle_mod, mix, scale=(0.5, 0.25, 2.0), base=base)
    want = np.array([0.5] * 4 + [0.25] * 4 + [2.0] * 16) + base
    np.testing.assert_array_equal(out["logits"][0], want)


def test_split_sigmoid_closed_form(oracle_mod):
    # sigmoid(log 3) = 3/4, sigmoid(-log 3) = 1/4.
    base = np.zeros(MIX, np.float32)
    mix = np.zeros((1, MIX))
    mix[0, 0], mix[0, 5] = math.log(3.0), -math.log(3.0)
    out = _split(oracle_mod, mix, scale=(1.0, 1.0, 1.0), base=base, pre_eps=1e-3)
    assert out["pre"][0, 0] == pytest.approx(0.75 + 1e-3, abs=1e-15)
    assert out["post"][0, 1] == pytest.approx(2.0 * 0.25, abs=1e-15)
    assert out["pre"][0, 1] == pytest.approx(0.5 + 1e-3, abs=1e-15)


@pytest.mark.parametrize("c0", [0, 3, 4, 7, 8, 9, 14, 23])
def test_split_order_and_comb_row_major(oracle_mod, c0):
    # a single large logit shows where each mix slot lands.
    base = np.zeros(MIX, np.float32)
    base[c0] = 40.0
    out = _split(oracle_mod, np.zeros((1, MIX)), base=base)
    pre, post, comb = out["pre"][0], out["post"][0], out["comb"][0]
    if c0 < 4:
        assert pre[c0] == pytest.approx(1.0 + 1e-6, abs=1e-12)
        assert np.allclose(np.delete(pre, c0), 0.5 + 1e-6)
    elif c0 < 8:
        assert post[c0 - 4] == pytest.approx(2.0, abs=1e-12)
        assert np.allclose(np.delete(post, c0 - 4), 1.0)
    else:
        j0, i0 = divmod(c0 - 8, 4)
        # convergence towards the permutation-like limit is sublinear; after
        # 20 iterations the dominant slot holds ~0.96 of its row and column.
        assert comb[j0, i0] > 0.9
        assert np.all(np.delete(comb[j0], i0) < 0.05)
        assert np.all(np.delete(comb[:, i0], j0) < 0.05)


def test_sinkhorn_eps_in_denominators_closed_form(oracle_mod):
    # all-zero logits, one iteration, eps = 0.5 (exaggerated):
    # rows: 1/(4 + eps) = x; columns: x / (4x + eps).
    eps = 0.5
    out = _split(oracle_mod, np.zeros((1, MIX)), sink_eps=eps, iters=1)
    x = 1.0 / (4.0 + eps)
    np.testing.assert_allclose(out["comb"][0], x / (4 * x + eps), rtol=1e-15)


def test_sinkhorn_columns_are_normalised_last(oracle_mod):
    # eps = 0: after any iteration count the column sums are exactly 1 (up to
    # rounding); the row sums of a non-converged matrix are not.
    rng = np.random.default_rng(2)
    base = np.zeros(MIX, np.float32)
    base[8:] = rng.standard_normal(16) * 3
    for iters in (1, 2, 5):
        comb = _split(oracle_mod, np.zeros((1, MIX)), base=base, sink_eps=0.0, iters=iters)["comb"][0]
        np.testing.assert_allclose(comb.sum(axis=0), 1.0, atol=1e-14)   # sum over j
    comb1 = _split(oracle_mod, np.zeros((1, MIX)), base=base, sink_eps=0.0, iters=1)["comb"][0]
    assert np.max(np.abs(comb1.sum(axis=1) - 1.0)) > 1e-3


def test_sinkhorn_rank_one_logits_uniform_after_one_iteration(oracle_mod):
    # logits a_j + b_i: exp is rank one, every row is a multiple of the same
    # vector, so the row step makes all rows equal and the column step gives 1/4.
    a = np.array([0.3, -1.2, 2.0, 0.7])
    b = np.array([-0.4, 1.1, 0.0, -2.5])
    base = np.zeros(MIX, np.float32)
    base[8:] = (a[:, None] + b[None, :]).reshape(16)
    comb = _split(oracle_mod, np.zeros((1, MIX)), base=base, sink_eps=0.0, iters=1)["comb"][0]
    np.testing.assert_allclose(comb, 0.25, atol=1e-7)    # base is stored as float32


def test_sinkhorn_converges_to_2x2_block_closed_form(oracle_mod):
    # Block-diagonal exp(logits) (off-block logits -80 => ~1e-35): each 2x2 block
    # [[a, b], [c, d]] scales to [[p, 1-p], [1-p, p]], p = sqrt(ad)/(sqrt(ad)+sqrt(bc)).
    L = np.full((4, 4), -80.0)
    blk1 = np.array([[0.5, -1.0], [2.0, 0.25]])
    blk2 = np.array([[1.5, 0.0], [-0.75, 1.0]])
    L[:2, :2], L[2:, 2:] = blk1, blk2
    base = np.zeros(MIX, np.float32)
    base[8:] = L.reshape(16)
    comb = _split(oracle_mod, np.zeros((1, MIX)), base=base, sink_eps=0.0, iters=2000)["comb"][0]
    for (r0, blk) in ((0, blk1), (2, blk2)):
        a, b_, c, d = np.exp(blk.astype(np.float32).astype(np.float64)).reshape(4)
        p = math.sqrt(a * d) / (math.sqrt(a * d) + math.sqrt(b_ * c))
        np.testing.assert_allclose(comb[r0:r0 + 2, r0:r0 + 2], [[p, 1 - p], [1 - p, p]], atol=1e-12)
    assert comb[:2, 2:].max() < 1e-30 and comb[2:, :2].max() < 1e-30


def test_sinkhorn_doubly_stochastic_when_converged(oracle_mod):
    rng = np.random.default_rng(9)
    mix = np.zeros((64, MIX))
    base = np.zeros(MIX, np.float32)
    out = oracle_mod.split_sinkhorn(mix + rng.standard_normal((64, MIX)) * 3.0,
                                    np.array([0, 0, 1], np.float32), base, 1e-6, 1e-6, 2.0, 2000)
    comb = out["comb"]
    assert np.max(np.abs(comb.sum(axis=1) - 1)) < 2e-6
    assert np.max(np.abs(comb.sum(axis=2) - 1)) < 2e-6
    assert np.all(comb > 0)


def test_gate_ranges(oracle_mod):
    rng = np.random.default_rng(1)
    out = oracle_mod.split_sinkhorn(rng.standard_normal((256, MIX)) * 4,
                                    np.array([1, 1, 1], np.float32),
                                    (rng.standard_normal(MIX) * 3).astype(np.float32),
                                    1e-6, 1e-6, 2.0, 20)
    assert np.all(out["pre"] > 1e-6) and np.all(out["pre"] < 1 + 1e-6)
    assert np.all(out["post"] > 0) and np.all(out["post"] < 2)


# --------------------------------------------------------------------------- a4 combine + norm
def test_combine_norm_one_hot_pre_constant_stream(oracle_mod):
    # stream i constant c_i, pre = e_i, w = 1  =>  x_norm = bf16(c_i / sqrt(c_i^2 + eps)).
    cs = [0.5, -2.0, 0.125, 3.0]
    R = np.zeros((1, HC, H), np.uint16)
    for i, c in enumerate(cs):
        R[0, i, :] = bf(c)
    w = bf(np.ones(H))
    eps = 0.75
    for i, c in enumerate(cs):
        pre = np.zeros((1, HC))
        pre[0, i] = 1.0
        xn = oracle_mod.combine_norm(R, pre, w, eps)
        want = oracle_mod.to_bf16(np.array([c / math.sqrt(c * c + eps)]))[0]
        assert np.all(xn == want), (i, xn[0, :4], want)


def test_combine_norm_gates_are_per_row(oracle_mod):
    # four rows with the same constant streams c_i, row m gated by e_(3-m):
    # row m's x_norm is the closed form of stream 3-m, so each row must read
    # its own gates
    cs = [0.5, -2.0, 0.125, 3.0]
    R = np.zeros((HC, HC, H), np.uint16)
    for i, c in enumerate(cs):
        R[:, i, :] = bf(c)
    pre = np.zeros((HC, HC))
    for m in range(HC):
        pre[m, HC - 1 - m] = 1.0
    eps = 0.75
    xn = oracle_mod.combine_norm(R, pre, bf(np.ones(H)), eps)
    for m in range(HC):
        c = cs[HC - 1 - m]
        want = oracle_mod.to_bf16(np.array([c / math.sqrt(c * c + eps)]))[0]
        assert np.all(xn[m] == want), (m, xn[m, :4], want)


def test_combine_norm_weighted_sum_and_per_column_weight(oracle_mod):
    # pre = (a, b, 0, 0) on constant streams: y = a c0 + b c1 everywhere; the
    # weight multiplies column h.  Exact: y/|y| = sign(y) when eps = 0.
    R = np.zeros((1, HC, H), np.uint16)
    R[0, 0, :], R[0, 1, :], R[0, 2, :], R[0, 3, :] = bf(1.0), bf(-3.0), bf(100.0), bf(7.0)
    w = bf(np.random.default_rng(3).uniform(0.5, 1.5, H))
    pre = np.array([[0.25, 0.5, 0.0, 0.0]])         # y = 0.25 - 1.5 = -1.25
    xn = oracle_mod.combine_norm(R, pre, w, 0.0)
    np.testing.assert_array_equal(xn[0], w ^ np.uint16(0x8000))


def test_combine_norm_mean_is_over_hidden_5120(oracle_mod):
    # y = c on the first half of the columns, 0 on the rest: mean(y^2) = c^2/2,
    # so x_norm = sqrt(2) * sign(c) * w there (eps = 0).
    R = np.zeros((1, HC, H), np.uint16)
    R[0, 2, : H // 2] = bf(0.375)
    w = bf(np.ones(H))
    pre = np.array([[0.0, 0.0, 1.0, 0.0]])
    xn = oracle_mod.combine_norm(R, pre, w, 0.0)
    assert np.all(xn[0, : H // 2] == oracle_mod.to_bf16(np.array([math.sqrt(2.0)]))[0])
    assert np.all(xn[0, H // 2:] == 0)


def test_combine_norm_scale_invariance_and_column_permutation(oracle_mod):
    rng = np.random.default_rng(7)
    R = _random_rows(2, seed=8)
    pre = rng.uniform(0.0, 1.0, (2, HC))
    w = bf(1 + 0.1 * rng.standard_normal(H))
    a = oracle_mod.combine_norm(R, pre, w, 0.0)
    b = oracle_mod.combine_norm(bf(unbf(R) * 4.0), pre, w, 0.0)
    np.testing.assert_array_equal(a, b)
    perm = rng.permutation(H)
    c = oracle_mod.combine_norm(R[:, :, perm], pre, w[perm], 0.0)
    np.testing.assert_array_equal(c, a[:, perm])


def test_combine_norm_unfused_rounding_within_one_ulp(oracle_mod):
    R = _random_rows(4, seed=12)
    pre = np.random.default_rng(0).uniform(0.0, 1.0, (4, HC))
    w = bf(1 + 0.1 * np.random.default_rng(1).standard_normal(H))
    a = unbf(oracle_mod.combine_norm(R, pre, w, 1e-6))
    b = unbf(oracle_mod.combine_norm(R, pre, w, 1e-6, round_y=True))
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(a), 1e-30))) - 7)
    assert np.all(np.abs(a - b) <= ulp)


# --------------------------------------------------------------------------- a5 post
def test_post_identity_comb_returns_residual_bits(oracle_mod):
    R = _random_rows(3, seed=21, scale=20.0)
    y = bf(np.random.default_rng(0).standard_normal((3, H)))
    out = oracle_mod.post(R, y, np.zeros((3, HC), np.float32), np.tile(np.eye(4, dtype=np.float32), (3, 1, 1)))
    np.testing.assert_array_equal(out, R)


def test_post_permutation_orientation(oracle_mod):
    # comb[j][i] = 1 iff j = pi(i)  =>  R_out[i] = R[pi(i)]: the sum runs over the
    # first index of comb (hc_post_torch_impl sums comb[:, j, i] * R[:, j] over j).
    R = _random_rows(2, seed=22)
    y = bf(np.zeros((2, H)))
    pi = [2, 0, 3, 1]
    comb = np.zeros((2, HC, HC), np.float32)
    for i, j in enumerate(pi):
        comb[:, j, i] = 1.0
    out = oracle_mod.post(R, y, np.zeros((2, HC), np.float32), comb)
    for i, j in enumerate(pi):
        np.testing.assert_array_equal(out[:, i], R[:, j])


def test_post_gate_only(oracle_mod):
    y = bf(np.random.default_rng(1).standard_normal((2, H)))
    R = _random_rows(2, seed=23)
    pw = np.array([[1.0, 0.5, 0.25, 2.0]] * 2, np.float32)
    out = oracle_mod.post(R, y, pw, np.zeros((2, HC, HC), np.float32))
    for i in range(HC):
        np.testing.assert_array_equal(out[:, i], bf(unbf(y) * pw[0, i]))


def test_post_exact_integer_brute_force(oracle_mod):
    # small-integer R and y, dyadic post/comb: every sum is exact and small
    # enough to be a bf16 value, so the result is fixed by integer arithmetic.
    rng = np.random.default_rng(5)
    rows = 3
    Ri = rng.integers(-8, 9, (rows, HC, H))
    yi = rng.integers(-8, 9, (rows, H))
    pq = rng.integers(-4, 5, (rows, HC))          # post = pq / 4
    cq = rng.integers(0, 5, (rows, HC, HC))       # comb = cq / 4
    out = oracle_mod.post(bf(Ri), bf(yi), (pq / 4).astype(np.float32), (cq / 4).astype(np.float32))
    want4 = pq[:, :, None] * yi[:, None, :] + np.einsum("mji,mjh->mih", cq, Ri)   # 4 * R_out
    assert np.abs(want4).max() / 4 < 256
    np.testing.assert_array_equal(unbf(out), want4 / 4.0)


# --------------------------------------------------------------------------- wiring
def test_pre_is_composition_of_parts(oracle_mod):
    R = synth.residual(0, 3)
    W = synth.weights(0)
    full = oracle_mod.pre(R, W.fn, W.scale, W.base, W.norm_w)
    mix, _ = oracle_mod.stats(R, W.fn, 1e-6)
    sp = oracle_mod.split_sinkhorn(mix, W.scale, W.base, 1e-6, 1e-6, 2.0, 20)
    xn = oracle_mod.combine_norm(R, sp["pre"], W.norm_w, 1e-6)
    np.testing.assert_array_equal(full["mix"], mix)
    for k in ("logits", "pre", "post", "comb"):
        np.testing.assert_array_equal(full[k], sp[k])
    np.testing.assert_array_equal(full["x_norm"], xn)
