"""Parity of mhc_fused_post_pre (hc_post of one sublayer, then hc_pre of the
next on its result; deepseek_v4.py, the mhc_fused_post_pre path between
sublayers) against the oracle, through the C ABI.

R_out is checked against the oracle's hc_post (and must carry mhc_post's
bits exactly); the next pre's outputs are checked against the oracle's pre
applied to the R_out the GPU produced -- the composition's definition -- with
the pre pass's tolerances.  Row shards reproduce the whole chunk's bits.
"""
import numpy as np
import pytest

import synth
from tests import parity as P

pytestmark = pytest.mark.gpu

HC, H, K, MIX = 4, 5120, 20480, 24
NEXT = 100          # seed offset of the next sublayer's weights


@pytest.fixture(scope="module")
def torch():
    import torch as t
    assert t.cuda.is_available(), "GPU tests need a CUDA device"
    return t


@pytest.fixture(scope="module")
def mhc(torch):
    from hyper_connection_residual_mhc_gb300 import build as b
    b.build()
    import hyper_connection_residual_mhc_gb300 as m
    m.lib()
    return m


def _bf(torch, bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _f(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _bits(torch, t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class Chain:
    """A residual, a sublayer output, this sublayer's post/comb (from the
    oracle's pre of R) and the next sublayer's weights."""

    def __init__(self, torch, oracle, rows, seed):
        self.rows = rows
        self.R = synth.residual(seed, rows)
        self.y = synth.sublayer_out(seed, rows)
        W = synth.weights(seed)
        o = P.oracle_rows_parallel(oracle.pre, self.R, rows=rows, fn=W.fn, scale=W.scale,
                                   base=W.base, w=W.norm_w, want_x_norm=False)
        self.post = o["post"].astype(np.float32)
        self.comb = o["comb"].astype(np.float32)
        self.Wn = synth.weights(seed + NEXT)
        self.d = dict(R=_bf(torch, self.R), y=_bf(torch, self.y), post=_f(torch, self.post),
                      comb=_f(torch, self.comb), fn=_f(torch, self.Wn.fn),
                      scale=_f(torch, self.Wn.scale), base=_f(torch, self.Wn.base),
                      w=_bf(torch, self.Wn.norm_w))

    def gpu(self, torch, mhc, lo=0, hi=None, logical_rows=None):
        hi = self.rows if hi is None else hi
        d = self.d
        n = hi - lo
        pre = torch.empty((n, HC), dtype=torch.float32, device="cuda")
        mix = torch.empty((n, MIX), dtype=torch.float32, device="cuda")
        R2, xn, po, co = mhc.mhc_fused_post_pre(
            d["R"][lo:hi], d["y"][lo:hi], d["post"][lo:hi], d["comb"][lo:hi], d["fn"], d["scale"],
            d["base"], d["w"], logical_rows=logical_rows, pre_out=pre, mix_out=mix)
        return {"R_out": R2, "x_norm": xn, "post": po, "comb": co, "pre": pre, "mix": mix}


def _check(torch, oracle, c, g, idx=None):
    sel = (lambda a: a) if idx is None else (lambda a: a[idx])
    R, y, post, comb = sel(c.R), sel(c.y), sel(c.post), sel(c.comb)
    R2 = sel(_bits(torch, g["R_out"]))
    ref_R2 = oracle.post(R, y, post, comb)
    P.check_bf16(R2, ref_R2, "R_out", term_mag=P.post_term_magnitude(R, y, post, comb))
    # the next pre, on the residual the GPU produced
    o = P.oracle_rows_parallel(oracle.pre, R2, rows=R2.shape[0], fn=c.Wn.fn, scale=c.Wn.scale,
                               base=c.Wn.base, w=c.Wn.norm_w)
    P.check_mix(sel(g["mix"].cpu().numpy().astype(np.float64)), o["mix"])
    P.check_gates(sel(g["pre"].cpu().numpy().astype(np.float64)),
                  sel(g["post"].cpu().numpy().astype(np.float64)), o, c.Wn.scale, R2, c.Wn.fn)
    P.check_abs(sel(g["comb"].cpu().numpy().astype(np.float64)), o["comb"], 1e-6, "comb")
    P.check_bf16(sel(_bits(torch, g["x_norm"])), o["x_norm"], "x_norm",
                 term_mag=P.combine_term_magnitude(R2, o["pre"], c.Wn.norm_w, 1e-6))


@pytest.mark.parametrize("rows", [1, 7, 48, 49, 128, 129, 1500])
def test_fused_post_pre_every_row(torch, mhc, oracle_mod, rows):
    c = Chain(torch, oracle_mod, rows, 200 + rows)
    g = c.gpu(torch, mhc)
    torch.cuda.synchronize()
    _check(torch, oracle_mod, c, g)


def test_fused_R_out_has_mhc_post_bits(torch, mhc, oracle_mod):
    c = Chain(torch, oracle_mod, 300, 5)
    g = c.gpu(torch, mhc)
    d = c.d
    ref = mhc.mhc_post(d["R"], d["y"], d["post"], d["comb"])
    assert torch.equal(g["R_out"], ref)


@pytest.mark.parametrize("rows", [1, 7, 48])
def test_fused_decode_sizes_equal_post_then_pre_bits(torch, mhc, oracle_mod, rows):
    # at decode sizes the fused call is one launch (hc_post on the loaded
    # columns, then the decode pre on R'); it must give exactly what
    # mhc_post followed by mhc_pre gives
    c = Chain(torch, oracle_mod, rows, 400 + rows)
    g = c.gpu(torch, mhc)
    d = c.d
    R2 = mhc.mhc_post(d["R"], d["y"], d["post"], d["comb"])
    pre = torch.empty((rows, HC), dtype=torch.float32, device="cuda")
    mix = torch.empty((rows, MIX), dtype=torch.float32, device="cuda")
    xn, po, co = mhc.mhc_pre(R2, d["fn"], d["scale"], d["base"], d["w"], pre_out=pre, mix_out=mix)
    torch.cuda.synchronize()
    ref = {"R_out": R2, "x_norm": xn, "post": po, "comb": co, "pre": pre, "mix": mix}
    for k, v in ref.items():
        assert torch.equal(g[k], v), k


def test_fused_full_size_sampled_rows(torch, mhc, oracle_mod):
    rows = 16384
    R = synth.residual(4, rows)
    y = synth.sublayer_out(4, rows)
    c = Chain.__new__(Chain)
    c.rows, c.R, c.y = rows, R, y
    W = synth.weights(4)
    # this sublayer's post/comb from the GPU pre (tested elsewhere) keeps setup fast
    dR = _bf(torch, R)
    _, post, comb = mhc.mhc_pre(dR, _f(torch, W.fn), _f(torch, W.scale), _f(torch, W.base),
                                _bf(torch, W.norm_w))
    c.post = post.cpu().numpy()
    c.comb = comb.cpu().numpy()
    c.Wn = synth.weights(4 + NEXT)
    c.d = dict(R=dR, y=_bf(torch, y), post=post, comb=comb, fn=_f(torch, c.Wn.fn),
               scale=_f(torch, c.Wn.scale), base=_f(torch, c.Wn.base), w=_bf(torch, c.Wn.norm_w))
    g = c.gpu(torch, mhc)
    torch.cuda.synchronize()
    rng = np.random.default_rng(11)
    idx = np.unique(np.concatenate([[0, 127, 128, rows // 2, rows - 1], rng.integers(0, rows, 24)]))
    _check(torch, oracle_mod, c, g, idx)


@pytest.mark.parametrize("rows", [1500, 2048])
def test_fused_shards_and_repeat_are_bit_exact(torch, mhc, oracle_mod, rows):
    # 2048 rows: the 8-CTA build (from 2048 logical rows)
    c = Chain(torch, oracle_mod, rows, 33)
    full = c.gpu(torch, mhc)
    again = c.gpu(torch, mhc)
    for k in full:
        assert torch.equal(full[k], again[k]), k
    s = rows // 4
    for r in range(4):
        part = c.gpu(torch, mhc, r * s, (r + 1) * s, logical_rows=rows)
        for k in full:
            assert torch.equal(part[k], full[k][r * s:(r + 1) * s]), (k, r)


@pytest.mark.parametrize("rows", [7, 48, 49, 1500, 2100])   # 2100: the 8-CTA build, ragged
def test_fused_mxfp8_against_the_oracle(torch, mhc, oracle_mod, rows):
    # the fused boundary with the next x_norm as MXFP8 (prefill_sp.py,
    # _mxfp8_quantize on the attention input): R_out, x_norm, post and comb
    # are the bits of mhc_fused_post_pre_prepared, which the tests above
    # check against the oracle; the codes and scales equal the oracle's
    # quantization of that x_norm bit for bit
    c = Chain(torch, oracle_mod, rows, 600 + rows)
    d = c.d
    h = mhc.mhc_prepare_weights(d["fn"])
    R2, xn, q, s, po, co = mhc.mhc_fused_post_pre_mxfp8(d["R"], d["y"], d["post"], d["comb"], h,
                                                         d["scale"], d["base"], d["w"])
    ref = mhc.mhc_fused_post_pre_prepared(d["R"], d["y"], d["post"], d["comb"], h, d["scale"],
                                          d["base"], d["w"])
    torch.cuda.synchronize()
    for name, a, b in zip(("R_out", "x_norm", "post", "comb"), (R2, xn, po, co), ref):
        assert torch.equal(a, b), name
    q_ref, s_ref = oracle_mod.mxfp8_quantize(_bits(torch, xn))
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    # and the whole chain against the oracle's post then pre
    g = {"R_out": R2, "x_norm": xn, "post": po, "comb": co}
    o_R2 = oracle_mod.post(c.R, c.y, c.post, c.comb)
    P.check_bf16(_bits(torch, R2), o_R2, "R_out",
                 term_mag=P.post_term_magnitude(c.R, c.y, c.post, c.comb))
    o = P.oracle_rows_parallel(oracle_mod.pre, _bits(torch, R2), rows=rows, fn=c.Wn.fn,
                               scale=c.Wn.scale, base=c.Wn.base, w=c.Wn.norm_w)
    P.check_abs(co.cpu().numpy(), o["comb"], 1e-6, "comb")
    P.check_bf16(_bits(torch, g["x_norm"]), o["x_norm"], "x_norm",
                 term_mag=P.combine_term_magnitude(_bits(torch, R2), o["pre"], c.Wn.norm_w, 1e-6))
    h.release()
    assert mhc.mhc_kernel_status() == 0


def test_fused_mxfp8_row_shards(torch, mhc, oracle_mod):
    rows = 1500
    c = Chain(torch, oracle_mod, rows, 700)
    d = c.d
    h = mhc.mhc_prepare_weights(d["fn"])
    args = lambda lo, hi: (d["R"][lo:hi], d["y"][lo:hi], d["post"][lo:hi], d["comb"][lo:hi], h,
                           d["scale"], d["base"], d["w"])
    full = mhc.mhc_fused_post_pre_mxfp8(*args(0, rows))
    parts = [mhc.mhc_fused_post_pre_mxfp8(*args(r0, r0 + 375), logical_rows=rows)
             for r0 in range(0, rows, 375)]
    torch.cuda.synchronize()
    for k in range(6):
        assert torch.equal(full[k], torch.cat([p[k] for p in parts])), k
    h.release()
