"""Non-default scalars on every pre path: the one-pass tensor-core launch
(> 48 rows; its resident 16-CTA build, and its streamed 8-CTA build for chunks
of 2048 rows and more), the decode-size launch (<= 48 rows) and the fused
post->pre, against the
oracle run with the same scalars (deepseek_v4.py, DeepseekV4DecoderLayer.hc_pre
passes rms_eps, hc_pre_eps, hc_sinkhorn_eps, post_mult and sinkhorn_repeat
through to the kernels).  Catches a scalar that is accepted but not used."""
import numpy as np
import pytest

import synth
from tests import parity as P

pytestmark = pytest.mark.gpu

HC, H, K, MIX = 4, 5120, 20480, 24
SCALARS = dict(rms_eps=0.25, hc_pre_eps=0.125, hc_sinkhorn_eps=0.5, norm_eps=0.0625, post_mult=3.0,
               iters=3)


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


def _params(mhc):
    s = SCALARS
    return mhc.default_params(rms_eps=s["rms_eps"], hc_pre_eps=s["hc_pre_eps"],
                              hc_sinkhorn_eps=s["hc_sinkhorn_eps"], norm_eps=s["norm_eps"],
                              post_mult=s["post_mult"], sinkhorn_iters=s["iters"])


def _check(torch, g, o, R, W):
    P.check_mix(g["mix"].cpu().numpy(), o["mix"])
    P.check_gates(g["pre"].cpu().numpy(), g["post"].cpu().numpy(), o, W.scale, R, W.fn,
                  post_mult=SCALARS["post_mult"], rms_eps=SCALARS["rms_eps"])
    P.check_abs(g["comb"].cpu().numpy(), o["comb"], 1e-6, "comb")
    P.check_bf16(_bits(torch, g["x_norm"]), o["x_norm"], "x_norm",
                 term_mag=P.combine_term_magnitude(R, o["pre"], W.norm_w, SCALARS["norm_eps"]))


def _oracle(oracle, R, W):
    s = SCALARS
    return P.oracle_rows_parallel(oracle.pre, R, rows=R.shape[0], fn=W.fn, scale=W.scale,
                                  base=W.base, w=W.norm_w, rms_eps=s["rms_eps"],
                                  hc_pre_eps=s["hc_pre_eps"], hc_sinkhorn_eps=s["hc_sinkhorn_eps"],
                                  norm_eps=s["norm_eps"], post_mult=s["post_mult"],
                                  iters=s["iters"])


# decode-size launch; the one-pass launch, resident build; the streamed build
# (200 rows as a shard of a 2048-row chunk)
@pytest.mark.parametrize("rows,logical", [(8, 8), (200, 200), (200, 2048)])
def test_pre_with_other_scalars(torch, mhc, oracle_mod, rows, logical):
    R = synth.residual(70 + rows, rows)
    W = synth.weights(70 + rows)
    pre = torch.empty((rows, HC), dtype=torch.float32, device="cuda")
    mix = torch.empty((rows, MIX), dtype=torch.float32, device="cuda")
    xn, post, comb = mhc.mhc_pre(_bf(torch, R), _f(torch, W.fn), _f(torch, W.scale),
                                 _f(torch, W.base), _bf(torch, W.norm_w), logical_rows=logical,
                                 params=_params(mhc), pre_out=pre, mix_out=mix)
    torch.cuda.synchronize()
    g = {"x_norm": xn, "post": post, "comb": comb, "pre": pre, "mix": mix}
    _check(torch, g, _oracle(oracle_mod, R, W), R, W)


# the prepared call: the one-pass launch streaming fn from the handle's image
# (16-CTA clusters below 2048 logical rows, 8-CTA from there on)
@pytest.mark.parametrize("rows,logical", [(200, 200), (200, 2048)])
def test_prepared_pre_with_other_scalars(torch, mhc, oracle_mod, rows, logical):
    R = synth.residual(80 + rows, rows)
    W = synth.weights(80 + rows)
    handle = mhc.mhc_prepare_weights(_f(torch, W.fn))
    pre = torch.empty((rows, HC), dtype=torch.float32, device="cuda")
    mix = torch.empty((rows, MIX), dtype=torch.float32, device="cuda")
    xn, post, comb = mhc.mhc_pre_prepared(_bf(torch, R), handle, _f(torch, W.scale),
                                          _f(torch, W.base), _bf(torch, W.norm_w),
                                          logical_rows=logical, params=_params(mhc),
                                          pre_out=pre, mix_out=mix)
    torch.cuda.synchronize()
    handle.release()
    g = {"x_norm": xn, "post": post, "comb": comb, "pre": pre, "mix": mix}
    _check(torch, g, _oracle(oracle_mod, R, W), R, W)


def test_fused_post_pre_with_other_scalars(torch, mhc, oracle_mod):
    rows = 200
    R = synth.residual(91, rows)
    y = synth.sublayer_out(91, rows)
    W = synth.weights(91)
    Wn = synth.weights(191)
    o = oracle_mod.pre(R, W.fn, W.scale, W.base, W.norm_w, want_x_norm=False)
    post, comb = o["post"].astype(np.float32), o["comb"].astype(np.float32)
    pre = torch.empty((rows, HC), dtype=torch.float32, device="cuda")
    mix = torch.empty((rows, MIX), dtype=torch.float32, device="cuda")
    R2, xn, po, co = mhc.mhc_fused_post_pre(
        _bf(torch, R), _bf(torch, y), _f(torch, post), _f(torch, comb), _f(torch, Wn.fn),
        _f(torch, Wn.scale), _f(torch, Wn.base), _bf(torch, Wn.norm_w), params=_params(mhc),
        pre_out=pre, mix_out=mix)
    torch.cuda.synchronize()
    R2b = _bits(torch, R2)
    g = {"x_norm": xn, "post": po, "comb": co, "pre": pre, "mix": mix}
    _check(torch, g, _oracle(oracle_mod, R2b, Wn), R2b, Wn)
