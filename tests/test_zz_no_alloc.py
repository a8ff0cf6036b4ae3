"""The allocation-free pre entry point (mhc_pre_noalloc).

Callers that cannot hand libmhc device scratch -- a framework whose caching
allocator owns the device memory, an operator/plugin enqueue that must not
allocate, a serving loop that cannot afford cudaMalloc/cudaFree, a C/FFI
caller without a device allocator -- use mhc_pre_noalloc, whose scratch is a
fixed device array inside the library.  This checks, through the C ABI, that it
gives what mhc_pre gives (within the parity tolerances of the other tests) on
two calls in a row with different inputs and sizes, so that nothing left in
the shared scratch by the first call leaks into the second, and that it
rejects a row count above its fixed limit.

This file is collected last on purpose: run alone in a fresh process or after
every other test, it sets up its own inputs.
"""
import numpy as np
import pytest

import synth
from tests import parity as P

pytestmark = pytest.mark.gpu

HC, H, MIX = 4, 5120, 24


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from hyper_connection_residual_mhc_gb300 import build as b
    b.build()
    import hyper_connection_residual_mhc_gb300 as m
    m.lib()
    return torch, m


def _inputs(torch, rows, seed):
    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()

    def f32(a):
        return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()

    R = synth.residual(seed, rows)
    W = synth.weights(seed)
    return R, W, bf(R), f32(W.fn), f32(W.scale), f32(W.base), bf(W.norm_w)


def _outputs(torch, rows):
    return (torch.empty((rows, H), dtype=torch.bfloat16, device="cuda"),
            torch.empty((rows, HC), dtype=torch.float32, device="cuda"),
            torch.empty((rows, HC, HC), dtype=torch.float32, device="cuda"),
            torch.empty((rows, HC), dtype=torch.float32, device="cuda"),
            torch.empty((rows, MIX), dtype=torch.float32, device="cuda"))


def _bits(torch, t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def test_noalloc_matches_mhc_pre_on_two_calls_in_a_row(env):
    torch, m = env
    assert m.mhc_pre_noalloc_max_rows() == 16384
    # two mhc_pre_noalloc calls back to back, larger first, so the second runs
    # on scratch the first one left full of its own values; then the
    # workspace-taking mhc_pre on the same inputs as the reference.
    cases = []
    for rows, seed in ((1500, 41), (701, 42)):
        R, W, dR, dfn, dscale, dbase, dw = _inputs(torch, rows, seed)
        cases.append((rows, R, W, (dR, dfn, dscale, dbase, dw), _outputs(torch, rows)))
    for rows, R, W, args, (xn, post, comb, pre, mix) in cases:
        m.mhc_pre_noalloc(*args, xn, post, comb, pre_out=pre, mix_out=mix)
    for rows, R, W, args, got in cases:
        rxn, rpost, rcomb, rpre, rmix = _outputs(torch, rows)
        m.mhc_pre(*args, x_norm=rxn, post=rpost, comb=rcomb, pre_out=rpre, mix_out=rmix)
        torch.cuda.synchronize()
        xn, post, comb, pre, mix = got
        ref_pre = rpre.cpu().numpy()
        P.check_mix(mix.cpu().numpy(), rmix.cpu().numpy())
        P.check_abs(pre.cpu().numpy(), ref_pre, 1e-6, "pre")
        P.check_abs(post.cpu().numpy(), rpost.cpu().numpy(), 1e-6, "post")
        P.check_abs(comb.cpu().numpy(), rcomb.cpu().numpy(), 1e-6, "comb")
        P.check_bf16(_bits(torch, xn), _bits(torch, rxn), "x_norm",
                     term_mag=P.combine_term_magnitude(R, ref_pre, W.norm_w, 1e-6))


def test_noalloc_rejects_rows_above_its_scratch(env):
    torch, m = env
    rows = m.mhc_pre_noalloc_max_rows() + 1
    # only shapes matter: the check fires on the host before anything runs
    R = torch.empty((rows, HC, H), dtype=torch.bfloat16, device="cuda")
    _, _, dR, dfn, dscale, dbase, dw = _inputs(torch, 1, 43)
    xn, post, comb, _, _ = _outputs(torch, rows)
    with pytest.raises(m.MhcError) as e:
        m.mhc_pre_noalloc(R, dfn, dscale, dbase, dw, xn, post, comb)
    assert e.value.code == -9
