"""The allocation-free pre entry point (mhc_pre_noalloc).

Callers that cannot hand libmhc device scratch -- a framework whose caching
allocator owns the device memory, an operator/plugin enqueue that must not
allocate, a serving loop that cannot afford cudaMalloc/cudaFree, a C/FFI
caller without a device allocator -- call mhc_pre_noalloc.  mhc_pre's kernels
take no scratch, so it is mhc_pre without the workspace argument.  Checked
here through the C ABI:
  * against the fp64 oracle element by element, on two calls in a row with
    different sizes and inputs (one-pass launch), and at 8 rows (decode-size
    launch); on sampled rows of a 2100-row chunk (the one-pass build that
    keeps fn resident, where mhc_pre streams it from its workspace);
  * bit-equal to mhc_pre on the same inputs below 2048 rows;
  * 4 row shards of a 2048-row chunk (logical_rows = 2048) give the full
    call's bits;
  * the host-side row limit (also covered without a GPU in test_abi_host).

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
    return R, W, (bf(R), f32(W.fn), f32(W.scale), f32(W.base), bf(W.norm_w))


def _outputs(torch, rows):
    return (torch.empty((rows, H), dtype=torch.bfloat16, device="cuda"),
            torch.empty((rows, HC), dtype=torch.float32, device="cuda"),
            torch.empty((rows, HC, HC), dtype=torch.float32, device="cuda"),
            torch.empty((rows, HC), dtype=torch.float32, device="cuda"),
            torch.empty((rows, MIX), dtype=torch.float32, device="cuda"))


def _bits(torch, t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _noalloc(m, args, outs, logical_rows=None):
    xn, post, comb, pre, mix = outs
    m.mhc_pre_noalloc(*args, xn, post, comb, logical_rows=logical_rows, pre_out=pre, mix_out=mix)


def _check_oracle(torch, oracle_mod, R, W, outs):
    xn, post, comb, pre, mix = outs
    o = P.oracle_rows_parallel(oracle_mod.pre, R, rows=R.shape[0], fn=W.fn, scale=W.scale,
                               base=W.base, w=W.norm_w)
    P.check_mix(mix.cpu().numpy(), o["mix"])
    P.check_gates(pre.cpu().numpy(), post.cpu().numpy(), o, W.scale, R, W.fn)
    P.check_abs(comb.cpu().numpy(), o["comb"], 1e-6, "comb")
    P.check_bf16(_bits(torch, xn), o["x_norm"], "x_norm",
                 term_mag=P.combine_term_magnitude(R, o["pre"], W.norm_w, 1e-6))


def _assert_same_bits(torch, a, b, what):
    for name, x, y in zip(("x_norm", "post", "comb", "pre", "mix"), a, b):
        assert np.array_equal(x.contiguous().view(torch.int32 if x.dtype == torch.float32
                                                  else torch.int16).cpu().numpy(),
                              y.contiguous().view(torch.int32 if y.dtype == torch.float32
                                                  else torch.int16).cpu().numpy()), \
            f"{what}: {name} bits differ"


@pytest.mark.parametrize("sizes", [((1500, 41), (701, 42)), ((8, 43), (3, 44))],
                         ids=["one-pass", "decode"])
def test_noalloc_against_the_oracle_two_calls_in_a_row(env, oracle_mod, sizes):
    torch, m = env
    cases = []
    for rows, seed in sizes:
        R, W, args = _inputs(torch, rows, seed)
        cases.append((R, W, args, _outputs(torch, rows)))
    for R, W, args, outs in cases:          # back to back, larger first
        _noalloc(m, args, outs)
    torch.cuda.synchronize()
    for R, W, args, outs in cases:
        _check_oracle(torch, oracle_mod, R, W, outs)
        ref = _outputs(torch, R.shape[0])
        xn, post, comb, pre, mix = ref
        m.mhc_pre(*args, x_norm=xn, post=post, comb=comb, pre_out=pre, mix_out=mix)
        torch.cuda.synchronize()
        _assert_same_bits(torch, outs, ref, f"noalloc vs mhc_pre at {R.shape[0]} rows")


def test_noalloc_above_the_streamed_threshold_against_the_oracle(env, oracle_mod):
    # 2100 rows: mhc_pre runs the 8-CTA build on fn's image in its workspace;
    # noalloc, without one, the 16-CTA build with fn resident.  Both meet the
    # oracle; their bits may differ by summation order.
    torch, m = env
    rows = 2100
    R, W, args = _inputs(torch, rows, 46)
    outs = _outputs(torch, rows)
    _noalloc(m, args, outs)
    ref = _outputs(torch, rows)
    xn, post, comb, pre, mix = ref
    m.mhc_pre(*args, x_norm=xn, post=post, comb=comb, pre_out=pre, mix_out=mix)
    torch.cuda.synchronize()
    idx = np.r_[0:64, 1000:1064, rows - 64:rows]
    o = P.oracle_rows_parallel(oracle_mod.pre, R[idx], rows=len(idx), fn=W.fn, scale=W.scale,
                               base=W.base, w=W.norm_w)
    for got in (outs, ref):
        g_xn, g_post, g_comb, g_pre, g_mix = got
        P.check_mix(g_mix.cpu().numpy()[idx], o["mix"])
        P.check_gates(g_pre.cpu().numpy()[idx], g_post.cpu().numpy()[idx], o, W.scale, R[idx], W.fn)
        P.check_abs(g_comb.cpu().numpy()[idx], o["comb"], 1e-6, "comb")
        P.check_bf16(_bits(torch, g_xn)[idx], o["x_norm"], "x_norm",
                     term_mag=P.combine_term_magnitude(R[idx], o["pre"], W.norm_w, 1e-6))
    assert m.mhc_kernel_status() == 0


def test_noalloc_row_shards_give_the_whole_chunk_bits(env):
    torch, m = env
    rows = 2048
    R, W, args = _inputs(torch, rows, 45)
    whole = _outputs(torch, rows)
    _noalloc(m, args, whole)
    parts = []
    for lo in range(0, rows, rows // 4):
        hi = lo + rows // 4
        sub = (args[0][lo:hi],) + args[1:]
        outs = _outputs(torch, hi - lo)
        _noalloc(m, sub, outs, logical_rows=rows)
        parts.append(outs)
    torch.cuda.synchronize()
    joined = tuple(torch.cat([p[i] for p in parts]) for i in range(5))
    _assert_same_bits(torch, joined, whole, "4 shards of 2048 rows")


def test_noalloc_row_limit(env):
    torch, m = env
    assert m.mhc_pre_noalloc_max_rows() == 1 << 24
