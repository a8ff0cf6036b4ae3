"""Prepared weights (mhc_prepare_weights / mhc_pre_prepared).

The handle holds a copy of fn and the one-pass kernel's bf16 hi/lo operand image,
written by a prep kernel through the same conversion routine the kernel uses
itself, so mhc_pre_prepared must give exactly mhc_pre's bits -- on the decode
path (which reads the fp32 copy) and on the tensor-core path (which streams
fn's tiles from the image instead of converting fn).
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

HC, H, MIX = 4, 5120, 24


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


def _run(torch, call, rows):
    pre = torch.empty((rows, HC), dtype=torch.float32, device="cuda")
    mix = torch.empty((rows, MIX), dtype=torch.float32, device="cuda")
    xn, post, comb = call(pre, mix)
    torch.cuda.synchronize()
    return {"x_norm": xn, "post": post, "comb": comb, "pre": pre, "mix": mix}


@pytest.mark.parametrize("rows", [8, 49, 129, 1500, 4096])
def test_prepared_equals_mhc_pre_bits(torch, mhc, rows):
    W = synth.weights(9)
    R = _bf(torch, synth.residual(9, rows))
    fn = torch.from_numpy(W.fn).cuda()
    scale = torch.from_numpy(W.scale).cuda()
    base = torch.from_numpy(W.base).cuda()
    w = _bf(torch, W.norm_w)
    ref = _run(torch, lambda pre, mix: mhc.mhc_pre(R, fn, scale, base, w, pre_out=pre,
                                                   mix_out=mix), rows)
    handle = mhc.mhc_prepare_weights(fn)
    got = _run(torch, lambda pre, mix: mhc.mhc_pre_prepared(R, handle, scale, base, w,
                                                            pre_out=pre, mix_out=mix), rows)
    for k in ref:
        assert torch.equal(got[k], ref[k]), k
    # the handle keeps its own copy: changing the caller's fn afterwards
    # changes nothing
    fn.zero_()
    again = _run(torch, lambda pre, mix: mhc.mhc_pre_prepared(R, handle, scale, base, w,
                                                              pre_out=pre, mix_out=mix), rows)
    for k in ref:
        assert torch.equal(again[k], ref[k]), k
    handle.release()
    assert mhc.mhc_kernel_status() == 0


@pytest.mark.parametrize("rows", [1500, 4096])
def test_prepared_row_shards_reproduce_whole_chunk_bits(torch, mhc, rows):
    # prefill_sp.py, sp_logical_rows / shard_range: rank r of 4 runs rows
    # [r*M/4, (r+1)*M/4) with the whole chunk's row count as the key; 1500
    # rows take the 16-CTA streamed build, 4096 the 8-CTA one
    W = synth.weights(14)
    R = _bf(torch, synth.residual(14, rows))
    scale = torch.from_numpy(W.scale).cuda()
    base = torch.from_numpy(W.base).cuda()
    w = _bf(torch, W.norm_w)
    handle = mhc.mhc_prepare_weights(torch.from_numpy(W.fn).cuda())
    full = _run(torch, lambda pre, mix: mhc.mhc_pre_prepared(R, handle, scale, base, w,
                                                             pre_out=pre, mix_out=mix), rows)
    s = rows // 4
    for r in range(4):
        lo, hi = r * s, (r + 1) * s
        got = _run(torch, lambda pre, mix: mhc.mhc_pre_prepared(
            R[lo:hi], handle, scale, base, w, logical_rows=rows, pre_out=pre, mix_out=mix), s)
        for k in full:
            assert torch.equal(got[k], full[k][lo:hi]), (k, r)
    handle.release()
    assert mhc.mhc_kernel_status() == 0


def test_released_handle_is_refused(torch, mhc):
    W = synth.weights(3)
    handle = mhc.mhc_prepare_weights(torch.from_numpy(W.fn).cuda())
    handle.release()
    handle.release()                       # a second release is a no-op
    R = torch.zeros((4, HC, H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        mhc.mhc_pre_prepared(R, handle, torch.from_numpy(W.scale).cuda(),
                             torch.from_numpy(W.base).cuda(), _bf(torch, W.norm_w))


@pytest.mark.parametrize("rows", [8, 1500])
def test_fused_prepared_equals_fused_bits(torch, mhc, rows):
    # the next sublayer's fn through a handle; the prepared call runs with the
    # smaller workspace (no room for fn's image)
    W, Wn = synth.weights(12), synth.weights(13)
    R = _bf(torch, synth.residual(12, rows))
    y = _bf(torch, synth.sublayer_out(12, rows))
    _, post, comb = mhc.mhc_pre(R, torch.from_numpy(W.fn).cuda(), torch.from_numpy(W.scale).cuda(),
                                torch.from_numpy(W.base).cuda(), _bf(torch, W.norm_w))
    fn = torch.from_numpy(Wn.fn).cuda()
    scale = torch.from_numpy(Wn.scale).cuda()
    base = torch.from_numpy(Wn.base).cuda()
    w = _bf(torch, Wn.norm_w)
    ref = mhc.mhc_fused_post_pre(R, y, post, comb, fn, scale, base, w)
    handle = mhc.mhc_prepare_weights(fn)
    ws = torch.empty((max(256, mhc.mhc_pre_workspace_bytes(rows)),), dtype=torch.uint8,
                     device="cuda")
    got = mhc.mhc_fused_post_pre_prepared(R, y, post, comb, handle, scale, base, w, workspace=ws)
    torch.cuda.synchronize()
    for name, a, b in zip(("R_out", "x_norm", "post", "comb"), got, ref):
        assert torch.equal(a, b), name
    handle.release()
    assert mhc.mhc_kernel_status() == 0
