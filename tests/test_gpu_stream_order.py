"""Stream order across back-to-back calls.

Chunks of up to 2048 rows launch with programmatic stream serialization, so
a kernel's blocks can be resident before the previous kernel on the stream
has finished; each kernel must wait for it before touching memory.  Here
several mhc_pre + mhc_post steps run on one stream with no synchronisation
between them, each step on a different R, all steps sharing one post / comb
buffer: step i + 1's pre writes the buffer that step i's post reads
(write-after-read), and each post reads what its own pre wrote
(read-after-write).  Every step's outputs must be bit-identical to the same
step run alone.  Sizes cover the one-launch decode pre (48 rows), the
one-pass pre with the attribute (128: the resident 16-CTA build; 2048: the
streamed 8-CTA build, after its fn-image launch) and without it (4096).
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

HC, H = 4, 5120
STEPS = 4


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


def _dev_bf16(torch, bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("rows", [48, 128, 2048, 4096])
def test_back_to_back_steps_keep_stream_order(torch, mhc, rows):
    W = synth.weights(7)
    fn = torch.from_numpy(W.fn).cuda()
    scale = torch.from_numpy(W.scale).cuda()
    base = torch.from_numpy(W.base).cuda()
    w = _dev_bf16(torch, W.norm_w)
    y = _dev_bf16(torch, synth.sublayer_out(7, rows))
    Rs = [_dev_bf16(torch, synth.residual(20 + i, rows)) for i in range(STEPS)]
    ws = torch.empty((max(256, mhc.mhc_pre_workspace_bytes(rows)),), dtype=torch.uint8,
                     device="cuda")

    # each step alone, synchronised before and after
    ref = []
    for R in Rs:
        torch.cuda.synchronize()
        xn, post, comb = mhc.mhc_pre(R, fn, scale, base, w, workspace=ws)
        R2 = mhc.mhc_post(R, y, post, comb)
        torch.cuda.synchronize()
        ref.append((xn.clone(), R2.clone()))

    # the same steps back to back on one stream, sharing the gate buffers
    post = torch.empty((rows, HC), dtype=torch.float32, device="cuda")
    comb = torch.empty((rows, HC, HC), dtype=torch.float32, device="cuda")
    xns = [torch.empty((rows, H), dtype=torch.bfloat16, device="cuda") for _ in range(STEPS)]
    R2s = [torch.empty_like(Rs[0]) for _ in range(STEPS)]
    s = torch.cuda.current_stream()
    torch.cuda.synchronize()
    for _ in range(3):                          # a few rounds: the race window is timing-dependent
        for i, R in enumerate(Rs):
            mhc.mhc_pre(R, fn, scale, base, w, workspace=ws, x_norm=xns[i], post=post, comb=comb,
                        stream=s)
            mhc.mhc_post(R, y, post, comb, out=R2s[i], stream=s)
        torch.cuda.synchronize()
        for i in range(STEPS):
            assert torch.equal(xns[i].view(torch.int16), ref[i][0].view(torch.int16)), ("x_norm", i)
            assert torch.equal(R2s[i].view(torch.int16), ref[i][1].view(torch.int16)), ("R_out", i)
    assert mhc.mhc_kernel_status() == 0
