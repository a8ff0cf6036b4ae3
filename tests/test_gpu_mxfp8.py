"""MXFP8 output of x_norm (prefill_sp.py, _mxfp8_quantize and swizzle_128x4)
against the oracle, bit for bit.

The codes and scales are integer decisions taken from bf16 values, so both
sides start from the same bf16 bits: the GPU's own x_norm for mhc_pre_mxfp8
(whose bits are mhc_pre's, checked here too), synthetic rows for the
standalone quantizer.
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

HC, H = 4, 5120


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


def _bits(torch, t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def special_rows(rows, cols, seed):
    """bf16 rows whose 32-column blocks span many magnitudes, plus the edge
    cases: an all-zero block, signed zeros, values that saturate (block amax
    in [448, 512) after scaling), bf16 subnormals, ties of E4M3 rounding."""
    rng = np.random.default_rng(seed)
    nb = cols // 32
    e = rng.integers(-40, 40, size=(rows, nb)).astype(float)
    x = rng.standard_normal((rows, cols)) * np.repeat(2.0 ** e, 32, axis=1)
    if nb >= 2:
        x[0, 0:32] = 0.0
        x[0, 32:64] = -0.0
        x[0, 33] = 1.9375                        # amax 1.9375 -> 496 after scaling: saturates
        x[0, 34] = -1.8125                       # 464: saturates
        x[0, 35] = 1.0 + 1 / 16                  # 272: tie 256 / 288 -> 256
        x[0, 36] = 2.0 ** -133                   # smallest bf16 subnormal
        x[0, 37] = -(2.0 ** -18)                 # t = -2^-10: ties to -0
    if rows > 1 and nb >= 1:
        x[1, 0:32] = 2.0 ** -130 * np.arange(1, 33)     # a block of bf16 subnormals
    return oracle.to_bf16(x)


@pytest.mark.parametrize("rows,cols", [(1, 32), (37, 96), (5, 5120), (1000, 5120)])
def test_quantize_matches_oracle(torch, mhc, rows, cols):
    xb = special_rows(rows, cols, seed=rows + cols)
    q, s = mhc.mhc_quantize_mxfp8(_bf(torch, xb))
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.mxfp8_quantize(xb)
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)


@pytest.mark.parametrize("rows,groups", [(1, 4), (128, 160), (300, 8), (1500, 160)])
def test_swizzle_matches_oracle(torch, mhc, rows, groups):
    rng = np.random.default_rng(rows * 7 + groups)
    s = rng.integers(1, 256, size=(rows, groups), dtype=np.uint8)
    out = mhc.mhc_swizzle_scales_128x4(torch.from_numpy(s).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), oracle.swizzle_128x4(s))


@pytest.mark.parametrize("rows", [8, 48, 1500, 4096])
def test_pre_mxfp8(torch, mhc, rows):
    # 4096 rows: the streamed 8-CTA build of the one-pass kernel (from 2048 rows)
    W = synth.weights(10)
    R = _bf(torch, synth.residual(10, rows))
    fn = torch.from_numpy(W.fn).cuda()
    scale = torch.from_numpy(W.scale).cuda()
    base = torch.from_numpy(W.base).cuda()
    w = _bf(torch, W.norm_w)
    h = mhc.mhc_prepare_weights(fn)
    xn_ref, post_ref, comb_ref = mhc.mhc_pre_prepared(R, h, scale, base, w)
    xn, q, s, post, comb = mhc.mhc_pre_mxfp8(R, h, scale, base, w)
    torch.cuda.synchronize()
    assert torch.equal(xn, xn_ref) and torch.equal(post, post_ref) and torch.equal(comb, comb_ref)
    q_ref, s_ref = oracle.mxfp8_quantize(_bits(torch, xn))
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    # the whole chunk's scales, tiled: the oracle's tiling of the same bytes
    sw = mhc.mhc_swizzle_scales_128x4(s)
    torch.cuda.synchronize()
    assert np.array_equal(sw.cpu().numpy(), oracle.swizzle_128x4(s_ref))
    h.release()
    assert mhc.mhc_kernel_status() == 0


@pytest.mark.parametrize("rows", [1500, 4096])
def test_pre_mxfp8_row_shards(torch, mhc, rows):
    # 4 shards (logical_rows = rows): every output, codes and scales
    # included, equals the whole-chunk call's
    W = synth.weights(11)
    R = _bf(torch, synth.residual(11, rows))
    h = mhc.mhc_prepare_weights(torch.from_numpy(W.fn).cuda())
    scale = torch.from_numpy(W.scale).cuda()
    base = torch.from_numpy(W.base).cuda()
    w = _bf(torch, W.norm_w)
    full = mhc.mhc_pre_mxfp8(R, h, scale, base, w)
    sh = rows // 4
    parts = [mhc.mhc_pre_mxfp8(R[r0:r0 + sh], h, scale, base, w, logical_rows=rows)
             for r0 in range(0, rows, sh)]
    torch.cuda.synchronize()
    for k in range(5):
        assert torch.equal(full[k], torch.cat([p[k] for p in parts])), k
    h.release()
