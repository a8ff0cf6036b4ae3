"""Parity of mhc_hc_head (the final stream collapse) on the GPU against the
oracle (deepseek_v4.py, hc_head_torch), through the C ABI.

Same workloads and tolerances as the pre pass: the 4 mixes to 1e-4 of the
row's mix scale, the gates to 1e-6, y to 2 bf16 ulp (or 2e-2 on the x40
columns, or 2 ulp of the largest pre_i R_i term where the streams cancel).
Row shards reproduce the whole chunk's bits.
"""
import numpy as np
import pytest

import synth
from tests import parity as P

pytestmark = pytest.mark.gpu

HC, H, K = 4, 5120, 20480
WL = {w.rows: w for w in synth.WORKLOADS}


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


def _dev_f32(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _bits(torch, t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _term_mag(R_bits, pre):
    R = P.unbf(R_bits)
    return np.max(np.abs(np.asarray(pre, np.float64))[:, :, None] * np.abs(R), axis=1)


def _run(torch, mhc, dR, hw, lo=0, hi=None, logical_rows=None):
    hi = dR.shape[0] if hi is None else hi
    n = hi - lo
    pre = torch.empty((n, HC), dtype=torch.float32, device="cuda")
    mix = torch.empty((n, HC), dtype=torch.float32, device="cuda")
    y = mhc.mhc_hc_head(dR[lo:hi], _dev_f32(torch, hw.fn), _dev_f32(torch, hw.scale),
                        _dev_f32(torch, hw.base), logical_rows=logical_rows, pre_out=pre,
                        mix_out=mix)
    return y, pre, mix


def _check(torch, y, pre, mix, R, o, idx=None):
    sel = (lambda a: a) if idx is None else (lambda a: a[idx])
    P.check_mix(sel(mix.cpu().numpy().astype(np.float64)), o["mix"], "head mix")
    P.check_abs(sel(pre.cpu().numpy().astype(np.float64)), o["pre"], 1e-6, "head pre")
    P.check_bf16(sel(_bits(torch, y)), o["y"], "head y", term_mag=_term_mag(R, o["pre"]))


@pytest.mark.parametrize("rows", [1, 7, 128, 129, 257, 1500])
def test_hc_head_every_row(torch, mhc, oracle_mod, rows):
    seed = WL[rows].seed if rows in WL else 40 + rows
    R = synth.residual(seed, rows)
    hw = synth.head_weights(seed)
    y, pre, mix = _run(torch, mhc, _dev_bf16(torch, R), hw)
    torch.cuda.synchronize()
    o = P.oracle_rows_parallel(oracle_mod.hc_head, R, rows=rows, fn=hw.fn, scale=hw.scale,
                               base=hw.base)
    _check(torch, y, pre, mix, R, o)


@pytest.mark.parametrize("rows", [4096, 16384])
def test_hc_head_full_size_sampled_rows(torch, mhc, oracle_mod, rows):
    seed = WL[rows].seed
    R = synth.residual(seed, rows)
    hw = synth.head_weights(seed)
    y, pre, mix = _run(torch, mhc, _dev_bf16(torch, R), hw)
    torch.cuda.synchronize()
    rng = np.random.default_rng(rows)
    idx = np.unique(np.concatenate([[0, 127, 128, rows // 2, rows - 1], rng.integers(0, rows, 20)]))
    o = oracle_mod.hc_head(R[idx], hw.fn, hw.scale, hw.base)
    _check(torch, y, pre, mix, R[idx], o, idx)


# non-default eps on both kernels: each is passed through, not a constant
@pytest.mark.parametrize("rows", [100, 700])
def test_hc_head_other_eps(torch, mhc, oracle_mod, rows):
    R = synth.residual(60 + rows, rows)
    hw = synth.head_weights(60 + rows)
    pre = torch.empty((rows, HC), dtype=torch.float32, device="cuda")
    mix = torch.empty((rows, HC), dtype=torch.float32, device="cuda")
    y = mhc.mhc_hc_head(_dev_bf16(torch, R), _dev_f32(torch, hw.fn), _dev_f32(torch, hw.scale),
                        _dev_f32(torch, hw.base), norm_eps=0.25, hc_eps=0.125, pre_out=pre,
                        mix_out=mix)
    torch.cuda.synchronize()
    o = P.oracle_rows_parallel(oracle_mod.hc_head, R, rows=rows, fn=hw.fn, scale=hw.scale,
                               base=hw.base, norm_eps=0.25, hc_eps=0.125)
    _check(torch, y, pre, mix, R, o)


@pytest.mark.parametrize("rows", [256, 2048])    # the <= 256-row kernel and the tile kernel
def test_hc_head_row_shards_and_repeat_are_bit_exact(torch, mhc, rows):
    R = synth.residual(WL[rows].seed if rows in WL else 50, rows)
    hw = synth.head_weights(2)
    dR = _dev_bf16(torch, R)
    full = _run(torch, mhc, dR, hw)
    again = _run(torch, mhc, dR, hw)
    for a, b in zip(full, again):
        assert torch.equal(a, b)
    s = rows // 4
    for r in range(4):
        part = _run(torch, mhc, dR, hw, r * s, (r + 1) * s, logical_rows=rows)
        for a, b in zip(part, full):
            assert torch.equal(a, b[r * s:(r + 1) * s]), r


def test_hc_head_gates_equal_pre_pass_gates(torch, mhc):
    # with hc_head's parameters set to the layer's first 4 fn rows, scale[0]
    # and base[0:4] (norm_eps = rms_eps, hc_eps = hc_pre_eps), hc_head's pre
    # gates are the pre pass's pre gates.  The two kernels form the dots
    # differently (fp32 on the CUDA cores; bf16 hi/lo on the tensor cores),
    # so they agree to the gate tolerance both meet against the oracle.
    rows = 300
    R = synth.residual(6, rows)
    W = synth.weights(6)
    dR = _dev_bf16(torch, R)
    hw = synth.HeadWeights(fn=np.ascontiguousarray(W.fn[:4]), base=W.base[:4].copy(),
                           scale=W.scale[:1].copy())
    _, pre_h, _ = _run(torch, mhc, dR, hw)
    pre_p = torch.empty((rows, HC), dtype=torch.float32, device="cuda")
    mhc.mhc_pre(dR, _dev_f32(torch, W.fn), _dev_f32(torch, W.scale), _dev_f32(torch, W.base),
                _dev_bf16(torch, W.norm_w), pre_out=pre_p)
    d = (pre_h - pre_p).abs().max().item()
    assert d <= 1e-6, d


def test_hc_head_validation(torch, mhc):
    R = torch.zeros((4, HC, H), dtype=torch.bfloat16, device="cuda")
    hw = synth.head_weights(0)
    with pytest.raises(mhc.MhcError) as e:
        mhc.mhc_hc_head(R, _dev_f32(torch, hw.fn), _dev_f32(torch, hw.scale),
                        _dev_f32(torch, hw.base), norm_eps=-1.0)
    assert e.value.code == -4
    with pytest.raises(mhc.MhcError) as e:
        mhc.mhc_hc_head(R, _dev_f32(torch, hw.fn), _dev_f32(torch, hw.scale),
                        _dev_f32(torch, hw.base), logical_rows=2)
    assert e.value.code == -2
    y = mhc.mhc_hc_head(R[:0], _dev_f32(torch, hw.fn), _dev_f32(torch, hw.scale),
                        _dev_f32(torch, hw.base))
    assert y.shape == (0, H)
