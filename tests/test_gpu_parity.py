"""Parity of the CUDA path (through the C ABI) against the CPU oracle.

All inputs come from the seeded generator in ``synth``; the oracle and the GPU
see the same bits.  Workloads: M = 128 (seed 0), 1500 (seed 1), 2048 (seed 2),
4096 (seed 3), 16384 (seed 4).  The two small ones are checked element by
element on every row; the large ones on sampled rows (rows are independent,
so the oracle computes just those rows) and by the bit-exact row-shard
property, which holds at any size.
"""
import numpy as np
import pytest

import synth
from tests import parity as P

pytestmark = pytest.mark.gpu

HC, H, K, MIX = 4, 5120, 20480, 24
WL = {w.rows: w for w in synth.WORKLOADS}


@pytest.fixture(scope="session")
def torch():
    import torch as t
    assert t.cuda.is_available(), "GPU tests need a CUDA device"
    return t


@pytest.fixture(scope="session")
def mhc(torch):
    from hyper_connection_residual_mhc_gb300 import build as b
    b.build()
    import hyper_connection_residual_mhc_gb300 as m
    m.lib()
    return m


def dev_bf16(torch, bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev_f32(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host_f(t):
    return t.detach().cpu().numpy().astype(np.float64)


class Case:
    """Inputs of one workload, on host and device, plus cached oracle results."""

    def __init__(self, torch, rows, seed, y_tensor=synth.T_Y):
        self.rows, self.seed = rows, seed
        self.R = synth.residual(seed, rows)
        self.y = synth.sublayer_out(seed, rows, tensor=y_tensor)
        self.W = synth.weights(seed)
        self.dR = dev_bf16(torch, self.R)
        self.dy = dev_bf16(torch, self.y)
        self.dfn = dev_f32(torch, self.W.fn)
        self.dscale = dev_f32(torch, self.W.scale)
        self.dbase = dev_f32(torch, self.W.base)
        self.dw = dev_bf16(torch, self.W.norm_w)

    def gpu_pre(self, torch, mhc, lo=0, hi=None, logical_rows=None):
        hi = self.rows if hi is None else hi
        n = hi - lo
        pre_out = torch.empty((n, HC), dtype=torch.float32, device="cuda")
        mix_out = torch.empty((n, MIX), dtype=torch.float32, device="cuda")
        xn, post, comb = mhc.mhc_pre(self.dR[lo:hi], self.dfn, self.dscale, self.dbase, self.dw,
                                     logical_rows=logical_rows, pre_out=pre_out, mix_out=mix_out)
        return {"x_norm": xn, "post": post, "comb": comb, "pre": pre_out, "mix": mix_out}

    def oracle_pre(self, oracle, rows_idx=None):
        R = self.R if rows_idx is None else self.R[rows_idx]
        return P.oracle_rows_parallel(oracle.pre, R, rows=R.shape[0], fn=self.W.fn,
                                      scale=self.W.scale, base=self.W.base, w=self.W.norm_w)


def _bits(torch, t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _check_pre(torch, g, o, c, rows_idx=None):
    sel = (lambda a: a) if rows_idx is None else (lambda a: a[rows_idx])
    P.check_mix(sel(host_f(g["mix"])), o["mix"])
    R = c.R if rows_idx is None else c.R[rows_idx]
    P.check_gates(sel(host_f(g["pre"])), sel(host_f(g["post"])), o, c.W.scale, R, c.W.fn)
    P.check_abs(sel(host_f(g["comb"])), o["comb"], 1e-6, "comb")
    P.check_bf16(sel(_bits(torch, g["x_norm"])), o["x_norm"], "x_norm",
                 term_mag=P.combine_term_magnitude(R, o["pre"], c.W.norm_w, 1e-6))


_cases = {}


def case(torch, rows):
    if rows not in _cases:
        _cases.clear()        # keep one large workload resident at a time
        _cases[rows] = Case(torch, rows, WL[rows].seed)
    return _cases[rows]


# --------------------------------------------------------------------------- full parity
@pytest.mark.parametrize("rows", [128, 1500])
def test_pre_parity_every_row(torch, mhc, oracle_mod, rows):
    c = case(torch, rows)
    g = c.gpu_pre(torch, mhc)
    torch.cuda.synchronize()
    _check_pre(torch, g, c.oracle_pre(oracle_mod), c)


@pytest.mark.parametrize("rows", [128, 1500])
def test_post_parity_every_row(torch, mhc, oracle_mod, rows):
    c = case(torch, rows)
    o = c.oracle_pre(oracle_mod)
    post32, comb32 = o["post"].astype(np.float32), o["comb"].astype(np.float32)
    out = mhc.mhc_post(c.dR, c.dy, dev_f32(torch, post32), dev_f32(torch, comb32))
    ref = P.oracle_rows_parallel(oracle_mod.post, c.R, c.y, post32, comb32, rows=rows)
    P.check_bf16(_bits(torch, out), ref, "R_out",
                 term_mag=P.post_term_magnitude(c.R, c.y, post32, comb32))


def test_pre_then_post_chain_every_row(torch, mhc, oracle_mod):
    c = case(torch, 128)
    g = c.gpu_pre(torch, mhc)
    out = mhc.mhc_post(c.dR, c.dy, g["post"], g["comb"])
    o = c.oracle_pre(oracle_mod)
    post32, comb32 = o["post"].astype(np.float32), o["comb"].astype(np.float32)
    ref = oracle_mod.post(c.R, c.y, post32, comb32)
    # comb differs by <= 1e-6 between the two sides; with |R| <= ~100 that is
    # well under 2 ulp of the largest term of every sum.
    P.check_bf16(_bits(torch, out), ref, "R_out chained",
                 term_mag=P.post_term_magnitude(c.R, c.y, post32, comb32))


# --------------------------------------------------------------------------- full sizes, sampled
def _sample_rows(rows, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, 129, rows // 4 - 1, rows // 4, rows // 2, rows - 129, rows - 2, rows - 1]
    pick = np.concatenate([[r for r in fixed if 0 <= r < rows], rng.integers(0, rows, 21)])
    return np.unique(pick)


@pytest.mark.parametrize("rows", [2048, 4096, 16384])
def test_full_size_sampled_rows(torch, mhc, oracle_mod, rows):
    c = case(torch, rows)
    idx = _sample_rows(rows, rows)
    g = c.gpu_pre(torch, mhc)
    out = mhc.mhc_post(c.dR, c.dy, g["post"], g["comb"])
    torch.cuda.synchronize()
    o = c.oracle_pre(oracle_mod, idx)
    _check_pre(torch, g, o, c, idx)
    post_g = host_f(g["post"])[idx].astype(np.float32)
    comb_g = host_f(g["comb"])[idx].astype(np.float32)
    ref = oracle_mod.post(c.R[idx], c.y[idx], post_g, comb_g)
    P.check_bf16(_bits(torch, out)[idx], ref, "R_out",
                 term_mag=P.post_term_magnitude(c.R[idx], c.y[idx], post_g, comb_g))


def test_chunk_larger_than_the_headline_sampled_rows(torch, mhc, oracle_mod):
    # 40001 rows: 1251 tiles of 32 rows over the co-resident clusters of the
    # streamed build (many rounds), a 1-row last tile, and 1.6 GB of R --
    # sizes past every workload above
    rows = 40001
    c = Case(torch, rows, 77)
    idx = np.unique(np.concatenate([[0, 127, 128, 20000, rows - 65, rows - 1],
                                    np.random.default_rng(77).integers(0, rows, 24)]))
    g = c.gpu_pre(torch, mhc)
    out = mhc.mhc_post(c.dR, c.dy, g["post"], g["comb"])
    torch.cuda.synchronize()
    _check_pre(torch, g, c.oracle_pre(oracle_mod, idx), c, idx)
    post_g = host_f(g["post"])[idx].astype(np.float32)
    comb_g = host_f(g["comb"])[idx].astype(np.float32)
    ref = oracle_mod.post(c.R[idx], c.y[idx], post_g, comb_g)
    P.check_bf16(_bits(torch, out)[idx], ref, "R_out",
                 term_mag=P.post_term_magnitude(c.R[idx], c.y[idx], post_g, comb_g))
    assert mhc.mhc_kernel_status() == 0
    _cases.clear()


def test_post_alone_with_second_seed_output(torch, mhc, oracle_mod):
    # M=4096: mhc_post on its own with y drawn from a second stream
    c = Case(torch, 4096, 3, y_tensor=synth.T_Y2)
    idx = _sample_rows(4096, 7)
    g = c.gpu_pre(torch, mhc)
    out = mhc.mhc_post(c.dR, c.dy, g["post"], g["comb"])
    post_g = host_f(g["post"])[idx].astype(np.float32)
    comb_g = host_f(g["comb"])[idx].astype(np.float32)
    ref = oracle_mod.post(c.R[idx], c.y[idx], post_g, comb_g)
    P.check_bf16(_bits(torch, out)[idx], ref, "R_out",
                 term_mag=P.post_term_magnitude(c.R[idx], c.y[idx], post_g, comb_g))


# --------------------------------------------------------------------------- row-shard invariance
@pytest.mark.parametrize("rows", [1500, 2048, 16384])
def test_row_shards_reproduce_whole_chunk_bits(torch, mhc, rows):
    # prefill_sp.py, sp_logical_rows / shard_range: rank r of 4 runs rows
    # [r*M/4, (r+1)*M/4) with the whole chunk's row count as the key.
    c = case(torch, rows)
    full = c.gpu_pre(torch, mhc)
    full_out = mhc.mhc_post(c.dR, c.dy, full["post"], full["comb"])
    W = 4
    s = rows // W
    for r in range(W):
        lo, hi = r * s, (r + 1) * s
        g = c.gpu_pre(torch, mhc, lo, hi, logical_rows=rows)
        out = mhc.mhc_post(c.dR[lo:hi], c.dy[lo:hi], g["post"], g["comb"], logical_rows=rows)
        for k in ("x_norm", "post", "comb", "pre", "mix"):
            assert torch.equal(g[k], full[k][lo:hi]), (k, r)
        assert torch.equal(out, full_out[lo:hi]), ("R_out", r)


def test_repeat_calls_are_bit_identical(torch, mhc):
    c = case(torch, 1500)
    a = c.gpu_pre(torch, mhc)
    b = c.gpu_pre(torch, mhc)
    for k in a:
        assert torch.equal(a[k], b[k]), k
    oa = mhc.mhc_post(c.dR, c.dy, a["post"], a["comb"])
    ob = mhc.mhc_post(c.dR, c.dy, a["post"], a["comb"])
    assert torch.equal(oa, ob)


# --------------------------------------------------------------------------- exact special cases
def test_post_special_cases_bit_exact(torch, mhc):
    rows = 300
    R = synth.residual(9, rows)
    y = synth.sublayer_out(9, rows)
    dR, dy = dev_bf16(torch, R), dev_bf16(torch, y)
    zeros4 = torch.zeros((rows, HC), dtype=torch.float32, device="cuda")
    eye = torch.eye(HC, dtype=torch.float32, device="cuda").expand(rows, HC, HC).contiguous()
    assert torch.equal(mhc.mhc_post(dR, dy, zeros4, eye), dR)           # R' = R
    pi = [2, 0, 3, 1]
    perm = torch.zeros((rows, HC, HC), dtype=torch.float32, device="cuda")
    for i, j in enumerate(pi):
        perm[:, j, i] = 1.0
    out = mhc.mhc_post(dR, dy, zeros4, perm)
    for i, j in enumerate(pi):
        assert torch.equal(out[:, i], dR[:, j]), i                     # R'_i = R_pi(i)
    ones4 = torch.ones((rows, HC), dtype=torch.float32, device="cuda")
    out = mhc.mhc_post(dR, dy, ones4, torch.zeros_like(perm))
    for i in range(HC):
        assert torch.equal(out[:, i], dy), i                           # R'_i = y


def test_combine_norm_one_hot_and_random_pre(torch, mhc, oracle_mod):
    rows = 64
    R = synth.residual(12, rows)
    W = synth.weights(12)
    rng = np.random.default_rng(3)
    pre = rng.uniform(0, 1, (rows, HC))
    pre[:HC] = np.eye(HC)
    pre32 = pre.astype(np.float32)
    out = mhc.mhc_combine_norm(dev_bf16(torch, R), dev_f32(torch, pre32), dev_bf16(torch, W.norm_w), 1e-6)
    ref = oracle_mod.combine_norm(R, pre32.astype(np.float64), W.norm_w, 1e-6)
    P.check_bf16(_bits(torch, out), ref, "x_norm",
                 term_mag=P.combine_term_magnitude(R, pre32, W.norm_w, 1e-6))


# --------------------------------------------------------------------------- edges
@pytest.mark.parametrize("rows", [1, 3, 7, 129])
def test_tiny_and_ragged_row_counts(torch, mhc, oracle_mod, rows):
    c = Case(torch, rows, 20 + rows)
    g = c.gpu_pre(torch, mhc)
    _check_pre(torch, g, c.oracle_pre(oracle_mod), c)
    out = mhc.mhc_post(c.dR, c.dy, g["post"], g["comb"])
    post_g, comb_g = host_f(g["post"]).astype(np.float32), host_f(g["comb"]).astype(np.float32)
    ref = oracle_mod.post(c.R, c.y, post_g, comb_g)
    P.check_bf16(_bits(torch, out), ref, "R_out",
                 term_mag=P.post_term_magnitude(c.R, c.y, post_g, comb_g))


def test_zero_rows_launch_nothing(torch, mhc):
    R = torch.empty((0, HC, H), dtype=torch.bfloat16, device="cuda")
    W = synth.weights(0)
    xn, post, comb = mhc.mhc_pre(R, dev_f32(torch, W.fn), dev_f32(torch, W.scale),
                                 dev_f32(torch, W.base), dev_bf16(torch, W.norm_w))
    assert xn.shape == (0, H) and post.shape == (0, HC) and comb.shape == (0, HC, HC)
    out = mhc.mhc_post(R, torch.empty((0, H), dtype=torch.bfloat16, device="cuda"), post, comb)
    assert out.shape == (0, HC, H)


def test_outputs_do_not_write_outside_their_rows(torch, mhc):
    # outputs live inside larger buffers filled with a sentinel; after pre and
    # post on rows 8..8+n the sentinel around them must be untouched.
    n, pad = 131, 8
    c = Case(torch, n, 31)
    xbuf = torch.full(((n + 2 * pad) * H,), -7.0, dtype=torch.bfloat16, device="cuda")
    pbuf = torch.full(((n + 2 * pad) * HC,), -7.0, dtype=torch.float32, device="cuda")
    cbuf = torch.full(((n + 2 * pad) * 16,), -7.0, dtype=torch.float32, device="cuda")
    obuf = torch.full(((n + 2 * pad) * K,), -7.0, dtype=torch.bfloat16, device="cuda")
    xn = xbuf[pad * H:(pad + n) * H].view(n, H)
    po = pbuf[pad * HC:(pad + n) * HC].view(n, HC)
    co = cbuf[pad * 16:(pad + n) * 16].view(n, HC, HC)
    ro = obuf[pad * K:(pad + n) * K].view(n, HC, H)
    mhc.mhc_pre(c.dR, c.dfn, c.dscale, c.dbase, c.dw, x_norm=xn, post=po, comb=co)
    mhc.mhc_post(c.dR, c.dy, po, co, out=ro)
    torch.cuda.synchronize()
    for buf, width in ((xbuf, H), (pbuf, HC), (cbuf, 16), (obuf, K)):
        assert torch.all(buf[:pad * width] == -7.0) and torch.all(buf[(pad + n) * width:] == -7.0)


def test_host_validation_rejects_before_launch(torch, mhc):
    c = Case(torch, 16, 5)
    flat = c.dR.view(-1)
    mis = flat[2:2 + 15 * K].view(15, HC, H)          # 4-byte offset: not 16-byte aligned
    with pytest.raises(mhc.MhcError) as e:
        mhc.mhc_post(mis, c.dy[:15], torch.zeros((15, HC), device="cuda"),
                     torch.zeros((15, HC, HC), device="cuda"))
    assert e.value.code == -3
    with pytest.raises(mhc.MhcError) as e:           # output aliases an input
        mhc.mhc_post(c.dR, c.dy, torch.zeros((16, HC), device="cuda"),
                     torch.zeros((16, HC, HC), device="cuda"), out=c.dR)
    assert e.value.code == -5
    with pytest.raises(mhc.MhcError) as e:           # logical_rows < rows
        mhc.mhc_post(c.dR, c.dy, torch.zeros((16, HC), device="cuda"),
                     torch.zeros((16, HC, HC), device="cuda"), logical_rows=8)
    assert e.value.code == -2
    with pytest.raises(mhc.MhcError) as e:
        mhc.mhc_pre(c.dR, c.dfn, c.dscale, c.dbase, c.dw,
                    params=mhc.default_params(sinkhorn_iters=0))
    assert e.value.code == -4


def test_no_kernel_gave_up_a_wait(torch, mhc):
    # every bounded wait of the fused kernel completed during this session
    torch.cuda.synchronize()
    assert mhc.mhc_kernel_status() == 0, mhc.mhc_kernel_status_detail()
