"""Decode-size chunks (logical_rows <= 48): mhc_pre runs as one launch of
16-CTA clusters on the CUDA cores (a group of up to 8 rows per cluster, K split
over the cluster; partials, gates and sums of y^2 exchanged by asynchronous
stores into distributed shared memory, counted on mbarriers).
Parity against the oracle with the pre pass's tolerances, on both sides of the
48-row switch, plus the row-shard bits within a decode chunk.
"""
import numpy as np
import pytest

import synth
from tests import parity as P
from tests.test_gpu_parity import Case, _bits, _check_pre, host_f  # noqa: F401

pytestmark = pytest.mark.gpu

HC, H, K, MIX = 4, 5120, 20480, 24


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


@pytest.mark.parametrize("rows", [1, 2, 7, 8, 9, 41, 47, 48, 49])
def test_decode_sizes_every_row(torch, mhc, oracle_mod, rows):
    c = Case(torch, rows, 60 + rows)
    g = c.gpu_pre(torch, mhc)
    torch.cuda.synchronize()
    _check_pre(torch, g, c.oracle_pre(oracle_mod), c)


def test_decode_chunk_shards_are_bit_exact(torch, mhc):
    rows = 45
    c = Case(torch, rows, 77)
    full = c.gpu_pre(torch, mhc)
    for lo, hi in ((0, 1), (1, 20), (20, 44), (44, 45)):
        g = c.gpu_pre(torch, mhc, lo, hi, logical_rows=rows)
        for k in ("x_norm", "post", "comb", "pre", "mix"):
            assert torch.equal(g[k], full[k][lo:hi]), (k, lo, hi)
    again = c.gpu_pre(torch, mhc)
    for k in full:
        assert torch.equal(full[k], again[k]), k


def test_same_rows_through_both_paths_agree(torch, mhc, oracle_mod):
    # 40 rows as a decode chunk of their own, and as a shard of a 4096-row
    # chunk (the tensor-core path): both within tolerance of the oracle
    c = Case(torch, 40, 91)
    dec = c.gpu_pre(torch, mhc)
    big = c.gpu_pre(torch, mhc, logical_rows=4096)
    torch.cuda.synchronize()
    o = c.oracle_pre(oracle_mod)
    _check_pre(torch, dec, o, c)
    _check_pre(torch, big, o, c)
    # the two paths sum in different orders: equal gates to fp32 rounding
    assert (dec["pre"] - big["pre"]).abs().max().item() <= 2e-6


def test_decode_waits_all_complete(torch, mhc):
    # groups of 1..6 rows a cluster (one or two 16-byte stores of y^2
    # partials per warp and CTA pair), full and partial last groups, then the
    # status word: no bounded wait of the decode kernel may have expired
    assert mhc.mhc_kernel_status(reset=True) == 0
    for rows, logical in ((1, 1), (5, 5), (40, 40), (45, 45), (48, 48), (3, 48), (7, 48)):
        c = Case(torch, rows, 120 + rows)
        c.gpu_pre(torch, mhc, logical_rows=logical)
    torch.cuda.synchronize()
    assert mhc.mhc_kernel_status() == 0
