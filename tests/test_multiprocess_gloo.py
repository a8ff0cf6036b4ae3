"""The N>1 host path on CPU: two gloo ranks shard a chunk's rows with
`shard.row_range`, each runs the oracle on its own rows only, and the
gathered shards must equal one whole-chunk run; the bench's max-over-ranks
timing reduction is checked on the same process group.  No GPU is used."""
import os
import socket

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_row_range_partitions_every_size():
    from hyper_connection_residual_mhc_gb300.shard import row_range
    for rows in (0, 1, 3, 7, 128, 1500, 2048):
        for world in (1, 2, 3, 4, 8):
            spans = [row_range(r, world, rows) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == rows
            for (a, b), (c, d) in zip(spans, spans[1:]):
                assert b == c and a <= b
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        row_range(2, 2, 10)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, rows, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist

    import oracle
    import synth
    from hyper_connection_residual_mhc_gb300.shard import max_over_ranks, row_range
    try:
        dist.init_process_group("gloo", rank=rank, world_size=world)
        lo, hi = row_range(rank, world, rows)
        R = synth.residual(11, hi - lo, row0=lo)        # this rank draws only its rows
        W = synth.weights(11)
        o = oracle.pre(R, W.fn, W.scale, W.base, W.norm_w)
        mine = torch.from_numpy(np.concatenate(
            [o["comb"].reshape(hi - lo, -1), o["post"], o["x_norm"].astype(np.float64)], axis=1))
        sizes = [row_range(r, world, rows) for r in range(world)]
        most = max(b - a for a, b in sizes)          # gloo gathers equal shapes: pad, then trim
        padded = torch.zeros((most, mine.shape[1]), dtype=mine.dtype)
        padded[:hi - lo] = mine
        parts = [torch.zeros_like(padded) for _ in sizes]
        dist.all_gather(parts, padded)
        t = max_over_ranks(1.0 + rank, dist)
        if rank == 0:
            q.put(("ok", torch.cat([p[:b - a] for p, (a, b) in zip(parts, sizes)]).numpy(), t))
        dist.barrier()
        dist.destroy_process_group()
    except Exception as e:          # report, never hang the parent
        q.put(("err", repr(e), None))


def test_two_gloo_ranks_match_the_whole_chunk(oracle_mod):
    import multiprocessing as mp

    import oracle
    import synth
    rows, world = 37, 2                  # odd: the ranks get 19 and 18 rows
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, rows, q)) for r in range(world)]
    for p in procs:
        p.start()
    try:
        status, got, t = q.get(timeout=240)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert status == "ok", got
    R = synth.residual(11, rows)
    W = synth.weights(11)
    o = oracle.pre(R, W.fn, W.scale, W.base, W.norm_w)
    whole = np.concatenate([o["comb"].reshape(rows, -1), o["post"],
                            o["x_norm"].astype(np.float64)], axis=1)
    assert np.array_equal(got, whole)
    assert t == 2.0                      # the slowest rank's time
    assert all(p.exitcode == 0 for p in procs)
