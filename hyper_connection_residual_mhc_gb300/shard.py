"""Row sharding of one chunk over ranks (host logic only, no GPU work).

The hc work is row-local (prefill_sp.py, `sp_logical_rows`: every rank runs
the same row-wise kernels on its own slice of the chunk with no exchange), so
a chunk of M rows splits into contiguous row ranges, one per rank, and each
rank calls the library on its range with ``logical_rows = M``.  Because the
kernels' per-row arithmetic never depends on the launch, the concatenated
shards are bit-identical to one whole-chunk call.
"""
from __future__ import annotations


def row_range(rank: int, world: int, rows: int) -> tuple[int, int]:
    """Rows [lo, hi) of a `rows`-row chunk owned by `rank` of `world`.

    The first ``rows % world`` ranks take one row more; every row is owned
    by exactly one rank, ranges are contiguous and in rank order.
    """
    if world < 1 or not 0 <= rank < world or rows < 0:
        raise ValueError(f"bad shard: rank={rank} world={world} rows={rows}")
    q, r = divmod(rows, world)
    lo = rank * q + min(rank, r)
    return lo, lo + q + (1 if rank < r else 0)


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The largest `value` over all ranks of the default process group (the
    job's wall time is its slowest rank's); `value` itself without one."""
    if dist is None or not dist.is_available() or not dist.is_initialized():
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
