"""Receiver-range sharding of one layer (host-side logic, no arithmetic).

The CSR offsets passed to the library are absolute edge indices, so a
receiver range [a, b) of a graph is the call with row_offsets[a : b+1],
N = b - a and out[a : b]; the edge arrays (vec, src, R) are passed whole.
Ranges are disjoint in the output, so shards need no reduction.  On a box
with one GPU per process the bench runs independent replicas; these helpers
are what a multi-GPU deployment (and the CPU tests) use to split the work.
"""
import numpy as np


def receiver_ranges(n_receivers, parts, row_offsets=None):
    """Contiguous [a, b) ranges covering 0..n_receivers, one per part.

    With row_offsets the cut points balance edges + receivers (the cost of
    the fused layer is about one edge per edge plus a few per receiver);
    without, receiver counts are equal.
    """
    n = int(n_receivers)
    parts = max(1, int(parts))
    if row_offsets is None:
        cuts = [(n * k) // parts for k in range(parts + 1)]
    else:
        off = np.asarray(row_offsets, dtype=np.int64)
        cost = (off - off[0]) + 4 * np.arange(n + 1)
        total = int(cost[-1])
        cuts = [0] + [int(np.searchsorted(cost, total * k / parts, side="left"))
                      for k in range(1, parts)] + [n]
        cuts = list(np.maximum.accumulate(cuts))
    return [(cuts[k], cuts[k + 1]) for k in range(parts)]


def shard_args(row_offsets, out, a, b):
    """(row_offsets view, out view) for receivers [a, b) (no copies)."""
    return row_offsets[a:b + 1], out[a:b]


def max_over_ranks(value, group=None):
    """Maximum of a per-rank float over the process group (timing)."""
    import torch
    import torch.distributed as dist

    if not dist.is_available() or not dist.is_initialized():
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64)
    if dist.get_backend(group) == "nccl":
        t = t.cuda()
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())
