"""World-size-2 gloo tests (CPU) of the receiver-range split and the
max-over-ranks timing used by the multi-process bench."""
import os
import socket

import numpy as np
import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist

    from equivariant_gnn_message_gb300.inputs import make_workload
    from equivariant_gnn_message_gb300.sharding import max_over_ranks, receiver_ranges
    from oracle import layer

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = make_workload(n_atoms=80, cutoff=5.0, channels=4, weights="shared", storage="f32", seed=3)
        a, b = receiver_ranges(wl.n_atoms, world, wl.off)[rank]
        part = layer.message_pass(wl.vec, wl.x, wl.off, wl.src, w=wl.w, receivers=np.arange(a, b))
        import torch

        parts = [None] * world
        dist.all_gather_object(parts, (a, b, part))
        worst = max_over_ranks(1.0 + rank)
        if rank == 0:
            full = layer.message_pass(wl.vec, wl.x, wl.off, wl.src, w=wl.w)
            glued = np.concatenate([p for (_, _, p) in sorted(parts, key=lambda t: t[0])])
            cover = sorted((pa, pb) for (pa, pb, _) in parts)
            q.put((np.max(np.abs(glued - full)), cover, worst))
    finally:
        dist.destroy_process_group()


def test_two_rank_receiver_split_and_max_timing():
    import multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    err, cover, worst = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert err < 1e-12
    assert cover[0][0] == 0 and cover[-1][1] == 80 and cover[0][1] == cover[1][0]
    assert worst == 2.0


@pytest.mark.parametrize("parts", [1, 2, 3, 7])
def test_receiver_ranges_cover_and_balance(parts):
    from equivariant_gnn_message_gb300.inputs import make_workload
    from equivariant_gnn_message_gb300.sharding import receiver_ranges

    wl = make_workload("pages_1k_c32")
    for off in (None, wl.off):
        r = receiver_ranges(wl.n_atoms, parts, off)
        assert r[0][0] == 0 and r[-1][1] == wl.n_atoms
        assert all(r[k][1] == r[k + 1][0] for k in range(parts - 1))
        if off is not None and parts > 1:
            edges = [wl.off[b] - wl.off[a] for a, b in r]
            assert max(edges) - min(edges) < 0.05 * wl.n_edges
