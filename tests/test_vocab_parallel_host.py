"""Host side of the vocabulary-parallel head, on the CPU.

The vocabulary is cut into whole 64-id blocks per rank (vocab_share), and the
ranks exchange their per-row records with one all-gather in rank order
(gather_records): the layout lmh_merge_records reads.  These tests check the
partition arithmetic, and run the exchange on two gloo ranks with records
that carry their rank and row, so a misplaced or reordered record shows.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("V", [64, 65, 4100, 128256, 151936, 248320])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_shares_partition_the_vocabulary(V, world):
    from top_reduction_gb300 import lmh as L
    if (V + 63) // 64 < world:
        pytest.skip("fewer blocks than ranks")
    shares = [L.vocab_share(V, r, world) for r in range(world)]
    pos = 0
    for b, n in shares:
        assert b == pos and n >= 1 and b % 64 == 0
        pos = b + n
    assert pos == V
    sizes = [n for _, n in shares[:-1]]
    assert max(sizes, default=0) - min(sizes, default=0) <= 64  # whole blocks, spread evenly


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, rows, rb, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from top_reduction_gb300 import lmh as L
        rec = torch.zeros((rows, rb), dtype=torch.uint8)
        rec[:, 0] = rank
        rec[:, 1] = torch.arange(rows, dtype=torch.uint8)
        rec[:, 2:] = (7 * rank + 1) % 256
        allrec = L.gather_records(rec)
        out_q.put((rank, allrec.numpy().tolist()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_gather_records_in_rank_order():
    world, rows, rb = 2, 5, 16 + 8 * 3
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, rows, rb, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    import numpy as np
    for rank in range(world):
        a = np.array(res[rank], dtype=np.uint8)
        assert a.shape == (world, rows, rb)
        for p in range(world):
            assert np.all(a[p, :, 0] == p)
            assert np.array_equal(a[p, :, 1], np.arange(rows))
            assert np.all(a[p, :, 2:] == (7 * p + 1) % 256)
