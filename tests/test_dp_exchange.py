"""The data-parallel exchange of sequence-sharded calls on CPU: world-size
2 and 3 gloo ranks gather integer counts (summed exactly) and per-sequence
records of unequal lengths, concatenated in rank order byte for byte."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

from grad_row_online_gb300 import dp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _records(rank: int, n: int) -> torch.Tensor:
    g = torch.Generator().manual_seed(1000 + rank)
    return torch.randint(0, 256, (n, 32), dtype=torch.uint8, generator=g)


def _rank(rank: int, world: int, sizes, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    counts = torch.tensor([10 * (rank + 1), rank + 1], dtype=torch.int64)
    total = dp.gather_counts(counts)
    recs = dp.gather_totals(_records(rank, sizes[rank]))
    dist.barrier()
    q.put((rank, total.tolist(), recs.numpy().tobytes(), tuple(recs.shape)))
    dist.destroy_process_group()


@pytest.mark.parametrize("sizes", [(3, 5), (4, 0, 2)])
def test_gather_in_rank_order(sizes):
    world = len(sizes)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, sizes, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in range(world))
    want = torch.cat([_records(r, n) for r, n in enumerate(sizes)])
    for rank, total, recs, shape in got:
        assert total == [sum(10 * (r + 1) for r in range(world)), sum(range(1, world + 1))]
        assert shape == tuple(want.shape)
        assert recs == want.numpy().tobytes()  # every rank holds the same bytes


def test_single_process_is_the_identity():
    c = torch.tensor([7, 2], dtype=torch.int64)
    assert dp.gather_counts(c).tolist() == [7, 2]
    r = _records(0, 4)
    assert torch.equal(dp.gather_totals(r), r)


@pytest.mark.parametrize("n,world", [(12, 1), (12, 5), (3, 4), (1024, 8)])
def test_shard_bounds_partition_in_rank_order(n, world):
    bounds = [dp.shard_bounds(n, world, r) for r in range(world)]
    assert bounds[0][0] == 0 and bounds[-1][1] == n
    for (a, b), (c, d) in zip(bounds, bounds[1:]):
        assert b == c and a <= b
    sizes = [b - a for a, b in bounds]
    assert max(sizes) - min(sizes) <= 1


def _tp_rank(rank: int, world: int, nck, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    rows = 5
    g = torch.Generator().manual_seed(77 + rank)
    parts = {"part_p": torch.randn(nck[rank], rows, 4, generator=g),
             "part_r": torch.randn(nck[rank], rows, 4, generator=g),
             # rank r holds the action of rows r, r + world, ...
             "action_logits": torch.tensor([[float(10 * j + 1) if j % world == rank else 0.0
                                             for j in range(rows)]] * 2)}
    out = dp.gather_vocab_partials(parts)
    dist.barrier()
    q.put((rank, out["part_p"].numpy().tobytes(), out["part_r"].shape[0],
           out["action_logits"].tolist()))
    dist.destroy_process_group()


def test_vocab_partials_exchange():
    nck = (2, 1, 3)
    world = len(nck)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_tp_rank, args=(r, world, nck, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in range(world))
    want = []
    for r in range(world):
        g = torch.Generator().manual_seed(77 + r)
        want.append(torch.randn(nck[r], 5, 4, generator=g))
    want = torch.cat(want).numpy().tobytes()
    for rank, pp, n_r, act in got:
        assert pp == want and n_r == sum(nck)
        assert act == [[float(10 * j + 1) for j in range(5)]] * 2


@pytest.mark.parametrize("V,world", [(8969, 1), (8969, 2), (8969, 3), (151936, 4), (100, 4)])
def test_vocab_shard_bounds_are_whole_chunks(V, world):
    C = 4096
    b = [dp.vocab_shard_bounds(V, C, world, r) for r in range(world)]
    assert b[0][0] == 0 and b[-1][1] == V
    for (x, y), (z, _) in zip(b, b[1:]):
        assert y == z
    for x, y in b:
        assert x == y or x % C == 0  # a nonempty slice starts on a chunk boundary
