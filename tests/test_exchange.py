"""Sort across ranks by one exchange of top-digit buckets, on CPU ranks.

The plan (bucket ranges per rank, send counts) is checked on its own; then
two and three gloo ranks run the whole exchange (all-gather of the
top-digit counts, plan, all-to-all of keys and values) with the CPU oracle
standing in for the per-rank GPU steps, and the concatenation of the ranks'
pieces must equal the oracle's stable sort of the concatenated input, keys
and index values element by element.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from bitonic_networks_gb300 import exchange, synth


def check_plan(h: np.ndarray):
    p = exchange.plan(h)
    world = h.shape[0]
    s = p.owner_start
    assert s[0] == 0 and s[-1] == 256 and np.all(np.diff(s) >= 0)
    # every key goes to the owner of its bucket
    for b in range(256):
        owner = int(np.searchsorted(s, b, side="right") - 1)
        assert s[owner] <= b < s[owner + 1]
    assert np.array_equal(p.send.sum(axis=1), h.sum(axis=1))          # each rank sends all its keys
    assert np.array_equal(p.recv_total, p.send.sum(axis=0))
    assert p.recv_total.sum() == h.sum()
    # rank r's first bucket starts where r * total / world keys lie before it
    tot = h.sum(axis=0)
    excl = np.concatenate([[0], np.cumsum(tot)[:-1]])
    for r in range(1, world):
        target = -(-r * int(tot.sum()) // world)
        b = int(s[r])
        if b < 256 and s[r] > s[r - 1]:
            assert excl[b] >= target
            assert b == 0 or excl[b - 1] < target or s[r] == s[r - 1]
    return p


@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_plan_uniform_balances(world):
    rng = np.random.default_rng(world)
    h = rng.integers(900, 1100, size=(world, 256))
    p = check_plan(h)
    avg = h.sum() / world
    assert np.all(np.abs(p.recv_total - avg) <= h.sum(axis=0).max() + 1)


def test_plan_skewed_and_empty():
    h = np.zeros((3, 256), dtype=np.int64)
    h[:, 0] = 1000          # one bucket holds almost everything
    h[:, 7] = 10
    h[1, 200] = 5
    p = check_plan(h)
    assert p.recv_total[0] == 3000    # the big bucket is not split
    check_plan(np.zeros((2, 256), dtype=np.int64))
    p = check_plan(np.eye(4, 256, dtype=np.int64) * 3)   # one bucket per rank
    assert p.recv_total.tolist() == [3, 3, 3, 3]


def test_plan_rejects_bad_shapes():
    with pytest.raises(ValueError):
        exchange.plan(np.zeros((2, 255)))
    with pytest.raises(ValueError):
        exchange.plan(-np.ones((2, 256)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def oracle_ops():
    """Host stand-ins for the per-rank GPU steps: the CPU oracle."""
    import oracle

    def u32(t):
        return t.numpy().view(np.uint32)

    def top_hist(keys):
        return torch.from_numpy(oracle.digit_histograms(u32(keys), 0, 24, 32)[0].astype(np.int64))

    def group(keys, values):
        k, v = oracle.radix_sort_pairs(u32(keys), None if values is None else u32(values), 0, 24, 32)
        return (torch.from_numpy(k.view(np.int32).copy()),
                None if v is None else torch.from_numpy(v.view(np.int32).copy()))

    def sort(keys, values):
        k, v = oracle.radix_sort_pairs(u32(keys), None if values is None else u32(values), 0, 0, 32)
        return (torch.from_numpy(k.view(np.int32).copy()),
                None if v is None else torch.from_numpy(v.view(np.int32).copy()))

    return exchange.LocalOps(top_hist=top_hist, group=group, sort=sort)


def shard(kind: str, rank: int, world: int):
    sizes = {"uniform": [70_001, 50_000, 90_017], "and3": [40_000, 0, 65_537],
             "distinct16": [30_000, 30_001, 1]}[kind][:world]
    gen = {"uniform": synth.uniform_keys, "and3": synth.and3_keys, "distinct16": synth.distinct16_keys}[kind]
    start = sum(sizes[:rank])
    k = gen(sizes[rank], 500 + 17 * rank) if sizes[rank] else np.zeros(0, dtype=np.uint32)
    v = np.arange(start, start + sizes[rank], dtype=np.uint32)   # global input index
    return k, v


def _rank(rank, world, port, kind, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        k, v = shard(kind, rank, world)
        rk, rv, p = exchange.sort_across_ranks(torch.from_numpy(k.view(np.int32)),
                                               torch.from_numpy(v.view(np.int32)), ops=oracle_ops())
        q.put((rank, rk.numpy().view(np.uint32).copy(), rv.numpy().view(np.uint32).copy(),
               p.owner_start.tolist()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("kind", ["uniform", "and3", "distinct16"])
def test_gloo_ranks_sort_by_exchange(world, kind):
    import oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, kind, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted((q.get(timeout=180) for _ in range(world)), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    keys = np.concatenate([got[r][1] for r in range(world)])
    vals = np.concatenate([got[r][2] for r in range(world)])
    all_k = np.concatenate([shard(kind, r, world)[0] for r in range(world)])
    all_v = np.concatenate([shard(kind, r, world)[1] for r in range(world)])
    exp_k, exp_v = oracle.radix_sort_pairs(all_k, all_v, 0, 0, 32)
    assert np.array_equal(keys, exp_k)
    assert np.array_equal(vals, exp_v)     # stable: equal keys keep the global input order
    assert all(got[r][3] == got[0][3] for r in range(world))   # every rank made the same plan
