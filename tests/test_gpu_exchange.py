"""The bucket-exchange sort on the GPU with its real local steps (gsort), as a
one-rank NCCL group (every run here has one GPU, and two ranks must not share
one GPU).  With one rank the plan gives rank 0 every bucket and the exchange
moves everything to itself; the local steps (top-digit histogram, grouping
by the top digit, full sort) run on the device and the result must equal the
oracle's stable sort."""
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

import oracle
from bitonic_networks_gb300 import exchange, synth
from gpu_util import assert_bits_equal, dev, host_u32

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.fixture(scope="module")
def one_rank_group():
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0, world_size=1)
    yield
    dist.destroy_process_group()


@pytest.mark.parametrize("n,kind", [(300_001, "uniform"), (1 << 20, "and3"), (5, "uniform"), (0, "uniform")])
def test_exchange_one_rank_matches_oracle(one_rank_group, n, kind):
    gen = {"uniform": synth.uniform_keys, "and3": synth.and3_keys}[kind]
    k = gen(n, 777) if n else np.zeros(0, dtype=np.uint32)
    v = synth.index_values(n) if n else np.zeros(0, dtype=np.uint32)
    kt = dev(k) if n else torch.zeros(0, dtype=torch.int32, device="cuda")
    vt = dev(v) if n else torch.zeros(0, dtype=torch.int32, device="cuda")
    rk, rv, p = exchange.sort_across_ranks(kt, vt)
    assert p.owner_start.tolist() == [0, 256]
    exp_k, exp_v = oracle.radix_sort_pairs(k, v, 0, 0, 32)
    assert_bits_equal(host_u32(rk), exp_k, f"keys {kind} n={n}")
    assert_bits_equal(host_u32(rv), exp_v, f"values {kind} n={n}")
