"""GPU 2-way split (partition) by every predicate, and the 1-bit split sort,
vs the CPU oracle bit for bit: several tiles with ragged tails, values,
unaligned buffers, all-true and all-false inputs, and n = 0."""
import numpy as np
import pytest
import torch

import oracle
from bitonic_networks_gb300 import gsort, synth

pytestmark = pytest.mark.gpu

SIZES = [1, 2, 31, 8191, 8192, 8193, 3 * 8192 + 11, 100_003, 1_000_001]


def to_dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a.copy()).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy().view(np.uint32)


def check_partition(x, values, what, **kw):
    flags = kw.get("flags")
    xt = to_dev(x)
    vt = to_dev(values) if values is not None else None
    ft = torch.from_numpy(flags.copy()).cuda() if flags is not None else None
    args = dict(kw)
    args["flags"] = ft
    o, vo, nt = gsort.partition(xt, vt, **args)
    eo, ev, m = oracle.default().partition(x, values, **kw)
    assert int(nt.item()) == m, f"{what}: num_true {int(nt.item())} != {m}"
    assert np.array_equal(host(o), np.asarray(eo).view(np.uint32)), f"{what}: elements"
    if values is not None:
        assert np.array_equal(host(vo), ev), f"{what}: values"


@pytest.mark.parametrize("n", SIZES)
def test_partition_predicates(n):
    u = synth.uniform_keys(n, 300 + n)
    idx = synth.index_values(n)
    rng = np.random.default_rng(n)
    flags = (rng.random(n) < 0.37).astype(np.uint8)
    check_partition(u, idx, f"flags n={n}", pred=0, flags=flags)
    for b in (0, 13, 31):
        check_partition(u, idx, f"bit set {b} n={n}", pred=1, param=b)
        check_partition(u, None, f"bit clear {b} n={n}", pred=2, param=b)
    check_partition(u, idx, f"less u32 n={n}", pred=3, kind=0, param=int(u[n // 2]))
    s = u.view(np.int32)
    check_partition(s, idx, f"less i32 n={n}", pred=3, kind=2, param=int(u[n // 3]))
    f = synth.normal_f32_with_specials(n, 400 + n)
    for pv in (0.0, -0.0, 1.25, float("-inf")):
        check_partition(f, idx, f"less f32 {pv} n={n}", pred=3, kind=1,
                        param=int(np.float32(pv).view(np.uint32)))
    c = synth.compaction_input(n, 500 + n)
    check_partition(c, idx, f"positive n={n}", pred=4)


def test_partition_all_true_all_false_and_empty():
    n = 50_000
    u = synth.uniform_keys(n, 9)
    check_partition(u | np.uint32(1), None, "all true", pred=1, param=0)
    check_partition(u & ~np.uint32(1), None, "all false", pred=1, param=0)
    o, vo, nt = gsort.partition(torch.empty(0, dtype=torch.int32, device="cuda"), pred=1)
    assert o.numel() == 0 and int(nt.item()) == 0


def test_partition_unaligned():
    n = 40_000
    u = synth.uniform_keys(n, 10)
    base = torch.empty(n + 3, dtype=torch.int32, device="cuda")
    xv = base[1:n + 1]
    xv.copy_(to_dev(u))
    o, _, nt = gsort.partition(xv, pred=2, param=5)
    eo, _, m = oracle.default().partition(u, None, pred=2, param=5)
    assert int(nt.item()) == m and np.array_equal(host(o), eo)


@pytest.mark.parametrize("n", [1, 8193, 100_003, 1 << 20])
@pytest.mark.parametrize("bits", [(0, 32), (3, 17), (31, 32), (0, 8), (5, 5)])
def test_split_sort_matches_oracle(n, bits):
    k = synth.and3_keys(n, 700 + n)
    v = synth.index_values(n)
    ko, vo = gsort.split_sort(to_dev(k), to_dev(v), bits[0], bits[1])
    ek, ev = oracle.default().split_sort(k, v, bits[0], bits[1])
    assert np.array_equal(host(ko), ek) and np.array_equal(host(vo), ev)


def test_split_sort_in_place_and_keys_only():
    n = 77_777
    k = synth.uniform_keys(n, 12)
    t = to_dev(k)
    gsort.split_sort(t, None, 0, 32, keys_out=t)
    assert np.array_equal(host(t), np.sort(k))
    t2 = to_dev(k)
    v2 = to_dev(synth.index_values(n))
    gsort.split_sort(t2, v2, 0, 7, keys_out=t2, values_out=v2)   # odd pass count, in place
    ek, ev = oracle.default().split_sort(k, synth.index_values(n), 0, 7)
    assert np.array_equal(host(t2), ek) and np.array_equal(host(v2), ev)
