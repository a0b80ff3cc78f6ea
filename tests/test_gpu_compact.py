"""GPU stream compaction vs the CPU oracle, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from bitonic_networks_gb300 import gsort, synth
from gpu_util import assert_bits_equal, dev, host_u32, offset_view

pytestmark = pytest.mark.gpu


def check(x: np.ndarray, out_off: int = 0, in_off: int = 0):
    n = x.size
    xi = dev(x)
    if in_off:
        xi = offset_view(xi, n, in_off)
    out = None
    if out_off:
        out = offset_view(torch.full((n,), 7.0, device="cuda"), n, out_off)
    got, nk = gsort.compact_positive(xi, out=out)
    exp, m = oracle.compact_positive(x)
    assert int(nk.item()) == m
    assert_bits_equal(host_u32(got), exp, f"compaction n={n}")


@pytest.mark.parametrize("n", [1, 2, 7, 31, 8191, 8192, 8193, 3 * 8192 + 5, 100_003, 1 << 20])
def test_mixed_matches_oracle(n):
    check(synth.compaction_input(n, 100 + n))


def test_worked_example():
    x = np.array([1.0, -2.0, 3.0, 0.0, -1.0, 4.0], dtype=np.float32)
    got, nk = gsort.compact_positive(dev(x))
    assert int(nk.item()) == 3
    assert host_u32(got).tolist() == np.array([1, 3, 4, 0, 0, 0], dtype=np.float32).view(
        np.uint32).tolist()


@pytest.mark.parametrize("n", [1, 9000, 70_001])
def test_specials(n):
    x = synth.compaction_input(n, 200 + n)
    b = x.view(np.uint32)
    b[0::11] = 0x7FC00000   # NaN: dropped
    b[1::13] = 0x80000000   # -0: dropped
    b[2::17] = 0x00000001   # +subnormal: kept
    b[3::19] = 0x7F800000   # +inf: kept
    b[4::23] = 0xFF800000   # -inf: dropped
    b[5::29] = 0x80000001   # -subnormal: dropped
    check(x)


@pytest.mark.parametrize("n", [1, 5000, 8192 * 4])
def test_all_kept_none_kept(n):
    check(np.abs(synth.compaction_input(n, 300)) + np.float32(0.5))
    check(-np.abs(synth.compaction_input(n, 301)) - np.float32(0.5))
    check(np.zeros(n, dtype=np.float32))


@pytest.mark.parametrize("offs", [(1, 0), (0, 1), (2, 3), (3, 2)])
def test_misaligned(offs):
    check(synth.compaction_input(50_001, 400), in_off=offs[0], out_off=offs[1])


def test_empty():
    e = torch.empty(0, dtype=torch.float32, device="cuda")
    out, nk = gsort.compact_positive(e)
    assert out.numel() == 0 and int(nk.item()) == 0


def test_repeated_with_shared_workspace():
    n = 123_457
    ws = torch.empty(gsort.compact_workspace_bytes(n), dtype=torch.uint8, device="cuda")
    for s in range(4):
        x = synth.compaction_input(n, 500 + s)
        got, nk = gsort.compact_positive(dev(x), workspace=ws)
        exp, m = oracle.compact_positive(x)
        assert int(nk.item()) == m
        assert_bits_equal(host_u32(got), exp, f"repeat {s}")
