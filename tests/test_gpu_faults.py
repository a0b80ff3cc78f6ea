"""Failure detection without a GPU fault: a test-only option makes one tile
never publish its counts, so the look-back waits behind it run out after a
short, bounded number of polls.  The kernels then record GSORT_ETIMEOUT in the
workspace and return; the host reads the status, and the context stays usable
(the next call succeeds)."""
import numpy as np
import pytest
import torch

import oracle
from bitonic_networks_gb300 import gsort, synth
from gpu_util import assert_bits_equal, dev, host_u32

pytestmark = pytest.mark.gpu

ETIMEOUT = -6


# 2^16 keys take the one-launch small-input kernel (a stalled CTA never reaches
# the grid barrier); 2^19 keys the per-pass kernels (a stalled tile never
# publishes, so the look-backs behind it wait)
@pytest.mark.parametrize("n", [8 * 8192, 64 * 8192])
@pytest.mark.parametrize("stall", [0, 1, 3])
def test_radix_wait_gives_up_and_reports(stall, n):
    k = synth.uniform_keys(n, 1)
    with pytest.raises(gsort.GsortError) as e:
        gsort.sort_pairs(dev(k), dev(synth.index_values(n)), spin_limit=2000, stall_tile=stall)
    assert e.value.code == ETIMEOUT
    # the device is still healthy: a normal call right after is exact
    got = gsort.sort_keys(dev(k))
    assert_bits_equal(host_u32(got), oracle.radix_sort_keys(k), "after timeout")


# keys only, every bit: the first pass reserves bin places with atomic cursors
# and waits for nothing; the stalled tile then never publishes in the second
# pass, whose look-backs give up
@pytest.mark.parametrize("stall", [0, 3])
def test_keys_only_wait_gives_up_and_reports(stall):
    n = 64 * 8192
    k = synth.uniform_keys(n, 4)
    with pytest.raises(gsort.GsortError) as e:
        gsort.sort_pairs(dev(k), None, spin_limit=2000, stall_tile=stall)
    assert e.value.code == ETIMEOUT
    got = gsort.sort_keys(dev(k))
    assert_bits_equal(host_u32(got), oracle.radix_sort_keys(k), "after timeout")


@pytest.mark.parametrize("stall", [0, 2])
def test_compaction_wait_gives_up_and_reports(stall):
    n = 8 * 8192
    x = synth.compaction_input(n, 2)
    with pytest.raises(gsort.GsortError) as e:
        gsort.compact_positive(dev(x), spin_limit=2000, stall_tile=stall)
    assert e.value.code == ETIMEOUT
    got, nk = gsort.compact_positive(dev(x))
    exp, m = oracle.compact_positive(x)
    assert int(nk.item()) == m
    assert_bits_equal(host_u32(got), exp, "after timeout")


def test_last_tile_stall_is_harmless_to_others():
    # a stall id beyond the grid: no timeout
    n = 64 * 8192
    k = synth.uniform_keys(n, 3)
    ko, _ = gsort.sort_pairs(dev(k), None, spin_limit=2000, stall_tile=10**6)  # no such tile
    assert_bits_equal(host_u32(ko), oracle.radix_sort_keys(k), "stall id beyond the grid")
