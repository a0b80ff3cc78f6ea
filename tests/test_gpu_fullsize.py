"""Parity at the full problem sizes, in the launch configuration the bench
times (default variant): every output element compared with the CPU oracle,
which finishes each of these in seconds."""
import numpy as np
import pytest
import torch

import oracle
from bitonic_networks_gb300 import gsort, synth
from gpu_util import assert_bits_equal, dev, host_u32

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.mark.parametrize("name", ["uniform_u32_65536", "uniform_u32_2^28", "and3_u32_2^28",
                                  "distinct16_u32_2^28"])
def test_keys_full_size(name):
    w = synth.WORKLOADS[name]
    k = synth.make_keys(w["gen"], w["n"], w["seed"])
    t = dev(k)
    got = host_u32(gsort.sort_keys(t))
    del t
    torch.cuda.empty_cache()
    assert_bits_equal(got, oracle.radix_sort_keys(k), name)


def test_pairs_full_size():
    w = synth.WORKLOADS["pairs_u32_2^24"]
    k = synth.make_keys(w["gen"], w["n"], w["seed"])
    v = synth.index_values(w["n"])
    ko, vo = gsort.sort_pairs(dev(k), dev(v))
    ek, ev = oracle.radix_sort_pairs(k, v, 0, 0, 32)
    assert_bits_equal(host_u32(ko), ek, "pairs keys")
    assert_bits_equal(host_u32(vo), ev, "pairs values (stability)")


def test_float_pairs_full_size():
    w = synth.WORKLOADS["normal_f32_pairs_2^26"]
    x = synth.make_keys(w["gen"], w["n"], w["seed"])
    v = synth.index_values(w["n"])
    ko, vo = gsort.sort_pairs(dev(x), dev(v))
    ek, ev = oracle.radix_sort_pairs(x, v, 1, 0, 32)
    assert_bits_equal(host_u32(ko), ek, "float keys")
    assert_bits_equal(host_u32(vo), ev, "float values")


def test_segments_full_size():
    w = synth.WORKLOADS["segments_16384x1024"]
    a = synth.segments(w["segments"], w["length"], w["seed"])
    t = dev(a)
    gsort.segmented_sort_(t)
    assert_bits_equal(host_u32(t), oracle.segmented_sort(a), "segments")


def test_compaction_full_size():
    w = synth.WORKLOADS["compact_f32_2^28"]
    x = synth.make_keys(w["gen"], w["n"], w["seed"])
    got, nk = gsort.compact_positive(dev(x))
    exp, m = oracle.compact_positive(x)
    assert int(nk.item()) == m
    assert_bits_equal(host_u32(got), exp, "compaction")
