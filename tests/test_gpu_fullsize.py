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


# ---- the "next" rows at the sizes the bench rows time

def test_u64_full_size():
    w = synth.WORKLOADS["uniform_u64_2^27"]
    k = synth.make_keys(w["gen"], w["n"], w["seed"])
    t = torch.from_numpy(k.view(np.int64)).cuda()
    got, _ = gsort.sort(t, kind=gsort.KEY_U64)
    got = got.cpu().numpy().view(np.uint64)
    del t
    torch.cuda.empty_cache()
    exp, _ = oracle.default().radix_sort(k, None, 3)
    assert np.array_equal(got, exp), "u64 keys"


def test_segments_mixed_full_size():
    w = synth.WORKLOADS["segments_mixed_2^26"]
    k = synth.make_keys(w["gen"], w["n"], w["seed"])
    off = synth.segment_offsets(w["n"], w["mix"], w["seed"])
    v = synth.index_values(w["n"])
    ko, vo = gsort.segmented_sort(dev(k), dev(off), dev(v), kind=gsort.KEY_U32)
    ek, ev = oracle.default().segmented_sort_general(k, off, v, 0)
    assert_bits_equal(host_u32(ko), ek, "segmented keys")
    assert_bits_equal(host_u32(vo), ev, "segmented values")


def test_partition_full_size():
    w = synth.WORKLOADS["partition_f32_2^28"]
    x = synth.make_keys(w["gen"], w["n"], w["seed"])
    o, _, nt = gsort.partition(dev(x), pred=gsort.PRED_POSITIVE)
    eo, _, m = oracle.default().partition(x, None, pred=4)
    assert int(nt.item()) == m
    assert_bits_equal(host_u32(o), eo, "partition")


def test_split_sort_full_size():
    w = synth.WORKLOADS["split_sort_u32_2^25"]
    k = synth.make_keys(w["gen"], w["n"], w["seed"])
    v = synth.index_values(w["n"])
    ko, vo = gsort.split_sort(dev(k), dev(v))
    ek, ev = oracle.default().split_sort(k, v, 0, 32)
    assert_bits_equal(host_u32(ko), ek, "split sort keys")
    assert_bits_equal(host_u32(vo), ev, "split sort values")
