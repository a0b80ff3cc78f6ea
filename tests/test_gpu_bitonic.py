"""GPU segmented bitonic sort vs the CPU oracle (each segment sorted)."""
import numpy as np
import pytest
import torch

import oracle
from bitonic_networks_gb300 import gsort, synth
from gpu_util import assert_bits_equal, dev, host_u32

pytestmark = pytest.mark.gpu

LENGTHS = [1, 2, 3, 5, 16, 31, 32, 33, 63, 64, 65, 100, 127, 128, 129, 255, 256, 257, 500,
           511, 512, 513, 1000, 1023, 1024]


@pytest.mark.parametrize("length", LENGTHS)
@pytest.mark.parametrize("segments", [1, 5, 4097])
def test_uniform_segments(length, segments):
    a = synth.segments(segments, length, 10 * length + segments)
    t = dev(a)
    gsort.segmented_sort_(t)
    assert_bits_equal(host_u32(t), oracle.segmented_sort(a), f"L={length} S={segments}")


@pytest.mark.parametrize("length", [8, 100, 1024])
def test_adversarial_segments(length):
    S = 64
    a = synth.segments(S, length, 77 + length)
    a[0] = 0xFFFFFFFF                         # all padding value
    a[1] = 0
    a[2] = np.sort(a[2])
    a[3] = np.sort(a[3])[::-1]
    a[4] = a[4] & np.uint32(1)                # 0/1 keys
    a[5] = a[5] & np.uint32(0x80000001)
    a[6, ::2] = 0xFFFFFFFF
    t = dev(a)
    gsort.segmented_sort_(t)
    assert_bits_equal(host_u32(t), oracle.segmented_sort(a), f"adversarial L={length}")


def test_exercise_example():
    # the 8-key tracing exercise, padded internally to a warp's 32 slots
    a = np.array([[5, 2, 8, 1, 9, 3, 7, 4]], dtype=np.uint32)
    t = dev(a)
    gsort.segmented_sort_(t)
    assert host_u32(t).tolist() == [[1, 2, 3, 4, 5, 7, 8, 9]]


def test_zero_one_principle_16():
    # every 0/1 input of one 16-key segment (the 0-1 principle)
    m = np.arange(1 << 16, dtype=np.uint32)
    a = ((m[:, None] >> np.arange(16, dtype=np.uint32)[None, :]) & 1).astype(np.uint32)
    t = dev(a)
    gsort.segmented_sort_(t)
    assert_bits_equal(host_u32(t), np.sort(a, axis=1), "0-1 principle, L=16")


def test_no_segments_and_untouched_neighbours():
    a = synth.segments(10, 300, 5)
    t = dev(a.ravel())
    body = t[300:300 * 9].view(8, 300)          # sort the middle 8 segments only
    gsort.segmented_sort_(body)
    got = host_u32(t).reshape(10, 300)
    assert_bits_equal(got[0], a[0], "segment before")
    assert_bits_equal(got[9], a[9], "segment after")
    assert_bits_equal(got[1:9], oracle.segmented_sort(a[1:9]), "middle")
    e = torch.empty((0, 64), dtype=torch.int32, device="cuda")
    gsort.segmented_sort_(e)
