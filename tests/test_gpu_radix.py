"""GPU radix sort vs the CPU oracle, bit for bit: keys, pairs with bit
ranges, float keys, in-place, misaligned buffers, every launch variant, and
the digit-histogram step on its own."""
import numpy as np
import pytest
import torch

import oracle
from bitonic_networks_gb300 import gsort, synth, _lib
from gpu_util import assert_bits_equal, dev, host_u32, offset_view

pytestmark = pytest.mark.gpu

# sizes spanning several tiles (4096 and 8192 keys) with ragged tails
SIZES = [1, 2, 3, 31, 32, 33, 1000, 4095, 4096, 4097, 8191, 8192, 8193, 3 * 8192 + 7,
         65536, 81946, 1_000_003]


def gen_keys(kind: str, n: int, seed: int) -> np.ndarray:
    if kind == "uniform":
        return synth.uniform_keys(n, seed)
    if kind == "and3":
        return synth.and3_keys(n, seed)
    if kind == "distinct16":
        return synth.distinct16_keys(n, seed)
    if kind == "equal":
        return np.full(n, 0xDEADBEEF, dtype=np.uint32)
    if kind == "sorted":
        return np.sort(synth.uniform_keys(n, seed))
    if kind == "reversed":
        return np.sort(synth.uniform_keys(n, seed))[::-1].copy()
    if kind == "extremes":
        k = synth.uniform_keys(n, seed)
        k[::3] = 0
        k[1::3] = 0xFFFFFFFF
        return k
    raise ValueError(kind)


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("kind", ["uniform", "and3", "distinct16", "equal", "sorted",
                                  "reversed", "extremes"])
def test_keys_match_oracle(n, kind):
    k = gen_keys(kind, n, 1000 + n)
    got = gsort.sort_keys(dev(k))
    assert_bits_equal(host_u32(got), oracle.radix_sort_keys(k), f"keys {kind} n={n}")


BIT_RANGES = [(0, 32), (0, 8), (4, 20), (8, 8), (0, 1), (31, 32), (3, 29), (7, 31),
              (24, 32), (0, 16), (16, 32), (1, 32), (0, 24)]


@pytest.mark.parametrize("n", [1, 4097, 8193, 100_003])
@pytest.mark.parametrize("bits", BIT_RANGES)
def test_pairs_bit_ranges_match_oracle(n, bits):
    b, e = bits
    k = synth.and3_keys(n, 2000 + n) ^ synth.uniform_keys(n, 3000 + n) & np.uint32(0x00FF00FF)
    v = synth.index_values(n)
    ko, vo = gsort.sort_pairs(dev(k), dev(v), b, e)
    ek, ev = oracle.radix_sort_pairs(k, v, 0, b, e)
    assert_bits_equal(host_u32(ko), ek, f"keys n={n} bits={bits}")
    assert_bits_equal(host_u32(vo), ev, f"values n={n} bits={bits}")


def float_keys(n: int, seed: int) -> np.ndarray:
    x = synth.normal_f32_with_specials(n, seed)
    if n >= 64:
        bits = x.view(np.uint32)
        bits[5::61] = 0x7FC00000          # +NaN (documented placement: after +inf)
        bits[7::67] = 0xFFC00001          # -NaN (before -inf)
        bits[11::71] = 0x00000001         # +subnormal
        bits[13::73] = 0x80000003         # -subnormal
        x[17::79] = np.float32(1.25)      # ties
    return x


@pytest.mark.parametrize("n", [1, 2, 100, 4097, 3 * 8192 + 5, 1 << 20])
def test_float_pairs_match_oracle(n):
    x = float_keys(n, 4000 + n)
    v = synth.index_values(n)
    ko, vo = gsort.sort_pairs(dev(x), dev(v))
    ek, ev = oracle.radix_sort_pairs(x, v, 1, 0, 32)
    assert_bits_equal(host_u32(ko), ek, f"float keys n={n}")
    assert_bits_equal(host_u32(vo), ev, f"float values n={n}")
    kk = gsort.sort_keys(dev(x))
    assert_bits_equal(host_u32(kk), ek, f"float keys only n={n}")


@pytest.mark.parametrize("bits", [(0, 32), (0, 24), (0, 8), (5, 6)])
@pytest.mark.parametrize("n", [4097, 50_001])
def test_in_place(n, bits):
    b, e = bits
    k = synth.uniform_keys(n, 5000 + n) & np.uint32(0xFF0FFFFF)
    v = synth.index_values(n)
    tk, tv = dev(k), dev(v)
    ko, vo = gsort.sort_pairs(tk, tv, b, e, keys_out=tk, values_out=tv)
    assert ko.data_ptr() == tk.data_ptr()
    ek, ev = oracle.radix_sort_pairs(k, v, 0, b, e)
    assert_bits_equal(host_u32(tk), ek, f"in-place keys {bits}")
    assert_bits_equal(host_u32(tv), ev, f"in-place values {bits}")
    # keys only, in place
    t = dev(k)
    gsort.sort_pairs(t, None, b, e, keys_out=t)
    assert_bits_equal(host_u32(t), oracle.radix_sort_pairs(k, None, 0, b, e)[0], "in-place keys only")


@pytest.mark.parametrize("offs", [(1, 0, 2, 3), (3, 1, 0, 2), (2, 2, 1, 1)])
def test_misaligned_buffers(offs):
    n = 3 * 8192 + 11
    k = synth.uniform_keys(n, 6000)
    v = synth.index_values(n)
    ki = offset_view(dev(k), n, offs[0])
    ko = offset_view(dev(k), n, offs[1])
    vi = offset_view(dev(v), n, offs[2])
    vo = offset_view(dev(v), n, offs[3])
    gsort.sort_pairs(ki, vi, keys_out=ko, values_out=vo)
    ek, ev = oracle.radix_sort_pairs(k, v, 0, 0, 32)
    assert_bits_equal(host_u32(ko), ek, "misaligned keys")
    assert_bits_equal(host_u32(vo), ev, "misaligned values")
    h = gsort.digit_histograms(ki)
    assert_bits_equal(host_u32(h), oracle.digit_histograms(k), "misaligned histogram")


@pytest.mark.parametrize("variant", range(_lib.load().gsort_radix_num_variants()))
def test_every_variant(variant):
    n = 1_000_003
    k = synth.and3_keys(n, 7000)
    v = synth.index_values(n)
    ko, vo = gsort.sort_pairs(dev(k), dev(v), variant=variant)
    ek, ev = oracle.radix_sort_pairs(k, v, 0, 0, 32)
    assert_bits_equal(host_u32(ko), ek, f"variant {variant} keys")
    assert_bits_equal(host_u32(vo), ev, f"variant {variant} values")
    x = float_keys(n, 7001)
    kx = gsort.sort_pairs(dev(x), None, variant=variant)[0]
    assert_bits_equal(host_u32(kx), oracle.radix_sort_keys(x, 1), f"variant {variant} floats")
    for m in (1, 4097, 12289):
        km = gsort.sort_pairs(dev(k[:m]), None, variant=variant)[0]
        assert_bits_equal(host_u32(km), oracle.radix_sort_keys(k[:m]), f"variant {variant} n={m}")


@pytest.mark.parametrize("bits", [(0, 32), (3, 21), (0, 1), (8, 31), (16, 24)])
@pytest.mark.parametrize("n", [1, 4096, 100_003])
def test_digit_histograms_match_oracle(n, bits):
    b, e = bits
    k = synth.and3_keys(n, 8000 + n)
    h = gsort.digit_histograms(dev(k), b, e)
    assert_bits_equal(host_u32(h), oracle.digit_histograms(k, 0, b, e), f"hist {bits}")
    x = float_keys(n, 8001 + n)
    # float keys: histogram of the mapped keys
    k32 = dev(x)
    hf = torch.empty((4, 256), dtype=torch.int32, device="cuda")
    lib = _lib.load()
    rc = lib.gsort_digit_histograms(k32.data_ptr(), n, 1, 0, 32, hf.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    assert_bits_equal(host_u32(hf), oracle.digit_histograms(x, 1, 0, 32), "float hist")


def test_repeated_calls_reuse_workspace():
    n = 200_003
    ws = torch.empty(gsort.radix_workspace_bytes(n, True), dtype=torch.uint8, device="cuda")
    for seed in range(5):
        k = synth.distinct16_keys(n, 9000 + seed)
        v = synth.index_values(n)
        ko, vo = gsort.sort_pairs(dev(k), dev(v), workspace=ws)
        ek, ev = oracle.radix_sort_pairs(k, v, 0, 0, 32)
        assert_bits_equal(host_u32(ko), ek, f"reuse {seed} keys")
        assert_bits_equal(host_u32(vo), ev, f"reuse {seed} values")


def test_empty_and_host_tensors():
    e = torch.empty(0, dtype=torch.int32, device="cuda")
    assert gsort.sort_keys(e).numel() == 0
    k = synth.uniform_keys(1000, 10)
    got = gsort.sort_keys(torch.from_numpy(k.view(np.int32).copy()))   # CPU tensor round trip
    assert not got.is_cuda
    assert_bits_equal(got.numpy(), oracle.radix_sort_keys(k), "host round trip")


def test_stream_is_respected():
    n = 300_001
    k = synth.uniform_keys(n, 11)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        t = dev(k)
        out = gsort.sort_keys(t, check=False)
    s.synchronize()
    assert_bits_equal(host_u32(out), oracle.radix_sort_keys(k), "side stream")
