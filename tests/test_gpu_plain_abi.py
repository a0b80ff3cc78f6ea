"""The plain boundary calls, made directly through ctypes, vs the CPU oracle.

gsort_radix_keys, gsort_radix_pairs, gsort_compact_positive and
gsort_segmented_bitonic are the calls the problem statement names.  The
Python wrapper goes through their option-taking forms, so these tests call
the plain symbols themselves: device buffers and the workspace come from
torch, the stream is torch's current stream, and every output element is
compared bit for bit with the oracle.  A second group repeats small sorts of
at most four tiles over many seeds, so that the look-back between tiles runs
in many different interleavings.
"""
import numpy as np
import pytest
import torch

import oracle
from bitonic_networks_gb300 import _lib, gsort, synth
from gpu_util import assert_bits_equal, dev, host_u32, offset_view

pytestmark = pytest.mark.gpu

KEY_U32, KEY_F32 = 0, 1


def stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def check_status(lib, ws: torch.Tensor):
    rc = lib.gsort_check(ws.data_ptr(), stream())
    assert rc == 0, lib.gsort_status_string(rc)


def radix_keys(k: np.ndarray, kind: int, in_place: bool = False, off: int = 0):
    lib = _lib.load()
    n = k.size
    kin = dev(k)
    if off:
        kin = offset_view(kin, n, off)
    kout = kin if in_place else torch.full((n,), -1, dtype=torch.int32, device="cuda")
    ws = torch.empty(lib.gsort_radix_workspace_bytes(n, 0), dtype=torch.uint8, device="cuda")
    rc = lib.gsort_radix_keys(kin.data_ptr(), kout.data_ptr(), n, kind, ws.data_ptr(), ws.numel(),
                              stream())
    assert rc == 0, lib.gsort_status_string(rc)
    check_status(lib, ws)
    return host_u32(kout)


def radix_pairs(k: np.ndarray, v: np.ndarray, kind: int, begin_bit: int, end_bit: int):
    lib = _lib.load()
    n = k.size
    kin, vin = dev(k), dev(v)
    kout = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    vout = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    ws = torch.empty(lib.gsort_radix_workspace_bytes(n, 1), dtype=torch.uint8, device="cuda")
    rc = lib.gsort_radix_pairs(kin.data_ptr(), kout.data_ptr(), vin.data_ptr(), vout.data_ptr(), n,
                               kind, begin_bit, end_bit, ws.data_ptr(), ws.numel(), stream())
    assert rc == 0, lib.gsort_status_string(rc)
    check_status(lib, ws)
    return host_u32(kout), host_u32(vout)


@pytest.mark.parametrize("n", [1, 3, 65_536, 300_007, 1 << 21])
def test_radix_keys_u32(n):
    k = synth.uniform_keys(n, 11_000 + n % 97)
    assert_bits_equal(radix_keys(k, KEY_U32), oracle.radix_sort_keys(k), f"gsort_radix_keys n={n}")


@pytest.mark.parametrize("n", [5, 70_001, 1 << 20])
def test_radix_keys_f32_specials(n):
    x = synth.normal_f32_with_specials(n, 11_100 + n % 89)
    b = x.view(np.uint32)
    b[::101] = 0x7FC00000   # +NaN: after +inf under the order map
    b[1::103] = 0xFFC00000  # -NaN: before -inf
    b[2::107] = 0x00000001  # subnormals of both signs
    b[3::109] = 0x80000001
    exp = oracle.radix_sort_keys(x, 1)
    assert_bits_equal(radix_keys(x, KEY_F32), exp, f"gsort_radix_keys f32 n={n}")


def test_radix_keys_in_place_and_misaligned():
    k = synth.uniform_keys(400_003, 11_200)
    exp = oracle.radix_sort_keys(k)
    assert_bits_equal(radix_keys(k, KEY_U32, in_place=True), exp, "in place")
    assert_bits_equal(radix_keys(k, KEY_U32, in_place=True, off=1), exp, "in place, 4-byte aligned")


@pytest.mark.parametrize("bits", [(0, 32), (0, 13), (7, 32), (5, 21), (16, 16)])
@pytest.mark.parametrize("kind", [KEY_U32, KEY_F32])
def test_radix_pairs(bits, kind):
    n = 250_001
    k = synth.and3_keys(n, 11_300 + bits[0] * 7 + bits[1])
    if kind == KEY_F32:
        k = k & np.uint32(0xBFFFFFFF)   # finite floats, both signs
    v = synth.index_values(n)
    got_k, got_v = radix_pairs(k, v, kind, *bits)
    exp_k, exp_v = oracle.radix_sort_pairs(k.view(np.float32) if kind == KEY_F32 else k, v, kind, *bits)
    assert_bits_equal(got_k, exp_k, f"gsort_radix_pairs keys {bits} kind {kind}")
    assert_bits_equal(got_v, exp_v, f"gsort_radix_pairs values {bits} kind {kind}")


@pytest.mark.parametrize("n", [1, 8193, 1_000_003])
def test_compact_positive(n):
    lib = _lib.load()
    x = synth.compaction_input(n, 11_400 + n % 83)
    b = x.view(np.uint32)
    b[::71] = 0x7FC00000    # NaN: dropped
    b[1::73] = 0x80000000   # -0: dropped
    b[2::79] = 0x00000001   # +subnormal: kept
    xi = dev(x)
    out = torch.full((n,), 7.0, dtype=torch.float32, device="cuda")
    kept = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    ws = torch.empty(lib.gsort_compact_workspace_bytes(n), dtype=torch.uint8, device="cuda")
    rc = lib.gsort_compact_positive(xi.data_ptr(), out.data_ptr(), n, kept.data_ptr(), ws.data_ptr(),
                                    ws.numel(), stream())
    assert rc == 0, lib.gsort_status_string(rc)
    check_status(lib, ws)
    exp, m = oracle.compact_positive(x)
    assert int(kept.item()) == m
    assert_bits_equal(host_u32(out), exp, f"gsort_compact_positive n={n}")


@pytest.mark.parametrize("shape", [(16384, 1024), (333, 1000), (7, 1), (1000, 33)])
def test_segmented_bitonic(shape):
    lib = _lib.load()
    s, length = shape
    k = synth.segments(s, length, 11_500 + length)
    t = dev(k.ravel())
    rc = lib.gsort_segmented_bitonic(t.data_ptr(), s, length, stream())
    assert rc == 0, lib.gsort_status_string(rc)
    torch.cuda.synchronize()
    exp = oracle.segmented_sort(k.reshape(s, length))
    assert_bits_equal(host_u32(t), exp, f"gsort_segmented_bitonic {shape}")


# Look-back races: sorts of two to four tiles, repeated over many seeds with
# one workspace (the histogram kernel and each pass clear the look-back words
# the next pass uses).  Variants 1 and 2 tile such small inputs (variant 0
# sorts them in one cooperative launch).
@pytest.mark.parametrize("variant,tile", [(1, 8192), (2, 4096)])
@pytest.mark.parametrize("tiles", [2, 3, 4])
def test_lookback_many_seeds(variant, tile, tiles):
    n = tiles * tile - 333
    ws = torch.empty(gsort.radix_workspace_bytes(n, True), dtype=torch.uint8, device="cuda")
    v = synth.index_values(n)
    vd = dev(v)
    for seed in range(12_000 + 1000 * tiles + 100 * variant, 12_000 + 1000 * tiles + 100 * variant + 100):
        if seed % 2:   # pairs of skewed keys: every pass stable
            k = synth.and3_keys(n, seed)
            got_k, got_v = gsort.sort_pairs(dev(k), vd, 0, 32, workspace=ws, variant=variant)
            exp_k, exp_v = oracle.radix_sort_pairs(k, v, 0, 0, 32)
            assert_bits_equal(host_u32(got_v), exp_v, f"values seed {seed}")
        else:          # keys only: order-free first pass and warps
            k = synth.uniform_keys(n, seed)
            got_k, _ = gsort.sort_pairs(dev(k), None, 0, 32, workspace=ws, variant=variant)
            exp_k = oracle.radix_sort_keys(k)
        assert_bits_equal(host_u32(got_k), exp_k, f"keys seed {seed}")
