"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every symbol include/gsort.h declares, sizes workspaces as documented, and
rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "gsort.h")


@pytest.fixture(scope="module")
def lib():
    from bitonic_networks_gb300 import _lib
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(gsort_\w+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_four_calls():
    names = declared_functions()
    for n in ("gsort_radix_keys", "gsort_radix_pairs", "gsort_compact_positive",
              "gsort_segmented_bitonic"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from bitonic_networks_gb300 import _lib
    names = declared_functions()
    assert names, "no declarations parsed"
    for name in names:
        assert hasattr(lib, name), f"libgsort.so does not export {name}"
        assert name in _lib.SIGNATURES, f"binding lacks a signature for {name}"


def test_status_strings_and_version(lib):
    assert lib.gsort_status_string(0) == b"GSORT_OK"
    for code in range(-6, 0):
        assert lib.gsort_status_string(code).startswith(b"GSORT_E")
    assert lib.gsort_version() >= 100
    assert lib.gsort_radix_num_variants() >= 1
    for v in range(lib.gsort_radix_num_variants()):
        assert lib.gsort_radix_variant_name(v)
    assert lib.gsort_radix_variant_name(99) is None


def test_workspace_sizes(lib):
    HDR = 8192

    def up(x):
        return -(-x // 256) * 256
    for n in (1, 4095, 4096, 4097, 65536, 1 << 18, (1 << 18) + 1, 1 << 24, (1 << 30) - 1):
        tiles = (n + 4095) // 4096
        state = 2 * up(tiles * 1024)   # two alternating regions of look-back words
        keys = up(n * 4)
        # up to 2^18 keys: three count buffers of the one-launch sort, a row per 2048 keys
        small = up(3 * ((n + 2047) // 2048) * 1024) if n <= 1 << 18 else 0
        starts = 8 * 1024   # bin starts of up to 8 passes
        assert lib.gsort_radix_workspace_bytes(n, 0) == HDR + starts + state + keys + small
        assert lib.gsort_radix_workspace_bytes(n, 1) == HDR + starts + state + 2 * keys + small
        ctiles = (n + 8191) // 8192
        assert lib.gsort_compact_workspace_bytes(n) == HDR + up(ctiles * 128)   # a line per tile
    assert lib.gsort_radix_workspace_bytes(-1, 0) == 0
    assert lib.gsort_radix_workspace_bytes(1 << 30, 0) == 0
    assert lib.gsort_compact_workspace_bytes(1 << 30) == 0


def test_general_workspace_sizes(lib):
    HDR = 8192

    def up(x):
        return -(-x // 256) * 256
    for n in (1, 4097, 1 << 20, (1 << 30) - 1):
        tiles = (n + 4095) // 4096
        state = 2 * up(tiles * 1024)
        for kind in (0, 1, 2):     # 32-bit kinds: the same layout as gsort_radix_workspace_bytes
            for wv in (0, 1):
                assert lib.gsort_radix_sort_workspace_bytes(n, kind, wv) == \
                    lib.gsort_radix_workspace_bytes(n, wv)
        for kind in (3, 4, 5):     # 64-bit kinds: 8 KiB of bin starts and 8 KiB of histograms, 8-byte keys
            assert lib.gsort_radix_sort_workspace_bytes(n, kind, 0) == HDR + 2 * 8192 + state + up(8 * n)
            assert lib.gsort_radix_sort_workspace_bytes(n, kind, 1) == \
                HDR + 2 * 8192 + state + up(8 * n) + up(4 * n)
    assert lib.gsort_radix_sort_workspace_bytes(10, 6, 0) == 0
    assert lib.gsort_radix_sort_workspace_bytes(10, -1, 0) == 0
    assert lib.gsort_radix_sort_workspace_bytes(1 << 30, 3, 0) == 0


def test_general_argument_errors(lib):
    big = 1 << 40
    f = lib.gsort_radix_sort
    assert f(A, B, None, None, 0, 3, 1, 0, 64, None, 0, None) == 0            # n == 0: no-op
    assert f(A, B, None, None, 10, 6, 0, 0, 32, W, big, None) == EINVAL        # no such kind
    assert f(A, B, None, None, 10, 0, 2, 0, 32, W, big, None) == EINVAL        # unknown flag
    assert f(A, B, None, None, 10, 2, 0, 0, 33, W, big, None) == EINVAL        # 32-bit kind, 33 bits
    assert f(A, B, None, None, 10, 3, 0, 0, 65, W, big, None) == EINVAL
    assert f(A + 4, B, None, None, 10, 3, 0, 0, 64, W, big, None) == EALIGN    # 64-bit keys: 8-byte aligned
    assert f(A, B + 4, None, None, 10, 5, 0, 0, 64, W, big, None) == EALIGN
    assert f(A, A + 8, None, None, 10, 3, 0, 0, 64, W, big, None) == EINVAL   # partial overlap (8-byte keys)
    # output values must not fall inside the 8-byte keys (10 keys = 80 bytes)
    assert f(A, B, B + 0x1000, A + 40, 10, 3, 0, 0, 64, W, big, None) == EINVAL
    assert f(A, B, A + 0x1000, B + 72, 10, 3, 0, 0, 64, W, big, None) == EINVAL
    assert f(A, B, None, None, 10, 3, 0, 0, 64, W, 100, None) == EWS
    assert f(A, B, None, None, 10, 3, 0, 0, 64, None, big, None) == EWS
    opt = __import__("bitonic_networks_gb300._lib", fromlist=["Options"]).Options(0, -1, None, 0, 1)
    assert lib.gsort_radix_sort_ex(A, B, None, None, 10, 3, 0, 0, 64, W, big, None,
                                   ctypes.byref(opt)) == EINVAL            # 64-bit keys: variant 0 only
    # the 32-bit calls refuse 64-bit kinds
    assert lib.gsort_radix_pairs(A, B, None, None, 10, 3, 0, 32, W, big, None) == EINVAL
    assert lib.gsort_radix_keys(A, B, 10, 4, W, big, None) == EINVAL
    h = lib.gsort_digit_histograms
    assert h(A, 10, 3, 0, 65, B, None) == EINVAL
    assert h(A + 4, 10, 3, 0, 64, B, None) == EALIGN
    assert h(A, 10, 6, 0, 8, B, None) == EINVAL


def test_segmented_sort_argument_errors(lib):
    big = 1 << 40
    O = 0x30000000
    f = lib.gsort_segmented_sort
    assert f(A, B, None, None, 0, O, 5, 0, 0, None, 0, None) == 0              # n == 0: no-op
    assert f(A, B, None, None, 10, O, 0, 0, 0, W, big, None) == EINVAL         # keys but no segment
    assert f(A, B, None, None, -1, O, 1, 0, 0, W, big, None) == EINVAL
    assert f(A, B, None, None, 1 << 30, O, 1, 0, 0, W, big, None) == ETOOBIG
    assert f(A, B, None, None, 10, O, 1, 3, 0, W, big, None) == EINVAL         # 64-bit kind
    assert f(A, B, None, None, 10, O, 1, 0, 4, W, big, None) == EINVAL         # unknown flag
    assert f(A, B, None, None, 10, None, 1, 0, 0, W, big, None) == EINVAL
    assert f(A, B, None, None, 10, O + 2, 1, 0, 0, W, big, None) == EALIGN
    assert f(A, B, A + 0x1000, None, 10, O, 1, 0, 0, W, big, None) == EINVAL   # values half given
    assert f(A, A + 4, None, None, 10, O, 1, 0, 0, W, big, None) == EINVAL     # partial overlap
    assert f(A, B, None, None, 10, B + 8, 1, 0, 0, W, big, None) == EINVAL     # offsets inside the output
    assert f(A, B, None, None, 10, O, 1, 0, 0, W, 64, None) == EWS
    assert f(A, B, None, None, 10, O, 1, 0, 0, W + 8, big, None) == EALIGN
    assert f(A, B, None, None, 10, O, 1, 0, 0, O, big, None) == EINVAL         # workspace over the offsets
    ws = lib.gsort_segmented_sort_workspace_bytes
    assert ws(-1, 1, 0) == 0 and ws(10, -1, 0) == 0 and ws(1 << 30, 1, 0) == 0
    assert ws(1 << 20, 1, 1) > ws(1 << 20, 1, 0) > 4 * (1 << 20)


def test_partition_and_split_sort_argument_errors(lib):
    big = 1 << 40
    F = 0x50000000
    p = lib.gsort_partition
    assert p(A, B, None, None, 0, 1, 0, 3, None, None, W, big, None) == 0         # n == 0 (no num_true)
    assert p(A, B, None, None, -1, 1, 0, 3, None, None, W, big, None) == EINVAL
    assert p(A, B, None, None, 10, 5, 0, 3, None, None, W, big, None) == EINVAL   # no such predicate
    assert p(A, B, None, None, 10, 1, 0, 32, None, None, W, big, None) == EINVAL  # bit 32
    assert p(A, B, None, None, 10, 3, 3, 0, None, None, W, big, None) == EINVAL   # LESS on a 64-bit kind
    assert p(A, B, None, None, 10, 0, 0, 0, None, None, W, big, None) == EINVAL   # flags missing
    assert p(A, A + 8, None, None, 10, 1, 0, 0, None, None, W, big, None) == EINVAL   # in/out overlap
    assert p(A, A, None, None, 10, 1, 0, 0, None, None, W, big, None) == EINVAL   # no in place
    assert p(A, B, None, None, 10, 0, 0, 0, B + 4, None, W, big, None) == EINVAL  # flags inside out
    assert p(A + 2, B, None, None, 10, 1, 0, 0, None, None, W, big, None) == EALIGN
    assert p(A, B, None, None, 10, 1, 0, 0, None, W + 4, W + 0x1000, big, None) == EALIGN   # num_true
    assert p(A, B, None, None, 10, 1, 0, 0, None, None, W, 16, None) == EWS
    s = lib.gsort_split_sort
    assert s(A, B, None, None, 0, 0, 32, None, 0, None) == 0
    assert s(A, B, None, None, 10, 0, 33, W, big, None) == EINVAL
    assert s(A, B, None, None, 10, 5, 4, W, big, None) == EINVAL
    assert s(A, A + 4, None, None, 10, 0, 32, W, big, None) == EINVAL
    assert s(A, B, None, None, 10, 0, 32, W, 64, None) == EWS
    assert lib.gsort_split_sort_workspace_bytes(1 << 20, 1) > lib.gsort_split_sort_workspace_bytes(1 << 20, 0)
    assert lib.gsort_partition_workspace_bytes(-1) == 0


def test_launch_count(lib):
    assert lib.gsort_radix_launch_count(100, 0, 32, 0) == 1          # up to 65,536 keys: one cluster kernel
    assert lib.gsort_radix_launch_count(1 << 16, 0, 32, 0) == 1
    assert lib.gsort_radix_launch_count((1 << 16) + 1, 0, 32, 0) == 2  # then one cooperative kernel
    assert lib.gsort_radix_launch_count(1 << 18, 0, 32, 1) == 2
    # header clear, histogram (its last CTA writes the bin starts), the passes
    assert lib.gsort_radix_launch_count((1 << 18) + 1, 0, 32, 0) == 6
    assert lib.gsort_radix_launch_count(1 << 20, 0, 8, 0) == 3
    assert lib.gsort_radix_launch_count(1 << 20, 0, 24, 1) == 6
    assert lib.gsort_radix_launch_count(0, 0, 32, 0) == 0
    assert lib.gsort_radix_launch_count(100, 5, 5, 0) == 0
    assert lib.gsort_radix_sort_launch_count(100, 3, 0, 64, 0) == 11      # 2 + 8 passes + hist clear
    assert lib.gsort_radix_sort_launch_count(100, 5, 0, 56, 1) == 11      # 7 passes, in place: + copy
    assert lib.gsort_radix_sort_launch_count(1 << 20, 2, 0, 32, 0) == 6
    assert lib.gsort_radix_sort_launch_count(100, 2, 0, 32, 0) == 1


# Fake device addresses: validation rejects these calls before any CUDA call.
A = 0x10000000
B = 0x20000000
W = 0x40000000
EINVAL, EALIGN, EWS, ETOOBIG = -1, -2, -3, -4


def test_radix_argument_errors(lib):
    big = 1 << 40
    f = lib.gsort_radix_pairs
    assert f(A, B, None, None, 0, 0, 0, 32, None, 0, None) == 0          # n == 0: no-op
    assert f(A, B, None, None, -1, 0, 0, 32, W, big, None) == EINVAL
    assert f(A, B, None, None, 1 << 30, 0, 0, 32, W, big, None) == ETOOBIG
    assert f(A, B, None, None, 10, 6, 0, 32, W, big, None) == EINVAL      # bad kind
    assert f(A, B, None, None, 10, 0, 5, 4, W, big, None) == EINVAL       # begin > end
    assert f(A, B, None, None, 10, 0, 0, 33, W, big, None) == EINVAL
    assert f(A, B, None, None, 10, 0, -1, 8, W, big, None) == EINVAL
    assert f(None, B, None, None, 10, 0, 0, 32, W, big, None) == EINVAL
    assert f(A, B, A + 0x1000, None, 10, 0, 0, 32, W, big, None) == EINVAL   # values half given
    assert f(A + 2, B, None, None, 10, 0, 0, 32, W, big, None) == EALIGN
    assert f(A, B + 1, None, None, 10, 0, 0, 32, W, big, None) == EALIGN
    assert f(A, A + 4, None, None, 10, 0, 0, 32, W, big, None) == EINVAL     # partial overlap
    assert f(A, B, None, None, 10, 0, 0, 32, None, big, None) == EWS
    assert f(A, B, None, None, 10, 0, 0, 32, W, 100, None) == EWS
    assert f(A, B, None, None, 10, 0, 0, 32, W + 16, big, None) == EALIGN     # ws not 256-aligned
    assert f(A, B, None, None, 10, 0, 0, 32, A, big, None) == EINVAL          # ws overlaps keys
    # keys and values must not share memory
    assert f(A, B, A + 0x100000, B, 10, 0, 0, 32, W, big, None) == EINVAL
    assert lib.gsort_radix_keys(A, B, -5, 0, W, big, None) == EINVAL
    assert lib.gsort_radix_keys(A, B, 10, 7, W, big, None) == EINVAL
    opt = __import__("bitonic_networks_gb300._lib", fromlist=["Options"]).Options(0, -1, None, 0, 999)
    assert lib.gsort_radix_pairs_ex(A, B, None, None, 10, 0, 0, 32, W, big, None,
                                    ctypes.byref(opt)) == EINVAL            # no such variant


def test_compaction_and_segment_argument_errors(lib):
    big = 1 << 40
    f = lib.gsort_compact_positive
    assert f(A, B, -1, None, W, big, None) == EINVAL
    assert f(A, B, 1 << 30, None, W, big, None) == ETOOBIG
    assert f(None, B, 10, None, W, big, None) == EINVAL
    assert f(A + 1, B, 10, None, W, big, None) == EALIGN
    assert f(A, A + 8, 10, None, W, big, None) == EINVAL                      # overlap
    assert f(A, B, 10, W + 4, W + 0x1000, big, None) == EALIGN                # num_kept alignment
    assert f(A, B, 10, None, None, big, None) == EWS
    assert f(A, B, 10, None, W, 16, None) == EWS
    g = lib.gsort_segmented_bitonic
    assert g(A, 10, 0, None) == EINVAL
    assert g(A, 10, 1025, None) == EINVAL
    assert g(A, -1, 16, None) == EINVAL
    assert g(A, 1 << 31, 16, None) == ETOOBIG
    assert g(A, 0, 16, None) == 0
    assert g(A, 10, 1, None) == 0
    assert g(None, 10, 16, None) == EINVAL
    assert g(A + 2, 10, 16, None) == EALIGN
    h = lib.gsort_digit_histograms
    assert h(A, 10, 0, 0, 32, None, None) == EINVAL
    assert h(A, 10, 0, 0, 40, B, None) == EINVAL
    assert h(A, 10, 0, 0, 32, B + 2, None) == EALIGN
    assert h(A, 1000, 0, 0, 32, A + 64, None) == EINVAL                       # output inside keys
    assert h(A, 10, 0, 7, 7, B, None) == 0
    assert lib.gsort_check(None, None) == EINVAL
