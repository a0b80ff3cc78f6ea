"""GPU radix sort of every key kind (u32, f32, i32, u64, f64, i64), ascending
and descending, vs the CPU oracle bit for bit: keys only and pairs, bit
ranges, in place, several tiles with ragged tails, and the 64-bit digit
histograms."""
import numpy as np
import pytest
import torch

import oracle
from bitonic_networks_gb300 import gsort, synth

pytestmark = pytest.mark.gpu

KINDS = [0, 1, 2, 3, 4, 5]
NAMES = {0: "u32", 1: "f32", 2: "i32", 3: "u64", 4: "f64", 5: "i64"}
# 32-bit keys: 8192-key tiles; 64-bit keys: 4096-key tiles
SIZES = [1, 2, 33, 4095, 4096, 4097, 8193, 3 * 8192 + 5, 100_003]


def _orc():
    return oracle.default()


def to_dev(a: np.ndarray) -> torch.Tensor:
    """numpy keys -> CUDA tensor of the same bytes (unsigned types as signed views)."""
    a = np.ascontiguousarray(a)
    view = {np.dtype(np.uint32): np.int32, np.dtype(np.uint64): np.int64}.get(a.dtype)
    if view is not None:
        a = a.view(view)
    return torch.from_numpy(a.copy()).cuda()


def host_bytes(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy().view(np.uint8)


def assert_same_bytes(got: torch.Tensor, exp: np.ndarray, what: str):
    g = host_bytes(got)
    e = np.ascontiguousarray(exp).view(np.uint8)
    assert g.shape == e.shape, f"{what}: {g.shape} != {e.shape}"
    if not np.array_equal(g, e):
        w = np.ascontiguousarray(exp).dtype.itemsize
        bad = np.flatnonzero((g.reshape(-1, w) != e.reshape(-1, w)).any(axis=1))
        raise AssertionError(f"{what}: {bad.size} keys differ, first at {int(bad[0])}")


def run(keys, vals, kind, desc, begin=0, end=None, in_place=False):
    kt = to_dev(keys)
    vt = None if vals is None else to_dev(vals)
    if in_place:
        ko, vo = gsort.sort(kt, vt, descending=desc, kind=kind, begin_bit=begin, end_bit=end,
                            keys_out=kt, values_out=vt)
    else:
        ko, vo = gsort.sort(kt, vt, descending=desc, kind=kind, begin_bit=begin, end_bit=end)
    ek, ev = _orc().radix_sort(keys, vals, kind, desc, begin, end)
    tag = f"{NAMES[kind]} desc={desc} n={keys.size} bits={begin}..{end} in_place={in_place}"
    assert_same_bytes(ko, ek, "keys " + tag)
    if vals is not None:
        assert_same_bytes(vo, ev, "values " + tag)


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("desc", [False, True])
def test_pairs_every_kind(n, kind, desc):
    keys = synth.keys_of_kind(kind, n, 500 + 7 * kind + n)
    run(keys, synth.index_values(n), kind, desc)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("desc", [False, True])
def test_keys_only_every_kind(kind, desc):
    n = 70_001
    run(synth.keys_of_kind(kind, n, 900 + kind), None, kind, desc)


@pytest.mark.parametrize("kind", [3, 5])
@pytest.mark.parametrize("bits", [(0, 64), (13, 51), (0, 9), (60, 61), (32, 64), (0, 32), (7, 63),
                                  (20, 20)])
@pytest.mark.parametrize("desc", [False, True])
def test_64bit_bit_ranges(kind, bits, desc):
    n = 20_011
    keys = synth.keys_of_kind(kind, n, 1300 + bits[0] * 64 + bits[1])
    run(keys, synth.index_values(n), kind, desc, bits[0], bits[1])


@pytest.mark.parametrize("kind", [1, 2])
@pytest.mark.parametrize("bits", [(0, 32), (3, 29), (31, 32), (0, 8)])
@pytest.mark.parametrize("desc", [False, True])
def test_32bit_kinds_bit_ranges(kind, bits, desc):
    n = 20_011
    keys = synth.keys_of_kind(kind, n, 1700 + bits[0] * 64 + bits[1])
    run(keys, synth.index_values(n), kind, desc, bits[0], bits[1])


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("end", [None, 56])   # 56 bits: an odd pass count for 64-bit keys
def test_in_place(kind, end):
    n = 9_001
    if end is not None and kind not in (3, 5):
        end = 24                                # 3 passes for 32-bit keys
    keys = synth.keys_of_kind(kind, n, 2100 + kind)
    run(keys, synth.index_values(n), kind, True, 0, end, in_place=True)
    run(keys, None, kind, False, 0, end, in_place=True)


def test_specials_every_float_kind():
    for kind, dt in ((1, np.float32), (4, np.float64)):
        tiny = np.finfo(dt).tiny
        base = np.array([0.0, -0.0, np.inf, -np.inf, 1.0, -1.0, tiny / 2, -tiny / 2,
                         np.finfo(dt).max, -np.finfo(dt).max, 2.5, -2.5], dtype=dt)
        keys = np.tile(base, 700)
        for desc in (False, True):
            run(keys, np.arange(keys.size, dtype=np.uint32), kind, desc)


def test_signed_extremes():
    for kind, dt in ((2, np.int32), (5, np.int64)):
        info = np.iinfo(dt)
        base = np.array([info.min, info.max, 0, -1, 1, info.min + 1, info.max - 1], dtype=dt)
        keys = np.tile(base, 1500)
        for desc in (False, True):
            run(keys, np.arange(keys.size, dtype=np.uint32), kind, desc)


@pytest.mark.parametrize("kind", [3, 4, 5])
@pytest.mark.parametrize("bits", [(0, 64), (5, 61), (56, 64)])
def test_64bit_histograms(kind, bits):
    n = 123_457
    keys = synth.keys_of_kind(kind, n, 2500 + kind)
    got = gsort.digit_histograms(to_dev(keys), bits[0], bits[1], kind=kind)
    exp = _orc().digit_histograms_general(keys, kind, bits[0], bits[1])
    assert np.array_equal(got.cpu().numpy().view(np.uint32).reshape(exp.shape), exp)


def test_large_u64_pairs():
    n = 1 << 22
    keys = synth.keys_of_kind(3, n, 4242)
    run(keys, synth.index_values(n), 3, False)


def test_large_f64_descending():
    n = 3_000_017
    keys = synth.keys_of_kind(4, n, 4343)
    run(keys, synth.index_values(n), 4, True)
