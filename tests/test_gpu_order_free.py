"""GPU keys-only sorts over every bit of the key vs the CPU oracle, bit for
bit, on inputs built so that the order-free ranking of the digit pass meets
both of its cases in every pass: warps whose keys all agree in the bits
below the current digit (ranked by plain shared atomics) next to warps
whose keys differ there (ranked by the stable multisplit).  Sizes are above
the one-launch small-input limit, so the tiled digit pass runs."""
import numpy as np
import pytest
import torch

import oracle
from bitonic_networks_gb300 import gsort, synth

pytestmark = pytest.mark.gpu

N = (1 << 21) + 12_345   # ragged last tile


def to_dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    view = {np.dtype(np.uint32): np.int32, np.dtype(np.uint64): np.int64}.get(a.dtype)
    if view is not None:
        a = a.view(view)
    return torch.from_numpy(a.copy()).cuda()


def host_bytes(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy().view(np.uint8)


def keys32(shape: str, n: int, seed: int) -> np.ndarray:
    """Input recipes (no sorting arithmetic): how many keys share the low
    bits decides which warps of each pass may rank in any order."""
    u = synth.uniform_keys(n, seed)
    w = synth.uniform_keys(n, seed + 1)
    if shape == "low3":        # 3 low bytes only: pass 1 sees three long runs
        return (u & np.uint32(0xFFFFFF00)) | (w % np.uint32(3))
    if shape == "mid_groups":  # ~3000 distinct low halves: pass 2 groups of ~700 keys
        return (u & np.uint32(0xFFFF0000)) | ((w % np.uint32(3000)) * np.uint32(17))
    if shape == "top_only":    # only the top byte varies: passes 0-2 see equal digits
        return (u & np.uint32(0xFF000000)) | np.uint32(0x00ABCDEF)
    if shape == "skewed_low":  # low byte 0 for 98 % of keys: pass 2 sees one long run, then
        # runs of ~160 keys, so warps there straddle three or more runs (stable ranks after
        # 16-byte loads of a pass whose runs are long on average)
        lo = np.where(w % np.uint32(50) == 0, (w >> np.uint32(8)) % np.uint32(255) + np.uint32(1), 0)
        return (u & np.uint32(0xFFFFFF00)) | lo.astype(np.uint32)
    if shape == "uniform":
        return u
    if shape == "and3":
        return synth.and3_keys(n, seed)
    if shape == "distinct16":
        return synth.distinct16_keys(n, seed)
    if shape == "sorted":
        return np.sort(u)
    if shape == "reversed":
        return np.sort(u)[::-1].copy()
    raise ValueError(shape)


SHAPES = ["low3", "mid_groups", "top_only", "skewed_low", "uniform", "and3", "distinct16", "sorted",
          "reversed"]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("variant", [0, 1, 2])
def test_u32_keys_every_variant(shape, variant):
    k = keys32(shape, N, 7100 + SHAPES.index(shape))
    got, _ = gsort.sort_pairs(to_dev(k), None, 0, 32, variant=variant)
    exp = oracle.radix_sort_keys(k)
    assert np.array_equal(host_bytes(got), exp.view(np.uint8)), f"{shape} variant {variant}"


@pytest.mark.parametrize("kind", [1, 2])
@pytest.mark.parametrize("desc", [False, True])
@pytest.mark.parametrize("shape", ["low3", "mid_groups", "uniform"])
def test_mapped_32bit_keys(kind, desc, shape):
    k = keys32(shape, N, 7300 + kind)
    if kind == 1:
        # finite floats of both signs, ties, both zeros
        k = k & np.uint32(0xBFFFFFFF)
        k[::97] = 0x80000000
        k[1::89] = 0
    got, _ = gsort.sort(to_dev(k.view(np.float32) if kind == 1 else k.view(np.int32)), None,
                        descending=desc, kind=kind)
    exp, _ = oracle.default().radix_sort(k.view(np.float32) if kind == 1 else k.view(np.int32),
                                         None, kind, desc, 0, None)
    assert np.array_equal(host_bytes(got), np.ascontiguousarray(exp).view(np.uint8))


@pytest.mark.parametrize("kind", [3, 4, 5])
@pytest.mark.parametrize("desc", [False, True])
@pytest.mark.parametrize("shape", ["low_runs", "skewed_low", "uniform"])
def test_64bit_keys(kind, desc, shape):
    n = (1 << 20) + 777
    base = synth.keys64(n, 7500 + kind)
    if shape == "low_runs":
        # the low 40 bits take 5 values, so the first five passes see long runs
        base = (base & np.uint64(0xFFFFFF0000000000)) | (base % np.uint64(5))
    if shape == "skewed_low":
        # low byte 0 for 98 % of keys: warps of pass 2 straddle many short runs
        w = synth.keys64(n, 7600 + kind)
        lo = np.where(w % np.uint64(50) == 0, (w >> np.uint64(8)) % np.uint64(255) + np.uint64(1), 0)
        base = (base & np.uint64(0xFFFFFFFFFFFFFF00)) | lo.astype(np.uint64)
    if kind == 4:
        base = base & np.uint64(0xBFFFFFFFFFFFFFFF)   # finite doubles
    dt = {3: np.uint64, 4: np.float64, 5: np.int64}[kind]
    keys = base.view(dt)
    got, _ = gsort.sort(to_dev(keys), None, descending=desc, kind=kind)
    exp, _ = oracle.default().radix_sort(keys, None, kind, desc, 0, None)
    assert np.array_equal(host_bytes(got), np.ascontiguousarray(exp).view(np.uint8))


@pytest.mark.parametrize("shape", ["low3", "mid_groups", "uniform"])
def test_segmented_keys_long_segments(shape):
    lens = [9000, 70_000, 1, 0, 300_000, 16_385, 8192, 123_457]
    n = sum(lens)
    k = keys32(shape, n, 7700)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.uint32)
    got, _ = gsort.segmented_sort(to_dev(k), to_dev(off), kind=0)
    exp, _ = oracle.default().segmented_sort_general(k, off, None, 0, False)
    assert np.array_equal(host_bytes(got), np.ascontiguousarray(exp).view(np.uint8))


@pytest.mark.parametrize("variant", [0, 1, 2])
@pytest.mark.parametrize("shape", ["uniform", "low3", "distinct16"])
def test_u32_keys_in_place(shape, variant):
    k = keys32(shape, N, 7900 + SHAPES.index(shape))
    t = to_dev(k)
    got, _ = gsort.sort_pairs(t, None, 0, 32, keys_out=t, variant=variant)
    assert got.data_ptr() == t.data_ptr()
    assert np.array_equal(host_bytes(t), oracle.radix_sort_keys(k).view(np.uint8)), f"{shape} in place"
