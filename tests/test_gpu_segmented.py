"""GPU variable-length segmented sort vs the CPU oracle, bit for bit: segment
length mixes on both sides of the 1024-key warp limit and of the 8192-key
tile, every 32-bit key kind, both directions, keys only and pairs
(stability), in place, empty and one-key segments, and offsets that break
the rules (reported as GSORT_EINVAL by gsort_check, nothing else touched)."""
import numpy as np
import pytest
import torch

import oracle
from bitonic_networks_gb300 import gsort, synth

pytestmark = pytest.mark.gpu

EINVAL = -1


def to_dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a.copy()).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy().view(np.uint32)


def offsets_of(lens) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(lens, dtype=np.int64))]).astype(np.uint32)


def check(keys, lens, kind=0, desc=False, values=True, in_place=False):
    off = offsets_of(lens)
    n = int(off[-1])
    assert keys.size == n
    vals = synth.index_values(n) if values else None
    kt = to_dev(keys)
    vt = to_dev(vals) if values else None
    ot = to_dev(off)
    if in_place:
        ko, vo = gsort.segmented_sort(kt, ot, vt, descending=desc, kind=kind, keys_out=kt,
                                      values_out=vt)
    else:
        ko, vo = gsort.segmented_sort(kt, ot, vt, descending=desc, kind=kind)
    ek, ev = oracle.default().segmented_sort_general(keys, off, vals, kind, desc)
    tag = f"kind={kind} desc={desc} values={values} in_place={in_place} segments={len(lens)} n={n}"
    got = host(ko)
    exp = np.ascontiguousarray(ek).view(np.uint32)
    if not np.array_equal(got, exp):
        bad = np.flatnonzero(got != exp)
        seg = np.searchsorted(off, bad[0], side="right") - 1
        raise AssertionError(f"keys {tag}: {bad.size} differ, first at {bad[0]} "
                             f"(segment {seg}, length {lens[seg]})")
    if values:
        assert np.array_equal(host(vo), ev), f"values {tag}"


def mixed_lengths(seed, n_target, hi=3000):
    rng = np.random.default_rng(seed)
    lens, total = [], 0
    while total < n_target:
        r = rng.random()
        L = int(rng.integers(0, 3)) if r < 0.2 else int(rng.integers(3, 40)) if r < 0.5 \
            else int(rng.integers(40, 1100)) if r < 0.9 else int(rng.integers(1100, hi))
        lens.append(L)
        total += L
    return lens


def keys_for(kind, n, seed):
    return synth.keys_of_kind(kind, n, seed) if n else np.zeros(0, dtype=np.uint32)


@pytest.mark.parametrize("kind", [0, 1, 2])
@pytest.mark.parametrize("desc", [False, True])
@pytest.mark.parametrize("values", [False, True])
def test_mixed_lengths(kind, desc, values):
    lens = mixed_lengths(10 + kind, 60_000)
    check(keys_for(kind, sum(lens), 20 + kind), lens, kind, desc, values)


# every class boundary: warp network sizes (32 .. 1024), the 1024/1025 switch
# to the tiled radix path, one and several tiles with ragged ends
EDGE_LENGTHS = [0, 1, 2, 3, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257, 511, 512, 513,
                1023, 1024, 1025, 1026, 2047, 4096, 8191, 8192, 8193, 16384, 16385, 30001]


@pytest.mark.parametrize("values", [False, True])
def test_edge_lengths(values):
    lens = EDGE_LENGTHS + EDGE_LENGTHS[::-1]
    check(keys_for(0, sum(lens), 77), lens, 0, False, values)


@pytest.mark.parametrize("length", [2, 17, 32, 100, 1000, 1024, 1025, 5000, 8192, 70000])
def test_equal_lengths(length):
    count = max(1, 200_000 // length)
    lens = [length] * count
    check(keys_for(0, sum(lens), 1000 + length), lens, 0, False, True)


def test_heavy_duplicates_are_stable():
    lens = [5, 900, 1024, 1025, 3000, 9000, 40, 1]
    n = sum(lens)
    keys = (synth.uniform_keys(n, 5) % np.uint32(7)).astype(np.uint32)   # 7 distinct keys
    for desc in (False, True):
        check(keys, lens, 0, desc, True)
        check(keys, lens, 0, desc, False)   # keys only: one digit value per bin cursor


def test_single_segment_large():
    n = 1_000_003
    check(keys_for(0, n, 8), [n], 0, False, True)
    check(keys_for(2, n, 9), [n], 2, True, False)


def test_many_tiny_segments():
    rng = np.random.default_rng(4)
    lens = rng.integers(0, 6, 100_000).tolist()
    check(keys_for(0, sum(lens), 10), lens, 0, False, True)


def test_in_place():
    lens = mixed_lengths(5, 50_000)
    n = sum(lens)
    for kind in (0, 1):
        check(keys_for(kind, n, 30 + kind), lens, kind, True, True, in_place=True)
        check(keys_for(kind, n, 40 + kind), lens, kind, False, False, in_place=True)


def test_empty_input_and_empty_segments():
    check(np.zeros(0, dtype=np.uint32), [0, 0, 0], 0, False, True)
    check(keys_for(0, 10, 3), [0, 0, 10, 0], 0, False, True)


@pytest.mark.parametrize("bad", ["first", "last", "decreasing", "beyond"])
def test_bad_offsets_reported(bad):
    n = 50_000
    keys = to_dev(synth.uniform_keys(n, 6))
    off = offsets_of([100, 20_000, 2000, n - 22_100])
    if bad == "first":
        off[0] = 5
    elif bad == "last":
        off[-1] = n - 1
    elif bad == "decreasing":
        off[2] = 50
    else:
        off[2] = n + 1000
    with pytest.raises(gsort.GsortError) as e:
        gsort.segmented_sort(keys, to_dev(off), None, kind=0)
    assert e.value.code == EINVAL
    # the context is healthy afterwards
    ok_off = offsets_of([n])
    ko, _ = gsort.segmented_sort(keys, to_dev(ok_off), None, kind=0)
    assert np.array_equal(host(ko), np.sort(host(keys)))


def test_keys_not_16_byte_aligned():
    """Keys that start 4 or 8 bytes past a 16-byte boundary (the histogram
    takes its 16-byte loads only from aligned keys)."""
    lens = [70_001, 3, 1025, 9000, 500, 20_000]
    off = to_dev(offsets_of(lens))
    n = sum(lens)
    for shift in (1, 2):
        keys = keys_for(0, n, 60 + shift)
        buf = torch.zeros(n + 4, dtype=torch.int32, device="cuda")
        kt = buf[shift:shift + n]
        kt.copy_(to_dev(keys))
        assert kt.data_ptr() % 16 == 4 * shift
        ko, _ = gsort.segmented_sort(kt, off, kind=0)
        ek, _ = oracle.default().segmented_sort_general(keys, offsets_of(lens), None, 0, False)
        assert np.array_equal(host(ko), np.ascontiguousarray(ek).view(np.uint32)), f"shift {shift}"


def test_concurrent_callers_on_their_own_streams():
    """Two host threads sort at once, each on a stream of its own (the small
    segments' networks of every call run on streams the library shares
    between calls)."""
    import threading

    lens = mixed_lengths(31, 120_000, hi=20_000)
    off_h = offsets_of(lens)
    n = sum(lens)
    keys = [keys_for(0, n, 90 + t) for t in range(2)]
    expect = [np.ascontiguousarray(oracle.default().segmented_sort_general(k, off_h, None, 0, False)[0])
              .view(np.uint32) for k in keys]
    errors = []

    def worker(t):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                kt = to_dev(keys[t])
                ot = to_dev(off_h)
                for _ in range(20):
                    ko, _ = gsort.segmented_sort(kt, ot, kind=0)
                    got = ko.cpu().numpy().view(np.uint32)
                    if not np.array_equal(got, expect[t]):
                        errors.append(f"thread {t}: result differs")
                        return
        except Exception as e:   # reported below
            errors.append(f"thread {t}: {e!r}")

    th = [threading.Thread(target=worker, args=(t,)) for t in range(2)]
    for x in th:
        x.start()
    for x in th:
        x.join()
    assert not errors, errors

