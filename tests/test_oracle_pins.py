"""Pins of the CPU oracle against things other than itself.

Each pin_* function checks one part of the oracle against a value printed on
the reference pages, a closed form, an invariant, a library routine the
problem reduces to (Python's stable sorted(), numpy), or brute force over all
tiny inputs.  The mutation tests at the bottom plant plausible mistakes in
copies of oracle.c and check that some pin catches each of them.
"""
import itertools

import numpy as np
import pytest

import oracle
from conftest import load_golden
from bitonic_networks_gb300 import synth

U32 = np.uint32


def _f32(vals):
    return np.array([float(v) for v in vals], dtype=np.float32)


def _bits(a):
    return np.asarray(a, dtype=np.float32).view(U32)


# ------------------------------------------------------------ worked examples

def pin_radix_worked_example(orc):
    g = load_golden("radix_worked_example.txt")
    inp = np.array([int(v) for v in g["input"]], dtype=U32)
    exp = [int(v) for v in g["expected"]]
    assert orc.radix_sort_keys(inp).tolist() == exp


def pin_compaction_worked_example(orc):
    g = load_golden("compaction_worked_example.txt")
    out, m = orc.compact_positive(_f32(g["input"]))
    assert m == int(g["kept"][0])
    assert np.array_equal(_bits(out), _bits(_f32(g["expected"])))


def pin_bitonic_exercise(orc):
    g = load_golden("bitonic_exercise.txt")
    inp = np.array([int(v) for v in g["input"]], dtype=U32)
    exp = [int(v) for v in g["expected"]]
    assert orc.bitonic_network(inp).tolist() == exp
    assert orc.segmented_sort(inp.reshape(1, -1)).ravel().tolist() == exp


def test_radix_worked_example(orc):
    pin_radix_worked_example(orc)


def test_compaction_worked_example(orc):
    pin_compaction_worked_example(orc)


def test_bitonic_exercise(orc):
    pin_bitonic_exercise(orc)


# ---------------------------------------------------------------- float map

def _total_order_chunks(chunk=1 << 24):
    """All non-NaN float32 bit patterns in increasing IEEE totalOrder:
    -inf ... -min_subnormal, -0, +0, +min_subnormal ... +inf."""
    hi = 0xFF800000
    while hi >= 0x80000000:
        lo = max(0x80000000, hi - chunk + 1)
        yield np.arange(hi, lo - 1, -1, dtype=np.int64).astype(U32)
        hi = lo - 1
    lo = 0
    while lo <= 0x7F800000:
        hi = min(0x7F800000, lo + chunk - 1)
        yield np.arange(lo, hi + 1, dtype=np.int64).astype(U32)
        lo = hi + 1


def pin_transform_monotone_exhaustive(orc, chunk=1 << 24):
    """Strictly increasing along totalOrder over every non-NaN pattern, and
    inverted exactly by the inverse map."""
    prev = None
    count = 0
    for c in _total_order_chunks(chunk):
        u = orc.f32_bits_to_ordered_array(c)
        assert np.all(u[1:] > u[:-1])
        if prev is not None:
            assert u[0] > prev
        prev = u[-1]
        assert np.array_equal(orc.ordered_to_f32_bits_array(u), c)
        count += c.size
    assert count == (1 << 32) - 2 * ((1 << 23) - 1)


def pin_transform_matches_float_compare(orc, n=1 << 20):
    """For random non-NaN pairs, the mapped order equals the hardware's IEEE
    comparison, with -0 placed before +0."""
    a = synth.u32(11, n)
    b = synth.u32(12, n)
    fa, fb = a.view(np.float32), b.view(np.float32)
    ok = ~(np.isnan(fa) | np.isnan(fb))
    fa, fb, a, b = fa[ok], fb[ok], a[ok], b[ok]
    ua = orc.f32_bits_to_ordered_array(a)
    ub = orc.f32_bits_to_ordered_array(b)
    zero_rule = (fa == 0) & (fb == 0) & np.signbit(fa) & ~np.signbit(fb)
    assert np.array_equal(ua < ub, (fa < fb) | zero_rule)


def test_transform_exhaustive(orc):
    pin_transform_monotone_exhaustive(orc)


def test_transform_vs_float_compare(orc):
    pin_transform_matches_float_compare(orc)
    # NaN placement (documented, not promised): +NaN above +inf, -NaN below -inf
    pinf, ninf = 0x7F800000, 0xFF800000
    assert orc.f32_bits_to_ordered(0x7FC00000) > orc.f32_bits_to_ordered(pinf)
    assert orc.f32_bits_to_ordered(0xFFC00000) < orc.f32_bits_to_ordered(ninf)
    for nan in (0x7FC00000, 0xFFC00001, 0x7F800001):
        assert orc.ordered_to_f32_bits(orc.f32_bits_to_ordered(nan)) == nan


# -------------------------------------------------------- histograms, scans

def pin_histograms_constructed(orc):
    """Keys assembled from known digits: each pass's histogram must equal the
    bincount of the digits that were put there (bits outside the range are
    random and must be ignored)."""
    n = 20000
    rnd = [synth.u32(100 + i, n) for i in range(6)]
    d = [(r & U32(0xFF)) for r in rnd[:4]]
    keys = d[0] | (d[1] << U32(8)) | (d[2] << U32(16)) | (d[3] << U32(24))
    h = orc.digit_histograms(keys, 0, 0, 32)
    assert h.shape == (4, 256)
    for p in range(4):
        assert np.array_equal(h[p], np.bincount(d[p], minlength=256))
    # bits [3, 21): digits of width 8, 8, 2; junk below bit 3 and from bit 21
    junk_lo = rnd[4] & U32(7)
    junk_hi = rnd[5] >> U32(21)
    d2 = d[2] & U32(3)
    keys = junk_lo | (d[0] << U32(3)) | (d[1] << U32(11)) | (d2 << U32(19)) | (junk_hi << U32(21))
    h = orc.digit_histograms(keys, 0, 3, 21)
    assert h.shape == (3, 256)
    assert np.array_equal(h[0], np.bincount(d[0], minlength=256))
    assert np.array_equal(h[1], np.bincount(d[1], minlength=256))
    assert np.array_equal(h[2], np.bincount(d2, minlength=256))
    assert np.all(h.sum(axis=1) == n)


def pin_scan_bins(orc):
    h = np.stack([synth.u32(7 + p, 256) & U32(0xFFFF) for p in range(4)])
    base = orc.exclusive_scan_bins(h)
    assert np.array_equal(base, (np.cumsum(h, axis=1, dtype=np.uint64) - h).astype(U32))


def test_histograms(orc):
    pin_histograms_constructed(orc)
    f = synth.normal_f32_with_specials(5000, 3)
    # kind 1 equals kind 0 on the mapped keys; every pass sums to n
    hf = orc.digit_histograms(f, 1, 0, 32)
    assert np.array_equal(hf, orc.digit_histograms(orc.f32_bits_to_ordered_array(f), 0, 0, 32))
    assert np.all(hf.sum(axis=1) == f.size)


def test_scan_bins(orc):
    pin_scan_bins(orc)


# ------------------------------------------------------------------- sorting

def _masked(k, b, e):
    return (int(k) >> b) & ((1 << (e - b)) - 1)


def pin_sort_vs_python_sorted(orc):
    """Stable sort by the masked key == Python's stable sorted()."""
    for n, dup_mask in ((1, 0xFFFFFFFF), (97, 0x0F0F0F0F), (1000, 0xFFFFFFFF), (3001, 0x80000103)):
        k = synth.u32(n, n) & U32(dup_mask)
        v = synth.index_values(n)
        assert orc.radix_sort_keys(k).tolist() == sorted(k.tolist())
        for b, e in ((0, 32), (0, 8), (4, 20), (8, 8), (0, 1), (31, 32), (3, 29), (7, 31), (24, 32)):
            order = sorted(range(n), key=lambda i: _masked(k[i], b, e))
            ko, vo = orc.radix_sort_pairs(k, v, 0, b, e)
            assert ko.tolist() == k[order].tolist(), (n, b, e)
            assert vo.tolist() == order, (n, b, e)


def _float_sort_key(x):
    return (x, 0 if np.signbit(x) else 1)


def pin_float_sort_vs_python_sorted(orc):
    x = synth.normal_f32_with_specials(3000, 5)
    x[::97] = np.float32(1.5)       # repeated values
    x[5::101] = np.float32(-1.5)
    v = synth.index_values(x.size)
    order = sorted(range(x.size), key=lambda i: _float_sort_key(float(x[i])))
    ko, vo = orc.radix_sort_pairs(x, v, 1, 0, 32)
    assert np.array_equal(_bits(ko), _bits(x[order]))
    assert vo.tolist() == order


def pin_sort_vs_numpy(orc):
    n = 1 << 20
    k = synth.uniform_keys(n, 21)
    assert np.array_equal(orc.radix_sort_keys(k), np.sort(k))
    k2 = k & U32(0x00FF00FF)
    ko, vo = orc.radix_sort_pairs(k2, synth.index_values(n), 0, 0, 32)
    order = np.argsort(k2, kind="stable")
    assert np.array_equal(ko, k2[order])
    assert np.array_equal(vo, order.astype(U32))
    f = synth.normal_f32_with_specials(n, 22)
    ko, vo = orc.radix_sort_pairs(f, synth.index_values(n), 1, 0, 32)
    order = np.lexsort((np.where(np.signbit(f), 0, 1), f))
    assert np.array_equal(_bits(ko), _bits(f[order]))
    assert np.array_equal(vo, order.astype(U32))


def _check_sorted_perm_stable(inp, ko, vo, keyf):
    """vo (the index payload) is a permutation, each key travelled with its
    index, keys are ordered by keyf, and equal keys keep input order."""
    assert sorted(vo) == list(range(len(inp)))
    assert [inp[i] for i in vo] == list(ko)
    for a in range(len(ko) - 1):
        ka, kb = keyf(ko[a]), keyf(ko[a + 1])
        assert ka <= kb
        if ka == kb:
            assert vo[a] < vo[a + 1]


def pin_bruteforce_tiny(orc, max_len=5):
    """Every sequence of length <= max_len over small alphabets: the output
    is a permutation of the input pairs, ordered, and stable."""
    alpha = [0, 1, 2, 0xFFFFFFFF]
    for L in range(0, max_len + 1):
        for seq in itertools.product(alpha, repeat=L):
            k = np.array(seq, dtype=U32)
            ko, vo = orc.radix_sort_pairs(k, np.arange(L, dtype=U32), 0, 0, 32)
            _check_sorted_perm_stable(list(seq), ko.tolist(), vo.tolist(), lambda x: x)
    alpha = [0, 1, 2, 3, 0x80000001, 0xFFFFFFFE]
    for L in range(0, 5):
        for seq in itertools.product(alpha, repeat=L):
            k = np.array(seq, dtype=U32)
            ko, vo = orc.radix_sort_pairs(k, np.arange(L, dtype=U32), 0, 1, 2)
            _check_sorted_perm_stable(list(seq), ko.tolist(), vo.tolist(),
                                      lambda x: (x >> 1) & 1)
    falpha = [float("-inf"), -1.0, -0.0, 0.0, 1.0, float("inf")]
    for L in range(0, 5):
        for seq in itertools.product(falpha, repeat=L):
            f = np.array(seq, dtype=np.float32)
            ko, vo = orc.radix_sort_pairs(f, np.arange(L, dtype=U32), 1, 0, 32)
            assert np.array_equal(_bits(ko), _bits(f[vo]))
            assert sorted(vo.tolist()) == list(range(L))
            kk = [_float_sort_key(float(x)) for x in ko]
            for a in range(L - 1):
                assert kk[a] <= kk[a + 1]
                if kk[a] == kk[a + 1]:
                    assert vo[a] < vo[a + 1]


def pin_three_pass_cross_check(orc):
    """The 2-bit, three-pass restatement agrees with the 8-bit oracle."""
    for n in (1, 511, 512, 513, 5000, 81946):
        k = synth.u32(300 + n, n) & U32(0xF0FFFF0F)
        ids = synth.index_values(n)
        k2, i2 = orc.radix2_three_pass(k, ids)
        k8, i8 = orc.radix_sort_pairs(k, ids, 0, 0, 32)
        assert np.array_equal(k2, k8) and np.array_equal(i2, i8)


def test_sort_vs_python_sorted(orc):
    pin_sort_vs_python_sorted(orc)


def test_float_sort_vs_python_sorted(orc):
    pin_float_sort_vs_python_sorted(orc)


def test_sort_vs_numpy(orc):
    pin_sort_vs_numpy(orc)


def test_bruteforce_tiny(orc):
    pin_bruteforce_tiny(orc)


def test_three_pass_cross_check(orc):
    pin_three_pass_cross_check(orc)


def test_empty_and_bad_ranges(orc):
    e = np.zeros(0, dtype=U32)
    assert orc.radix_sort_keys(e).size == 0
    assert orc.num_passes(0, 32) == 4 and orc.num_passes(3, 29) == 4
    assert orc.num_passes(8, 8) == 0 and orc.num_passes(0, 1) == 1
    assert orc.num_passes(5, 4) == -1 and orc.num_passes(0, 33) == -1
    k = synth.u32(5, 100)
    ko, vo = orc.radix_sort_pairs(k, synth.index_values(100), 0, 9, 9)   # no bits: identity
    assert np.array_equal(ko, k) and np.array_equal(vo, synth.index_values(100))


# ---------------------------------------------------------------- compaction

def pin_compaction_vs_numpy(orc):
    x = synth.compaction_input(100003, 9)
    out, m = orc.compact_positive(x)
    keep = x > 0
    assert m == int(keep.sum())
    assert np.array_equal(_bits(out[:m]), _bits(x[keep]))
    assert np.all(_bits(out[m:]) == 0)


def pin_compaction_specials(orc):
    sub = np.array([1, 0x80000001], dtype=U32).view(np.float32)   # +/- smallest subnormal
    x = np.array([np.nan, -np.nan, 0.0, -0.0, sub[0], sub[1], np.inf, -np.inf, 1.0],
                 dtype=np.float32)
    out, m = orc.compact_positive(x)
    assert m == 3
    assert _bits(out[:3]).tolist() == [1, 0x7F800000, 0x3F800000]
    assert _bits(out[3:]).tolist() == [0] * 6
    out, m = orc.compact_positive(np.zeros(0, dtype=np.float32))
    assert m == 0 and out.size == 0


def test_compaction_vs_numpy(orc):
    pin_compaction_vs_numpy(orc)


def test_compaction_specials(orc):
    pin_compaction_specials(orc)


# ----------------------------------------------------------------- segments

def pin_segmented_vs_numpy(orc):
    for L in (1, 2, 3, 31, 32, 33, 100, 1000, 1024):
        a = synth.segments(17, L, 40 + L)
        if L > 4:
            a[3] = a[3] & U32(0xF)          # duplicates
            a[5] = np.sort(a[5])            # already sorted
            a[6] = np.sort(a[6])[::-1]      # reversed
        assert np.array_equal(orc.segmented_sort(a), np.sort(a, axis=1))


def pin_bitonic_zero_one(orc):
    """0-1 principle: a comparator network sorts every input iff it sorts
    every 0/1 input.  All 2^16 binary inputs of length 16."""
    for m in range(1 << 16):
        bits = np.array([(m >> i) & 1 for i in range(16)], dtype=U32)
        assert orc.bitonic_network(bits).tolist() == sorted(bits.tolist())


def pin_bitonic_padding(orc):
    """Padding a length-L input with 0xFFFFFFFF up to a power of two, then
    keeping the first L outputs, sorts it (any L)."""
    for L in (1, 2, 3, 5, 17, 31, 33, 63, 64):
        Lp = 1 << max(0, (L - 1).bit_length())
        a = synth.u32(500 + L, L)
        a[::3] = U32(0xFFFFFFFF)
        padded = np.concatenate([a, np.full(Lp - L, 0xFFFFFFFF, dtype=U32)])
        assert orc.bitonic_network(padded)[:L].tolist() == sorted(a.tolist())


def test_segmented_vs_numpy(orc):
    pin_segmented_vs_numpy(orc)


def test_bitonic_zero_one(orc):
    pin_bitonic_zero_one(orc)


def test_bitonic_padding(orc):
    pin_bitonic_padding(orc)


# ------------------------------------------------------------ planted mistakes

# --------------------------------------------- f1: every key kind, both directions

import math

KINDS = {"u32": 0, "f32": 1, "i32": 2, "u64": 3, "f64": 4, "i64": 5}
KIND_DTYPE = {0: np.uint32, 1: np.float32, 2: np.int32, 3: np.uint64, 4: np.float64, 5: np.int64}


def _py_key(kind):
    """Python sort key of one numpy element: integer value, or (value, sign) for
    floats so that -0.0 sorts before +0.0 (IEEE totalOrder on non-NaN values)."""
    if kind in (1, 4):
        return lambda v: (float(v), math.copysign(1.0, float(v)))
    return lambda v: int(v)


def _edge_keys(kind, n, seed):
    rng = np.random.default_rng(seed)
    dt = np.dtype(KIND_DTYPE[kind])
    if kind in (1, 4):
        vals = rng.standard_normal(n) * 10.0 ** rng.integers(-5, 6, n)
        specials = [0.0, -0.0, np.inf, -np.inf, 1.0, -1.0, np.finfo(dt).tiny / 4,
                    -np.finfo(dt).tiny / 4, np.finfo(dt).max, -np.finfo(dt).max]
        vals[: len(specials)] = specials
        vals = vals.astype(dt)
        vals[rng.integers(0, n, n // 4)] = vals[rng.integers(0, n, n // 4)]   # duplicates
    else:
        info = np.iinfo(dt)
        vals = rng.integers(info.min, info.max, n, dtype=dt, endpoint=True)
        specials = [info.min, info.max, 0, 1]
        if info.min < 0:
            specials += [-1]
        vals[: len(specials)] = np.array(specials, dtype=dt)
        vals[rng.integers(0, n, n // 4)] = vals[rng.integers(0, n, n // 4)]
    rng.shuffle(vals)
    return vals


def _python_stable(keys, kind, descending):
    key = _py_key(kind)
    order = sorted(range(len(keys)), key=lambda i: key(keys[i]), reverse=descending)
    return np.array(order, dtype=np.uint32)


def pin_general_vs_python_sorted(orc):
    # Python's sorted() is stable, also with reverse=True (equal keys keep
    # their input order), which is the order the descending sort promises.
    for kind in range(6):
        for desc in (False, True):
            keys = _edge_keys(kind, 3000, 100 + kind)
            idx = np.arange(keys.size, dtype=np.uint32)
            ko, vo = orc.radix_sort(keys, idx, kind, desc)
            exp = _python_stable(keys, kind, desc)
            assert np.array_equal(vo, exp), (kind, desc)
            assert np.array_equal(ko.view(np.uint8), keys[exp].view(np.uint8)), (kind, desc)


def pin_general_bit_range(orc):
    rng = np.random.default_rng(7)
    keys = rng.integers(0, 2**64 - 1, 2000, dtype=np.uint64, endpoint=True)
    keys[1::3] = keys[0::3][: keys[1::3].size]        # equal keys
    idx = np.arange(keys.size, dtype=np.uint32)
    for b, e in [(0, 64), (13, 51), (40, 64), (0, 9), (60, 61)]:
        for desc in (False, True):
            ko, vo = orc.radix_sort(keys, idx, 3, desc, b, e)
            mask = (1 << (e - b)) - 1
            exp = sorted(range(keys.size), key=lambda i: (int(keys[i]) >> b) & mask, reverse=desc)
            assert vo.tolist() == exp, (b, e, desc)
            assert np.array_equal(ko, keys[exp])


def pin_general_bruteforce(orc, max_len=4):
    alphabets = {
        2: [-2**31, -1, 0, 1, 2**31 - 1],
        3: [0, 1, 2**63, 2**64 - 1],
        4: [-np.inf, -1.0, -0.0, 0.0, 1.0, np.inf],
        5: [-2**63, -1, 0, 2**63 - 1],
    }
    for kind, alpha in alphabets.items():
        dt = KIND_DTYPE[kind]
        key = _py_key(kind)
        for length in range(1, max_len + 1):
            for combo in itertools.product(range(len(alpha)), repeat=length):
                keys = np.array([alpha[c] for c in combo], dtype=dt)
                idx = np.arange(length, dtype=np.uint32)
                for desc in (False, True):
                    ko, vo = orc.radix_sort(keys, idx, kind, desc)
                    assert sorted(vo.tolist()) == list(range(length))        # a permutation
                    assert np.array_equal(ko.view(np.uint8), keys[vo].view(np.uint8))
                    ks = [key(v) for v in ko]
                    for i in range(length - 1):
                        if desc:
                            assert ks[i] >= ks[i + 1]
                        else:
                            assert ks[i] <= ks[i + 1]
                        if ks[i] == ks[i + 1]:
                            assert vo[i] < vo[i + 1]                        # stable


def pin_general_maps(orc):
    rng = np.random.default_rng(11)
    for kind in range(6):
        w = 8 * np.dtype(KIND_DTYPE[kind]).itemsize
        bits = [int(x) for x in rng.integers(0, 2**w - 1, 400, dtype=np.uint64, endpoint=True)]
        for desc in (False, True):
            for b in bits:                                   # the map is a bijection on bit patterns
                u = orc.key_to_ordered(b, kind, desc)
                assert 0 <= u < 2**w
                assert orc.ordered_to_key(u, kind, desc) == b
        # monotone along values sorted by Python
        keys = _edge_keys(kind, 500, 200 + kind)
        if kind in (1, 4):
            keys = keys[~np.isnan(keys)]
        key = _py_key(kind)
        ordered = sorted(keys.tolist(), key=key)
        as_bits = np.array(ordered, dtype=KIND_DTYPE[kind]).view(np.uint32 if w == 32 else np.uint64)
        us = [orc.key_to_ordered(int(b), kind) for b in as_bits]
        ud = [orc.key_to_ordered(int(b), kind, True) for b in as_bits]
        for i in range(len(us) - 1):
            same = key(ordered[i]) == key(ordered[i + 1])
            assert (us[i] == us[i + 1]) if same else (us[i] < us[i + 1])
            assert (ud[i] == ud[i + 1]) if same else (ud[i] > ud[i + 1])


def pin_general_histograms(orc):
    keys = _edge_keys(5, 3000, 5)
    h = orc.digit_histograms_general(keys, 5)
    assert h.shape == (8, 256) and (h.sum(axis=1) == keys.size).all()
    u = np.array([orc.key_to_ordered(int(b), 5) for b in keys.view(np.uint64)], dtype=np.uint64)
    for p in range(8):
        assert np.array_equal(h[p], np.bincount(((u >> np.uint64(8 * p)) & np.uint64(255)).astype(np.int64),
                                                minlength=256))


def test_general_vs_python_sorted(orc):
    pin_general_vs_python_sorted(orc)


def test_general_bit_range(orc):
    pin_general_bit_range(orc)


def test_general_bruteforce(orc):
    pin_general_bruteforce(orc)


def test_general_maps(orc):
    pin_general_maps(orc)


def test_general_histograms(orc):
    pin_general_histograms(orc)


def test_general_matches_32bit_oracle(orc):
    # the two oracle entry points agree on the kinds they share
    keys = synth.uniform_keys(5000, 3)
    idx = np.arange(5000, dtype=np.uint32)
    a = orc.radix_sort_pairs(keys, idx, 0, 3, 29)
    b = orc.radix_sort(keys, idx, 0, False, 3, 29)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ------------------------------------------------ f2: variable-length segments

def _segment_lengths(rng, n_target):
    lens = []
    total = 0
    while total < n_target:
        r = rng.random()
        L = int(rng.integers(0, 3)) if r < 0.3 else int(rng.integers(3, 40)) if r < 0.8 \
            else int(rng.integers(40, 3000))
        lens.append(L)
        total += L
    return np.array(lens, dtype=np.int64)


def pin_segmented_general(orc):
    rng = np.random.default_rng(31)
    for kind in (0, 1, 2):
        for desc in (False, True):
            lens = _segment_lengths(rng, 6000)
            off = np.concatenate([[0], np.cumsum(lens)]).astype(np.uint32)
            n = int(off[-1])
            keys = _edge_keys(kind, n, 400 + kind) if n else np.zeros(0, KIND_DTYPE[kind])
            idx = np.arange(n, dtype=np.uint32)
            ko, vo = orc.segmented_sort_general(keys, off, idx, kind, desc)
            key = _py_key(kind)
            for s in range(lens.size):
                a, b = int(off[s]), int(off[s + 1])
                exp = sorted(range(a, b), key=lambda i: key(keys[i]), reverse=desc)
                assert vo[a:b].tolist() == exp, (kind, desc, s)
            assert np.array_equal(ko.view(np.uint8), keys[vo].view(np.uint8))


def test_segmented_general(orc):
    pin_segmented_general(orc)


def test_segmented_general_rejects_bad_offsets(orc):
    keys = np.arange(10, dtype=np.uint32)[::-1].copy()
    for off in ([1, 10], [0, 9], [0, 6, 4, 10], [0, 11]):
        with pytest.raises(RuntimeError):
            orc.segmented_sort_general(keys, np.array(off), None, 0)
    ko, _ = orc.segmented_sort_general(keys, np.array([0, 0, 10, 10]), None, 0)
    assert ko.tolist() == list(range(10))


# ------------------------------------------------------ f3: 2-way split

def _total_order_less(x, p):
    """numpy IEEE totalOrder 'x < p' for float32 arrays without NaN."""
    return (x < p) | ((x == p) & np.signbit(x) & ~np.signbit(np.float32(p)))


def pin_partition_vs_numpy(orc):
    rng = np.random.default_rng(21)
    n = 5000
    u = synth.uniform_keys(n, 21)
    idx = np.arange(n, dtype=np.uint32)
    cases = []
    flags = (rng.random(n) < 0.3).astype(np.uint8)
    cases.append((u, dict(pred=0, flags=flags), flags.astype(bool)))
    for b in (0, 7, 31):
        cases.append((u, dict(pred=1, param=b), ((u >> np.uint32(b)) & np.uint32(1)) == 1))
        cases.append((u, dict(pred=2, param=b), ((u >> np.uint32(b)) & np.uint32(1)) == 0))
    piv = int(u[17])
    cases.append((u, dict(pred=3, kind=0, param=piv), u < np.uint32(piv)))
    s32 = u.view(np.int32)
    cases.append((s32, dict(pred=3, kind=2, param=int(np.uint32(s32[5].view(np.uint32)))), s32 < s32[5]))
    f = synth.normal_f32_with_specials(n, 22)
    for pv in (0.0, -0.0, 0.5, -np.inf):
        pbits = int(np.float32(pv).view(np.uint32))
        cases.append((f, dict(pred=3, kind=1, param=pbits), _total_order_less(f, np.float32(pv))))
    cases.append((f, dict(pred=4), f > 0))
    for x, kw, mask in cases:
        out, vo, m = orc.partition(x, idx, **kw)
        assert m == int(mask.sum()), kw
        exp = np.concatenate([idx[mask], idx[~mask]])
        assert np.array_equal(vo, exp), kw
        assert np.array_equal(np.asarray(out).view(np.uint32), np.asarray(x).view(np.uint32)[exp]), kw


def pin_partition_worked_example(orc):
    g = load_golden("compaction_worked_example.txt")
    x = _f32(g["input"])
    out, _, m = orc.partition(x, None, pred=4)
    kept = int(g["kept"][0])
    assert m == kept
    assert np.array_equal(_bits(out[:m]), _bits(_f32(g["expected"])[:kept]))


def pin_split_sort(orc):
    rng = np.random.default_rng(23)
    keys = synth.uniform_keys(3000, 23)
    keys[::5] = keys[1::5][: keys[::5].size]
    idx = np.arange(keys.size, dtype=np.uint32)
    for b, e in [(0, 32), (3, 17), (31, 32), (0, 1), (8, 24)]:
        ko, vo = orc.split_sort(keys, idx, b, e)
        mask = (1 << (e - b)) - 1
        exp = sorted(range(keys.size), key=lambda i: (int(keys[i]) >> b) & mask)
        assert vo.tolist() == exp, (b, e)
        assert np.array_equal(ko, keys[exp])
        k8, v8 = orc.radix_sort_pairs(keys, idx, 0, b, e)     # the 8-bit oracle agrees
        assert np.array_equal(ko, k8) and np.array_equal(vo, v8)


def test_partition_vs_numpy(orc):
    pin_partition_vs_numpy(orc)


def test_partition_worked_example(orc):
    pin_partition_worked_example(orc)


def test_split_sort(orc):
    pin_split_sort(orc)


MUTANTS = {
    # a reversed scatter: each pass is no longer stable
    "unstable_scatter": ("for (int64_t i = 0; i < n; ++i) {\n            uint32_t d = digit_of",
                         "for (int64_t i = n - 1; i >= 0; --i) {\n            uint32_t d = digit_of"),
    # digits taken 7 bits apart instead of 8
    "digit_stride": ("digit_of(uint32_t k, int begin_bit, int end_bit, int p)\n{\n    int lo = begin_bit + 8 * p;",
                     "digit_of(uint32_t k, int begin_bit, int end_bit, int p)\n{\n    int lo = begin_bit + 7 * p;"),
    # the integer sign trick applied to floats (negatives not reversed)
    "float_map_sign_only": ("        return ~bits;\n    return bits | 0x80000000u;",
                            "        return bits ^ 0x80000000u;\n    return bits | 0x80000000u;"),
    # >= instead of > in the compaction predicate
    "compaction_ge": ("if (x > 0.0f) {", "if (x >= 0.0f) {"),
    # bitonic direction from the wrong bit
    "bitonic_direction": ("int ascending = (i & k) == 0;", "int ascending = (i & j) == 0;"),
    # last digit not narrowed to the remaining bits
    "last_digit_width": ("int lo = begin_bit + 8 * p;\n    int width = end_bit - lo;\n    if (width > 8)\n        width = 8;\n    return (uint32_t)(((uint64_t)k",
                         "int lo = begin_bit + 8 * p;\n    int width = end_bit - lo;\n    width = 8;\n    return (uint32_t)(((uint64_t)k"),
    # f1: reversed scatter in the general sort (not stable)
    "general_unstable": ("for (int64_t i = 0; i < n; ++i) {\n            uint32_t slot = next[digit_of64",
                         "for (int64_t i = n - 1; i >= 0; --i) {\n            uint32_t slot = next[digit_of64"),
    # f1: 64-bit digits 7 bits apart
    "digit64_stride": ("digit_of64(uint64_t k, int begin_bit, int end_bit, int p)\n{\n    int lo = begin_bit + 8 * p;",
                       "digit_of64(uint64_t k, int begin_bit, int end_bit, int p)\n{\n    int lo = begin_bit + 7 * p;"),
    # f1: signed 64-bit offset by 2^62 instead of 2^63
    "i64_offset": ("case 5: u = bits + 0x8000000000000000ull; break;",
                   "case 5: u = bits + 0x4000000000000000ull; break;"),
    # f1: negative doubles only get the sign bit flipped
    "f64_sign_only": ("        if (bits >> 63)\n            u = ~bits;",
                      "        if (bits >> 63)\n            u = bits ^ 0x8000000000000000ull;"),
    # f1: descending complement at 32 bits for every width
    # f2: the last segment is left unsorted
    "segmented_last": ("for (int64_t s = 0; s < num_segments; ++s) {\n        uint32_t a = offsets[s];",
                       "for (int64_t s = 0; s + 1 < num_segments; ++s) {\n        uint32_t a = offsets[s];"),
    # f3: the false side of a split in reverse order
    "partition_false_reversed": ("    int64_t k = m;\n    for (int64_t i = 0; i < n; ++i) {",
                                 "    int64_t k = m;\n    for (int64_t i = n - 1; i >= 0; --i) {"),
    # f3: bit test of the wrong bit
    "partition_bit": ("case 1: return ((x >> param) & 1u) == 1u;", "case 1: return ((x >> (param + 1)) & 1u) == 1u;"),
    "descending_width": ("    }\n    if (descending)\n        u = (w == 64 ? 0xFFFFFFFFFFFFFFFFull : 0xFFFFFFFFull) - u;",
                         "    }\n    if (descending)\n        u = 0xFFFFFFFFull - u;"),
}

PINS = [pin_radix_worked_example, pin_compaction_worked_example, pin_bitonic_exercise,
        pin_transform_matches_float_compare, pin_histograms_constructed,
        pin_sort_vs_python_sorted, pin_float_sort_vs_python_sorted,
        pin_compaction_specials, pin_bitonic_zero_one, pin_segmented_vs_numpy,
        pin_general_vs_python_sorted, pin_general_bit_range, pin_general_maps,
        pin_segmented_general, pin_partition_vs_numpy, pin_partition_worked_example,
        pin_split_sort]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found"
    path = tmp_path / "oracle_mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.Oracle(oracle.compile_source(str(path), str(tmp_path / "libmutant.so")))
    failed = []
    for pin in PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
