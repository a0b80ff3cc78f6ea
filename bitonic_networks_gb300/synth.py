"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module holds input generators only -- none of the sorting arithmetic.
It is the one piece of code that both the CPU oracle's callers and the GPU
library's callers use, so that both sides see the same bytes.

Every stream is counter-based: word i of stream `seed` is splitmix64(seed, i)
(Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
2014; the finaliser constants are the published ones).  Results are therefore
identical on every machine and independent of numpy's own generators.

The workloads mirror the shapes of the reference pages' problems: uniform
32-bit keys, key/index pairs, low-entropy keys, float keys with signed zeros
and infinities, batched 1024-key segments, and the three-way mix of negative,
zero and positive floats of the stream-compaction example.
"""
from __future__ import annotations

import numpy as np

_M64 = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15
SEED_BASE = 0x9E3779B9
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def stream_seed(seed: int, k: int) -> int:
    """Seed of the k-th independent sub-stream of `seed`."""
    z = np.array([(seed + (k + 1) * 0xD1B54A32D192ED03) & _M64], dtype=np.uint64)
    return int(_mix(z)[0])


def splitmix64(seed: int, n: int, start: int = 0) -> np.ndarray:
    """Words start .. start+n-1 of the counter-based stream `seed` (uint64)."""
    out = np.empty(n, dtype=np.uint64)
    s = np.uint64(seed & _M64)
    g = np.uint64(_GAMMA)
    with np.errstate(over="ignore"):
        for lo in range(0, n, _CHUNK):
            hi = min(n, lo + _CHUNK)
            idx = np.arange(start + lo + 1, start + hi + 1, dtype=np.uint64)
            out[lo:hi] = _mix(s + idx * g)
    return out


def u32(seed: int, n: int) -> np.ndarray:
    """Uniform 32-bit words: the low half of each splitmix64 word."""
    out = np.empty(n, dtype=np.uint32)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        out[lo:hi] = (splitmix64(seed, hi - lo, lo) & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    return out


def u01(seed: int, n: int, start: int = 0) -> np.ndarray:
    """Uniform doubles in (0, 1) with 24-bit resolution (never 0, never a
    subnormal, exactly representable in float32)."""
    out = np.empty(n, dtype=np.float64)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        w = splitmix64(seed, hi - lo, start + lo)
        out[lo:hi] = ((w >> np.uint64(40)) | np.uint64(1)).astype(np.float64) * (2.0 ** -24)
    return out


# ----------------------------------------------------------------- workloads

def uniform_keys(n: int, seed: int = SEED_BASE) -> np.ndarray:
    """n uniform uint32 keys over the full 32-bit range."""
    return u32(seed, n)


def and3_keys(n: int, seed: int = SEED_BASE) -> np.ndarray:
    """Low-entropy keys: AND of three independent uniform words
    (each bit is 1 with probability 1/8)."""
    a = u32(stream_seed(seed, 0), n)
    a &= u32(stream_seed(seed, 1), n)
    a &= u32(stream_seed(seed, 2), n)
    return a


def distinct16_keys(n: int, seed: int = SEED_BASE) -> np.ndarray:
    """Heavy duplicates: each key is one of 16 distinct values, chosen
    uniformly (value table drawn from one stream, choices from another)."""
    table = []
    j = 0
    tseed = stream_seed(seed, 0)
    while len(table) < 16:
        v = int(u32(tseed, j + 1)[j])
        if v not in table:
            table.append(v)
        j += 1
    table = np.array(table, dtype=np.uint32)
    pick = np.empty(n, dtype=np.uint32)
    cseed = stream_seed(seed, 1)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        pick[lo:hi] = table[(splitmix64(cseed, hi - lo, lo) & np.uint64(15)).astype(np.int64)]
    return pick


def index_values(n: int) -> np.ndarray:
    """Payload = original position 0..n-1 (makes stability visible)."""
    return np.arange(n, dtype=np.uint32)


def normal_f32_with_specials(n: int, seed: int = SEED_BASE) -> np.ndarray:
    """float32 ~ Normal(0, 1) (Box-Muller in float64, rounded once), with
    exactly n//100 each of +0.0, -0.0, +inf and -inf at positions taken from
    a seeded random permutation (no NaN)."""
    u1 = u01(stream_seed(seed, 0), n)
    u2 = u01(stream_seed(seed, 1), n)
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    del u1, u2
    x = z.astype(np.float32)
    del z
    q = n // 100
    if q > 0:
        r = splitmix64(stream_seed(seed, 2), n)
        chosen = np.argpartition(r, 4 * q - 1)[: 4 * q]
        chosen = chosen[np.argsort(r[chosen], kind="stable")]
        x[chosen[0 * q:1 * q]] = np.float32(0.0)
        x[chosen[1 * q:2 * q]] = np.float32(-0.0)
        x[chosen[2 * q:3 * q]] = np.float32(np.inf)
        x[chosen[3 * q:4 * q]] = np.float32(-np.inf)
    return x


def normal_with_specials(n: int, dtype=np.float64, seed: int = SEED_BASE) -> np.ndarray:
    """normal_f32_with_specials at another float width (float64: no rounding)."""
    u1 = u01(stream_seed(seed, 0), n)
    u2 = u01(stream_seed(seed, 1), n)
    x = (np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)).astype(dtype)
    q = n // 100
    if q > 0:
        r = splitmix64(stream_seed(seed, 2), n)
        chosen = np.argpartition(r, 4 * q - 1)[: 4 * q]
        chosen = chosen[np.argsort(r[chosen], kind="stable")]
        for j, v in enumerate((0.0, -0.0, np.inf, -np.inf)):
            x[chosen[j * q:(j + 1) * q]] = dtype(v)
    return x


def keys64(n: int, seed: int = SEED_BASE) -> np.ndarray:
    """uint64 keys uniform over [0, 2^64): one splitmix64 word per key."""
    return splitmix64(stream_seed(seed, 3), n)


def keys_of_kind(kind: int, n: int, seed: int = SEED_BASE) -> np.ndarray:
    """Seeded keys of a key kind (0 u32, 1 f32, 2 i32, 3 u64, 4 f64, 5 i64),
    uniform over the bit patterns for integers, normal with +-0 and +-inf
    for floats, with a share of repeated keys so that stability matters."""
    if kind in (0, 2):
        k = uniform_keys(n, seed).view(np.int32 if kind == 2 else np.uint32)
    elif kind in (3, 5):
        k = keys64(n, seed).view(np.int64 if kind == 5 else np.uint64)
    else:
        k = normal_with_specials(n, np.float32 if kind == 1 else np.float64, seed)
    if n >= 8:
        r = splitmix64(stream_seed(seed, 4), n // 8) % np.uint64(n)
        k = k.copy()
        k[r.astype(np.int64)] = k[: n // 8]   # about an eighth of the keys repeat earlier ones
    return k


def segment_offsets(n: int, mix: str, seed: int = SEED_BASE) -> np.ndarray:
    """uint32 offsets (0 first, n last) of segments covering n keys:
    "small": lengths uniform in [1, 1024]; "large": uniform in [8192, 2^20];
    "mixed": log-uniform in [1, 2^17] (most segments short, most keys in
    long segments).  The last segment takes what is left."""
    rng_words = splitmix64(stream_seed(seed, 5), max(16, 4 * n // 512 + 64))
    u = (rng_words >> np.uint64(11)).astype(np.float64) / float(1 << 53)
    if mix == "small":
        lens = 1 + np.floor(u * 1024).astype(np.int64)
    elif mix == "large":
        lens = 8192 + np.floor(u * (2**20 - 8192)).astype(np.int64)
    elif mix == "mixed":
        lens = np.floor(np.exp2(u * 17)).astype(np.int64)
    else:
        raise ValueError(mix)
    ends = np.cumsum(lens)
    k = int(np.searchsorted(ends, n))
    if k >= lens.size:
        raise ValueError("not enough segment lengths drawn")
    off = np.concatenate([[0], ends[:k], [n]]).astype(np.uint32)
    return off


def compaction_input(n: int, seed: int = SEED_BASE) -> np.ndarray:
    """float32 drawn from {-U(0,1), 0.0, +U(0,1)} with probabilities
    0.4 / 0.2 / 0.4 (category from one stream, magnitude from another)."""
    out = np.empty(n, dtype=np.float32)
    sa, sb = stream_seed(seed, 0), stream_seed(seed, 1)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        a = u01(sa, hi - lo, lo)
        b = u01(sb, hi - lo, lo)
        v = np.where(a < 0.4, -b, np.where(a < 0.6, 0.0, b))
        out[lo:hi] = v.astype(np.float32)
    return out


def segments(num_segments: int, segment_len: int, seed: int = SEED_BASE) -> np.ndarray:
    """[num_segments, segment_len] uniform uint32 keys."""
    return u32(seed, num_segments * segment_len).reshape(num_segments, segment_len)


# Named workloads: the five problem configurations (seed = SEED_BASE + id).
WORKLOADS = {
    "uniform_u32_65536": dict(kind="keys", n=65536, gen="uniform", seed=SEED_BASE + 0),
    "pairs_u32_2^24": dict(kind="pairs", n=1 << 24, gen="uniform", seed=SEED_BASE + 1),
    "and3_u32_2^28": dict(kind="keys", n=1 << 28, gen="and3", seed=SEED_BASE + 2),
    "distinct16_u32_2^28": dict(kind="keys", n=1 << 28, gen="distinct16", seed=SEED_BASE + 3),
    "uniform_u32_2^28": dict(kind="keys", n=1 << 28, gen="uniform", seed=SEED_BASE + 5),
    "normal_f32_pairs_2^26": dict(kind="f32pairs", n=1 << 26, gen="normal_specials", seed=SEED_BASE + 4),
    "segments_16384x1024": dict(kind="segments", n=16384 * 1024, segments=16384, length=1024,
                                gen="uniform", seed=SEED_BASE + 6),
    "compact_f32_2^28": dict(kind="compact", n=1 << 28, gen="compaction", seed=SEED_BASE + 7),
    # the "next" rows: other key kinds, variable-length segments, 2-way split
    "uniform_u64_2^27": dict(kind="u64", n=1 << 27, gen="keys64", seed=SEED_BASE + 8),
    "segments_mixed_2^26": dict(kind="segsort", n=1 << 26, gen="uniform", mix="mixed",
                                seed=SEED_BASE + 9),
    "partition_f32_2^28": dict(kind="partition", n=1 << 28, gen="compaction", seed=SEED_BASE + 10),
    "split_sort_u32_2^25": dict(kind="splitsort", n=1 << 25, gen="uniform", seed=SEED_BASE + 11),
}


def make_keys(gen: str, n: int, seed: int) -> np.ndarray:
    if gen == "uniform":
        return uniform_keys(n, seed)
    if gen == "and3":
        return and3_keys(n, seed)
    if gen == "distinct16":
        return distinct16_keys(n, seed)
    if gen == "normal_specials":
        return normal_f32_with_specials(n, seed)
    if gen == "compaction":
        return compaction_input(n, seed)
    if gen == "keys64":
        return keys64(n, seed)
    raise ValueError(gen)
