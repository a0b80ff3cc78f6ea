"""ctypes binding of oracle.c -- TEST INFRASTRUCTURE ONLY.

Argument marshalling only: every computation happens in oracle.c.  The shared
object is compiled with the host C compiler on first use (or by
__graft_entry__.build()), without -ffast-math so that float comparisons keep
IEEE semantics (subnormals are not flushed).

`Oracle(path)` wraps any build of oracle.c; the module-level functions use
the default build.  The mutation tests compile deliberately broken copies of
oracle.c and load them through the same class.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_default = None

_u32p = ctypes.POINTER(ctypes.c_uint32)
_i64 = ctypes.c_int64
_int = ctypes.c_int


def compile_source(src: str, out_path: str) -> str:
    """Compile one C file into a shared object at out_path."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    cc = os.environ.get("CC", "gcc")
    tmp = out_path + f".tmp{os.getpid()}"
    subprocess.run([cc, "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                    "-o", tmp, src], check=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so (skipped when up to date)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(SOURCE)):
        return _LIB_PATH
    return compile_source(SOURCE, _LIB_PATH)


def _as_u32(a) -> np.ndarray:
    """View float32/uint32/int32 data as a contiguous uint32 array (bit patterns)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32 or a.dtype == np.int32:
        a = a.view(np.uint32)
    if a.dtype != np.uint32:
        raise TypeError(f"expected 32-bit data, got {a.dtype}")
    return a


# numpy dtype of each key kind (u32, f32, i32, u64, f64, i64)
KIND_DTYPES = (np.uint32, np.float32, np.int32, np.uint64, np.float64, np.int64)


def _as_kind(a, kind: int) -> np.ndarray:
    """Contiguous 1-D array of the key kind's dtype (same bits, no conversion)."""
    a = np.ascontiguousarray(a).ravel()
    want = np.dtype(KIND_DTYPES[kind])
    if a.dtype != want:
        if a.dtype.itemsize != want.itemsize:
            raise TypeError(f"kind {kind} wants {want.itemsize}-byte keys, got {a.dtype}")
        a = a.view(want)
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_u32p)


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


class Oracle:
    """One loaded build of oracle.c."""

    _SIGS = {
        "oracle_f32_bits_to_ordered": (ctypes.c_uint32, [ctypes.c_uint32]),
        "oracle_ordered_to_f32_bits": (ctypes.c_uint32, [ctypes.c_uint32]),
        "oracle_f32_bits_to_ordered_array": (None, [_u32p, _u32p, _i64]),
        "oracle_ordered_to_f32_bits_array": (None, [_u32p, _u32p, _i64]),
        "oracle_num_passes": (_int, [_int, _int]),
        "oracle_digit_histograms": (_int, [_u32p, _i64, _int, _int, _int, _u32p]),
        "oracle_exclusive_scan_bins": (None, [_u32p, _int, _u32p]),
        "oracle_radix_sort_pairs": (_int, [_u32p, _u32p, _u32p, _u32p, _i64, _int, _int, _int]),
        "oracle_radix_sort_keys": (_int, [_u32p, _u32p, _i64, _int]),
        "oracle_compact_positive": (_i64, [_u32p, _u32p, _i64]),
        "oracle_segmented_sort": (_int, [_u32p, _i64, _int]),
        "oracle_bitonic_network": (_int, [_u32p, _int]),
        "oracle_radix2_three_pass": (_int, [_u32p, _u32p, _u32p, _u32p, _i64]),
        "oracle_kind_bytes": (_int, [_int]),
        "oracle_key_to_ordered": (ctypes.c_uint64, [ctypes.c_uint64, _int, _int]),
        "oracle_ordered_to_key": (ctypes.c_uint64, [ctypes.c_uint64, _int, _int]),
        "oracle_digit_histograms_general": (_int, [ctypes.c_void_p, _i64, _int, _int, _int, _int,
                                                   _u32p]),
        "oracle_radix_sort_general": (_int, [ctypes.c_void_p, _u32p, ctypes.c_void_p, _u32p, _i64,
                                             _int, _int, _int, _int]),
        "oracle_segmented_sort_general": (_int, [_u32p, _u32p, _u32p, _u32p, _i64, _u32p, _i64,
                                                 _int, _int]),
        "oracle_partition": (_i64, [_u32p, _u32p, _u32p, _u32p, _i64, _int, _int, ctypes.c_uint32,
                                    ctypes.c_void_p]),
        "oracle_split_sort": (_int, [_u32p, _u32p, _u32p, _u32p, _i64, _int, _int]),
    }

    def __init__(self, path: str):
        self.lib = ctypes.CDLL(path)
        for name, (res, args) in self._SIGS.items():
            fn = getattr(self.lib, name)
            fn.restype = res
            fn.argtypes = args

    # a0 -----------------------------------------------------------------
    def f32_bits_to_ordered(self, bits: int) -> int:
        return int(self.lib.oracle_f32_bits_to_ordered(int(bits) & 0xFFFFFFFF))

    def ordered_to_f32_bits(self, u: int) -> int:
        return int(self.lib.oracle_ordered_to_f32_bits(int(u) & 0xFFFFFFFF))

    def f32_bits_to_ordered_array(self, bits) -> np.ndarray:
        b = _as_u32(bits).ravel()
        out = np.empty_like(b)
        self.lib.oracle_f32_bits_to_ordered_array(_ptr(b), _ptr(out), b.size)
        return out

    def ordered_to_f32_bits_array(self, u) -> np.ndarray:
        b = _as_u32(u).ravel()
        out = np.empty_like(b)
        self.lib.oracle_ordered_to_f32_bits_array(_ptr(b), _ptr(out), b.size)
        return out

    def num_passes(self, begin_bit: int, end_bit: int) -> int:
        return int(self.lib.oracle_num_passes(begin_bit, end_bit))

    # a1, a2 -------------------------------------------------------------
    def digit_histograms(self, keys, kind: int = 0, begin_bit: int = 0,
                         end_bit: int = 32) -> np.ndarray:
        """hist[passes, 256]."""
        k = _as_u32(keys).ravel()
        p = self.num_passes(begin_bit, end_bit)
        if p < 0:
            raise ValueError("bad bit range")
        hist = np.zeros((max(p, 1), 256), dtype=np.uint32)
        _check(self.lib.oracle_digit_histograms(_ptr(k), k.size, kind, begin_bit, end_bit,
                                                _ptr(hist)), "digit_histograms")
        return hist[:p]

    def exclusive_scan_bins(self, hist) -> np.ndarray:
        """base[passes, 256], the exclusive scan of each row."""
        h = _as_u32(hist).reshape(-1, 256)
        base = np.zeros_like(h)
        self.lib.oracle_exclusive_scan_bins(_ptr(h), h.shape[0], _ptr(base))
        return base

    # a3 -----------------------------------------------------------------
    def radix_sort_pairs(self, keys, vals=None, kind: int = 0, begin_bit: int = 0,
                         end_bit: int = 32):
        """(keys_out, vals_out or None); float32 keys come back as float32."""
        src_dtype = np.asarray(keys).dtype
        k = _as_u32(keys).ravel()
        ko = np.empty_like(k)
        v = vo = None
        if vals is not None:
            v = _as_u32(vals).ravel()
            if v.size != k.size:
                raise ValueError("keys and values differ in length")
            vo = np.empty_like(v)
        _check(self.lib.oracle_radix_sort_pairs(_ptr(k), _ptr(v), _ptr(ko), _ptr(vo), k.size,
                                                kind, begin_bit, end_bit), "radix_sort_pairs")
        if src_dtype == np.float32:
            ko = ko.view(np.float32)
        return ko, vo

    def radix_sort_keys(self, keys, kind: int = 0) -> np.ndarray:
        return self.radix_sort_pairs(keys, None, kind, 0, 32)[0]

    # f1: every key kind, both directions ------------------------------
    def key_to_ordered(self, bits: int, kind: int, descending: bool = False) -> int:
        return int(self.lib.oracle_key_to_ordered(int(bits) & (2**64 - 1), kind, int(descending)))

    def ordered_to_key(self, u: int, kind: int, descending: bool = False) -> int:
        return int(self.lib.oracle_ordered_to_key(int(u) & (2**64 - 1), kind, int(descending)))

    def digit_histograms_general(self, keys, kind: int, begin_bit: int = 0,
                                 end_bit: int | None = None, descending: bool = False):
        k = _as_kind(keys, kind)
        if end_bit is None:
            end_bit = 8 * k.itemsize
        p = (end_bit - begin_bit + 7) // 8
        hist = np.zeros((max(p, 1), 256), dtype=np.uint32)
        _check(self.lib.oracle_digit_histograms_general(
            k.ctypes.data, k.size, kind, int(descending), begin_bit, end_bit, _ptr(hist)),
            "digit_histograms_general")
        return hist[:p]

    def radix_sort(self, keys, vals=None, kind: int = 0, descending: bool = False,
                   begin_bit: int = 0, end_bit: int | None = None):
        """(keys_out with the input dtype, vals_out or None)."""
        k = _as_kind(keys, kind)
        if end_bit is None:
            end_bit = 8 * k.itemsize
        ko = np.empty_like(k)
        v = vo = None
        if vals is not None:
            v = _as_u32(vals).ravel()
            if v.size != k.size:
                raise ValueError("keys and values differ in length")
            vo = np.empty_like(v)
        _check(self.lib.oracle_radix_sort_general(k.ctypes.data, _ptr(v), ko.ctypes.data, _ptr(vo),
                                                  k.size, kind, int(descending), begin_bit,
                                                  end_bit), "radix_sort_general")
        return ko, vo

    # f2: variable-length segments --------------------------------------
    def segmented_sort_general(self, keys, offsets, vals=None, kind: int = 0,
                               descending: bool = False):
        """(keys_out with the input dtype, vals_out or None); raises on bad offsets."""
        k = _as_kind(keys, kind)
        off = np.ascontiguousarray(offsets, dtype=np.uint32).ravel()
        ko = np.empty_like(k)
        v = vo = None
        if vals is not None:
            v = _as_u32(vals).ravel()
            vo = np.empty_like(v)
        _check(self.lib.oracle_segmented_sort_general(
            _ptr(k.view(np.uint32)), _ptr(v), _ptr(ko.view(np.uint32)), _ptr(vo), k.size, _ptr(off),
            max(off.size - 1, 0), kind, int(descending)), "segmented_sort_general")
        return ko, vo

    # f3: 2-way split ---------------------------------------------------
    def partition(self, x, vals=None, pred: int = 1, kind: int = 0, param: int = 0, flags=None):
        """(out, vals_out or None, m) with out keeping the input dtype."""
        src_dtype = np.asarray(x).dtype
        xi = _as_u32(x).ravel()
        out = np.empty_like(xi)
        v = vo = None
        if vals is not None:
            v = _as_u32(vals).ravel()
            vo = np.empty_like(v)
        fl = None
        if flags is not None:
            fl = np.ascontiguousarray(flags, dtype=np.uint8).ravel()
        m = self.lib.oracle_partition(_ptr(xi), _ptr(v), _ptr(out), _ptr(vo), xi.size, pred, kind,
                                      int(param) & 0xFFFFFFFF,
                                      None if fl is None else fl.ctypes.data)
        if src_dtype in (np.float32, np.int32):
            out = out.view(src_dtype)
        return out, vo, int(m)

    def split_sort(self, keys, vals=None, begin_bit: int = 0, end_bit: int = 32):
        k = _as_u32(keys).ravel()
        ko = np.empty_like(k)
        v = vo = None
        if vals is not None:
            v = _as_u32(vals).ravel()
            vo = np.empty_like(v)
        _check(self.lib.oracle_split_sort(_ptr(k), _ptr(v), _ptr(ko), _ptr(vo), k.size, begin_bit,
                                          end_bit), "split_sort")
        return ko, vo

    # a4 -----------------------------------------------------------------
    def compact_positive(self, x):
        """(out float32, m)."""
        xi = _as_u32(np.asarray(x, dtype=np.float32)).ravel()
        out = np.empty_like(xi)
        m = self.lib.oracle_compact_positive(_ptr(xi), _ptr(out), xi.size)
        return out.view(np.float32), int(m)

    # a5 -----------------------------------------------------------------
    def segmented_sort(self, keys2d) -> np.ndarray:
        a = np.array(_as_u32(keys2d), copy=True)
        if a.ndim != 2:
            raise ValueError("expected a 2-D array [segments, length]")
        _check(self.lib.oracle_segmented_sort(_ptr(a), a.shape[0], a.shape[1]),
               "segmented_sort")
        return a

    def bitonic_network(self, keys) -> np.ndarray:
        a = np.array(_as_u32(keys), copy=True).ravel()
        _check(self.lib.oracle_bitonic_network(_ptr(a), a.size), "bitonic_network")
        return a

    # cross-check ---------------------------------------------------------
    def radix2_three_pass(self, keys, ids):
        k = _as_u32(keys).ravel()
        i = _as_u32(ids).ravel()
        ko = np.empty_like(k)
        io = np.empty_like(i)
        _check(self.lib.oracle_radix2_three_pass(_ptr(k), _ptr(i), _ptr(ko), _ptr(io), k.size),
               "radix2_three_pass")
        return ko, io


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def _fwd(name):
    def f(*a, **k):
        return getattr(default(), name)(*a, **k)
    f.__name__ = name
    f.__doc__ = getattr(Oracle, name).__doc__
    return f


f32_bits_to_ordered = _fwd("f32_bits_to_ordered")
ordered_to_f32_bits = _fwd("ordered_to_f32_bits")
f32_bits_to_ordered_array = _fwd("f32_bits_to_ordered_array")
ordered_to_f32_bits_array = _fwd("ordered_to_f32_bits_array")
num_passes = _fwd("num_passes")
digit_histograms = _fwd("digit_histograms")
exclusive_scan_bins = _fwd("exclusive_scan_bins")
radix_sort_pairs = _fwd("radix_sort_pairs")
radix_sort_keys = _fwd("radix_sort_keys")
compact_positive = _fwd("compact_positive")
segmented_sort = _fwd("segmented_sort")
bitonic_network = _fwd("bitonic_network")
radix2_three_pass = _fwd("radix2_three_pass")
