"""torch-facing wrappers of libgsort (argument marshalling only).

Every computation runs in the CUDA kernels of libgsort.so; these functions
allocate outputs and workspaces with torch, pass raw pointers and the current
CUDA stream, and raise GsortError on a non-zero status.  There is no CPU
fallback: CPU tensors are copied to the current CUDA device, processed there
and copied back.

sort_pairs/sort_keys take 32-bit keys: torch.uint32 or torch.int32 tensors are
sorted as unsigned 32-bit integers (an int32 tensor is a container of bit
patterns there), and torch.float32 tensors in IEEE totalOrder (-0.0 before
+0.0).  sort() takes every key kind, with the kind read from the dtype
(int32/int64 signed, uint32/uint64 unsigned, float32/float64 totalOrder)
unless given, in either direction.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from .build import build  # noqa: F401  (re-exported)

KEY_U32, KEY_F32, KEY_I32, KEY_U64, KEY_F64, KEY_I64 = 0, 1, 2, 3, 4, 5
DESCENDING = 1
_U32_DTYPES = (torch.int32,) + ((torch.uint32,) if hasattr(torch, "uint32") else ())
_KIND_OF_DTYPE = {torch.float32: KEY_F32, torch.int32: KEY_I32, torch.float64: KEY_F64,
                  torch.int64: KEY_I64}
if hasattr(torch, "uint32"):
    _KIND_OF_DTYPE[torch.uint32] = KEY_U32
if hasattr(torch, "uint64"):
    _KIND_OF_DTYPE[torch.uint64] = KEY_U64
_KIND_BYTES = {KEY_U32: 4, KEY_F32: 4, KEY_I32: 4, KEY_U64: 8, KEY_F64: 8, KEY_I64: 8}


class GsortError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        lib = _lib.load()
        msg = lib.gsort_status_string(code).decode()
        super().__init__(f"{what}: {msg}" if what else msg)
        self.code = code


def library_path() -> str:
    return _lib.library_path()


def _check(rc: int, what: str):
    if rc != 0:
        raise GsortError(rc, what)


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _key_kind(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return KEY_F32
    if t.dtype in _U32_DTYPES:
        return KEY_U32
    raise TypeError(f"keys must be uint32, int32 (as bit patterns) or float32, got {t.dtype}")


def _flat_cuda(t: torch.Tensor, name: str) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.view(-1)


def _workspace(nbytes: int, device, workspace=None) -> torch.Tensor:
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise GsortError(-3, "workspace")
        return workspace
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)


def radix_workspace_bytes(n: int, with_values: bool) -> int:
    return int(_lib.load().gsort_radix_workspace_bytes(n, 1 if with_values else 0))


def compact_workspace_bytes(n: int) -> int:
    return int(_lib.load().gsort_compact_workspace_bytes(n))


def _events_arg(events):
    if not events:
        return None, 0
    for e in events:            # torch creates the CUDA event on its first record
        if e.cuda_event == 0:
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    return arr, len(events)


def sort_pairs(keys: torch.Tensor, values: torch.Tensor | None = None, begin_bit: int = 0,
               end_bit: int = 32, *, keys_out: torch.Tensor | None = None,
               values_out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
               events=None, variant: int = 0, spin_limit: int = 0, stall_tile: int = -1,
               check: bool = True):
    """Stable sort of keys (and values) by key bits [begin_bit, end_bit).

    Returns (sorted_keys, sorted_values or None).  keys_out/values_out may be
    the inputs themselves (in place).  With check=True the call synchronises
    the stream and raises on a device-side error (a look-back timeout)."""
    if not keys.is_cuda:
        return _host_roundtrip(sort_pairs, keys, values, begin_bit, end_bit)
    k = _flat_cuda(keys, "keys")
    kind = _key_kind(k)
    v = None
    if values is not None:
        v = _flat_cuda(values, "values")
        if v.numel() != k.numel() or v.element_size() != 4:
            raise ValueError("values must be a 32-bit tensor with one entry per key")
    n = k.numel()
    ko = torch.empty_like(k) if keys_out is None else _flat_cuda(keys_out, "keys_out")
    vo = None
    if v is not None:
        vo = torch.empty_like(v) if values_out is None else _flat_cuda(values_out, "values_out")
    lib = _lib.load()
    ws = _workspace(radix_workspace_bytes(n, v is not None), k.device, workspace)
    ev, nev = _events_arg(events)
    opt = _lib.Options(spin_limit, stall_tile, ctypes.cast(ev, ctypes.POINTER(ctypes.c_void_p))
                       if ev is not None else None, nev, variant)
    with torch.cuda.device(k.device):
        rc = lib.gsort_radix_pairs_ex(
            k.data_ptr(), ko.data_ptr(), v.data_ptr() if v is not None else None,
            vo.data_ptr() if vo is not None else None, n, kind, begin_bit, end_bit,
            ws.data_ptr(), ws.numel(), _stream(k.device), ctypes.byref(opt))
        _check(rc, "gsort_radix_pairs")
        if check and n > 0 and begin_bit < end_bit:
            _check(lib.gsort_check(ws.data_ptr(), _stream(k.device)), "gsort_radix_pairs (device)")
    ko = ko.view(keys.shape) if keys_out is None else keys_out
    if vo is not None:
        vo = vo.view(values.shape) if values_out is None else values_out
    return ko, vo


def sort_workspace_bytes(n: int, kind: int, with_values: bool) -> int:
    return int(_lib.load().gsort_radix_sort_workspace_bytes(n, kind, 1 if with_values else 0))


def sort(keys: torch.Tensor, values: torch.Tensor | None = None, *, descending: bool = False,
         kind: int | None = None, begin_bit: int = 0, end_bit: int | None = None,
         keys_out: torch.Tensor | None = None, values_out: torch.Tensor | None = None,
         workspace: torch.Tensor | None = None, events=None, spin_limit: int = 0,
         stall_tile: int = -1, check: bool = True):
    """Stable radix sort of 32- or 64-bit keys (and 32-bit values), ascending
    or descending, by bits [begin_bit, end_bit) of the mapped key (default:
    the whole key).  Returns (sorted_keys, sorted_values or None)."""
    if not keys.is_cuda:
        return _host_roundtrip(
            lambda k, v: sort(k, v, descending=descending, kind=kind, begin_bit=begin_bit,
                              end_bit=end_bit), keys, values)
    k = _flat_cuda(keys, "keys")
    if kind is None:
        if k.dtype not in _KIND_OF_DTYPE:
            raise TypeError(f"no key kind for dtype {k.dtype}; pass kind=")
        kind = _KIND_OF_DTYPE[k.dtype]
    if _KIND_BYTES.get(kind) != k.element_size():
        raise TypeError(f"kind {kind} needs {_KIND_BYTES.get(kind)}-byte keys, got {k.dtype}")
    if end_bit is None:
        end_bit = 8 * k.element_size()
    v = None
    if values is not None:
        v = _flat_cuda(values, "values")
        if v.numel() != k.numel() or v.element_size() != 4:
            raise ValueError("values must be a 32-bit tensor with one entry per key")
    n = k.numel()
    ko = torch.empty_like(k) if keys_out is None else _flat_cuda(keys_out, "keys_out")
    vo = None
    if v is not None:
        vo = torch.empty_like(v) if values_out is None else _flat_cuda(values_out, "values_out")
    lib = _lib.load()
    ws = _workspace(sort_workspace_bytes(n, kind, v is not None), k.device, workspace)
    ev, nev = _events_arg(events)
    opt = _lib.Options(spin_limit, stall_tile, ctypes.cast(ev, ctypes.POINTER(ctypes.c_void_p))
                       if ev is not None else None, nev, 0)
    with torch.cuda.device(k.device):
        rc = lib.gsort_radix_sort_ex(
            k.data_ptr(), ko.data_ptr(), v.data_ptr() if v is not None else None,
            vo.data_ptr() if vo is not None else None, n, kind, DESCENDING if descending else 0,
            begin_bit, end_bit, ws.data_ptr(), ws.numel(), _stream(k.device), ctypes.byref(opt))
        _check(rc, "gsort_radix_sort")
        if check and n > 0 and begin_bit < end_bit:
            _check(lib.gsort_check(ws.data_ptr(), _stream(k.device)), "gsort_radix_sort (device)")
    ko = ko.view(keys.shape) if keys_out is None else keys_out
    if vo is not None:
        vo = vo.view(values.shape) if values_out is None else values_out
    return ko, vo


def segmented_sort_workspace_bytes(n: int, num_segments: int, with_values: bool) -> int:
    return int(_lib.load().gsort_segmented_sort_workspace_bytes(n, num_segments,
                                                                 1 if with_values else 0))


def segmented_sort(keys: torch.Tensor, offsets: torch.Tensor, values: torch.Tensor | None = None,
                   *, descending: bool = False, kind: int | None = None,
                   keys_out: torch.Tensor | None = None, values_out: torch.Tensor | None = None,
                   workspace: torch.Tensor | None = None, events=None, check: bool = True):
    """Stable sort of each segment [offsets[s], offsets[s+1]) of 32-bit keys
    (and 32-bit values).  offsets: int32/uint32 tensor of num_segments + 1
    entries, 0 first and len(keys) last.  Returns (keys, values or None)."""
    if not keys.is_cuda:
        return _host_roundtrip(
            lambda k, o, v: segmented_sort(k, o, v, descending=descending, kind=kind),
            keys, offsets, values)
    k = _flat_cuda(keys, "keys")
    if kind is None:
        if k.dtype not in _KIND_OF_DTYPE:
            raise TypeError(f"no key kind for dtype {k.dtype}; pass kind=")
        kind = _KIND_OF_DTYPE[k.dtype]
    if _KIND_BYTES.get(kind) != 4 or k.element_size() != 4:
        raise TypeError("segmented_sort takes 32-bit keys")
    off = _flat_cuda(offsets, "offsets")
    if off.element_size() != 4:
        raise TypeError("offsets must be a 32-bit tensor")
    v = None
    if values is not None:
        v = _flat_cuda(values, "values")
        if v.numel() != k.numel() or v.element_size() != 4:
            raise ValueError("values must be a 32-bit tensor with one entry per key")
    n, S = k.numel(), max(off.numel() - 1, 0)
    ko = torch.empty_like(k) if keys_out is None else _flat_cuda(keys_out, "keys_out")
    vo = None
    if v is not None:
        vo = torch.empty_like(v) if values_out is None else _flat_cuda(values_out, "values_out")
    lib = _lib.load()
    ws = _workspace(segmented_sort_workspace_bytes(n, S, v is not None), k.device, workspace)
    ev, nev = _events_arg(events)
    opt = _lib.Options(0, -1, ctypes.cast(ev, ctypes.POINTER(ctypes.c_void_p))
                       if ev is not None else None, nev, 0)
    with torch.cuda.device(k.device):
        rc = lib.gsort_segmented_sort_ex(
            k.data_ptr(), ko.data_ptr(), v.data_ptr() if v is not None else None,
            vo.data_ptr() if vo is not None else None, n, off.data_ptr(), S, kind,
            DESCENDING if descending else 0, ws.data_ptr(), ws.numel(), _stream(k.device),
            ctypes.byref(opt))
        _check(rc, "gsort_segmented_sort")
        if check and n > 0:
            _check(lib.gsort_check(ws.data_ptr(), _stream(k.device)), "gsort_segmented_sort (device)")
    ko = ko.view(keys.shape) if keys_out is None else keys_out
    if vo is not None:
        vo = vo.view(values.shape) if values_out is None else values_out
    return ko, vo


PRED_FLAGS, PRED_BIT_SET, PRED_BIT_CLEAR, PRED_LESS, PRED_POSITIVE = 0, 1, 2, 3, 4


def partition(x: torch.Tensor, values: torch.Tensor | None = None, *, pred: int = PRED_BIT_SET,
              param: int = 0, kind: int = KEY_U32, flags: torch.Tensor | None = None,
              out: torch.Tensor | None = None, values_out: torch.Tensor | None = None,
              workspace: torch.Tensor | None = None, check: bool = True):
    """Stable 2-way split of 32-bit elements: those whose predicate holds
    first, the others after, each side in input order.  Returns (out,
    values_out or None, num_true) with num_true a one-element int64 tensor."""
    if not x.is_cuda:
        raise ValueError("partition takes CUDA tensors")
    xi = _flat_cuda(x, "x")
    if xi.element_size() != 4:
        raise TypeError("partition takes 32-bit elements")
    v = None
    if values is not None:
        v = _flat_cuda(values, "values")
        if v.numel() != xi.numel() or v.element_size() != 4:
            raise ValueError("values must be a 32-bit tensor with one entry per element")
    fl = None
    if pred == PRED_FLAGS:
        if flags is None:
            raise ValueError("PRED_FLAGS needs flags")
        fl = _flat_cuda(flags, "flags")
        if fl.element_size() != 1 or fl.numel() != xi.numel():
            raise ValueError("flags must be a 1-byte tensor with one entry per element")
    n = xi.numel()
    o = torch.empty_like(xi) if out is None else _flat_cuda(out, "out")
    vo = None
    if v is not None:
        vo = torch.empty_like(v) if values_out is None else _flat_cuda(values_out, "values_out")
    nt = torch.empty(1, dtype=torch.int64, device=xi.device)
    lib = _lib.load()
    ws = _workspace(int(lib.gsort_partition_workspace_bytes(n)), xi.device, workspace)
    with torch.cuda.device(xi.device):
        rc = lib.gsort_partition(xi.data_ptr(), o.data_ptr(), v.data_ptr() if v is not None else None,
                                 vo.data_ptr() if vo is not None else None, n, pred, kind,
                                 int(param) & 0xFFFFFFFF, fl.data_ptr() if fl is not None else None,
                                 nt.data_ptr(), ws.data_ptr(), ws.numel(), _stream(xi.device))
        _check(rc, "gsort_partition")
        if check and n > 0:
            _check(lib.gsort_check(ws.data_ptr(), _stream(xi.device)), "gsort_partition (device)")
    o = o.view(x.shape) if out is None else out
    if vo is not None:
        vo = vo.view(values.shape) if values_out is None else values_out
    return o, vo, nt


def split_sort(keys: torch.Tensor, values: torch.Tensor | None = None, begin_bit: int = 0,
               end_bit: int = 32, *, keys_out: torch.Tensor | None = None,
               values_out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
               check: bool = True):
    """The 1-bit split LSD sort (one stable split per bit) of unsigned 32-bit keys."""
    if not keys.is_cuda:
        raise ValueError("split_sort takes CUDA tensors")
    k = _flat_cuda(keys, "keys")
    v = None if values is None else _flat_cuda(values, "values")
    n = k.numel()
    ko = torch.empty_like(k) if keys_out is None else _flat_cuda(keys_out, "keys_out")
    vo = None
    if v is not None:
        vo = torch.empty_like(v) if values_out is None else _flat_cuda(values_out, "values_out")
    lib = _lib.load()
    ws = _workspace(int(lib.gsort_split_sort_workspace_bytes(n, 1 if v is not None else 0)),
                    k.device, workspace)
    with torch.cuda.device(k.device):
        rc = lib.gsort_split_sort(k.data_ptr(), ko.data_ptr(), v.data_ptr() if v is not None else None,
                                  vo.data_ptr() if vo is not None else None, n, begin_bit, end_bit,
                                  ws.data_ptr(), ws.numel(), _stream(k.device))
        _check(rc, "gsort_split_sort")
        if check and n > 0 and begin_bit < end_bit:
            _check(lib.gsort_check(ws.data_ptr(), _stream(k.device)), "gsort_split_sort (device)")
    ko = ko.view(keys.shape) if keys_out is None else keys_out
    if vo is not None:
        vo = vo.view(values.shape) if values_out is None else values_out
    return ko, vo


def sort_keys(keys: torch.Tensor, **kw) -> torch.Tensor:
    """Ascending sort of 32-bit keys (all 32 bits)."""
    if not keys.is_cuda:
        return _host_roundtrip(sort_keys, keys)
    ko = kw.pop("keys_out", None)
    return sort_pairs(keys, None, 0, 32, keys_out=ko, **kw)[0]


def digit_histograms(keys: torch.Tensor, begin_bit: int = 0, end_bit: int | None = None, *,
                     kind: int | None = None) -> torch.Tensor:
    """[passes, 256] counts of each 8-bit digit of the (ascending) mapped key
    (int32 tensor holding uint32 counts).  Without `kind`, 32-bit tensors are
    read as sort_keys reads them (int32/uint32 unsigned, float32 totalOrder)
    and 64-bit tensors by their dtype."""
    k = _flat_cuda(keys, "keys")
    if kind is None:
        kind = _key_kind(k) if k.element_size() == 4 else _KIND_OF_DTYPE.get(k.dtype)
        if kind is None:
            raise TypeError(f"no key kind for dtype {k.dtype}; pass kind=")
    if end_bit is None:
        end_bit = 8 * k.element_size()
    passes = (end_bit - begin_bit + 7) // 8
    out = torch.empty((max(passes, 1), 256), dtype=torch.int32, device=k.device)
    with torch.cuda.device(k.device):
        _check(_lib.load().gsort_digit_histograms(k.data_ptr(), k.numel(), kind, begin_bit,
                                                   end_bit, out.data_ptr(), _stream(k.device)),
               "gsort_digit_histograms")
    return out[:passes]


def compact_positive(x: torch.Tensor, *, out: torch.Tensor | None = None,
                     num_kept: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                     events=None, spin_limit: int = 0, stall_tile: int = -1, check: bool = True):
    """Keeps x > 0 in order, zero-fills the rest.  Returns (out, num_kept)
    where num_kept is a one-element int64 CUDA tensor."""
    if not x.is_cuda:
        return _host_roundtrip(compact_positive, x)
    if x.dtype != torch.float32:
        raise TypeError("compact_positive takes float32")
    xi = _flat_cuda(x, "x")
    n = xi.numel()
    o = torch.empty_like(xi) if out is None else _flat_cuda(out, "out")
    nk = torch.empty(1, dtype=torch.int64, device=xi.device) if num_kept is None else num_kept
    lib = _lib.load()
    ws = _workspace(compact_workspace_bytes(n), xi.device, workspace)
    ev, nev = _events_arg(events)
    opt = _lib.Options(spin_limit, stall_tile, ctypes.cast(ev, ctypes.POINTER(ctypes.c_void_p))
                       if ev is not None else None, nev, 0)
    with torch.cuda.device(xi.device):
        rc = lib.gsort_compact_positive_ex(xi.data_ptr(), o.data_ptr(), n, nk.data_ptr(),
                                           ws.data_ptr(), ws.numel(), _stream(xi.device),
                                           ctypes.byref(opt))
        _check(rc, "gsort_compact_positive")
        if check and n > 0:
            _check(lib.gsort_check(ws.data_ptr(), _stream(xi.device)),
                   "gsort_compact_positive (device)")
    return (o.view(x.shape) if out is None else out), nk


def segmented_sort_(keys2d: torch.Tensor) -> torch.Tensor:
    """Sorts every row of a [segments, length <= 1024] 32-bit tensor in place."""
    if keys2d.dim() != 2:
        raise ValueError("expected a 2-D tensor [segments, length]")
    if not keys2d.is_cuda:
        out = _host_roundtrip(segmented_sort_, keys2d)
        keys2d.copy_(out)
        return keys2d
    if keys2d.dtype not in _U32_DTYPES:
        raise TypeError("segmented_sort_ takes uint32 or int32 (as unsigned bit patterns)")
    k = _flat_cuda(keys2d, "keys")
    with torch.cuda.device(k.device):
        _check(_lib.load().gsort_segmented_bitonic(k.data_ptr(), keys2d.shape[0], keys2d.shape[1],
                                                    _stream(k.device)), "gsort_segmented_bitonic")
    return keys2d


def _host_roundtrip(fn, *args):
    """Runs fn on the current CUDA device for CPU tensors: pinned host ->
    device copy, the GPU call, device -> host copy."""
    dev = torch.device("cuda", torch.cuda.current_device())
    moved = [a.pin_memory().to(dev, non_blocking=True) if isinstance(a, torch.Tensor) else a
             for a in args]
    res = fn(*moved)
    if isinstance(res, tuple):
        return tuple(r.to("cpu") if isinstance(r, torch.Tensor) else r for r in res)
    return res.to("cpu")
