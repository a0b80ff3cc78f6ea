"""Runs one library call on a seeded input, for profilers (ncu).

    python profile_cases.py OP [--n-log2 K] [--warmup W]
           [--reps R] [--variant V]

OP: keys (uint32 keys, 32 bits), pairs (uint32 key/index pairs), fpairs
(float keys with index values), compact (compaction input), segments (1024-key
segments, n/1024 of them), hist (the digit-histogram step alone), sort (any
key kind: --kind u32|f32|i32|u64|f64|i64 [--desc] [--values]), segsort
(variable-length segments, --mix small|mixed|large [--values] [--desc]),
partition (compaction input split by x > 0 [--values]), splitsort (the 1-bit
split sort of uint32 keys [--values]).
keys, hist and segsort take --dist uniform|and3|distinct16 (the key distribution).
--time prints the median CUDA-event time of the timed calls.
Each call is followed by a device-status check; the process exits non-zero on
any error, so a profiler only ever runs a command that finished cleanly.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

from bitonic_networks_gb300 import _lib, gsort, synth


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("op", choices=["keys", "pairs", "fpairs", "compact", "segments", "hist", "sort",
                                   "segsort", "partition", "splitsort"])
    ap.add_argument("--mix", choices=["small", "mixed", "large"], default="mixed")
    ap.add_argument("--dist", choices=["uniform", "and3", "distinct16"], default="uniform")
    ap.add_argument("--kind", choices=["u32", "f32", "i32", "u64", "f64", "i64"], default="u64")
    ap.add_argument("--desc", action="store_true")
    ap.add_argument("--values", action="store_true")
    ap.add_argument("--time", action="store_true")
    ap.add_argument("--n-log2", type=int, default=26)
    ap.add_argument("--warmup", type=int, default=1)
    ap.add_argument("--reps", type=int, default=1)
    ap.add_argument("--variant", type=int, default=0)
    a = ap.parse_args(argv)
    n = 1 << a.n_log2
    dev = torch.device("cuda", 0)

    def up(x: np.ndarray) -> torch.Tensor:
        x = np.ascontiguousarray(x)
        return torch.from_numpy(x.view(np.int32) if x.dtype == np.uint32 else x).to(dev)

    kinds = {"u32": 0, "f32": 1, "i32": 2, "u64": 3, "f64": 4, "i64": 5}
    kind = kinds[a.kind]
    if a.op == "partition":
        x = up(synth.compaction_input(n, 9))
        v = up(synth.index_values(n)) if a.values else None
    elif a.op == "splitsort":
        x = up(synth.uniform_keys(n, 10))
        v = up(synth.index_values(n)) if a.values else None
    elif a.op == "segsort":
        x = up({"uniform": synth.uniform_keys, "and3": synth.and3_keys,
                "distinct16": synth.distinct16_keys}[a.dist](n, 7))
        off_np = synth.segment_offsets(n, a.mix, 8)
        off = up(off_np)
        v = up(synth.index_values(n)) if a.values else None
        print(f"segsort {a.mix}: {off_np.size - 1} segments, "
              f"{int(((off_np[1:] - off_np[:-1]) <= 1024).sum())} of at most 1024 keys "
              f"holding {int((off_np[1:] - off_np[:-1])[(off_np[1:] - off_np[:-1]) <= 1024].sum())} keys")
    elif a.op == "sort":
        kx = synth.keys_of_kind(kind, n, 6)
        kx = kx.view({4: np.int32, 8: np.int64}[kx.dtype.itemsize]) if kx.dtype.kind == "u" else kx
        x = torch.from_numpy(np.ascontiguousarray(kx)).to(dev)
        v = up(synth.index_values(n)) if a.values else None
    elif a.op in ("keys", "hist"):
        x = up({"uniform": synth.uniform_keys, "and3": synth.and3_keys,
                "distinct16": synth.distinct16_keys}[a.dist](n, 1))
    elif a.op == "pairs":
        x, v = up(synth.uniform_keys(n, 2)), up(synth.index_values(n))
    elif a.op == "fpairs":
        x, v = up(synth.normal_f32_with_specials(n, 3)), up(synth.index_values(n))
    elif a.op == "compact":
        x = up(synth.compaction_input(n, 4))
    else:
        seg = up(synth.segments(n // 1024, 1024, 5))
        x = seg.clone()

    def once():
        if a.op == "partition":
            gsort.partition(x, v, pred=gsort.PRED_POSITIVE, check=not a.time)
        elif a.op == "splitsort":
            gsort.split_sort(x, v, 0, 32, check=not a.time)
        elif a.op == "segsort":
            gsort.segmented_sort(x, off, v, descending=a.desc, kind=0, check=not a.time)
        elif a.op == "sort":
            gsort.sort(x, v, descending=a.desc, kind=kind, check=not a.time)
        elif a.op == "keys":
            gsort.sort_pairs(x, None, variant=a.variant)
        elif a.op in ("pairs", "fpairs"):
            gsort.sort_pairs(x, v, variant=a.variant)
        elif a.op == "compact":
            gsort.compact_positive(x)
        elif a.op == "hist":
            gsort.digit_histograms(x)
        else:
            x.copy_(seg)
            gsort.segmented_sort_(x.view(-1, 1024))

    for _ in range(a.warmup):
        once()
    times = []
    for _ in range(a.reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        once()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    if a.time:
        ms = float(np.median(times))
        print(f"{a.op} {a.kind if a.op == 'sort' else ''} desc={a.desc} values={a.values}: "
              f"median {ms:.4f} ms per call over {a.reps}, {n / ms / 1e6:.2f} Gkeys/s")
    print(f"{a.op}: n=2^{a.n_log2} warmup={a.warmup} reps={a.reps} variant={a.variant} "
          f"({_lib.load().gsort_radix_variant_name(a.variant).decode()}) ok")
    return 0


if __name__ == "__main__":
    sys.exit(main())
