"""Benchmark of the sorting path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gsort|reference]

A step is one full LSD radix sort of 2^28 uniform uint32 keys (the problem
the headline metric is quoted on): init, the all-digit histogram and four
single-pass digit scatters (keys only, so the first pass is order-free).
Inputs are resident in HBM and larger than L2 (1 GiB of keys), so no flush is
needed between steps.  The JSON line also carries:
  roofline      the dominant kernel, k_digit_pass (digit passes 2-4):
                algorithmic bytes (4 B read + 4 B written per key) / its
                mean CUDA-event time, against the measured HBM copy bandwidth;
  first_pass    the same for k_digit_pass_free (the order-free first pass);
  sort_roofline the whole sort: 32 B per key (4 passes x 8 B) / step time;
  e2e           the same sort through the C ABI from pinned host buffers
                (host->device copy, sort, device->host copy in the timed region);
                e2e.overlapped: a double-buffered stream of such sorts, whose
                uploads, sorts and downloads overlap across steps;
  rows          the other problem configurations (pairs 2^24, float pairs 2^26,
                low-entropy 2^28 keys, 16384 x 1024 segments, 2^28 compaction);
  cpu_baseline  the CPU oracle (one core) sorting all 2^28 keys of the same
                workload on this host, repeated for about --cpu-seconds.
--impl reference times the CPU oracle alone, each step one sort of the same
2^28 keys (--ref-sample-log2 to sort a prefix instead; rank 0 only).  With --gpus N > 1 (torchrun) every rank sorts its own
2^28 keys (independent replicas, no collective on the data path); value is the
keys of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Gkeys/s for 2^28 uint32 keys & 2^24 k/v pairs; % of HBM roofline (ncu)"
WORKLOAD = "uniform_u32_2^28"
PASSES = 4
WORKLOAD_TEXT = (f"{WORKLOAD}: stable LSD radix sort of 2^28 uniform uint32 keys, keys only, "
                 "8-bit digits (4 passes)")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def traffic_record(kernel: str):
    """Per-launch DRAM bytes from a committed ncu capture, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    import hashlib
    h = hashlib.sha256()
    for rel in rec.get("sources", []):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    if h.hexdigest() != rec.get("source_sha256"):
        return None
    return rec


class Clocks:
    """nvidia-smi sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def reduce_max_ms(ms: float, dist, device) -> float:
    """The slowest rank's time (every rank gets it); ms itself without a process group."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(ms_per_step: float, keys_per_rank: int, world: int) -> float:
    """Whole-job Gkeys/s: the keys of all ranks over the slowest rank's step time."""
    return world * keys_per_rank / (ms_per_step * 1e-3) / 1e9


def time_oracle_sort(keys: np.ndarray, min_seconds: float, max_reps: int):
    import oracle
    reps, t_total = 0, 0.0
    while reps < max_reps and (reps == 0 or t_total < min_seconds):
        t0 = time.perf_counter()
        oracle.radix_sort_keys(keys)
        t_total += time.perf_counter() - t0
        reps += 1
    return keys.size * reps / t_total / 1e9, reps, t_total


def run_reference(args):
    """The CPU oracle as the reference arm: each step sorts the workload's first
    2^ref_sample_log2 keys (all of them by default)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from bitonic_networks_gb300 import synth
    w = synth.WORKLOADS[WORKLOAD]
    sample = 1 << args.ref_sample_log2
    keys = synth.make_keys(w["gen"], sample, w["seed"])
    import oracle
    oracle.build()
    for _ in range(args.warmup):
        oracle.radix_sort_keys(keys[: sample >> 4])
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.radix_sort_keys(keys)
        times.append(time.perf_counter() - t0)
    t = sum(times) / len(times)
    value = sample / t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "Gkeys/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u32", "data": "synthetic",
        "config": ({"workload": WORKLOAD_TEXT, "n": sample} if sample == w["n"] else
                   {"workload": f"{WORKLOAD} keys-only stable LSD radix sort, CPU oracle "
                                f"on a {sample}-key sample", "n": sample}),
        "cpu_baseline": {"value": value, "unit": "Gkeys/s", "cores": 1, "kind": "oracle",
                         "sample": f"first {sample} keys of the {WORKLOAD} workload per step, one core"},
        "e2e": {"value": value, "unit": "Gkeys/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gsort", choices=["gsort", "reference"])
    ap.add_argument("--variant", type=int, default=0)
    ap.add_argument("--no-rows", action="store_true", help="time only the headline sort")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-sample-log2", type=int, default=28)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "gsort":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args)

    import torch
    from bitonic_networks_gb300 import _lib, gsort, synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    device = torch.device("cuda", torch.cuda.current_device())
    lib = _lib.load()
    stream = torch.cuda.current_stream()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    w = synth.WORKLOADS[WORKLOAD]
    n = w["n"]
    keys_h = synth.make_keys(w["gen"], n, w["seed"] + 1000 * rank)
    keys = torch.from_numpy(keys_h.view(np.int32)).to(device)
    out = torch.empty_like(keys)
    ws = torch.empty(gsort.radix_workspace_bytes(n, False), dtype=torch.uint8, device=device)
    nev = 3 + PASSES

    def sort_once(events=None):
        ev_arr = None
        if events is not None:
            ev_arr = (ctypes.c_void_p * nev)(*[e.cuda_event for e in events])
        opt = _lib.Options(0, -1, ctypes.cast(ev_arr, ctypes.POINTER(ctypes.c_void_p))
                           if ev_arr is not None else None, nev if events else 0, args.variant)
        rc = lib.gsort_radix_pairs_ex(keys.data_ptr(), out.data_ptr(), None, None, n, 0, 0, 32,
                                      ws.data_ptr(), ws.numel(), stream.cuda_stream,
                                      ctypes.byref(opt))
        if rc != 0:
            raise gsort.GsortError(rc, "gsort_radix_pairs_ex")

    for _ in range(args.warmup):
        sort_once()
    if lib.gsort_check(ws.data_ptr(), stream.cuda_stream) != 0:
        raise RuntimeError("device-side error during warm-up")

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(args.steps)]
    for evs in events:          # torch creates the CUDA event on its first record
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize()
    clocks = Clocks(device.index)
    barrier()
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(args.steps):
        sort_once(events[s])
    t_end.record(stream)
    barrier()
    clk = clocks.stop()
    status = lib.gsort_check(ws.data_ptr(), stream.cuda_stream)
    if status != 0:
        raise RuntimeError(f"device-side error in the timed region: {status}")
    ms_total = reduce_max_ms(t_start.elapsed_time(t_end), dist, device)
    ms_step = ms_total / args.steps
    value = job_throughput(ms_step, n, world)

    pass_ms = [events[s][2 + p].elapsed_time(events[s][3 + p])
               for s in range(args.steps) for p in range(PASSES)]
    hist_ms = [events[s][1].elapsed_time(events[s][2]) for s in range(args.steps)]
    init_ms = [events[s][0].elapsed_time(events[s][1]) for s in range(args.steps)]
    pass_mean = sum(pass_ms) / len(pass_ms)
    # the first pass of this keys-only sort runs k_digit_pass_free, the other
    # three k_digit_pass (the dominant kernel: three launches per sort)
    each = [sum(pass_ms[s * PASSES + p] for s in range(args.steps)) / args.steps for p in range(PASSES)]
    stable_mean = sum(each[1:]) / (PASSES - 1)
    hbm_peak, peak_src = peaks()
    pass_bytes = 8 * n
    achieved = pass_bytes / (stable_mean * 1e-3) / 1e9
    first_gbs = pass_bytes / (each[0] * 1e-3) / 1e9
    trec = traffic_record("digit_pass")
    frec = traffic_record("digit_pass_free")
    sort_gbs = 32 * n / (ms_step * 1e-3) / 1e9

    # correctness spot check of the timed output (sorted, same multiset as a sample)
    o = out[: 1 << 20].cpu().view(torch.int32).numpy().view(np.uint32)
    assert np.all(o[1:] >= o[:-1]), "timed output is not sorted"

    line = {
        "metric": METRIC, "value": value, "unit": "Gkeys/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT,
                   "n": n, "variant": lib.gsort_radix_variant_name(args.variant).decode(),
                   "l2": "inputs larger than L2 (1 GiB keys + 1 GiB ping-pong), no flush",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "kernel": "k_digit_pass (digit passes 2-4 of the sort)",
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "peak_source": peak_src,
                     "traffic": (trec["dram_bytes_per_launch"] * n / trec["n"]) if trec else None,
                     "algorithmic_bytes_per_launch": pass_bytes,
                     "mean_launch_ms": stable_mean},
        "first_pass": {"kernel": "k_digit_pass_free (order-free first digit pass)",
                       "achieved": first_gbs, "peak": hbm_peak, "unit": "GB/s",
                       "frac": first_gbs / hbm_peak,
                       "traffic": (frec["dram_bytes_per_launch"] * n / frec["n"]) if frec else None,
                       "algorithmic_bytes_per_launch": pass_bytes, "launch_ms": each[0]},
        "sort_roofline": {"achieved": sort_gbs, "peak": hbm_peak, "unit": "GB/s",
                          "frac": sort_gbs / hbm_peak, "bytes_per_step": 32 * n,
                          "note": "32 B/key = 4 passes x (4 B read + 4 B written); the "
                                  "histogram read (4 B/key) is spent but not counted"},
        "kernels_ms": {"init": sum(init_ms) / len(init_ms), "histogram": sum(hist_ms) / len(hist_ms),
                       "digit_pass": pass_mean, "digit_pass_each": each},
        "gpu_launches": args.steps * lib.gsort_radix_launch_count(n, 0, 32, 0),
        "clocks": clk,
    }

    if rank == 0 and not args.no_e2e:
        line["e2e"] = e2e(lib, gsort, keys_h, n, device, stream, args)
    if rank == 0 and not args.no_rows:
        del keys, out, ws
        torch.cuda.empty_cache()
        line["rows"] = rows(lib, gsort, synth, device, stream, args, hbm_peak)
    if rank == 0 and not args.no_cpu:
        # the whole workload (every key of the timed sort), sorted once or more
        gk, reps, secs = time_oracle_sort(keys_h, args.cpu_seconds, 50)
        line["cpu_baseline"] = {"value": gk, "unit": "Gkeys/s", "cores": 1, "kind": "oracle",
                                "sample": f"all {n} keys of the {WORKLOAD} workload, "
                                          f"sorted {reps} times ({secs:.1f} s)",
                                "nproc": os.cpu_count()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def e2e(lib, gsort, keys_h, n, device, stream, args):
    """Host buffers through the C ABI: pinned H2D copy, sort, D2H copy."""
    import torch
    hin = torch.from_numpy(keys_h.view(np.int32)).pin_memory()
    hout = torch.empty_like(hin).pin_memory()
    din = torch.empty(n, dtype=torch.int32, device=device)
    dout = torch.empty_like(din)
    ws = torch.empty(gsort.radix_workspace_bytes(n, False), dtype=torch.uint8, device=device)

    def step():
        din.copy_(hin, non_blocking=True)
        rc = lib.gsort_radix_keys(din.data_ptr(), dout.data_ptr(), n, 0, ws.data_ptr(),
                                  ws.numel(), stream.cuda_stream)
        if rc != 0:
            raise gsort.GsortError(rc, "gsort_radix_keys")
        hout.copy_(dout, non_blocking=True)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    steps = max(3, min(args.steps, 10))
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    res = hout[: 1 << 16].numpy().view(np.uint32)
    assert np.all(res[1:] >= res[:-1]), "e2e output is not sorted"
    out = {"value": n / (ms * 1e-3) / 1e9, "unit": "Gkeys/s", "ms_per_step": ms,
           "h2d_bytes_per_step": 4 * n, "d2h_bytes_per_step": 4 * n}
    out["overlapped"] = e2e_overlapped(lib, gsort, hin, n, device, stream, ws, steps, args.warmup)
    return out


def e2e_overlapped(lib, gsort, hin, n, device, stream, ws, steps, warmup):
    """A stream of sorts from host memory: the same calls and copies per step,
    double-buffered, so that step i+1's upload runs beside step i's sort and
    step i-1's download (uploads, sorts and downloads on three streams, ordered
    by events).  Every step still copies its whole input in and its whole
    result out inside the timed region."""
    import torch
    up = torch.cuda.Stream(device)
    down = torch.cuda.Stream(device)
    din = [torch.empty(n, dtype=torch.int32, device=device) for _ in range(2)]
    dout = [torch.empty(n, dtype=torch.int32, device=device) for _ in range(2)]
    hout = [torch.empty_like(hin).pin_memory() for _ in range(2)]
    ev = lambda: torch.cuda.Event()
    uploaded = [ev(), ev()]
    sorted_ = [ev(), ev()]
    downloaded = [ev(), ev()]
    used = [False, False]

    def step(i):
        j = i % 2
        with torch.cuda.stream(up):
            if used[j]:
                up.wait_event(sorted_[j])          # the sort of step i-2 has read din[j]
            din[j].copy_(hin, non_blocking=True)
            uploaded[j].record(up)
        stream.wait_event(uploaded[j])
        if used[j]:
            stream.wait_event(downloaded[j])       # the download of step i-2 has read dout[j]
        rc = lib.gsort_radix_keys(din[j].data_ptr(), dout[j].data_ptr(), n, 0, ws.data_ptr(),
                                  ws.numel(), stream.cuda_stream)
        if rc != 0:
            raise gsort.GsortError(rc, "gsort_radix_keys")
        sorted_[j].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(sorted_[j])
            hout[j].copy_(dout[j], non_blocking=True)
            downloaded[j].record(down)
        used[j] = True

    for i in range(max(3, warmup)):
        step(i)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    up.wait_event(a)
    down.wait_event(a)
    for i in range(steps):
        step(i)
    stream.wait_event(downloaded[(steps - 1) % 2])
    stream.wait_event(downloaded[steps % 2])
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    for h in hout:
        res = h[: 1 << 16].numpy().view(np.uint32)
        assert np.all(res[1:] >= res[:-1]), "overlapped e2e output is not sorted"
    return {"value": n / (ms * 1e-3) / 1e9, "unit": "Gkeys/s", "ms_per_step": ms,
            "h2d_bytes_per_step": 4 * n, "d2h_bytes_per_step": 4 * n,
            "note": "double-buffered stream of sorts: uploads, sorts and downloads on three streams"}


def _median_ms(fn, stream, warm, reps):
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def rows(lib, gsort, synth, device, stream, args, peak):
    """One line per problem configuration (median of reps, CUDA events)."""
    import torch
    out = {}
    reps = max(5, args.steps)
    warm = max(3, args.warmup)

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(device)

    def sort_row(name, with_values, kind):
        w = synth.WORKLOADS[name]
        n = w["n"]
        k = dev(synth.make_keys(w["gen"], n, w["seed"]))
        ko = torch.empty_like(k)
        v = vo = None
        if with_values:
            v = dev(synth.index_values(n))
            vo = torch.empty_like(v)
        ws = torch.empty(gsort.radix_workspace_bytes(n, with_values), dtype=torch.uint8,
                         device=device)

        def fn():
            rc = lib.gsort_radix_pairs(k.data_ptr(), ko.data_ptr(),
                                       v.data_ptr() if v is not None else None,
                                       vo.data_ptr() if vo is not None else None, n, kind, 0, 32,
                                       ws.data_ptr(), ws.numel(), stream.cuda_stream)
            assert rc == 0
        ms = _median_ms(fn, stream, warm, reps)
        assert lib.gsort_check(ws.data_ptr(), stream.cuda_stream) == 0
        byts = (16 if with_values else 8) * PASSES * n
        gbs = byts / (ms * 1e-3) / 1e9
        out[name] = {"n": n, "ms": ms, "Gkeys/s": n / (ms * 1e-3) / 1e9, "GB/s": gbs,
                     "frac": gbs / peak, "bytes": byts}

    sort_row("pairs_u32_2^24", True, 0)
    sort_row("normal_f32_pairs_2^26", True, 1)
    sort_row("and3_u32_2^28", False, 0)
    sort_row("distinct16_u32_2^28", False, 0)
    sort_row("uniform_u32_65536", False, 0)
    torch.cuda.empty_cache()

    w = synth.WORKLOADS["segments_16384x1024"]
    segs = dev(synth.segments(w["segments"], w["length"], w["seed"]))
    work = segs.clone()

    def seg_fn():
        work.copy_(segs)
        rc = lib.gsort_segmented_bitonic(work.data_ptr(), w["segments"], w["length"],
                                         stream.cuda_stream)
        assert rc == 0
    ms_copy = _median_ms(lambda: work.copy_(segs), stream, warm, reps)
    ms = _median_ms(seg_fn, stream, warm, reps) - ms_copy
    n = w["n"]
    gbs = 8 * n / (ms * 1e-3) / 1e9
    ce = 55 * 512 * w["segments"]
    out["segments_16384x1024"] = {"n": n, "ms": ms, "Gkeys/s": n / (ms * 1e-3) / 1e9,
                                  "GB/s": gbs, "frac": gbs / peak,
                                  "compare_exchanges_per_s": ce / (ms * 1e-3),
                                  "note": "time of the restoring copy subtracted"}
    del segs, work
    torch.cuda.empty_cache()

    w = synth.WORKLOADS["compact_f32_2^28"]
    n = w["n"]
    x = dev(synth.make_keys(w["gen"], n, w["seed"]))
    o = torch.empty_like(x)
    nk = torch.empty(1, dtype=torch.int64, device=device)
    ws = torch.empty(gsort.compact_workspace_bytes(n), dtype=torch.uint8, device=device)

    def cfn():
        rc = lib.gsort_compact_positive(x.data_ptr(), o.data_ptr(), n, nk.data_ptr(),
                                        ws.data_ptr(), ws.numel(), stream.cuda_stream)
        assert rc == 0
    ms = _median_ms(cfn, stream, warm, reps)
    assert lib.gsort_check(ws.data_ptr(), stream.cuda_stream) == 0
    gbs = 8 * n / (ms * 1e-3) / 1e9
    out["compact_f32_2^28"] = {"n": n, "ms": ms, "Gkeys/s": n / (ms * 1e-3) / 1e9, "GB/s": gbs,
                               "frac": gbs / peak}
    del x, o, ws
    torch.cuda.empty_cache()

    # next rows: 64-bit keys, variable-length segments, 2-way split, 1-bit split sort
    w = synth.WORKLOADS["uniform_u64_2^27"]
    n = w["n"]
    k = torch.from_numpy(synth.make_keys(w["gen"], n, w["seed"]).view(np.int64)).to(device)
    ko = torch.empty_like(k)
    ws = torch.empty(lib.gsort_radix_sort_workspace_bytes(n, 3, 0), dtype=torch.uint8, device=device)

    def u64_fn():
        assert lib.gsort_radix_sort(k.data_ptr(), ko.data_ptr(), None, None, n, 3, 0, 0, 64,
                                    ws.data_ptr(), ws.numel(), stream.cuda_stream) == 0
    ms = _median_ms(u64_fn, stream, warm, reps)
    assert lib.gsort_check(ws.data_ptr(), stream.cuda_stream) == 0
    byts = 16 * 8 * n
    out["uniform_u64_2^27"] = {"n": n, "ms": ms, "Gkeys/s": n / (ms * 1e-3) / 1e9,
                               "GB/s": byts / (ms * 1e-3) / 1e9,
                               "frac": byts / (ms * 1e-3) / 1e9 / peak, "bytes": byts}
    del k, ko, ws
    torch.cuda.empty_cache()

    w = synth.WORKLOADS["segments_mixed_2^26"]
    n = w["n"]
    k = dev(synth.make_keys(w["gen"], n, w["seed"]))
    off_np = synth.segment_offsets(n, w["mix"], w["seed"])
    off = dev(off_np)
    ko = torch.empty_like(k)
    S = off_np.size - 1
    ws = torch.empty(lib.gsort_segmented_sort_workspace_bytes(n, S, 0), dtype=torch.uint8,
                     device=device)

    def seg_var_fn():
        assert lib.gsort_segmented_sort(k.data_ptr(), ko.data_ptr(), None, None, n, off.data_ptr(),
                                        S, 0, 0, ws.data_ptr(), ws.numel(), stream.cuda_stream) == 0
    ms = _median_ms(seg_var_fn, stream, warm, reps)
    assert lib.gsort_check(ws.data_ptr(), stream.cuda_stream) == 0
    lens = np.diff(off_np.astype(np.int64))
    n_small = int(lens[lens <= 1024].sum())
    byts = 8 * n_small + 32 * (n - n_small)   # one read + write for short segments, 4 passes for long
    out["segments_mixed_2^26"] = {"n": n, "segments": S, "keys_in_short_segments": n_small,
                                  "ms": ms, "Gkeys/s": n / (ms * 1e-3) / 1e9,
                                  "GB/s": byts / (ms * 1e-3) / 1e9,
                                  "frac": byts / (ms * 1e-3) / 1e9 / peak, "bytes": byts}
    del k, ko, off, ws
    torch.cuda.empty_cache()

    w = synth.WORKLOADS["partition_f32_2^28"]
    n = w["n"]
    x = dev(synth.make_keys(w["gen"], n, w["seed"]))
    o = torch.empty_like(x)
    nt = torch.empty(1, dtype=torch.int64, device=device)
    ws = torch.empty(lib.gsort_partition_workspace_bytes(n), dtype=torch.uint8, device=device)

    def part_fn():
        assert lib.gsort_partition(x.data_ptr(), o.data_ptr(), None, None, n, 4, 1, 0, None,
                                   nt.data_ptr(), ws.data_ptr(), ws.numel(), stream.cuda_stream) == 0
    ms = _median_ms(part_fn, stream, warm, reps)
    assert lib.gsort_check(ws.data_ptr(), stream.cuda_stream) == 0
    byts = 8 * n
    out["partition_f32_2^28"] = {"n": n, "ms": ms, "Gkeys/s": n / (ms * 1e-3) / 1e9,
                                 "GB/s": byts / (ms * 1e-3) / 1e9,
                                 "frac": byts / (ms * 1e-3) / 1e9 / peak, "bytes": byts,
                                 "note": "bytes = one read and one write; the counting read adds 4 B/element"}
    del x, o, ws
    torch.cuda.empty_cache()

    w = synth.WORKLOADS["split_sort_u32_2^25"]
    n = w["n"]
    k = dev(synth.make_keys(w["gen"], n, w["seed"]))
    ko = torch.empty_like(k)
    ws = torch.empty(lib.gsort_split_sort_workspace_bytes(n, 0), dtype=torch.uint8, device=device)

    def split_fn():
        assert lib.gsort_split_sort(k.data_ptr(), ko.data_ptr(), None, None, n, 0, 32,
                                    ws.data_ptr(), ws.numel(), stream.cuda_stream) == 0
    ms = _median_ms(split_fn, stream, warm, reps)
    assert lib.gsort_check(ws.data_ptr(), stream.cuda_stream) == 0
    byts = 8 * 32 * n
    out["split_sort_u32_2^25"] = {"n": n, "ms": ms, "Gkeys/s": n / (ms * 1e-3) / 1e9,
                                  "GB/s": byts / (ms * 1e-3) / 1e9,
                                  "frac": byts / (ms * 1e-3) / 1e9 / peak, "bytes": byts}
    return out


if __name__ == "__main__":
    sys.exit(main())
