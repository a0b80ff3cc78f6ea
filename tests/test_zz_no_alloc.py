"""The allocation-free compaction entry point, called through the C ABI.

gsort_compact_positive_noalloc serves callers that cannot give the library a
workspace (code that runs where device allocation is forbidden or too costly);
its scratch is a static device array inside libgsort.  These tests check, on
two calls in a row (the second call reuses the array the first one left
behind), that it returns exactly what the workspace-taking entry point returns
and what the CPU oracle's compaction gives, including NaN, both zeros,
subnormals and buffers that are 4-byte but not 16-byte aligned, and that sizes
beyond its stated maximum are refused.  The file name makes pytest collect it
last.
"""
import numpy as np
import pytest
import torch

import oracle
from bitonic_networks_gb300 import _lib, gsort, synth
from gpu_util import assert_bits_equal, dev, host_u32, offset_view

pytestmark = pytest.mark.gpu

MAX_N = 1 << 28          # GSORT_COMPACT_NOALLOC_MAX_N
ETOOBIG = -4


def noalloc(x: torch.Tensor, out_off: int = 0):
    lib = _lib.load()
    n = x.numel()
    out = torch.full((n,), 7.0, dtype=torch.float32, device=x.device)
    if out_off:
        out = offset_view(out, n, out_off)
    kept = torch.full((1,), -1, dtype=torch.int64, device=x.device)
    rc = lib.gsort_compact_positive_noalloc(x.data_ptr(), out.data_ptr(), n, kept.data_ptr(),
                                            torch.cuda.current_stream().cuda_stream)
    assert rc == 0, lib.gsort_status_string(rc)
    torch.cuda.synchronize()
    return out, int(kept.item())


def with_specials(n: int, seed: int) -> np.ndarray:
    x = synth.compaction_input(n, seed)
    b = x.view(np.uint32)
    b[0::11] = 0x7FC00000   # NaN: dropped
    b[1::13] = 0x80000000   # -0: dropped
    b[2::17] = 0x00000001   # +subnormal: kept
    b[3::19] = 0x7F800000   # +inf: kept
    b[4::23] = 0xFF800000   # -inf: dropped
    b[5::29] = 0x80000001   # -subnormal: dropped
    return x


@pytest.mark.parametrize("n", [1, 8193, 3 * 8192 + 5, 1_000_003])
def test_noalloc_matches_workspace_entry_point_and_oracle_twice(n):
    for call, seed in enumerate((900 + n, 901 + n)):
        x_np = with_specials(n, seed)
        x = dev(x_np)
        exp, exp_kept = gsort.compact_positive(x)
        got, got_kept = noalloc(x)
        assert got_kept == int(exp_kept.item()), f"call {call}"
        assert_bits_equal(host_u32(got), host_u32(exp), f"n={n} call {call} vs workspace entry point")
        ora, m = oracle.compact_positive(x_np)
        assert got_kept == m, f"call {call}"
        assert_bits_equal(host_u32(got), ora, f"n={n} call {call} vs oracle")


@pytest.mark.parametrize("offs", [(1, 0), (0, 3), (2, 1)])
def test_noalloc_misaligned_buffers(offs):
    n = 50_001
    for call, seed in enumerate((950, 951)):
        x_np = with_specials(n, seed + offs[0])
        x = offset_view(dev(x_np), n, offs[0]) if offs[0] else dev(x_np)
        got, got_kept = noalloc(x, out_off=offs[1])
        ora, m = oracle.compact_positive(x_np)
        assert got_kept == m, f"{offs} call {call}"
        assert_bits_equal(host_u32(got), ora, f"{offs} call {call} vs oracle")


def test_noalloc_refuses_more_than_its_maximum():
    lib = _lib.load()
    x = torch.zeros(4, dtype=torch.float32, device="cuda")
    rc = lib.gsort_compact_positive_noalloc(x.data_ptr(), x.data_ptr() + 1024, MAX_N + 1, None,
                                            torch.cuda.current_stream().cuda_stream)
    assert rc == ETOOBIG
