"""The allocation-free compaction entry point, called through the C ABI.

gsort_compact_positive_noalloc serves callers that cannot give the library a
workspace (code that runs where device allocation is forbidden or too costly);
its scratch is a static device array inside libgsort.  This test checks that
it returns exactly what the workspace-taking entry point returns, on two calls
in a row (the second call reuses the array the first one left behind), and
that sizes beyond its stated maximum are refused.  The file name makes pytest
collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from bitonic_networks_gb300 import _lib, gsort, synth
from gpu_util import assert_bits_equal, dev, host_u32

pytestmark = pytest.mark.gpu

MAX_N = 1 << 28          # GSORT_COMPACT_NOALLOC_MAX_N
ETOOBIG = -4


def noalloc(x: torch.Tensor):
    lib = _lib.load()
    n = x.numel()
    out = torch.full((n,), 7.0, dtype=torch.float32, device=x.device)
    kept = torch.full((1,), -1, dtype=torch.int64, device=x.device)
    rc = lib.gsort_compact_positive_noalloc(x.data_ptr(), out.data_ptr(), n, kept.data_ptr(),
                                            torch.cuda.current_stream().cuda_stream)
    assert rc == 0, lib.gsort_status_string(rc)
    torch.cuda.synchronize()
    return out, int(kept.item())


@pytest.mark.parametrize("n", [1, 8193, 3 * 8192 + 5, 1_000_003])
def test_noalloc_matches_workspace_entry_point_twice(n):
    for call, seed in enumerate((900 + n, 901 + n)):
        x = dev(synth.compaction_input(n, seed))
        exp, exp_kept = gsort.compact_positive(x)
        got, got_kept = noalloc(x)
        assert got_kept == int(exp_kept.item()), f"call {call}"
        assert_bits_equal(host_u32(got), host_u32(exp), f"n={n} call {call}")


def test_noalloc_refuses_more_than_its_maximum():
    lib = _lib.load()
    x = torch.zeros(4, dtype=torch.float32, device="cuda")
    rc = lib.gsort_compact_positive_noalloc(x.data_ptr(), x.data_ptr() + 1024, MAX_N + 1, None,
                                            torch.cuda.current_stream().cuda_stream)
    assert rc == ETOOBIG
