"""Small helpers shared by the GPU parity tests (no method arithmetic)."""
import numpy as np
import torch


def dev(a: np.ndarray) -> torch.Tensor:
    """numpy 32-bit array -> CUDA tensor with the same bytes (uint32 -> int32 view)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a.copy()).cuda()


def host_u32(t: torch.Tensor) -> np.ndarray:
    """CUDA tensor -> numpy uint32 bit patterns."""
    return t.detach().cpu().contiguous().view(torch.int32).numpy().view(np.uint32)


def assert_bits_equal(got: np.ndarray, exp: np.ndarray, what: str = ""):
    got = np.asarray(got).view(np.uint32).ravel()
    exp = np.asarray(exp).view(np.uint32).ravel()
    assert got.shape == exp.shape, f"{what}: shape {got.shape} != {exp.shape}"
    if not np.array_equal(got, exp):
        bad = np.flatnonzero(got != exp)
        i = int(bad[0])
        raise AssertionError(f"{what}: {bad.size} mismatches, first at {i}: "
                             f"got 0x{int(got[i]):08x} expected 0x{int(exp[i]):08x}")


def offset_view(t: torch.Tensor, n: int, off: int) -> torch.Tensor:
    """A length-n view of a fresh buffer starting `off` elements in (for
    pointers that are 4-byte but not 16-byte aligned)."""
    buf = torch.empty(n + off + 4, dtype=t.dtype, device=t.device)
    v = buf[off:off + n]
    v.copy_(t)
    return v
