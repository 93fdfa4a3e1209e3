"""Helpers shared by the GPU parity tests: host<->device moves of bf16 bit
patterns and the element-wise comparison the tests use.

Tolerances (written here once, used by every GPU parity test):
  FP8 GMM vs the FP8 CPU oracle: atol 1e-3, rtol 1e-2 — the bound that
      "GEMM Kernel 性能优化十问" Q9.2 gives for an FP8 kernel against an FP8 CPU
      reference (only accumulation-order differences allowed).
  bf16 GMM and tgmm vs the fp64 oracle: rtol 1e-2 plus atol 1e-3 (a pure
      relative bound fails on sums that cancel to ~0; the absolute term is far
      below one bf16 ulp of the typical output).
"""
import numpy as np
import torch

FP8_ATOL, FP8_RTOL = 1e-3, 1e-2
BF16_ATOL, BF16_RTOL = 1e-3, 1e-2


def dev():
    return torch.device("cuda:0")


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev())


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def bf16_to_np64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def assert_close(got, ref, atol, rtol, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values in the kernel output"
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    if np.any(bad):
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                             f"first at {tuple(i)}: got {got[tuple(i)]!r} want {ref[tuple(i)]!r}")


def poison_bf16(t: torch.Tensor) -> torch.Tensor:
    """Fill with NaN so that any element a kernel forgets to write shows up."""
    t.view(torch.int16).fill_(0x7FC0)
    return t


GUARD_BYTES = 4096
_GUARD_BEFORE, _GUARD_AFTER = 0xA5, 0x5A


class Guarded:
    """An output tensor with canary bands in front of it and behind it, in
    the same device allocation (the out-of-bounds check that stands in for a
    memory sanitizer): a kernel that writes past either end of its output
    changes a band, and check() then fails.  The tensor starts 4096 bytes
    into the allocation, so it keeps the 16-byte alignment the library needs;
    poison=True fills a bf16 tensor with NaN (unwritten elements show up)."""

    def __init__(self, shape, dtype, poison=True, device="cuda"):
        itemsize = torch.empty((), dtype=dtype).element_size()
        n = int(np.prod(shape)) * itemsize
        self.n = n
        self.raw = torch.empty(2 * GUARD_BYTES + n, dtype=torch.uint8, device=device)
        self.raw[:GUARD_BYTES].fill_(_GUARD_BEFORE)
        self.raw[GUARD_BYTES + n:].fill_(_GUARD_AFTER)
        self.t = self.raw[GUARD_BYTES:GUARD_BYTES + n].view(dtype).view(shape)
        if poison and dtype == torch.bfloat16:
            poison_bf16(self.t)
        elif poison:
            self.t.view(torch.uint8).fill_(0xEE)

    def check(self, what=""):
        torch.cuda.synchronize()
        before = self.raw[:GUARD_BYTES]
        after = self.raw[GUARD_BYTES + self.n:]
        assert torch.all(before == _GUARD_BEFORE), f"{what}: a write landed in the band before the output"
        assert torch.all(after == _GUARD_AFTER), f"{what}: a write landed in the band after the output"
