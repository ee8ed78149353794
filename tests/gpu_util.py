"""Helpers of the GPU parity tests: device copies of the synthetic inputs,
outputs with guard bands, and the tolerance check."""
import numpy as np
import pytest
import torch

SENTINEL = 1234.5
GUARD = 64  # fp32 elements of guard band on each side of an output


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__ as g
    g.build()


def dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to("cuda")


class Guarded:
    """fp32 device output of n elements between two guard bands."""

    def __init__(self, n: int, fill: float = float("nan")):
        self.n = n
        self.buf = torch.full((n + 2 * GUARD,), SENTINEL, dtype=torch.float32, device="cuda")
        self.buf[GUARD:GUARD + n] = fill

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr() + 4 * GUARD

    def get(self) -> np.ndarray:
        b = self.buf.cpu().numpy()
        assert np.all(b[:GUARD] == SENTINEL) and np.all(b[GUARD + self.n:] == SENTINEL), "guard band overwritten"
        return b[GUARD:GUARD + self.n].copy()


def assert_within(y, ref, a, what="", rel=1e-3, absol=1e-6):
    """|y - ref| <= rel * a + absol elementwise (the method's GEMV tolerance)."""
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - ref)
    tol = rel * a + absol
    bad = ~(err <= tol)
    if bad.any():
        i = np.flatnonzero(bad.ravel())[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first {i.tolist()} "
                             f"err {err.ravel()[i].tolist()} tol {tol.ravel()[i].tolist()}")
