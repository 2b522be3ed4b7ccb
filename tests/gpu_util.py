"""Helpers for the GPU parity tests: device copies, guarded outputs and the tolerance check."""

from __future__ import annotations

import numpy as np
import torch

SENTINEL = np.array([0x7FC0DEAD], np.uint32).view(np.float32)[0]  # a NaN no kernel writes
PAD = 64  # guard floats on each side of an output


def cu(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


class Guarded:
    """An output buffer with sentinel-filled guard zones on both sides (catches out-of-bounds writes)."""

    def __init__(self, *shape):
        n = int(np.prod(shape))
        self.n, self.shape = n, shape
        self.buf = torch.full((n + 2 * PAD,), float(SENTINEL), dtype=torch.float32, device="cuda")
        self.buf.view(torch.int32).fill_(int(np.array([SENTINEL]).view(np.int32)[0]))
        self.t = self.buf[PAD:PAD + n].view(*shape)

    def result(self) -> np.ndarray:
        torch.cuda.synchronize()
        host = self.buf.cpu().numpy()
        guard = np.concatenate([host[:PAD], host[PAD + self.n:]]).view(np.uint32)
        assert np.all(guard == np.uint32(0x7FC0DEAD)), "a kernel wrote outside its output"
        return host[PAD:PAD + self.n].reshape(self.shape)


def assert_close(y, ref, bound, what=""):
    """|y - ref| <= 1e-3 * bound + 1e-5 element-wise (bound = sum_k |w_k| |x_k| from the oracle)."""
    y = np.asarray(y, np.float64)
    assert y.shape == ref.shape, (y.shape, ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    err = np.abs(y - ref)
    lim = 1e-3 * bound + 1e-5
    bad = err > lim
    if np.any(bad):
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; first at {i}: got {y.flat[i]!r}, "
                             f"oracle {ref.flat[i]!r}, limit {lim.flat[i]:.3e}")
