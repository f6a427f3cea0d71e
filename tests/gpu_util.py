"""Shared helpers for the GPU parity tests (tolerances and data movement)."""
import numpy as np
import torch

from tensor_matmul_collective_gb300 import workloads as wl

DEV = torch.device("cuda:0")


def bound(ref: np.ndarray, K: int) -> np.ndarray:
    """Per-element tolerance for fp32-accumulated, 16-bit-rounded outputs:
    |gpu - ref| <= 1e-2 |ref| + 1e-2 sqrt(K / 4096), K the full contraction."""
    return 1e-2 * np.abs(ref) + 1e-2 * np.sqrt(K / 4096.0)


def assert_close(got, ref: np.ndarray, K: int, what: str = "") -> None:
    g = got.detach().to("cpu", torch.float64).numpy() if isinstance(got, torch.Tensor) else got
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - ref)
    b = bound(ref, K)
    bad = err > b
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; first at {tuple(i)}: "
                             f"got {g[tuple(i)]!r} ref {ref[tuple(i)]!r}")
    fro = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30)
    assert fro <= 5e-3, f"{what}: relative Frobenius error {fro:.3g}"


def bits(ts):
    return [wl.bits16(t) for t in ts]


def to_dev(ts):
    return [t.to(DEV) for t in ts]
