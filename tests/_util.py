"""Helpers shared by the tests (no quantization or GEMM arithmetic here)."""
from __future__ import annotations

import numpy as np
import pytest
import torch


def u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (on the CPU)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().view(np.uint8)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def sizes_to_ends(sizes) -> np.ndarray:
    return np.cumsum(np.asarray(sizes, dtype=np.int64))


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    major, minor = torch.cuda.get_device_capability()
    if (major, minor) != (10, 3):
        pytest.skip("kernels are built for sm_103a only")


# The GEMM acceptance bound: |gpu - o| <= 1e-2 |o| + 1e-3 rms(o), elementwise,
# against the fp64 oracle o; rms over the whole reference tensor (or the sample).
REL_TOL = 1e-2
RMS_TOL = 1e-3


def assert_gemm_close(gpu: np.ndarray, ref: np.ndarray, rms: float | None = None, what: str = ""):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape
    if rms is None:
        rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    bound = REL_TOL * np.abs(ref) + RMS_TOL * rms
    err = np.abs(gpu - ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        msg = ", ".join(f"{tuple(i)}: gpu={gpu[tuple(i)]:.6g} ref={ref[tuple(i)]:.6g}" for i in idx)
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} outside tolerance (rms={rms:.3g}); {msg}")


def sqnr_db(ref: np.ndarray, got: np.ndarray) -> float:
    num = float(np.sum(ref.astype(np.float64) ** 2))
    den = float(np.sum((ref.astype(np.float64) - got.astype(np.float64)) ** 2))
    return float("inf") if den == 0 else 10.0 * np.log10(num / den)
