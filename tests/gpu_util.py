"""Helpers shared by the GPU parity tests: moving synthetic inputs to the
device, reading results back, and the floating-point acceptance rule."""
from __future__ import annotations

import numpy as np
import pytest
import torch

# Elementwise acceptance for floating-point outputs against the float64
# oracle: |gpu - ref| <= TOL * (|ref| + rms(ref)), rms over the whole output.
TOL = 1e-2


def require_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def bf(a: np.ndarray, dev) -> torch.Tensor:
    """uint16 bf16 bit patterns -> torch.bfloat16 tensor on dev."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)


def u8(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(dev)


def i32(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns on the host."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(gpu: np.ndarray, ref: np.ndarray, tol: float = TOL, what: str = "") -> None:
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    err = np.abs(gpu - ref)
    bound = tol * (np.abs(ref) + rms)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {err.size} outside tolerance; worst at {i}: "
                             f"gpu={gpu[i]!r} ref={ref[i]!r} bound={bound[i]!r} rms={rms!r}")
