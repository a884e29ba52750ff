"""Helpers shared by the GPU parity tests (no method arithmetic here)."""
import numpy as np
import pytest
import torch

import mxfp8_precision_gemms_gb300 as m


def device():
    if not torch.cuda.is_available():
        pytest.fail("this test needs a CUDA GPU")
    return torch.device("cuda:0")


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    """numpy uint16 BF16 bit patterns -> CUDA bf16 tensor."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device())


def to_dev_u8(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(device())


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def filled(shape, value, dtype=torch.uint8):
    """Device buffer pre-filled with a sentinel, to catch bytes the kernel skipped."""
    return torch.full(shape if isinstance(shape, tuple) else (shape,), value, dtype=dtype,
                      device=device())


def assert_ok():
    st = m.mxfp8_last_device_status()
    assert st == m.MXFP8_OK, m.mxfp8_status_string(st)


def gemm_tolerance_check(gpu_bf16: torch.Tensor, ref: np.ndarray, what=""):
    """|gpu - ref| <= 1e-2 |ref| + 1e-3 rms(ref), elementwise."""
    g = gpu_bf16.float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    err = np.abs(g - ref)
    bound = 1e-2 * np.abs(ref) + 1e-3 * rms
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; first at {tuple(i)}: "
            f"gpu={g[tuple(i)]!r} ref={ref[tuple(i)]!r} rms={rms:.4g}")
    return float((err / np.maximum(bound, 1e-300)).max()) if ref.size else 0.0
