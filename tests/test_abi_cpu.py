"""Host-side checks of the C ABI that need no GPU: the library builds for
sm_103a, loads, exports every function include/mxfp8.h declares, and rejects
bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "mxfp8.h")


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if not n.startswith("__")))


@pytest.fixture(scope="module")
def lib():
    from mxfp8_precision_gemms_gb300 import _build
    _build.build()
    import mxfp8_precision_gemms_gb300 as m
    return m.lib()


def test_header_declares_the_boundary():
    names = header_functions()
    for n in ("fp8_quantize_mx", "fp8_quantize_tensor", "fp8_scaled_gemm", "fp8_grouped_gemm",
              "fp8_quantize_mx_grouped", "mxfp8_scale_bytes", "mxfp8_last_device_status"):
        assert n in names


def test_library_exports_every_header_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_scale_bytes_matches_oracle(lib):
    import oracle
    for rows, k in ((1, 32), (128, 128), (129, 4096), (8192, 4096), (4096, 8192), (300, 96)):
        assert lib.mxfp8_scale_bytes(rows, k) == oracle.scale_bytes(rows, k)
    assert lib.mxfp8_scale_bytes(0, 128) == 0
    assert lib.mxfp8_grouped_scale_bytes(1000, 256, 4) == (1000 // 128 + 1 + 4) * 2 * 512


def test_host_validation(lib):
    import mxfp8_precision_gemms_gb300 as m
    P = 0x10000  # an aligned fake device address: never dereferenced on these paths
    # null input
    assert lib.fp8_quantize_mx(None, 64, 64, 64, m.MX_ROWWISE, P, P, None, None, None) == m.MXFP8_ERR_INVALID_ARG
    # no orientation / unknown flags
    assert lib.fp8_quantize_mx(P, 64, 64, 64, 0, P, P, None, None, None) == m.MXFP8_ERR_INVALID_ARG
    assert lib.fp8_quantize_mx(P, 64, 64, 64, 9, P, P, None, None, None) == m.MXFP8_ERR_INVALID_ARG
    # cols % 32, colwise rows % 32
    assert lib.fp8_quantize_mx(P, 64, 48, 48, m.MX_ROWWISE, P, P, None, None, None) == m.MXFP8_ERR_UNSUPPORTED_SHAPE
    assert lib.fp8_quantize_mx(P, 48, 64, 64, m.MX_COLWISE, None, None, P, P, None) == m.MXFP8_ERR_UNSUPPORTED_SHAPE
    # misaligned pointer / stride
    assert lib.fp8_quantize_mx(P + 2, 64, 64, 64, m.MX_ROWWISE, P, P, None, None, None) == m.MXFP8_ERR_MISALIGNED
    assert lib.fp8_quantize_mx(P, 64, 64, 68, m.MX_ROWWISE, P, P, None, None, None) == m.MXFP8_ERR_MISALIGNED
    # empty input is a no-op
    assert lib.fp8_quantize_mx(None, 0, 64, 64, m.MX_ROWWISE, None, None, None, None, None) == m.MXFP8_OK
    # per-tensor
    assert lib.fp8_quantize_tensor(P, 100, 7, P, P, P, None, None) == m.MXFP8_ERR_INVALID_ARG
    assert lib.fp8_quantize_tensor(P, 100, 0, None, P, P, None, None) == m.MXFP8_ERR_INVALID_ARG
    assert lib.fp8_quantize_tensor(P + 1, 100, 0, P, P, P, None, None) == m.MXFP8_ERR_MISALIGNED
    assert lib.fp8_quantize_tensor(P, 100, 0, P, P, P, P + 8, None) == m.MXFP8_ERR_MISALIGNED
    assert lib.mxfp8_tensor_workspace_bytes() >= 8
    # batched per-tensor
    B = lib.fp8_quantize_tensor_batch
    xs = (ctypes.c_void_p * 17)(*([P] * 17))
    ns = (ctypes.c_int64 * 17)(*([64] * 17))
    arr = lambda a: ctypes.cast(a, ctypes.c_void_p)
    assert B(0, arr(xs), arr(ns), 0, P, P, arr(xs), P, None) == m.MXFP8_ERR_UNSUPPORTED_SHAPE
    assert B(17, arr(xs), arr(ns), 0, P, P, arr(xs), P, None) == m.MXFP8_ERR_UNSUPPORTED_SHAPE
    assert B(2, arr(xs), arr(ns), 3, P, P, arr(xs), P, None) == m.MXFP8_ERR_INVALID_ARG
    assert B(2, None, arr(ns), 0, P, P, arr(xs), P, None) == m.MXFP8_ERR_INVALID_ARG
    assert B(2, arr(xs), arr(ns), 0, P, P, arr(xs), None, None) == m.MXFP8_ERR_INVALID_ARG
    assert B(2, arr(xs), arr(ns), 0, P, P, arr(xs), P + 4, None) == m.MXFP8_ERR_MISALIGNED
    bad = (ctypes.c_void_p * 2)(P, P + 2)
    assert B(2, arr(bad), arr(ns), 0, P, P, arr(xs), P, None) == m.MXFP8_ERR_MISALIGNED
    neg = (ctypes.c_int64 * 2)(64, -1)
    assert B(2, arr(xs), arr(neg), 0, P, P, arr(xs), P, None) == m.MXFP8_ERR_INVALID_ARG
    # batched MX
    QB = lib.fp8_quantize_mx_batch
    r64 = (ctypes.c_int64 * 3)(64, 64, 64)
    c48 = (ctypes.c_int64 * 3)(64, 48, 64)
    r48 = (ctypes.c_int64 * 3)(64, 48, 64)
    l60 = (ctypes.c_int64 * 3)(64, 64, 60)
    fl = lambda *v: arr((ctypes.c_uint * 3)(*v))
    R, C, F = m.MX_ROWWISE, m.MX_COLWISE, m.MX_SCALE_FLOOR
    qs = arr(xs)
    assert QB(3, arr(xs), arr(r64), arr(r64), arr(r64), fl(R, 0, R), qs, qs, qs, qs, None) == m.MXFP8_ERR_INVALID_ARG
    assert QB(3, arr(xs), arr(r64), arr(r64), arr(r64), fl(R, 9, R), qs, qs, qs, qs, None) == m.MXFP8_ERR_INVALID_ARG
    assert QB(3, arr(xs), arr(r64), arr(r64), arr(r64), fl(R, R | F, R), qs, qs, qs, qs, None) == m.MXFP8_ERR_INVALID_ARG
    assert QB(0, arr(xs), arr(r64), arr(r64), arr(r64), fl(R, R, R), qs, qs, qs, qs, None) == m.MXFP8_ERR_UNSUPPORTED_SHAPE
    assert QB(17, arr(xs), arr(r64), arr(r64), arr(r64), fl(R, R, R), qs, qs, qs, qs, None) == m.MXFP8_ERR_UNSUPPORTED_SHAPE
    assert QB(3, arr(xs), arr(r64), arr(c48), arr(r64), fl(R, R, R), qs, qs, qs, qs, None) == m.MXFP8_ERR_UNSUPPORTED_SHAPE
    assert QB(3, arr(xs), arr(r48), arr(r64), arr(r64), fl(R, C, R), qs, qs, qs, qs, None) == m.MXFP8_ERR_UNSUPPORTED_SHAPE
    assert QB(3, arr(xs), arr(r64), arr(r64), arr(l60), fl(R, R, R), qs, qs, qs, qs, None) == m.MXFP8_ERR_INVALID_ARG
    assert QB(3, arr(xs), arr(r64), arr(r64), arr(r64), fl(R, R, R), None, qs, qs, qs, None) == m.MXFP8_ERR_INVALID_ARG
    assert QB(3, arr(xs), arr(r64), arr(r64), arr(r64), fl(R, C, R), qs, qs, None, None, None) == m.MXFP8_ERR_INVALID_ARG
    assert QB(3, arr(xs), arr(r64), arr(r64), arr(r64), None, qs, qs, qs, qs, None) == m.MXFP8_ERR_INVALID_ARG
    bad3 = (ctypes.c_void_p * 3)(P, P, P + 8)
    assert QB(3, arr(bad3), arr(r64), arr(r64), arr(r64), fl(R, R, R), qs, qs, qs, qs, None) == m.MXFP8_ERR_MISALIGNED
    z3 = (ctypes.c_int64 * 3)(0, 0, 0)
    assert QB(3, arr(xs), arr(z3), arr(r64), arr(r64), fl(R, C, R | C), None, None, None, None, None) == m.MXFP8_OK
    # GEMM
    G = lib.fp8_scaled_gemm
    assert G(5, 0, 0, P, P, P, P, 128, 128, 128, P, 128, None) == m.MXFP8_ERR_INVALID_ARG
    assert G(m.GEMM_MX, 1, 0, P, P, P, P, 128, 128, 128, P, 128, None) == m.MXFP8_ERR_UNSUPPORTED_SHAPE
    assert G(m.GEMM_MX, 0, 0, P, P, P, P, 128, 128, 48, P, 128, None) == m.MXFP8_ERR_UNSUPPORTED_SHAPE
    assert G(m.GEMM_MX, 0, 0, P, P, P, P, 128, 132, 128, P, 136, None) == m.MXFP8_ERR_MISALIGNED
    assert G(m.GEMM_MX, 0, 0, None, P, P, P, 128, 128, 128, P, 128, None) == m.MXFP8_ERR_INVALID_ARG
    assert G(m.GEMM_MX, 0, 0, P, P, P, P, 128, 128, 128, P, 64, None) == m.MXFP8_ERR_INVALID_ARG
    assert G(m.GEMM_MX, 0, 0, P + 16, P + 8, P, P, 128, 128, 128, P, 128, None) == m.MXFP8_ERR_MISALIGNED
    assert G(m.GEMM_MX, 0, 0, P, P, P, P, 0, 128, 128, P, 128, None) == m.MXFP8_OK
    # the pair: either problem's bad argument fails the call before any launch
    GP = lib.fp8_scaled_gemm_pair
    good = (0, 0, P, P, P, P, 128, 128, 128, P, 128)
    assert GP(5, *good, *good, None) == m.MXFP8_ERR_INVALID_ARG
    assert GP(m.GEMM_MX, *good, 0, 0, P, P, P, P, 128, 128, 48, P, 128, None) == m.MXFP8_ERR_UNSUPPORTED_SHAPE
    assert GP(m.GEMM_MX, 1, 0, P, P, P, P, 128, 128, 128, P, 128, *good, None) == m.MXFP8_ERR_UNSUPPORTED_SHAPE
    assert GP(m.GEMM_MX, *good, 0, 0, P, P, P, P, 128, 132, 128, P, 136, None) == m.MXFP8_ERR_MISALIGNED
    assert GP(m.GEMM_MX, *good, 0, 0, None, P, P, P, 128, 128, 128, P, 128, None) == m.MXFP8_ERR_INVALID_ARG
    # both empty: nothing to launch
    empty = (0, 0, P, P, P, P, 0, 128, 128, P, 128)
    assert GP(m.GEMM_MX, *empty, *empty, None) == m.MXFP8_OK
    # grouped
    GG = lib.fp8_grouped_gemm
    assert GG(P, P, P, P, P, 0, 128, 128, 128, P, 128, None) == m.MXFP8_ERR_INVALID_ARG
    assert GG(P, P, P, P, P, 2000, 128, 128, 128, P, 128, None) == m.MXFP8_ERR_UNSUPPORTED_SHAPE
    assert GG(P, P, P, P, None, 4, 128, 128, 128, P, 128, None) == m.MXFP8_ERR_INVALID_ARG
    assert GG(P, P, P, P, P, 4, 128, 128, 96 + 16, P, 128, None) == m.MXFP8_ERR_UNSUPPORTED_SHAPE
    assert lib.fp8_quantize_mx_grouped(P, 128, 64, 64, P, 4, m.MX_COLWISE, P, P, None) == m.MXFP8_ERR_INVALID_ARG
    assert lib.fp8_quantize_mx_grouped(P, 128, 64, 64, P, 0, 0, P, P, None) == m.MXFP8_ERR_INVALID_ARG
    # route weighting with the routing per token: k in 1..16, cols <= 2^30,
    # rowwise flags only, routing tables given (all checked before any device access)
    WT = lib.fp8_route_weight_quantize_mx_tokens
    assert WT(P, 64, 2048, 0, P, P, 512, 2048, None, 0, 0, P, P, None) == m.MXFP8_ERR_UNSUPPORTED_SHAPE
    assert WT(P, 64, 2048, 17, P, P, 512, 2048, None, 0, 0, P, P, None) == m.MXFP8_ERR_UNSUPPORTED_SHAPE
    assert WT(P, 64, (1 << 30) + 32, 8, P, P, 512, (1 << 30) + 32, None, 0, 0, P, P,
              None) == m.MXFP8_ERR_UNSUPPORTED_SHAPE
    assert WT(P, 64, 2048, 8, P, P, 512, 2048, None, 0, m.MX_COLWISE, P, P, None) == m.MXFP8_ERR_INVALID_ARG
    assert WT(P, 64, 2048, 8, None, P, 512, 2048, None, 0, 0, P, P, None) == m.MXFP8_ERR_INVALID_ARG
    # every failure leaves a message; status strings exist
    assert lib.mxfp8_last_error()
    for s in range(7):
        assert lib.mxfp8_status_string(s)


def test_ops_fail_loudly_without_cuda_tensors(lib):
    import torch
    import mxfp8_precision_gemms_gb300 as m
    x = torch.zeros(32, 32, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        m.fp8_quantize_mx(x)
