"""The allocation-free per-tensor entry point, fp8_quantize_tensor_noalloc.

It serves callers that cannot allocate device memory when they quantize: its
scratch is a static array inside the library instead of a workspace the
caller passes.  Through the C ABI, calls in a row (the array keeps the
previous call's contents, which the entry point must clear) must give the
oracle's bytes, amax and scale, and the same as fp8_quantize_tensor; n = 0
and odd n included.  This file is collected last so that a failure here
never hides the other tests' results; it passes both on its own in a fresh
process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import mxfp8_precision_gemms_gb300 as m
import oracle
import workloads

pytestmark = pytest.mark.gpu


def _call(fn, L, x, fmt, extra=()):
    n = x.numel()
    dev = torch.device("cuda:0")
    q = torch.full((max(n, 1),), 0xA5, dtype=torch.uint8, device=dev)
    amax = torch.full((1,), -1.0, dtype=torch.float32, device=dev)
    scale = torch.full((1,), -1.0, dtype=torch.float32, device=dev)
    st = fn(x.data_ptr() if n else None, n, fmt, amax.data_ptr(), scale.data_ptr(), q.data_ptr(),
            *extra, torch.cuda.current_stream().cuda_stream)
    assert st == m.MXFP8_OK, m.mxfp8_last_error()
    assert m.mxfp8_last_device_status() == m.MXFP8_OK
    return (q.cpu().numpy()[:n], amax.cpu().numpy().view(np.uint32)[0],
            scale.cpu().numpy().view(np.uint32)[0])


@pytest.mark.parametrize("fmt", [m.FP8_E4M3, m.FP8_E5M2])
def test_noalloc_matches_oracle_and_existing_entry_point(fmt):
    assert torch.cuda.is_available()
    dev = torch.device("cuda:0")
    L = m.lib()
    # different tensors in a row: no call may see the previous call's amax
    # (the large, outlier-scaled one first, then smaller ones)
    xs = [workloads.tensor4096(seed=7, device=dev, m=1024, n=8, k=2048)["X"].reshape(-1),
          workloads.normal((777, 40), 1e-3, 8, 0, device=dev).reshape(-1),
          workloads.normal((4099,), 3.0, 9, 0, device=dev),
          torch.empty(0, dtype=torch.bfloat16, device=dev),
          workloads.normal((1, 7), 0.5, 10, 0, device=dev).reshape(-1)]
    for x in xs:
        got = _call(L.fp8_quantize_tensor_noalloc, L, x, fmt)
        ref = _call(L.fp8_quantize_tensor, L, x, fmt, extra=(None,))
        a, s, q = oracle.quantize_tensor(workloads.bits(x), fmt)
        assert np.array_equal(got[0], q), x.numel()
        assert got[1] == np.float32(a).view(np.uint32), x.numel()
        assert got[2] == np.float32(s).view(np.uint32), x.numel()
        assert np.array_equal(got[0], ref[0]) and got[1:] == ref[1:], x.numel()
