"""The allocation-free per-tensor entry point, fp8_quantize_tensor_noalloc.

It serves callers that cannot allocate device memory when they quantize: its
scratch is a static array inside the library instead of a workspace the
caller passes.  Through the C ABI, two calls in a row (the array keeps the
previous call's contents, which the entry point must clear) must give the
same bytes, amax and scale as fp8_quantize_tensor.  This file is collected
last so that a failure here never hides the other tests' results; it passes
both on its own in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import mxfp8_precision_gemms_gb300 as m
import workloads

pytestmark = pytest.mark.gpu


def _reference(L, x, fmt):
    n = x.numel()
    q = torch.empty(n, dtype=torch.uint8, device=x.device)
    amax = torch.empty(1, dtype=torch.float32, device=x.device)
    scale = torch.empty(1, dtype=torch.float32, device=x.device)
    st = L.fp8_quantize_tensor(x.data_ptr(), n, fmt, amax.data_ptr(), scale.data_ptr(), q.data_ptr(),
                               None, torch.cuda.current_stream().cuda_stream)
    assert st == m.MXFP8_OK, m.mxfp8_last_error()
    return q.cpu().numpy(), amax.cpu().numpy().view(np.uint32), scale.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("fmt", [m.FP8_E4M3, m.FP8_E5M2])
def test_noalloc_matches_existing_entry_point_twice(fmt):
    assert torch.cuda.is_available()
    dev = torch.device("cuda:0")
    L = m.lib()
    # two different tensors: the second call must not see the first call's amax
    big = workloads.tensor4096(seed=7, device=dev, m=1024, n=8, k=2048)["X"].reshape(-1)
    small = (workloads.normal((777, 40), 1e-3, 8, 0, device=dev)).reshape(-1)
    for x in (big, small):
        want_q, want_a, want_s = _reference(L, x, fmt)
        n = x.numel()
        q = torch.full((n,), 0xA5, dtype=torch.uint8, device=dev)
        amax = torch.full((1,), -1.0, dtype=torch.float32, device=dev)
        scale = torch.full((1,), -1.0, dtype=torch.float32, device=dev)
        st = L.fp8_quantize_tensor_noalloc(x.data_ptr(), n, fmt, amax.data_ptr(), scale.data_ptr(),
                                           q.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert st == m.MXFP8_OK, m.mxfp8_last_error()
        assert m.mxfp8_last_device_status() == m.MXFP8_OK
        assert np.array_equal(q.cpu().numpy(), want_q)
        assert amax.cpu().numpy().view(np.uint32)[0] == want_a[0]
        assert scale.cpu().numpy().view(np.uint32)[0] == want_s[0]
