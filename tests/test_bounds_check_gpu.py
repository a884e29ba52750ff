"""The bounds-checked build (libmxfp8_bc.so, compiled with
-DMXFP8_BOUNDS_CHECK): every global access whose address the kernels compute
is guarded by the extent of the tensor it touches, and a failed check records
MXFP8_ERR_DEVICE_CHECK and skips the access.  Every entry point runs on
ragged shapes through that build: no check may fail, and every output must
equal the product library's bit for bit.  With the guard bands
(test_guard_bands_gpu.py) this stands in for a memory sanitizer, which is not
available here."""
import contextlib

import numpy as np
import pytest
import torch

import mxfp8_precision_gemms_gb300 as m
import workloads
from gpu_util import device
from mxfp8_precision_gemms_gb300 import _build

pytestmark = pytest.mark.gpu

COUNTS = [0, 130, 5, 0, 256, 1]


@contextlib.contextmanager
def library(path):
    """Route the binding's calls to the library at `path`, then back."""
    saved = (m.LIB_PATH, m._lib)
    m.LIB_PATH, m._lib = path, None
    try:
        yield
    finally:
        m.LIB_PATH, m._lib = saved


@pytest.fixture(scope="module")
def checked():
    return _build.build(bounds_check=True)


def same_bytes(a, b):
    a = a.detach().contiguous().view(-1).view(torch.uint8)
    b = b.detach().contiguous().view(-1).view(torch.uint8)
    return torch.equal(a, b)


def run_both(checked, fn):
    """fn() returns output tensors: run it on the bounds-checked build, then
    on the product build, and compare."""
    with library(checked):
        got = [t.clone() for t in fn()]
        st = m.mxfp8_last_device_status()
    want = fn()
    assert st == m.MXFP8_OK, f"an index check failed: {m.mxfp8_status_string(st)}"
    assert len(got) == len(want)
    for i, (a, b) in enumerate(zip(got, want)):
        assert same_bytes(a, b), f"output {i} differs from the product build's"


def bf16(shape, seed, scale=1.0):
    return workloads.normal(shape, scale, seed, 0, device())


def offsets(counts=COUNTS):
    return torch.from_numpy(workloads.offsets_from_counts(np.array(counts))).to(device())


def zeros_u8(n):
    return torch.zeros(max(1, n), dtype=torch.uint8, device=device())


def test_mx_quantizers(checked):
    x = bf16((288, 416), 1)           # colwise needs rows % 32 == 0
    xr = bf16((300, 416), 2)          # rowwise only: a ragged last row tile
    off = offsets()
    xg = bf16((int(off[-1]), 160), 3)

    def fn():
        both = m.fp8_quantize_mx(x, m.MX_ROWWISE | m.MX_COLWISE)
        col = m.fp8_quantize_mx(x, m.MX_COLWISE)
        row = m.fp8_quantize_mx(xr, m.MX_ROWWISE | m.MX_SCALE_FLOOR)
        sg = zeros_u8(m.mxfp8_grouped_scale_bytes(xg.shape[0], 160, len(COUNTS)))
        qg, sg = m.fp8_quantize_mx_grouped(xg, off, s=sg)
        return [both["q_row"], both["s_row"], both["q_col"], both["s_col"], col["q_col"],
                col["s_col"], row["q_row"], row["s_row"], qg, sg]
    run_both(checked, fn)


def test_mx_batches(checked):
    a, b = bf16((300, 416), 4), bf16((64, 96), 5)
    c, d = bf16((288, 416), 6), bf16((96, 128), 7)

    def fn():
        r = m.fp8_quantize_mx_batch([a, b])
        t = m.fp8_quantize_mx_batch([c, d], flags=[m.MX_ROWWISE | m.MX_COLWISE, m.MX_COLWISE])
        return [r[0]["q_row"], r[0]["s_row"], r[1]["q_row"], r[1]["s_row"], t[0]["q_row"],
                t[0]["s_row"], t[0]["q_col"], t[0]["s_col"], t[1]["q_col"], t[1]["s_col"]]
    run_both(checked, fn)


def test_per_tensor(checked):
    x = bf16((7, 1031), 8)            # n odd: the vector loops' scalar tails
    y = bf16((96, 200), 9, 3.0)
    scale = torch.tensor([0.25], dtype=torch.float32, device=device())
    s_out = torch.tensor([0.125], dtype=torch.float32, device=device())

    def fn():
        q1, a1, s1 = m.fp8_quantize_tensor(x, m.FP8_E4M3)
        q2, a2, s2 = m.fp8_quantize_tensor_batch([x, y], m.FP8_E5M2)
        q3, a3, n3 = m.fp8_quantize_tensor_scaled(y, scale, m.FP8_E5M2)
        q4, n4 = m.fp8_requantize_tensor(q1, s1, s_out)
        return [q1, a1, s1, *q2, a2, s2, q3, a3, n3, q4, n4]
    run_both(checked, fn)


def test_routed_conversions(checked):
    off = offsets()
    rows = int(off[-1])
    h = bf16((rows, 320), 12)
    tokens, k = rows // 4 + 3, 4
    dy = bf16((tokens, 160), 13, 1e-3)
    rng = np.random.default_rng(14)
    slots = rng.permutation(tokens * k)[:rows]
    tr = np.full(tokens * k, -1, np.int32)
    tr[slots] = np.arange(rows)
    tw = rng.uniform(0, 1, tokens * k).astype(np.float32)
    row_token = np.full(rows, -1, np.int32)
    row_weight = np.zeros(rows, np.float32)
    row_token[tr[slots]] = slots // k
    row_weight[tr[slots]] = tw[slots]
    tr_d = torch.from_numpy(tr.reshape(tokens, k)).to(device())
    tw_d = torch.from_numpy(tw.reshape(tokens, k)).to(device())
    rt_d = torch.from_numpy(row_token).to(device())
    rw_d = torch.from_numpy(row_weight).to(device())
    xq = bf16((rows, 160), 15)
    plain = bf16((300, 416), 16)

    def fn():
        G = len(COUNTS)
        sq = zeros_u8(m.mxfp8_grouped_scale_bytes(rows, 160, G))
        qq, sq = m.fp8_quantize_mx_grouped(xq, off, s=sq)
        dq = m.fp8_dequantize_mx(qq, sq, offsets=off)
        pq = m.fp8_quantize_mx(plain, m.MX_ROWWISE)
        dp = m.fp8_dequantize_mx(pq["q_row"], pq["s_row"])
        ss = zeros_u8(m.mxfp8_grouped_scale_bytes(rows, 160, G))
        qs, ss = m.fp8_swiglu_quantize_mx(h, offsets=off, s=ss)
        sw = zeros_u8(m.mxfp8_grouped_scale_bytes(rows, 160, G))
        qw, sw = m.fp8_route_weight_quantize_mx(dy, rt_d, rw_d, offsets=off, s=sw)
        qt, st = m.fp8_route_weight_quantize_mx_tokens(dy, tr_d, tw_d, rows, offsets=off)
        qp, sp = m.fp8_route_weight_quantize_mx_tokens(dy, tr_d, tw_d, rows)
        return [dq, dp, qs, ss, qw, sw, qt, st, qp, sp]
    run_both(checked, fn)


def test_gemms(checked):
    a, b = bf16((300, 416), 17), bf16((200, 416), 18, 0.02)
    off = offsets()
    total = int(off[-1])
    ag = bf16((total, 160), 19)
    bg = bf16((len(COUNTS) * 128, 160), 20, 0.02)
    x2, w2 = bf16((257, 320), 21), bf16((384, 320), 22, 0.02)

    def fn():
        qa = m.fp8_quantize_mx(a, m.MX_ROWWISE)
        qb = m.fp8_quantize_mx(b, m.MX_ROWWISE)
        c_mx = m.fp8_scaled_gemm(m.GEMM_MX, qa["q_row"], qa["s_row"], qb["q_row"], qb["s_row"])
        ta, _, sa = m.fp8_quantize_tensor(a)
        tb, _, sb = m.fp8_quantize_tensor(b)
        c_t = m.fp8_scaled_gemm(m.GEMM_TENSOR, ta, sa, tb, sb)
        sg = zeros_u8(m.mxfp8_grouped_scale_bytes(total, 160, len(COUNTS)))
        qg, sg = m.fp8_quantize_mx_grouped(ag, off, s=sg)
        qw = m.fp8_quantize_mx(bg, m.MX_ROWWISE)   # 128 rows per expert: each expert's own layout
        c_g = m.fp8_grouped_gemm(qg, sg, qw["q_row"].view(len(COUNTS), 128, 160), qw["s_row"], off)
        q2 = m.fp8_quantize_mx(x2, m.MX_ROWWISE)
        r2 = m.fp8_quantize_mx(w2, m.MX_ROWWISE)
        p0, p1 = m.fp8_scaled_gemm_pair(
            m.GEMM_MX, dict(a=qa["q_row"], a_scale=qa["s_row"], b=qb["q_row"], b_scale=qb["s_row"]),
            dict(a=q2["q_row"], a_scale=q2["s_row"], b=r2["q_row"], b_scale=r2["s_row"]))
        return [c_mx, c_t, c_g, p0, p1]
    run_both(checked, fn)
