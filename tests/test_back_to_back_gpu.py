"""Back-to-back quantize -> GEMM pairs on one stream.

The GEMMs are launched with programmatic stream serialization: a GEMM may
start while the quantizer before it on the stream is finishing, and waits for
that kernel's results after its prologue.  Each case enqueues several
quantize -> GEMM pairs that reuse one quantized-operand buffer, with no
synchronization in between, then recomputes every pair on its own (after a
device synchronization) and requires the same output bit for bit.  A GEMM
that read its operands, scales, per-tensor scale scalars or group offsets
before the kernel before it had finished would see the previous pair's
bytes; the rounds' inputs differ, so their outputs differ too (checked)."""
import pytest
import torch

import mxfp8_precision_gemms_gb300 as m
from gpu_util import assert_ok, device

pytestmark = pytest.mark.gpu

ROUNDS = 6


def _randn(shape, seed, scale=1.0):
    g = torch.Generator(device=device()).manual_seed(seed)
    return (torch.randn(shape, generator=g, device=device()) * scale).to(torch.bfloat16)


def _same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def _check_rounds(outs, alone):
    for i, (c, r) in enumerate(zip(outs, alone)):
        assert _same(c, r), f"round {i}: the back-to-back GEMM differs from the same GEMM run alone"
    assert not _same(outs[0], outs[1])


def test_mx_pairs_reuse_one_operand_buffer():
    dev = device()
    M, N, K = 2048, 1024, 4096
    xs = [_randn((M, K), 100 + i, 1.0 + i) for i in range(ROUNDS)]
    qw = m.fp8_quantize_mx(_randn((N, K), 7, 0.02))
    q = torch.empty((M, K), dtype=torch.uint8, device=dev)
    s = torch.empty(m.mxfp8_scale_bytes(M, K), dtype=torch.uint8, device=dev)
    outs = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(ROUNDS)]
    torch.cuda.synchronize()
    for i in range(ROUNDS):
        m.fp8_quantize_mx(xs[i], m.MX_ROWWISE, q_row=q, s_row=s)
        m.fp8_scaled_gemm(m.GEMM_MX, q, s, qw["q_row"], qw["s_row"], c=outs[i])
    torch.cuda.synchronize()
    assert_ok()
    alone = []
    for i in range(ROUNDS):
        qi = m.fp8_quantize_mx(xs[i])
        torch.cuda.synchronize()
        alone.append(m.fp8_scaled_gemm(m.GEMM_MX, qi["q_row"], qi["s_row"], qw["q_row"], qw["s_row"]))
        torch.cuda.synchronize()
    _check_rounds(outs, alone)


def test_per_tensor_pairs_reuse_payloads_and_scales():
    """The GEMM's epilogue reads the per-tensor scales the cooperative
    quantizer just wrote; each round scales X differently."""
    dev = device()
    n = 2048
    xs = [_randn((n, n), 200 + i, 0.5 * (i + 1)) for i in range(ROUNDS)]
    w = _randn((n, n), 9, 0.02)
    ws = torch.zeros(m.mxfp8_tensor_workspace_bytes(), dtype=torch.uint8, device=dev)
    qs = [torch.empty((n, n), dtype=torch.uint8, device=dev) for _ in range(2)]
    amax = torch.empty(2, dtype=torch.float32, device=dev)
    scale = torch.empty(2, dtype=torch.float32, device=dev)
    outs = [torch.empty((n, n), dtype=torch.bfloat16, device=dev) for _ in range(ROUNDS)]
    torch.cuda.synchronize()
    for i in range(ROUNDS):
        m.fp8_quantize_tensor_batch([xs[i], w], workspace=ws, qs=qs, amax=amax, scale=scale)
        m.fp8_scaled_gemm(m.GEMM_TENSOR, qs[0], scale[0:1], qs[1], scale[1:2], c=outs[i])
    torch.cuda.synchronize()
    assert_ok()
    alone = []
    for i in range(ROUNDS):
        (qx, qw), _, sc = m.fp8_quantize_tensor_batch([xs[i], w], workspace=ws)
        torch.cuda.synchronize()
        alone.append(m.fp8_scaled_gemm(m.GEMM_TENSOR, qx, sc[0:1], qw, sc[1:2]))
        torch.cuda.synchronize()
    _check_rounds(outs, alone)


def test_grouped_pairs_reuse_one_operand_buffer():
    dev = device()
    counts = [300, 0, 1000, 129, 2, 617]
    N, K = 512, 1024
    G = len(counts)
    off = torch.tensor([0] + list(torch.tensor(counts).cumsum(0).tolist()), dtype=torch.int32,
                       device=dev)
    total = sum(counts)
    xs = [_randn((total, K), 300 + i, 1.0 + 0.25 * i) for i in range(ROUNDS)]
    wd = _randn((G * N, K), 11, 0.02)
    qw = torch.empty((G, N, K), dtype=torch.uint8, device=dev)
    sb = m.mxfp8_scale_bytes(N, K)
    sw = torch.empty(G * sb, dtype=torch.uint8, device=dev)
    for g in range(G):
        m.fp8_quantize_mx(wd[g * N:(g + 1) * N], m.MX_ROWWISE, q_row=qw[g], s_row=sw[g * sb:(g + 1) * sb])
    q = torch.empty((total, K), dtype=torch.uint8, device=dev)
    s = torch.empty(m.mxfp8_grouped_scale_bytes(total, K, G), dtype=torch.uint8, device=dev)
    outs = [torch.empty((total, N), dtype=torch.bfloat16, device=dev) for _ in range(ROUNDS)]
    torch.cuda.synchronize()
    for i in range(ROUNDS):
        m.fp8_quantize_mx_grouped(xs[i], off, q=q, s=s)
        m.fp8_grouped_gemm(q, s, qw, sw, off, c=outs[i])
    torch.cuda.synchronize()
    assert_ok()
    alone = []
    for i in range(ROUNDS):
        qi, si = m.fp8_quantize_mx_grouped(xs[i], off)
        torch.cuda.synchronize()
        alone.append(m.fp8_grouped_gemm(qi, si, qw, sw, off))
        torch.cuda.synchronize()
    _check_rounds(outs, alone)


def test_backward_pairs_reuse_both_orientations():
    """The backward step: dY quantized both ways into reused buffers, then the
    dgrad + wgrad launch (fp8_scaled_gemm_pair) reading both orientations."""
    dev = device()
    T, din, dout = 1024, 768, 512
    dys = [_randn((T, dout), 400 + i, 1e-3 * (i + 1)) for i in range(ROUNDS)]
    qw = m.fp8_quantize_mx(_randn((dout, din), 13, 0.02), m.MX_COLWISE)   # W^T rows: din x dout
    qx = m.fp8_quantize_mx(_randn((T, din), 14), m.MX_COLWISE)            # X^T rows: din x T
    q_row = torch.empty((T, dout), dtype=torch.uint8, device=dev)
    s_row = torch.empty(m.mxfp8_scale_bytes(T, dout), dtype=torch.uint8, device=dev)
    q_col = torch.empty((dout, T), dtype=torch.uint8, device=dev)
    s_col = torch.empty(m.mxfp8_scale_bytes(dout, T), dtype=torch.uint8, device=dev)
    dx = [torch.empty((T, din), dtype=torch.bfloat16, device=dev) for _ in range(ROUNDS)]
    dw = [torch.empty((dout, din), dtype=torch.bfloat16, device=dev) for _ in range(ROUNDS)]
    torch.cuda.synchronize()
    for i in range(ROUNDS):
        m.fp8_quantize_mx(dys[i], m.MX_ROWWISE | m.MX_COLWISE, q_row=q_row, s_row=s_row,
                          q_col=q_col, s_col=s_col)
        m.fp8_scaled_gemm_pair(
            m.GEMM_MX,
            dict(a=q_row, a_scale=s_row, b=qw["q_col"], b_scale=qw["s_col"], c=dx[i]),
            dict(a=q_col, a_scale=s_col, b=qx["q_col"], b_scale=qx["s_col"], c=dw[i]))
    torch.cuda.synchronize()
    assert_ok()
    alone_dx, alone_dw = [], []
    for i in range(ROUNDS):
        qd = m.fp8_quantize_mx(dys[i], m.MX_ROWWISE | m.MX_COLWISE)
        torch.cuda.synchronize()
        a, b = m.fp8_scaled_gemm_pair(
            m.GEMM_MX,
            dict(a=qd["q_row"], a_scale=qd["s_row"], b=qw["q_col"], b_scale=qw["s_col"]),
            dict(a=qd["q_col"], a_scale=qd["s_col"], b=qx["q_col"], b_scale=qx["s_col"]))
        torch.cuda.synchronize()
        alone_dx.append(a)
        alone_dw.append(b)
    _check_rounds(dx, alone_dx)
    _check_rounds(dw, alone_dw)
