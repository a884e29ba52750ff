"""CUDA graphs and streams.  Every entry point is stream-ordered and issues
only kernel launches and memsets on the caller's stream (no allocation, no
synchronization), so a step built from them can be captured once into a CUDA
graph and replayed on new inputs, and independent steps can run on separate
streams at the same time.  Both must give the eager results bit for bit (the
same kernels run on the same bytes); one replay per test is also checked
against the oracle.  Each step runs once eagerly before capture, so
first-use set-up (kernel attributes, occupancy queries) happens outside it."""
import numpy as np
import pytest
import torch

import mxfp8_precision_gemms_gb300 as m
import oracle
from gpu_util import assert_ok, device, gemm_tolerance_check, host

pytestmark = pytest.mark.gpu


def _randn(shape, seed, scale=1.0):
    g = torch.Generator(device=device()).manual_seed(seed)
    return (torch.randn(shape, generator=g, device=device()) * scale).to(torch.bfloat16)


def _bits(t):
    return host(t.contiguous().view(torch.int16)).view(np.uint16)


def _capture(step):
    """Warm up on a side stream, then capture `step` into a graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    return g


def _same(a, b):
    return torch.equal(a.view(torch.uint8), b.view(torch.uint8))


class MxStep:
    """Quantize X and W rowwise (one batched launch), then C = X W^T."""

    def __init__(self, M, N, K):
        u8 = dict(dtype=torch.uint8, device=device())
        self.X = torch.empty((M, K), dtype=torch.bfloat16, device=device())
        self.W = torch.empty((N, K), dtype=torch.bfloat16, device=device())
        self.outs = [{"q_row": torch.empty((M, K), **u8), "s_row": torch.empty(m.mxfp8_scale_bytes(M, K), **u8)},
                     {"q_row": torch.empty((N, K), **u8), "s_row": torch.empty(m.mxfp8_scale_bytes(N, K), **u8)}]
        self.C = torch.empty((M, N), dtype=torch.bfloat16, device=device())

    def __call__(self):
        qx, qw = m.fp8_quantize_mx_batch([self.X, self.W], outs=self.outs)
        m.fp8_scaled_gemm(m.GEMM_MX, qx["q_row"], qx["s_row"], qw["q_row"], qw["s_row"], c=self.C)


def test_graph_replay_mx_quantize_and_gemm():
    M, N, K = 520, 768, 1024
    step = MxStep(M, N, K)
    step.X.copy_(_randn((M, K), 1))
    step.W.copy_(_randn((N, K), 2, 0.05))
    g = _capture(step)
    eager = MxStep(M, N, K)
    for seed in (3, 5, 7):
        x, w = _randn((M, K), seed), _randn((N, K), seed + 1, 0.05)
        step.X.copy_(x)
        step.W.copy_(w)
        g.replay()
        eager.X.copy_(x)
        eager.W.copy_(w)
        eager()
        torch.cuda.synchronize()
        assert_ok()
        for a, b in zip(step.outs, eager.outs):
            assert _same(a["q_row"], b["q_row"]) and _same(a["s_row"], b["s_row"]), seed
        assert _same(step.C, eager.C), seed
    ra = oracle.quantize_mx(_bits(step.X), oracle.ROWWISE)
    rb = oracle.quantize_mx(_bits(step.W), oracle.ROWWISE)
    assert np.array_equal(host(step.outs[0]["q_row"]), ra["q_row"])
    gemm_tolerance_check(step.C, oracle.gemm_mx(ra["q_row"], ra["s_row"], rb["q_row"], rb["s_row"]),
                         "graph replay")


def test_graph_replay_per_tensor_paths():
    """The single-launch per-tensor path (workspace memset + cooperative
    launch), the two-kernel path, the per-tensor GEMM and one delayed-scaling
    cast whose amax history advances on every replay."""
    M, N, K = 384, 256, 512
    X, W = _randn((M, K), 11), _randn((N, K), 12, 0.05)
    u8 = dict(dtype=torch.uint8, device=device())
    f32 = dict(dtype=torch.float32, device=device())
    ws = torch.zeros(m.mxfp8_tensor_workspace_bytes(), **u8)
    qx, qw = torch.empty((M, K), **u8), torch.empty((N, K), **u8)
    amax, scale = torch.empty(2, **f32), torch.empty(2, **f32)
    q2, a2, s2 = torch.empty(M * K, **u8), torch.empty(1, **f32), torch.empty(1, **f32)
    C = torch.empty((M, N), dtype=torch.bfloat16, device=device())
    hist = torch.zeros(8, **f32)
    pos = torch.zeros(1, dtype=torch.int32, device=device())
    qd, sd, ad = torch.empty(M * K, **u8), torch.empty(1, **f32), torch.empty(1, **f32)
    sat = torch.empty(1, dtype=torch.int64, device=device())

    def step():
        m.fp8_quantize_tensor_batch([X, W], m.FP8_E4M3, workspace=ws, qs=[qx, qw], amax=amax, scale=scale)
        m.fp8_quantize_tensor(X.view(-1), m.FP8_E4M3, q=q2, amax=a2, scale=s2)
        m.fp8_scaled_gemm(m.GEMM_TENSOR, qx, scale[0:1], qw, scale[1:2], c=C)
        m.fp8_quantize_tensor_delayed(X.view(-1), hist, pos, m.FP8_E5M2, q=qd, scale=sd, amax=ad, sat_count=sat)

    g = _capture(step)   # the warm-up already recorded one amax in the history
    h0 = host(hist).copy()
    for i in range(3):
        X.copy_(_randn((M, K), 20 + i, 1.0 + i))
        g.replay()
        torch.cuda.synchronize()
        assert_ok()
        wa, wsc, wq = oracle.quantize_tensor(_bits(X).reshape(-1), m.FP8_E4M3)
        assert host(amax)[0] == wa and host(scale)[0] == wsc
        assert np.array_equal(host(qx).reshape(-1), wq) and np.array_equal(host(q2), wq)
        assert host(a2)[0] == wa and host(s2)[0] == wsc
        assert host(pos)[0] == (2 + i) % 8, "the history position advances once per replay"
        assert host(hist)[(1 + i) % 8] == wa
    assert h0[0] != 0
    wb = oracle.quantize_tensor(_bits(W).reshape(-1), m.FP8_E4M3)
    ref = oracle.gemm_tensor(wq.reshape(M, K), m.FP8_E4M3, wsc, wb[2].reshape(N, K), m.FP8_E4M3, wb[1])
    gemm_tolerance_check(C, ref, "per-tensor graph replay")


def test_graph_replay_grouped_and_routed():
    """Grouped quantize + grouped GEMM, then the routed conversions, with the
    expert counts changed between replays (offsets live on the device)."""
    G, N, K, total, f = 4, 256, 256, 600, 128
    u8 = dict(dtype=torch.uint8, device=device())
    off = torch.zeros(G + 1, dtype=torch.int32, device=device())
    X = _randn((total, K), 31)
    Wt = _randn((G * N, K), 32, 0.05)
    qw = m.fp8_quantize_mx(Wt, m.MX_ROWWISE)
    qa = torch.empty((total, K), **u8)
    sa = torch.empty(m.mxfp8_grouped_scale_bytes(total, K, G), **u8)
    C = torch.empty((total, N), dtype=torch.bfloat16, device=device())
    H = _randn((total, 2 * f), 33, 2.0)
    qh, sh = torch.empty((total, f), **u8), torch.empty(m.mxfp8_grouped_scale_bytes(total, f, G), **u8)
    back = torch.empty((total, K), dtype=torch.bfloat16, device=device())
    tok = torch.from_numpy(np.random.default_rng(34).integers(0, 100, total).astype(np.int32)).to(device())
    wt = torch.rand(total, generator=torch.Generator(device=device()).manual_seed(35), device=device())
    dY = _randn((100, K), 36)
    qr, sr = torch.empty((total, K), **u8), torch.empty(m.mxfp8_grouped_scale_bytes(total, K, G), **u8)

    def step():
        m.fp8_quantize_mx_grouped(X, off, q=qa, s=sa)
        m.fp8_grouped_gemm(qa, sa, qw["q_row"].view(G, N, K), qw["s_row"], off, c=C)
        m.fp8_dequantize_mx(qa, sa, offsets=off, out=back)
        m.fp8_swiglu_quantize_mx(H, offsets=off, q=qh, s=sh)
        m.fp8_route_weight_quantize_mx(dY, tok, wt, offsets=off, q=qr, s=sr)

    off.copy_(torch.tensor([0, 150, 300, 450, 600], dtype=torch.int32))
    g = _capture(step)
    for counts in ([0, 300, 1, 299], [600, 0, 0, 0], [129, 128, 127, 216]):
        o = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        off.copy_(torch.from_numpy(o))
        g.replay()
        snap = [t.clone() for t in (qa, sa, C, back, qh, sh, qr, sr)]
        step()   # eager, same inputs
        torch.cuda.synchronize()
        assert_ok()
        for a, b in zip(snap, (qa, sa, C, back, qh, sh, qr, sr)):
            assert _same(a, b), counts
        wq, ws_ = oracle.quantize_mx_grouped(_bits(X), o)
        assert np.array_equal(host(qa), wq) and np.array_equal(host(sa)[:ws_.size], ws_)
        assert np.array_equal(_bits(back), oracle.dequantize_mx_grouped(wq, ws_, o))
        hq, hs = oracle.quantize_mx_grouped(oracle.swiglu_bf16(_bits(H)), o)
        assert np.array_equal(host(qh), hq) and np.array_equal(host(sh)[:hs.size], hs)


def test_two_streams_run_independent_steps():
    """Two MX steps issued alternately on two streams (running concurrently)
    give the same bytes as the same steps run one after the other."""
    shapes = [(700, 512, 768), (256, 1024, 2048)]
    steps = [MxStep(*s) for s in shapes]
    ref = [MxStep(*s) for s in shapes]
    for i, (a, b) in enumerate(zip(steps, ref)):
        x, w = _randn(a.X.shape, 40 + i), _randn(a.W.shape, 50 + i, 0.05)
        a.X.copy_(x); a.W.copy_(w); b.X.copy_(x); b.W.copy_(w)
    for b in ref:
        b()
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    for _ in range(4):
        for st, a in zip(streams, steps):
            with torch.cuda.stream(st):
                a()
    torch.cuda.synchronize()
    assert_ok()
    for a, b in zip(steps, ref):
        assert _same(a.C, b.C)
        for oa, ob in zip(a.outs, b.outs):
            assert _same(oa["q_row"], ob["q_row"]) and _same(oa["s_row"], ob["s_row"])
