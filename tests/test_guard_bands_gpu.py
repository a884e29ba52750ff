"""Guard bands around every output: the stand-in for a memory sanitizer
(compute-sanitizer is not available).  Each output buffer is the interior of
a larger allocation whose 512 bytes on either side hold a fill pattern; for
outputs with a row stride wider than the row (C with ldc > N, BF16 output
with ld > cols) the gap between rows is guarded too.  After every call the
guards must be untouched.  Shapes are ragged (partial tiles, partial 32-row
groups, partial K and N tiles) so that every edge of every kernel's index
arithmetic is exercised; the values themselves are checked by the parity
tests."""
import numpy as np
import pytest
import torch

import mxfp8_precision_gemms_gb300 as m
import workloads
from gpu_util import assert_ok, device, to_dev_bf16

pytestmark = pytest.mark.gpu

GUARD = 512   # bytes on each side: keeps every alignment the library needs
PAT = 0xC3


class Guarded:
    """An output tensor of `shape` and `dtype` (rows padded to `ld` elements
    when given) inside a pattern-filled allocation."""

    def __init__(self, shape, dtype=torch.uint8, ld=None):
        shape = shape if isinstance(shape, tuple) else (shape,)
        esize = torch.empty((), dtype=dtype).element_size()
        if ld is not None:
            assert len(shape) == 2 and ld >= shape[1]
            inner = shape[0] * ld * esize
        else:
            inner = int(np.prod(shape)) * esize
        self.inner = inner
        self.raw = torch.full((2 * GUARD + inner,), PAT, dtype=torch.uint8, device=device())
        body = self.raw[GUARD:GUARD + inner].view(dtype)
        if ld is not None:
            self.full = body.view(shape[0], ld)
            self.t = self.full[:, :shape[1]]
            self.cols = shape[1]
        else:
            self.full = None
            self.t = body.view(shape)

    def check(self, what):
        r = self.raw.cpu().numpy()
        assert np.all(r[:GUARD] == PAT), f"{what}: bytes written before the buffer"
        assert np.all(r[GUARD + self.inner:] == PAT), f"{what}: bytes written after the buffer"
        if self.full is not None and self.full.shape[1] > self.cols:
            gap = self.full[:, self.cols:].contiguous().view(torch.uint8).cpu().numpy()
            assert np.all(gap == PAT), f"{what}: bytes written between rows"


def bits(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return workloads.bits((torch.randn(*shape, generator=g) * scale).to(torch.bfloat16))


def check_all(outs, what):
    torch.cuda.synchronize()
    assert_ok()
    for name, g in outs.items():
        g.check(f"{what} {name}")


@pytest.mark.parametrize("rows,cols", [(192, 160), (1056, 96), (32, 4128), (4128, 160)])
@pytest.mark.parametrize("flags", [m.MX_ROWWISE, m.MX_COLWISE, m.MX_ROWWISE | m.MX_COLWISE])
def test_quantize_mx(rows, cols, flags):
    x = to_dev_bf16(bits((rows, cols), rows + cols))
    o = {}
    if flags & m.MX_ROWWISE:
        o["q_row"], o["s_row"] = Guarded((rows, cols)), Guarded(m.mxfp8_scale_bytes(rows, cols))
    if flags & m.MX_COLWISE:
        o["q_col"], o["s_col"] = Guarded((cols, rows)), Guarded(m.mxfp8_scale_bytes(cols, rows))
    m.fp8_quantize_mx(x, flags, **{k: g.t for k, g in o.items()})
    check_all(o, f"quantize_mx {rows}x{cols} flags {flags}")


def test_quantize_mx_grouped():
    counts = [0, 1, 127, 128, 129, 0, 300, 5]
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    total, cols = int(off[-1]), 96
    x = to_dev_bf16(bits((total, cols), 3))
    o = {"q": Guarded((total, cols)), "s": Guarded(m.mxfp8_grouped_scale_bytes(total, cols, len(counts)))}
    m.fp8_quantize_mx_grouped(x, torch.from_numpy(off).to(device()), q=o["q"].t, s=o["s"].t)
    check_all(o, "quantize_mx_grouped")


def test_quantize_mx_batch():
    shapes = [(192, 160), (100, 96), (32, 4128), (64, 32)]
    flags = [m.MX_ROWWISE | m.MX_COLWISE, m.MX_ROWWISE, m.MX_COLWISE, m.MX_COLWISE]
    xs = [to_dev_bf16(bits(sh, 10 + i)) for i, sh in enumerate(shapes)]
    guards, outs = {}, []
    for i, ((r, c), f) in enumerate(zip(shapes, flags)):
        o = {}
        if f & m.MX_ROWWISE:
            o["q_row"], o["s_row"] = Guarded((r, c)), Guarded(m.mxfp8_scale_bytes(r, c))
        if f & m.MX_COLWISE:
            o["q_col"], o["s_col"] = Guarded((c, r)), Guarded(m.mxfp8_scale_bytes(c, r))
        guards.update({f"{i} {k}": g for k, g in o.items()})
        outs.append({k: g.t for k, g in o.items()})
    m.fp8_quantize_mx_batch(xs, flags, outs=outs)
    check_all(guards, "quantize_mx_batch")


@pytest.mark.parametrize("n", [1, 15, 1000003])
def test_quantize_tensor(n):
    x = to_dev_bf16(bits((n,), n))
    for ws in (None, torch.zeros(m.mxfp8_tensor_workspace_bytes(), dtype=torch.uint8, device=device())):
        o = {"q": Guarded((n,)), "amax": Guarded((1,), torch.float32), "scale": Guarded((1,), torch.float32)}
        m.fp8_quantize_tensor(x, m.FP8_E4M3, q=o["q"].t, amax=o["amax"].t, scale=o["scale"].t, workspace=ws)
        check_all(o, f"quantize_tensor n={n} workspace={ws is not None}")


def test_quantize_tensor_batch():
    ns = [1, 17, 4099, 65536]
    xs = [to_dev_bf16(bits((n,), 20 + n)) for n in ns]
    o = {f"q{i}": Guarded((n,)) for i, n in enumerate(ns)}
    o["amax"], o["scale"] = Guarded((len(ns),), torch.float32), Guarded((len(ns),), torch.float32)
    m.fp8_quantize_tensor_batch(xs, m.FP8_E5M2, qs=[o[f"q{i}"].t for i in range(len(ns))],
                                amax=o["amax"].t, scale=o["scale"].t)
    check_all(o, "quantize_tensor_batch")


def test_scaled_and_delayed_casts():
    n = 100003
    x = to_dev_bf16(bits((n,), 5, 40.0))
    s = torch.tensor([2.0], dtype=torch.float32, device=device())
    o = {"q": Guarded((n,)), "amax": Guarded((1,), torch.float32), "sat": Guarded((1,), torch.int64)}
    m.fp8_quantize_tensor_scaled(x, s, m.FP8_E5M2, q=o["q"].t, amax=o["amax"].t, sat_count=o["sat"].t)
    check_all(o, "quantize_tensor_scaled")
    hist = Guarded((16,), torch.float32)
    hist.t.zero_()
    pos = Guarded((1,), torch.int32)
    pos.t.zero_()
    o = {"q": Guarded((n,)), "scale": Guarded((1,), torch.float32), "amax": Guarded((1,), torch.float32),
         "sat": Guarded((1,), torch.int64), "history": hist, "pos": pos}
    for _ in range(3):
        m.fp8_quantize_tensor_delayed(x, hist.t, pos.t, m.FP8_E4M3, q=o["q"].t, scale=o["scale"].t,
                                      amax=o["amax"].t, sat_count=o["sat"].t)
    check_all(o, "quantize_tensor_delayed")
    q_in = o["q"].t.clone()
    o2 = {"out": Guarded((n,)), "sat": Guarded((1,), torch.int64)}
    m.fp8_requantize_tensor(q_in, s, s * 0.5, m.FP8_E4M3, m.FP8_E5M2, out=o2["out"].t, sat_count=o2["sat"].t)
    check_all(o2, "requantize_tensor")


@pytest.mark.parametrize("M,N,K,ldc", [(200, 136, 96, 136), (130, 264, 4096, 272), (300, 512, 384, 520),
                                       (1000, 1024, 160, 1032), (1, 8, 32, 8)])
def test_mx_gemm(M, N, K, ldc):
    a = m.fp8_quantize_mx(to_dev_bf16(bits((M, K), 1)), m.MX_ROWWISE)
    b = m.fp8_quantize_mx(to_dev_bf16(bits((N, K), 2)), m.MX_ROWWISE)
    c = Guarded((M, N), torch.bfloat16, ld=ldc)
    m.fp8_scaled_gemm(m.GEMM_MX, a["q_row"], a["s_row"], b["q_row"], b["s_row"], c=c.t)
    check_all({"C": c}, f"mx gemm {M}x{N}x{K} ldc {ldc}")


def test_tensor_gemm():
    M, N, K = 260, 200, 256
    qa, _, sa = m.fp8_quantize_tensor(to_dev_bf16(bits((M, K), 3)))
    qb, _, sb = m.fp8_quantize_tensor(to_dev_bf16(bits((N, K), 4)))
    c = Guarded((M, N), torch.bfloat16, ld=208)
    m.fp8_scaled_gemm(m.GEMM_TENSOR, qa.view(M, K), sa, qb.view(N, K), sb, c=c.t)
    check_all({"C": c}, "tensor gemm")


def test_grouped_gemm_and_routed_conversions():
    counts = [40, 0, 300, 129, 1]
    G, N, K = len(counts), 256, 384
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    off_d = torch.from_numpy(off).to(device())
    total = int(off[-1])
    qa, sa = m.fp8_quantize_mx_grouped(to_dev_bf16(bits((total, K), 5)), off_d)
    qw = m.fp8_quantize_mx(to_dev_bf16(bits((G * N, K), 6)), m.MX_ROWWISE)
    c = Guarded((total, N), torch.bfloat16, ld=N + 8)
    m.fp8_grouped_gemm(qa, sa, qw["q_row"].view(G, N, K), qw["s_row"], off_d, c=c.t)
    check_all({"C": c}, "grouped gemm")
    # dequantize (BF16 rows with a wider stride), SwiGLU + quantize, route weighting + quantize
    d = Guarded((total, K), torch.bfloat16, ld=K + 16)
    m.fp8_dequantize_mx(qa, sa, offsets=off_d, out=d.t)
    check_all({"out": d}, "dequantize grouped")
    h = to_dev_bf16(bits((total, 2 * 96), 7, 3.0))
    o = {"q": Guarded((total, 96)), "s": Guarded(m.mxfp8_grouped_scale_bytes(total, 96, G))}
    m.fp8_swiglu_quantize_mx(h, offsets=off_d, q=o["q"].t, s=o["s"].t)
    check_all(o, "swiglu quantize grouped")
    tokens = 97
    dy = to_dev_bf16(bits((tokens, 160), 8))
    rng = np.random.default_rng(9)
    tok = torch.from_numpy(rng.integers(0, tokens, total).astype(np.int32)).to(device())
    wt = torch.from_numpy(rng.random(total).astype(np.float32)).to(device())
    o = {"q": Guarded((total, 160)), "s": Guarded(m.mxfp8_grouped_scale_bytes(total, 160, G))}
    m.fp8_route_weight_quantize_mx(dy, tok, wt, offsets=off_d, q=o["q"].t, s=o["s"].t)
    check_all(o, "route weight quantize grouped")


def test_gemm_pair():
    """Two GEMMs in one launch, both C with a wider row stride."""
    shapes = [((200, 136, 96), 144), ((300, 512, 384), 520)]
    gs, guards = [], {}
    for i, ((M, N, K), ldc) in enumerate(shapes):
        a = m.fp8_quantize_mx(to_dev_bf16(bits((M, K), 30 + i)), m.MX_ROWWISE)
        b = m.fp8_quantize_mx(to_dev_bf16(bits((N, K), 40 + i)), m.MX_ROWWISE)
        c = Guarded((M, N), torch.bfloat16, ld=ldc)
        guards[f"C{i}"] = c
        gs.append(dict(a=a["q_row"], a_scale=a["s_row"], b=b["q_row"], b_scale=b["s_row"], c=c.t))
    m.fp8_scaled_gemm_pair(m.GEMM_MX, gs[0], gs[1])
    check_all(guards, "gemm pair")


def test_route_weight_tokens_grouped():
    """The per-token route weighting: payload rows and the (zeroed first)
    group-padded scale array, with ragged groups and unused route slots."""
    counts = [40, 0, 300, 129, 1]
    G = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    off_d = torch.from_numpy(off).to(device())
    rows, k, cols = int(off[-1]), 4, 160
    tokens = rows // k + 3
    rng = np.random.default_rng(10)
    slots = rng.permutation(tokens * k)[:rows]
    tr = np.full(tokens * k, -1, np.int32)
    tr[slots] = np.arange(rows)
    dy = to_dev_bf16(bits((tokens, cols), 11))
    tw = torch.from_numpy(rng.random((tokens, k)).astype(np.float32)).to(device())
    o = {"q": Guarded((rows, cols)), "s": Guarded(m.mxfp8_grouped_scale_bytes(rows, cols, G))}
    m.fp8_route_weight_quantize_mx_tokens(dy, torch.from_numpy(tr.reshape(tokens, k)).to(device()), tw,
                                          rows, offsets=off_d, q=o["q"].t, s=o["s"].t)
    check_all(o, "route weight quantize per token")
