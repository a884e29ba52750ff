"""GPU parity of the routed-path conversions around the quantizer:
dequantization, fused SwiGLU + MX quantization (the correctly rounded BF16
hidden value, including values next to a BF16 rounding midpoint) and fused
route weighting + MX gradient quantization, plain and group-padded, on small
ragged shapes and at the workloads' full sizes; every byte against the
oracle."""
import numpy as np
import pytest
import torch

import mxfp8_precision_gemms_gb300 as m
import oracle
import workloads
from gpu_util import assert_ok, device, filled, host, to_dev_bf16, to_dev_u8

pytestmark = pytest.mark.gpu

SHAPES = [(1, 32), (127, 96), (128, 128), (300, 416), (513, 1056)]
GROUP_COUNTS = [[0, 130, 5, 0, 256, 1], [1], [0, 0, 700], [128, 128, 3]]


def _offsets(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


def _random_mx(rows, cols, seed, specials=True):
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 256, size=(rows, cols), dtype=np.uint8)
    if not specials:
        q[(q & 0x7F) == 0x7F] = 0x3C
    s = rng.integers(0, 256 if specials else 255, size=oracle.scale_bytes(rows, cols), dtype=np.uint8)
    return q, s


def _bits_equal_or_both_nan(got, want):
    gn = np.isnan(oracle.bf16_decode(got))
    wn = np.isnan(oracle.bf16_decode(want))
    assert np.array_equal(gn, wn), "NaN positions differ"
    d = (got != want) & ~wn
    assert not d.any(), f"{int(d.sum())} BF16 values differ, first at {np.argwhere(d)[0]}"


# ---------------------------------------------------------- dequantize --

@pytest.mark.parametrize("rows,cols", SHAPES)
def test_dequantize_random_codes_and_scales(rows, cols):
    """Every E4M3 code with every scale byte, including 0 (2^-127), 254
    (overflow to Inf), 255 (NaN) and NaN payload codes."""
    q, s = _random_mx(rows, cols, rows * 7 + cols)
    out = filled((rows, cols + 8), 0x7777, torch.int16).view(torch.bfloat16)
    m.fp8_dequantize_mx(to_dev_u8(q), to_dev_u8(s), out=out[:, :cols])
    assert_ok()
    got = host(out.view(torch.int16)).view(np.uint16)
    _bits_equal_or_both_nan(got[:, :cols], oracle.dequantize_mx(q, s))
    assert np.all(got[:, cols:] == 0x7777), "wrote past cols"


def test_dequantize_roundtrip_of_gpu_quantization():
    x = workloads.student_t((384, 640), 4, 3, 0, device())
    qd = m.fp8_quantize_mx(x, m.MX_ROWWISE | m.MX_COLWISE)
    back = m.fp8_dequantize_mx(qd["q_row"], qd["s_row"])
    back_t = m.fp8_dequantize_mx(qd["q_col"], qd["s_col"])
    assert_ok()
    want = oracle.quantize_mx(workloads.bits(x), oracle.ROWWISE | oracle.COLWISE)
    assert np.array_equal(host(back.view(torch.int16)).view(np.uint16),
                          oracle.dequantize_mx(want["q_row"], want["s_row"]))
    assert np.array_equal(host(back_t.view(torch.int16)).view(np.uint16),
                          oracle.dequantize_mx(want["q_col"], want["s_col"]))


@pytest.mark.parametrize("counts", GROUP_COUNTS)
def test_dequantize_grouped(counts):
    off = _offsets(counts)
    rows, cols = int(off[-1]), 160
    rng = np.random.default_rng(len(counts))
    x = oracle.bf16_round(rng.standard_normal((rows, cols)) * np.exp(rng.uniform(-20, 20, (rows, 1))))
    q, s = oracle.quantize_mx_grouped(x, off)
    s_full = np.zeros(oracle.grouped_scale_bytes(off, cols) + 512, np.uint8)
    s_full[: s.size] = s
    out = m.fp8_dequantize_mx(to_dev_u8(q), to_dev_u8(s_full),
                              offsets=torch.from_numpy(off).to(device()))
    assert_ok()
    assert np.array_equal(host(out.view(torch.int16)).view(np.uint16),
                          oracle.dequantize_mx_grouped(q, s, off))


def test_dequantize_grouped_bad_offsets_recorded():
    off = np.array([0, 50, 40, 100], np.int32)  # decreasing
    q = torch.zeros((100, 32), dtype=torch.uint8, device=device())
    s = torch.zeros(8192, dtype=torch.uint8, device=device())
    m.fp8_dequantize_mx(q, s, offsets=torch.from_numpy(off).to(device()))
    assert m.mxfp8_last_device_status() == m.MXFP8_ERR_DEVICE_CHECK
    assert_ok()  # cleared


def test_dequantize_full_size_mlp_up_activation():
    """Save/restore of the mlp_up activation X (8192 x 4096): GPU quantize,
    GPU dequantize, every BF16 value against the oracle."""
    x = workloads.mlp_up(seed=0, device=device())["X"]
    qd = m.fp8_quantize_mx(x, m.MX_ROWWISE)
    back = m.fp8_dequantize_mx(qd["q_row"], qd["s_row"])
    back2 = m.fp8_dequantize_mx(qd["q_row"], qd["s_row"])
    assert_ok()
    want = oracle.quantize_mx(workloads.bits(x), oracle.ROWWISE)
    ref = oracle.dequantize_mx(want["q_row"], want["s_row"])
    assert np.array_equal(host(back.view(torch.int16)).view(np.uint16), ref)
    assert torch.equal(back.view(torch.int16), back2.view(torch.int16))


# ----------------------------------------------------- SwiGLU + quantize --

def _swiglu_check(h_dev, offsets=None, floor=False):
    """Every payload and scale byte of the fused SwiGLU + MX quantization
    against the oracle's MX quantization of the correctly rounded BF16
    hidden value."""
    flags = m.MX_SCALE_FLOOR if floor else 0
    off_d = None if offsets is None else torch.from_numpy(offsets).to(device())
    q, s = m.fp8_swiglu_quantize_mx(h_dev, offsets=off_d, flags=flags)
    assert_ok()
    y = oracle.swiglu_bf16(workloads.bits(h_dev))
    fl = oracle.SCALE_FLOOR if floor else 0
    if offsets is None:
        want = oracle.quantize_mx(y, oracle.ROWWISE | fl)
        q_exp, s_exp = want["q_row"], want["s_row"]
    else:
        q_exp, s_exp = oracle.quantize_mx_grouped(y, offsets, oracle.ROWWISE | fl)
    qh, sh = host(q), host(s)[: s_exp.size]
    dq = np.argwhere(qh != q_exp)
    assert dq.size == 0, f"{len(dq)} payload bytes differ, first at {dq[:4].tolist()}"
    ds = np.nonzero(sh != s_exp)[0]
    assert ds.size == 0, f"{ds.size} scale bytes differ, first at {ds[:4]}"
    return y


# documented bound of the fast path: 4.5 * 2^-24 with u = 1 (exhaustive over
# the BF16 gates below), 7.5 * 2^-24 for a general u (three more half-ulp
# roundings at most)
SWIGLU_BOUND_U1 = 4.5 * 2.0 ** -24
SWIGLU_BOUND = 7.5 * 2.0 ** -24


def _swiglu_rel_err(gb, ub, bound):
    """Largest relative error of the fast path over values above 2^-100,
    after checking every value against bound * |y| + 2^-149."""
    y = host(m.mxfp8_debug_swiglu_f32(to_dev_bf16(gb), to_dev_bf16(ub))).astype(np.float64)
    assert_ok()
    want = oracle.swiglu(np.concatenate([gb[None, :], ub[None, :]], axis=1))[0]
    # well beyond fp32's range both are infinite (so is the BF16 value); right
    # at the edge either FLT_MAX or infinity is a correct fp32 result
    a = np.abs(want)
    over = a >= 2.0 ** 128 * (1 + 2.0 ** -20)
    edge = ~over & (a >= float(np.finfo(np.float32).max) * (1 - 2.0 ** -20))
    assert np.all(np.isinf(y[over]) & (np.sign(y[over]) == np.sign(want[over])))
    y, want = y[~(over | edge)], want[~(over | edge)]
    err = np.abs(y - want)
    assert np.all(err <= bound * np.abs(want) + 2.0 ** -149)
    big = np.abs(want) >= 2.0 ** -100
    return np.max(err[big] / np.abs(want[big]), initial=0.0)


def test_swiglu_fast_path_error_every_gate():
    """Every finite BF16 gate the fast path takes (g >= -80, |g| log2(e)
    within fp32's range) with u = 1: the
    fp32 value the quantizer rounds to BF16 is within the documented bound of
    g sigma(g) computed in FP64 by the oracle; with random ups, within the
    general bound."""
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    g = oracle.bf16_decode(allb)
    # past |g| log2(e) > fp32's largest value the fast path gives NaN (its
    # blocks are redone in FP64)
    huge = np.isfinite(g) & (np.abs(g) * np.log2(np.e) > float(np.finfo(np.float32).max) * (1 + 2.0 ** -20))
    yh = host(m.mxfp8_debug_swiglu_f32(to_dev_bf16(allb[huge]), to_dev_bf16(np.full(int(huge.sum()), 0x3F80, np.uint16))))
    assert_ok()  # the packed and scalar fast paths agree bit for bit
    assert huge.sum() > 0 and np.all(np.isnan(yh))
    edge = np.abs(g) * np.log2(np.e) > float(np.finfo(np.float32).max) * (1 - 2.0 ** -20)
    gb = allb[np.isfinite(g) & (g >= -80) & (g != 0) & ~edge]
    rel = _swiglu_rel_err(gb, np.full(gb.shape, 0x3F80, np.uint16), SWIGLU_BOUND_U1)
    assert rel <= SWIGLU_BOUND_U1, rel / 2.0 ** -24
    rng = np.random.default_rng(5)
    ub = oracle.bf16_round(rng.standard_normal(gb.size) * np.exp(rng.uniform(-20, 20, gb.size)))
    rel = _swiglu_rel_err(gb, ub, SWIGLU_BOUND)
    assert rel <= SWIGLU_BOUND, rel / 2.0 ** -24


def test_swiglu_fast_path_special_gates():
    """NaN gates propagate; gates from 87 up to 2^127 (e^-g flushes to 0)
    give g u exactly; +Inf and gates past ~2.4e38 give NaN in the fast path
    (the quantizer redoes a block with a NaN or Inf maximum in FP64); zero
    gates give 0."""
    gb = np.array([0x7F80, 0x7FC0, 0x42B0, 0x4300, 0x7F00, 0x7F7F, 0x0000, 0x8000], np.uint16)
    ub = np.array([0x3F80] * 6 + [0x4000, 0x4000], np.uint16)
    y = host(m.mxfp8_debug_swiglu_f32(to_dev_bf16(gb), to_dev_bf16(ub)))
    assert_ok()
    assert np.isnan(y[0]) and np.isnan(y[1]) and np.isnan(y[5])
    gd = oracle.bf16_decode(gb)
    assert y[2] == np.float32(gd[2]) and y[3] == np.float32(gd[3]) and y[4] == np.float32(gd[4])
    assert y[6] == 0 and y[7] == 0


@pytest.mark.parametrize("rows,f", SHAPES)
@pytest.mark.parametrize("floor", [False, True])
def test_swiglu_quantize_plain(rows, f, floor):
    rng = np.random.default_rng(rows + f)
    h = oracle.bf16_round(rng.standard_normal((rows, 2 * f)) * 3)
    _swiglu_check(to_dev_bf16(h), floor=floor)


def test_swiglu_quantize_extremes():
    """Gates far below -80 (the double path), BF16-subnormal gates, gates
    beyond 64, huge ups, zeros of both signs and values that underflow BF16."""
    rng = np.random.default_rng(21)
    rows, f = 256, 128
    g = rng.standard_normal((rows, f)) * np.exp(rng.uniform(-100, 6, (rows, 1)))
    u = rng.standard_normal((rows, f)) * np.exp(rng.uniform(-60, 60, (rows, 1)))
    g[:8] = -rng.uniform(80, 300, (8, f))
    g[8, :16] = 0.0
    u[9, :16] = -0.0
    g[10] = np.ldexp(rng.uniform(1, 2, f), rng.integers(-133, -100, f))
    g[11] = rng.uniform(60, 3000, f) * rng.choice([-1, 1], f)
    g[12] = rng.uniform(2.4e38, 3.3e38, f)  # a |g| L2E past fp32: NaN in the fast path
    u[12] = rng.standard_normal(f) * 2.0 ** -120
    g[13, :4] = [np.inf, -np.inf, np.inf, 1.0]
    u[13, :4] = [1.0, 1.0, 0.0, np.inf]
    h = oracle.bf16_round(np.concatenate([g, u], axis=1))
    _swiglu_check(to_dev_bf16(h))


@pytest.mark.parametrize("counts", GROUP_COUNTS)
def test_swiglu_quantize_grouped(counts):
    off = _offsets(counts)
    rng = np.random.default_rng(sum(counts))
    h = oracle.bf16_round(rng.standard_normal((int(off[-1]), 2 * 96)) * 2)
    _swiglu_check(to_dev_bf16(h), offsets=off)


def test_swiglu_quantize_16_byte_aligned():
    """h with a row stride that is a multiple of 16 bytes but not 32 (no
    256-bit accesses)."""
    rows, f = 150, 96
    rng = np.random.default_rng(31)
    wide = oracle.bf16_round(rng.standard_normal((rows, 2 * f + 8)) * 2)
    hd = to_dev_bf16(wide)[:, : 2 * f]
    assert hd.stride(0) % 16 == 8
    _swiglu_check(hd)


def test_swiglu_quantize_full_size():
    """The grouped workload's up/gate output (262144 x 1024, 64 experts):
    every byte exact, and the workload holds values whose fast fp32 value
    sits next to a BF16 midpoint (so the resolution runs)."""
    w = workloads.swiglu_hidden(seed=0, device=device())
    _swiglu_check(w["H"], offsets=w["offsets"])
    h = w["H"][:4096]
    f = h.shape[1] // 2
    y = host(m.mxfp8_debug_swiglu_f32(h[:, :f].contiguous().reshape(-1),
                                      h[:, f:].contiguous().reshape(-1)))
    assert_ok()
    low = y.view(np.uint32) & 0xFFFF
    assert int((np.abs(low.astype(np.int64) - 0x8000) <= 8).sum()) > 100


def _near_midpoint_pairs(n, seed, window=8):
    """(gate, up) BF16 pairs whose fp32-rounded SwiGLU value has its low 16
    bits within `window` of 0x8000: the fast path's own rounding of these
    cannot be trusted (found with the oracle's FP64 SwiGLU)."""
    rng = np.random.default_rng(seed)
    gs, us = [], []
    while sum(map(len, gs)) < n:
        k = 1 << 20
        g = oracle.bf16_round(rng.standard_normal(k) * np.exp(rng.uniform(-3, 2.5, k)))
        u = oracle.bf16_round(rng.standard_normal(k) * np.exp(rng.uniform(-30, 30, k)))
        y = oracle.swiglu(np.stack([g, u], axis=1))[:, 0].astype(np.float32)
        low = (y.view(np.uint32) & 0xFFFF).astype(np.int64)
        hit = (np.abs(low - 0x8000) <= window) & (np.abs(y) > 2.0 ** -70)
        gs.append(g[hit])
        us.append(u[hit])
    return np.concatenate(gs)[:n], np.concatenate(us)[:n]


def test_swiglu_quantize_near_midpoints():
    """Blocks seeded with values next to a BF16 rounding midpoint: one per
    block, several in one block, in neighbouring lanes of a warp, plus
    saturated gates whose g u is itself a midpoint.  The fast path's own
    BF16 rounding is wrong for some of them (checked through the fast-path
    hook), the quantized bytes never are."""
    g, u = _near_midpoint_pairs(1500, 51)
    sat_g = oracle.bf16_round(np.array([48.0, 56.0, 80.0, 3 * 2.0 ** 20, 13.0, 40.0]))
    sat_u = oracle.bf16_round(np.array([107 / 128, 37 / 64, -53 * 2.0 ** 10, -107 * 2.0 ** -30,
                                        21.0 / 1024, 107 / 64]))
    g = np.concatenate([g, sat_g])
    u = np.concatenate([u, sat_u])
    rows, f = 384, 256
    rng = np.random.default_rng(52)
    h = oracle.bf16_round(rng.standard_normal((rows, 2 * f)) * 2)
    # positions: most blocks get one value, the first 64 rows get four per block
    n = g.size
    pos = rng.choice(rows * f, size=n, replace=False)
    dense = (np.arange(64)[:, None] * f + np.arange(0, f, 8)[None, :]).reshape(-1)[: n // 4]
    pos[: dense.size] = dense
    pos = np.unique(pos)[:n]
    r, c = pos // f, pos % f
    h[r, c] = g[: pos.size]
    h[r, f + c] = u[: pos.size]
    y = _swiglu_check(to_dev_bf16(h))
    fast = host(m.mxfp8_debug_swiglu_f32(to_dev_bf16(h[r, c]), to_dev_bf16(h[r, f + c])))
    naive = oracle.bf16_round(fast.astype(np.float64))
    assert int((naive != y[r, c]).sum()) > 20  # the fast rounding alone is wrong there


def test_swiglu_quantize_product_past_fp32():
    """Gates in (1, 6) with ups near the BF16 maximum: g u leaves fp32's
    range while g sigma(g) u mostly stays finite (the block is redone in
    FP64); larger gates give values past the range (Inf, NaN scale)."""
    rng = np.random.default_rng(53)
    rows, f = 128, 128
    g = rng.uniform(1.01, 8.0, (rows, f))
    u = rng.uniform(2.0 ** 126, 3.3e38, (rows, f)) * rng.choice([-1, 1], (rows, f))
    g[::2] = rng.standard_normal((rows // 2, f))  # ordinary rows between them
    u[::2] = rng.standard_normal((rows // 2, f))
    h = oracle.bf16_round(np.concatenate([g, u], axis=1))
    y = _swiglu_check(to_dev_bf16(h))
    v = oracle.bf16_decode(y[1::2])
    hv = oracle.bf16_decode(h[1::2])
    past = np.abs(hv[:, :f] * hv[:, f:]) > float(np.finfo(np.float32).max)
    assert (past & np.isfinite(v)).sum() > 100 and np.isinf(v).any()


# ------------------------------------------- route weighting + quantize --

def _weighted_check(dy, tok, wt, offsets=None, floor=False):
    off_d = None if offsets is None else torch.from_numpy(offsets).to(device())
    q, s = m.fp8_route_weight_quantize_mx(dy, torch.from_numpy(tok).to(device()),
                                          torch.from_numpy(wt).to(device()), offsets=off_d,
                                          flags=m.MX_SCALE_FLOOR if floor else 0)
    st = m.mxfp8_last_device_status()
    g = oracle.route_weight(workloads.bits(dy), tok, wt)
    fl = oracle.SCALE_FLOOR if floor else 0
    if offsets is None:
        want = oracle.quantize_mx(g, oracle.ROWWISE | fl)
        q_exp, s_exp = want["q_row"], want["s_row"]
    else:
        q_exp, s_exp = oracle.quantize_mx_grouped(g, offsets, oracle.ROWWISE | fl)
    assert np.array_equal(host(q), q_exp)
    assert np.array_equal(host(s)[: s_exp.size], s_exp)
    return st


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("floor", [False, True])
def test_route_weight_quantize_plain(rows, cols, floor):
    rng = np.random.default_rng(rows * 3 + cols)
    tokens = max(1, rows // 3)
    dy = to_dev_bf16(oracle.bf16_round(rng.standard_normal((tokens, cols)) *
                                       np.exp(rng.uniform(-25, 5, (tokens, 1)))))
    tok = rng.integers(0, tokens, rows).astype(np.int32)
    wt = rng.uniform(0, 1, rows).astype(np.float32)
    assert _weighted_check(dy, tok, wt, floor=floor) == m.MXFP8_OK


def test_route_weight_quantize_16_byte_aligned():
    """dY rows 16 bytes apart from a 32-byte boundary (row stride cols + 8:
    the 16-byte load path)."""
    rng = np.random.default_rng(31)
    tokens, cols, rows = 50, 224, 300
    dyb = oracle.bf16_round(rng.standard_normal((tokens, cols)))
    wide = np.zeros((tokens, cols + 8), np.uint16)
    wide[:, :cols] = dyb
    dy = to_dev_bf16(wide)[:, :cols]
    tok = rng.integers(0, tokens, rows).astype(np.int32)
    wt = rng.uniform(0, 1, rows).astype(np.float32)
    assert _weighted_check(dy, tok, wt) == m.MXFP8_OK


def test_route_weight_quantize_extremes():
    """Exact-product ties, products below fp32's normal range (the double
    branch), overflow to Inf, zero weights, and an out-of-range token index
    (recorded; that row quantizes as zeros)."""
    rng = np.random.default_rng(22)
    tokens, cols, rows = 8, 64, 40
    dy = oracle.bf16_round(rng.standard_normal((tokens, cols)) * np.exp(rng.uniform(-80, 80, (tokens, 1))))
    dy[0, :8] = [0x3F80, 0xBF80, 0x0001, 0x8001, 0x7F7F, 0x0080, 0x3F81, 0x0000]
    tok = rng.integers(0, tokens, rows).astype(np.int32)
    tok[:6] = 0
    wt = rng.uniform(0, 1, rows).astype(np.float32)
    wt[:6] = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 2.0 ** -30, 1.5, 0.0, 2.0 ** -126], np.float32)
    wt[8:14] = np.array([-0.75, 2.0 ** 20, 2.0 ** -140, -(2.0 ** 100), 2.0 ** 126, -(2.0 ** -149)],
                        np.float32)  # negative, large, subnormal
    tok[7] = tokens  # out of range
    st = _weighted_check(to_dev_bf16(dy), tok, wt)
    assert st == m.MXFP8_ERR_DEVICE_CHECK


def _fp32_midpoint_pairs(n, seed):
    """(x, w) pairs whose fp32 product lands exactly on a BF16 rounding
    midpoint while the exact product does not: the double-rounding cases."""
    rng = np.random.default_rng(seed)
    xs_bits = np.arange(0x0080, 0x7F80, dtype=np.uint16)  # positive normal BF16
    xs = oracle.bf16_decode(xs_bits)
    found = []
    while len(found) < n:
        w = np.float32(rng.uniform(0.25, 1.0))
        p32 = (xs.astype(np.float32) * w).astype(np.float32)
        hit = ((p32.view(np.uint32) & 0xFFFF) == 0x8000) & (p32.astype(np.float64) != xs * np.float64(w))
        for i in np.nonzero(hit)[0][:2]:
            found.append((int(xs_bits[i]), w))
    return found[:n]


def test_route_weight_quantize_double_rounding_cases():
    """Products whose fp32 rounding sits on a BF16 midpoint take the exact
    path; one fp32 rounding followed by the BF16 rounding would be off by one
    unit in the last place there."""
    pairs = _fp32_midpoint_pairs(32, 23)
    cols = 64
    dy = np.zeros((len(pairs), cols), np.uint16)
    rng = np.random.default_rng(24)
    for i, (xb, _) in enumerate(pairs):
        dy[i] = oracle.bf16_round(rng.uniform(0.5, 1.0, cols))
        dy[i, i % cols] = xb
    tok = np.arange(len(pairs), dtype=np.int32)
    wt = np.array([w for _, w in pairs], np.float32)
    g = oracle.route_weight(dy, tok, wt)
    naive = (oracle.bf16_decode(dy).astype(np.float32) * wt[:, None]).astype(np.float32)
    naive_bits = oracle.bf16_round(naive.astype(np.float64))
    assert (naive_bits != g).sum() >= len(pairs) // 4  # the cases are real
    assert _weighted_check(to_dev_bf16(dy), tok, wt) == m.MXFP8_OK


@pytest.mark.parametrize("counts", GROUP_COUNTS)
def test_route_weight_quantize_grouped(counts):
    off = _offsets(counts)
    rows = int(off[-1])
    rng = np.random.default_rng(rows)
    tokens = max(1, rows // 4)
    dy = to_dev_bf16(oracle.bf16_round(rng.standard_normal((tokens, 224)) * 1e-3))
    tok = rng.integers(0, tokens, rows).astype(np.int32)
    wt = rng.uniform(0, 1, rows).astype(np.float32)
    assert _weighted_check(dy, tok, wt, offsets=off) == m.MXFP8_OK


def test_route_weight_quantize_full_size():
    """Combine backward of 32768 tokens x 2048, top-8 of 64 experts."""
    w = workloads.combine_backward(seed=0, device=device())
    assert _weighted_check(w["dY"], w["row_token"], w["row_weight"], offsets=w["offsets"]) == m.MXFP8_OK


# --------------------------- route weighting + quantize, per-token form --

def _tokens_check(dy, token_rows, token_weights, rows, offsets=None, floor=False):
    """fp8_route_weight_quantize_mx_tokens against the oracle (through the
    equivalent per-row routing) and against the per-row entry point."""
    off_d = None if offsets is None else torch.from_numpy(offsets).to(device())
    flags = m.MX_SCALE_FLOOR if floor else 0
    cols = dy.shape[1]
    # scale bytes pre-filled: every byte of the used layout (padding rows and
    # blocks past cols included) must be written by the call
    n_s = (m.mxfp8_scale_bytes(rows, cols) if offsets is None
           else m.mxfp8_grouped_scale_bytes(rows, cols, len(offsets) - 1))
    s_buf = filled((max(1, n_s),), 0x77, torch.uint8)
    q, s = m.fp8_route_weight_quantize_mx_tokens(
        dy, torch.from_numpy(token_rows).to(device()), torch.from_numpy(token_weights).to(device()),
        rows, offsets=off_d, flags=flags, s=s_buf)
    st = m.mxfp8_last_device_status()
    row_token = np.full(rows, -1, np.int32)
    row_weight = np.zeros(rows, np.float32)
    t_idx, j_idx = np.nonzero((token_rows >= 0) & (token_rows < rows))
    row_token[token_rows[t_idx, j_idx]] = t_idx
    row_weight[token_rows[t_idx, j_idx]] = token_weights[t_idx, j_idx]
    g = oracle.route_weight(workloads.bits(dy), row_token, row_weight)
    fl = oracle.SCALE_FLOOR if floor else 0
    if offsets is None:
        want = oracle.quantize_mx(g, oracle.ROWWISE | fl)
        q_exp, s_exp = want["q_row"], want["s_row"]
    else:
        q_exp, s_exp = oracle.quantize_mx_grouped(g, offsets, oracle.ROWWISE | fl)
    assert np.array_equal(host(q), q_exp)
    assert np.array_equal(host(s)[: s_exp.size], s_exp)
    q2, s2 = m.fp8_route_weight_quantize_mx(dy, torch.from_numpy(row_token).to(device()),
                                            torch.from_numpy(row_weight).to(device()), offsets=off_d,
                                            flags=flags)
    assert torch.equal(q, q2) and torch.equal(s[: s_exp.size], s2[: s_exp.size])
    return st


def _random_routing(tokens, k, rows, rng):
    perm = rng.permutation(tokens * k)[:rows] if rows <= tokens * k else None
    tr = np.full(tokens * k, -1, np.int64)
    tr[perm] = np.arange(rows)  # slot perm[i] routes to dispatched row i
    return tr.reshape(tokens, k).astype(np.int32), rng.uniform(0, 1, (tokens, k)).astype(np.float32)


@pytest.mark.parametrize("tokens,k,cols", [(7, 1, 32), (50, 8, 224), (33, 3, 416), (130, 16, 96)])
@pytest.mark.parametrize("floor", [False, True])
def test_route_weight_tokens_plain(tokens, k, cols, floor):
    rng = np.random.default_rng(tokens * 7 + k)
    rows = tokens * k - (tokens // 3)  # some slots unused (-1)
    tr, tw = _random_routing(tokens, k, rows, rng)
    dy = to_dev_bf16(oracle.bf16_round(rng.standard_normal((tokens, cols)) *
                                       np.exp(rng.uniform(-25, 5, (tokens, 1)))))
    assert _tokens_check(dy, tr, tw, rows, floor=floor) == m.MXFP8_OK


@pytest.mark.parametrize("counts", GROUP_COUNTS)
def test_route_weight_tokens_grouped(counts):
    off = _offsets(counts)
    rows = int(off[-1])
    k = 4
    tokens = (rows + k - 1) // k + 1
    rng = np.random.default_rng(rows + 5)
    tr, tw = _random_routing(tokens, k, rows, rng)
    dy = to_dev_bf16(oracle.bf16_round(rng.standard_normal((tokens, 224)) * 1e-3))
    assert _tokens_check(dy, tr, tw, rows, offsets=off) == m.MXFP8_OK


def test_route_weight_tokens_ties_and_bad_row():
    """The 32 constructed double-rounding cases (fp32 product on a BF16
    midpoint, exact product off it) through the per-token form, half of them
    with the value negated (the correction's direction follows the sign),
    plus a slot naming a row past the end (recorded, skipped)."""
    pairs = _fp32_midpoint_pairs(32, 23)
    cols, k = 64, 2
    tokens = len(pairs)
    rng = np.random.default_rng(25)
    dy = np.zeros((tokens, cols), np.uint16)
    for i, (xb, _) in enumerate(pairs):
        dy[i] = oracle.bf16_round(rng.uniform(0.5, 1.0, cols) * rng.choice([-1.0, 1.0], cols))
        dy[i, i % cols] = xb | (0x8000 if i % 2 else 0)
    rows = tokens  # slot 0 of token i -> row i; slot 1 unused
    tr = np.full((tokens, k), -1, np.int32)
    tr[:, 0] = np.arange(tokens)
    tw = np.zeros((tokens, k), np.float32)
    tw[:, 0] = [w for _, w in pairs]
    assert _tokens_check(to_dev_bf16(dy), tr, tw, rows) == m.MXFP8_OK
    tr[3, 1] = rows + 5
    assert _tokens_check(to_dev_bf16(dy), tr, tw, rows) == m.MXFP8_ERR_DEVICE_CHECK


def test_route_weight_tokens_full_size():
    """Combine backward of 32768 tokens x 2048, top-8 of 64 experts, routing
    given per token."""
    w = workloads.combine_backward(seed=0, device=device())
    rows = w["token_rows"].size
    assert _tokens_check(w["dY"], w["token_rows"], w["token_weights"], rows,
                         offsets=w["offsets"]) == m.MXFP8_OK


def test_route_weight_tokens_extremes():
    """The per-token form on blocks that mix BF16-subnormal products with a
    block maximum near 2^-100 (the scale folded into the weight still gives
    their signed zeros), products at the top of the range, subnormal and
    largest BF16 inputs, weights of 2^-30, 2^-126 and 0, negative, large and
    subnormal weights, exact-product ties, and blocks holding Inf or NaN."""
    rng = np.random.default_rng(26)
    tokens, cols, k = 24, 96, 3
    mag = np.exp(rng.uniform(-80, 80, (tokens, 1)))
    dy = oracle.bf16_round(rng.standard_normal((tokens, cols)) * mag)
    dy[0, :8] = [0x3F80, 0xBF80, 0x0001, 0x8001, 0x7F7F, 0x0080, 0x3F81, 0x0000]
    # row 1: a block spanning 2^-131 .. 2^-100 (BF16 subnormals beside a normal maximum)
    dy[1, :32] = oracle.bf16_round(np.ldexp(rng.uniform(1, 2, 32), rng.integers(-131, -100, 32)) *
                                   rng.choice([-1, 1], 32))
    dy[2, :32] = oracle.bf16_round(np.ldexp(rng.uniform(1, 2, 32), rng.integers(-140, -118, 32)))
    # blocks holding Inf, -Inf and NaN inputs: NaN scale, every payload byte 0x7F
    dy[3, 0], dy[3, 33], dy[3, 70] = 0x7F80, 0xFF80, 0x7FC0
    rows = tokens * k
    tr = np.arange(rows, dtype=np.int32).reshape(tokens, k)
    tw = rng.uniform(0, 1, (tokens, k)).astype(np.float32)
    tw[0] = [1 + 2.0 ** -8, 2.0 ** -30, 2.0 ** -126]
    tw[1] = [1.0, 0.75, 2.0 ** -20]
    tw[2] = [0.0, 1.5, 1 + 3 * 2.0 ** -8]
    # negative, large and subnormal weights: the folded weight's range and
    # sign (a subnormal weight never folds; a large one overflows some blocks)
    tw[4] = [-0.75, 2.0 ** 20, 2.0 ** -140]
    tw[5] = [-(1 + 2.0 ** -8), -(2.0 ** 100), 2.0 ** -149]
    tw[6] = [2.0 ** 126, -(2.0 ** -126), 3.0e38]
    assert _tokens_check(to_dev_bf16(dy), tr, tw, rows) == m.MXFP8_OK
