"""Pins of the FP64 oracle against facts fixed outside the oracle itself.

Every test here runs on the CPU.  The pins are: values printed on the pages
(tests/golden/*.txt), torch's own float8 conversions (an independent library
implementation of the same encodings), brute force over all FP8 codes and
all BF16 bit patterns, closed forms and invariants of the method, and numpy
matmuls of operands dequantized without the oracle.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from conftest import pow2_or_float, read_golden, read_golden_table

E4M3, E5M2 = oracle.E4M3, oracle.E5M2
ALL_CODES = np.arange(256, dtype=np.uint8)


def torch_fp8_decode(codes, fmt):
    dt = torch.float8_e4m3fn if fmt == E4M3 else torch.float8_e5m2
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(dt).to(torch.float64).numpy()


def torch_fp8_encode_f32(v32, fmt):
    """torch's RNE cast of fp32 values (NOT saturating: out of range -> NaN/Inf)."""
    dt = torch.float8_e4m3fn if fmt == E4M3 else torch.float8_e5m2
    return torch.from_numpy(np.asarray(v32, np.float32)).to(dt).view(torch.uint8).numpy()


def all_bf16_bits():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


def bf16_values_torch(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


# ------------------------------------------------------------ page values --

def test_bf16_worked_value():
    g = read_golden("bf16_worked_value.txt")
    x32 = np.float32(float(g["input_fp32"]))
    bits = oracle.bf16_round([float(x32)])[0]
    assert bits == int(g["bf16_bits"], 16)
    assert oracle.bf16_decode([bits])[0] == float(g["bf16_value"])


def test_fig50_block():
    g = read_golden("fig50_block.txt")
    x = float(g["x"])
    pos = int(g["position_1based"]) - 1
    rng = np.random.default_rng(50)
    # the other 31 values: any magnitudes at most 1.75, so x is the maximum
    block = rng.uniform(-1.75, 1.75, 32)
    block[pos] = x
    bits = oracle.bf16_round(block)
    assert oracle.bf16_decode([bits[pos]])[0] == x  # 2.28125 is a BF16 value
    out = oracle.quantize_mx(bits.reshape(1, 32), oracle.ROWWISE)
    s_byte = out["s_row"][oracle.swizzle_offset(0, 0, 32)]
    assert s_byte == int(g["scale_byte"])
    s = 2.0 ** (int(s_byte) - 127)
    assert x / s == float(g["x_over_s"])
    q = out["q_row"][0, pos]
    assert q == int(g["q_bits"], 2)
    assert oracle.fp8_decode([q])[0] == float(g["q_value"])
    xhat = s * oracle.fp8_decode([q])[0]
    assert xhat == float(g["xhat"])
    assert round(100 * (xhat - x) / x, 1) == float(g["rel_error_percent"])
    # the same byte for any block maximum in (1.75, 3.5]
    for amax in (1.75 + 2**-6, 2.28125, 3.0, 3.5):
        assert oracle.e8m0_scale_byte([amax])[0] == 120
    assert oracle.e8m0_scale_byte([1.75])[0] == 119


def test_scale_rule_a500():
    g = read_golden("scale_rule_a500.txt")
    a = float(g["amax"])
    block = np.zeros(32)
    block[0] = a
    bits = oracle.bf16_round(block)
    assert oracle.bf16_decode(bits[:1])[0] == 500.0
    fl = oracle.quantize_mx(bits.reshape(1, 32), oracle.ROWWISE | oracle.SCALE_FLOOR)
    rc = oracle.quantize_mx(bits.reshape(1, 32), oracle.ROWWISE)
    assert fl["s_row"][0] == int(g["floor_scale_byte"])
    assert 2.0 ** (int(fl["s_row"][0]) - 127) == float(g["floor_scale"])
    assert fl["q_row"][0, 0] == int(g["floor_q_bits"], 16)
    assert oracle.fp8_decode(fl["q_row"][0, :1])[0] == float(g["floor_q_value"])
    assert rc["s_row"][0] == int(g["rceil_scale_byte"])
    assert 2.0 ** (int(rc["s_row"][0]) - 127) == float(g["rceil_scale"])
    assert rc["q_row"][0, 0] == int(g["rceil_q_bits_derived"], 16)
    assert oracle.fp8_decode(rc["q_row"][0, :1])[0] == float(g["rceil_q_value_derived"])


def _format_facts(fmt):
    vals = oracle.fp8_decode(ALL_CODES, fmt)
    pos = vals[(ALL_CODES < 0x80) & np.isfinite(vals) & (vals > 0)]
    normal_codes = [c for c in range(1, 0x80)
                    if np.isfinite(vals[c]) and ((c >> (3 if fmt == E4M3 else 2)) != 0)]
    min_normal = min(vals[c] for c in normal_codes)
    above_one = min(v for v in pos if v > 1.0)
    return pos.max(), min_normal, pos.min(), above_one - 1.0


def test_format_table():
    rows = {r[0]: r[1:] for r in read_golden_table("format_table.txt")}
    for name, fmt in (("E4M3", E4M3), ("E5M2", E5M2)):
        mx, mn, sub, sp = _format_facts(fmt)
        want = [pow2_or_float(v) for v in rows[name]]
        assert (mx, mn, sub, sp) == tuple(want), name
    # FP8-LM Section 3.4 decimals
    assert abs(_format_facts(E4M3)[1] - 1.56e-2) < 1e-4
    assert abs(_format_facts(E4M3)[2] - 1.95e-3) < 1e-5
    assert abs(_format_facts(E5M2)[1] - 6.10e-5) < 1e-7
    assert abs(_format_facts(E5M2)[2] - 1.53e-5) < 1e-7
    # E8M0: bytes 0..254 are 2^-127 .. 2^127, 255 is NaN
    assert oracle.e8m0_scale_byte([2.0 ** -200])[0] == 0
    e8 = rows["E8M0"]
    assert pow2_or_float(e8[0]) == 2.0 ** (254 - 127)
    assert pow2_or_float(e8[1]) == 2.0 ** (0 - 127)
    # BF16
    b = oracle.bf16_decode(all_bf16_bits())
    fin = b[np.isfinite(b) & (b > 0)]
    bf = rows["BF16"]
    assert abs(fin.max() / float(bf[0]) - 1) < 1e-3
    assert fin[fin >= 2.0 ** -126].min() == pow2_or_float(bf[1])
    assert fin.min() == pow2_or_float(bf[2])
    assert fin[fin > 1.0].min() - 1.0 == pow2_or_float(bf[3])


def test_storage_eq57():
    g = read_golden("storage_eq57.txt")
    per_value = 1 + 1 / 32
    assert per_value == 33 / 32 == eval(g["bytes_per_value"])
    assert round(100 * (1 - per_value / 2), 1) == float(g["saving_vs_bf16_percent"])
    assert 2 * per_value == float(g["two_orientations_bytes_per_value"])
    for rows, cols in ((128, 128), (256, 4096), (96, 64), (1, 32)):
        x = oracle.bf16_round(np.random.default_rng(rows).normal(size=(rows, cols)))
        out = oracle.quantize_mx(x, oracle.ROWWISE)
        logical_scales = rows * cols // 32
        assert out["q_row"].size + logical_scales == rows * cols * 33 // 32
        # padded physical size follows the 128 x 4 tile geometry
        assert out["s_row"].size == math.ceil(rows / 128) * math.ceil(cols / 128) * 512
        if rows % 32 == 0:
            both = oracle.quantize_mx(x, oracle.ROWWISE | oracle.COLWISE)
            nbytes = both["q_row"].size + both["q_col"].size + 2 * logical_scales
            assert nbytes == 2 * rows * cols * 33 // 32


# ------------------------------------------------------ codecs vs torch --

@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_fp8_decode_all_codes_vs_torch(fmt):
    ours = oracle.fp8_decode(ALL_CODES, fmt)
    ref = torch_fp8_decode(ALL_CODES, fmt)
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.array_equal(ours[~both_nan], ref[~both_nan])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    # signed zeros
    assert math.copysign(1, ours[0x80]) == -1 and ours[0x80] == 0
    # NaN codes: E4M3 has exactly 0x7F / 0xFF, no infinity
    if fmt == E4M3:
        assert set(np.flatnonzero(np.isnan(ours))) == {0x7F, 0xFF}
        assert not np.isinf(ours).any()
    else:
        assert set(np.flatnonzero(np.isinf(ours))) == {0x7C, 0xFC}


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_fp8_codes_monotone_and_roundtrip(fmt):
    vals = oracle.fp8_decode(ALL_CODES, fmt)
    top = 0x7E if fmt == E4M3 else 0x7B
    pos = vals[: top + 1]
    assert np.all(np.diff(pos) > 0)
    finite = [c for c in range(256) if np.isfinite(vals[c])]
    enc = oracle.fp8_encode(vals[finite], fmt)
    assert np.array_equal(enc, np.array(finite, np.uint8))


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_fp8_encode_ties_to_even(fmt):
    vals = oracle.fp8_decode(ALL_CODES, fmt)
    top = 0x7E if fmt == E4M3 else 0x7B
    for c in range(top):
        mid = (vals[c] + vals[c + 1]) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.fp8_encode([mid], fmt)[0] == even
        assert oracle.fp8_encode([-mid], fmt)[0] == even | 0x80
        eps = (vals[c + 1] - vals[c]) * 1e-6
        assert oracle.fp8_encode([mid - eps], fmt)[0] == c
        assert oracle.fp8_encode([mid + eps], fmt)[0] == c + 1


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_fp8_encode_saturates(fmt):
    top = 0x7E if fmt == E4M3 else 0x7B
    mx = 448.0 if fmt == E4M3 else 57344.0
    for v in (mx, mx * (1 + 2**-10), mx * 1.5, mx * 4, 1e30, math.inf):
        assert oracle.fp8_encode([v], fmt)[0] == top
        assert oracle.fp8_encode([-v], fmt)[0] == top | 0x80
    assert oracle.fp8_encode([math.nan], fmt)[0] == 0x7F


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_fp8_encode_all_bf16_times_all_scales_vs_torch(fmt):
    """Every BF16 pattern divided by every E8M0 scale: the MX payload step."""
    b = all_bf16_bits()
    x = bf16_values_torch(b)
    x = x[np.isfinite(x)]
    limit = 464.0 if fmt == E4M3 else 61440.0  # torch rounds |v| >= limit to NaN/Inf
    mx = 448.0 if fmt == E4M3 else 57344.0
    checked = 0
    for e in range(-127, 128):
        v = np.ldexp(x, -e)
        # keep v exactly representable in fp32 so torch's fp32 cast sees it exactly
        keep = (np.abs(v) >= 2.0 ** -140) & (np.abs(v) < 2.0 ** 100) | (v == 0)
        v = v[keep]
        if v.size == 0:
            continue
        ours = oracle.fp8_encode(v, fmt)
        small = np.abs(v) < limit
        ref = torch_fp8_encode_f32(v[small].astype(np.float32), fmt)
        assert np.array_equal(ours[small], ref), e
        big = ~small
        want = np.where(np.signbit(v[big]), 0x80, 0) | (0x7E if fmt == E4M3 else 0x7B)
        assert np.array_equal(ours[big], want.astype(np.uint8))
        assert np.all(np.abs(oracle.fp8_decode(ours, fmt)) <= mx)
        checked += v.size
    assert checked > 5_000_000


def test_bf16_round_vs_torch():
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.normal(size=20000), rng.normal(size=20000) * 1e-38,
                        rng.normal(size=20000) * 1e30, [0.0, -0.0, 1.0, 3.1415927]])
    v32 = v.astype(np.float32)
    ref = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = oracle.bf16_round(v32.astype(np.float64))
    assert np.array_equal(ours, ref)
    # decode agrees with torch for every pattern (NaNs aside)
    b = all_bf16_bits()
    ref_d = bf16_values_torch(b)
    d = oracle.bf16_decode(b)
    ok = ~np.isnan(ref_d)
    assert np.array_equal(d[ok], ref_d[ok]) and np.isnan(d[~ok]).all()


# ------------------------------------------------------------ E8M0 rules --

def _positive_finite_bf16():
    b = all_bf16_bits()
    v = bf16_values_torch(b)
    return v[np.isfinite(v) & (v > 0)]


def test_rceil_all_bf16_amax():
    a = _positive_finite_bf16()
    byte = oracle.e8m0_scale_byte(a)
    e = byte.astype(np.int64) - 127
    # float evaluation of "amax / 448 rounded up to a power of two"
    ef = np.ceil(np.log2(a / 448.0)).astype(np.int64)
    assert np.array_equal(e, np.clip(ef, -127, 127))
    # the definition: smallest e with amax <= 448 * 2^e (where not clamped)
    free = e > -127
    assert np.all(a[free] <= np.ldexp(448.0, e[free]))
    assert np.all(a[free] > np.ldexp(448.0, e[free] - 1))
    assert np.all(a[~free] <= np.ldexp(448.0, -127))
    # rceil never saturates: amax / s <= 448
    assert np.all(a / np.ldexp(1.0, e) <= 448.0)


def test_floor_all_bf16_amax():
    a = _positive_finite_bf16()
    byte = oracle.e8m0_scale_byte(a, floor=True)
    e = byte.astype(np.int64) - 127
    _, x = np.frexp(a)
    assert np.array_equal(e, np.clip(x - 1 - 8, -127, 127))
    ef = np.floor(np.log2(a)).astype(np.int64) - 8
    assert np.array_equal(e, np.clip(ef, -127, 127))
    # floor is at most one binade finer than rceil
    rc = oracle.e8m0_scale_byte(a).astype(np.int64)
    assert np.all((rc - byte >= 0) & (rc - byte <= 1))


def test_zero_and_tiny_blocks():
    assert oracle.e8m0_scale_byte([0.0])[0] == 0
    assert oracle.e8m0_scale_byte([0.0], floor=True)[0] == 0
    assert oracle.e8m0_scale_byte([2.0 ** -133])[0] == 0
    x = np.zeros((1, 32), np.uint16)
    x[0, 5] = 0x8000  # -0
    out = oracle.quantize_mx(x)
    assert out["s_row"][0] == 0
    assert out["q_row"][0, 5] == 0x80 and out["q_row"][0, 0] == 0x00
    # a subnormal-only block: scale 2^-127, payload x * 2^127 is still exact
    sub = np.zeros((1, 32), np.uint16)
    sub[0, :] = np.arange(1, 33)  # bf16 subnormals k * 2^-133
    out = oracle.quantize_mx(sub)
    assert out["s_row"][0] == 0
    want = oracle.fp8_encode(np.arange(1, 33) * 2.0 ** -133 * 2.0 ** 127)
    assert np.array_equal(out["q_row"][0], want)


def test_negative_values_rounding_to_zero_keep_sign():
    block = np.full(32, 0.0)
    block[0] = 300.0
    block[1] = -1e-6
    out = oracle.quantize_mx(oracle.bf16_round(block).reshape(1, 32))
    assert out["q_row"][0, 1] == 0x80


def test_nonfinite_block():
    x = oracle.bf16_round(np.ones(64)).reshape(1, 64)
    x[0, 3] = 0x7FC0  # NaN
    x[0, 40] = 0x7F80  # Inf
    out = oracle.quantize_mx(x)
    assert out["s_row"][oracle.swizzle_offset(0, 0, 64)] == 0xFF
    assert out["s_row"][oracle.swizzle_offset(0, 1, 64)] == 0xFF
    assert np.all(out["q_row"] == 0x7F)


# ------------------------------------------------ MX quantize, whole matrix --

def _blocked_swizzle_index(rows, kblocks):
    """Byte position of every logical scale (r, j), built by array reshapes:
    pad to (R_t*128, K_t*4), view as (R_t, 4 groups, 32, K_t, 4), and order
    the bytes as (R_t, K_t, 32, 4 groups, 4).  Written without the oracle."""
    rt, kt = math.ceil(rows / 128), math.ceil(kblocks / 4)
    idx = np.arange(rt * 128 * kt * 4).reshape(rt, 4, 32, kt, 4)
    # idx[t, g, i, u, c] is the logical (row = t*128 + g*32 + i, block = u*4 + c)
    logical = idx.reshape(rt * 128, kt * 4)
    order = np.transpose(idx, (0, 3, 2, 1, 4)).reshape(-1)
    pos = np.empty_like(order)
    pos[order] = np.arange(order.size)
    return pos[logical.reshape(-1)].reshape(rt * 128, kt * 4)[:rows, :kblocks]


def _torch_mx_recipe(x_bits, floor=False):
    """Independent MX quantization with torch ops: block amax, power-of-two
    scale from a float evaluation, payload by torch's float8 cast of x / s."""
    x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).to(torch.float64)
    rows, cols = x.shape
    blocks = x.reshape(rows, cols // 32, 32)
    amax = blocks.abs().amax(dim=-1)
    if floor:
        e = torch.floor(torch.log2(amax)) - 8
    else:
        e = torch.ceil(torch.log2(amax / 448.0))
    e = torch.where(amax == 0, torch.full_like(e, -127), e).clamp(-127, 127)
    v = (blocks * torch.pow(2.0, -e).unsqueeze(-1)).to(torch.float32)
    vs = v.clamp(-448.0, 448.0)  # torch's cast does not saturate by itself
    q = vs.to(torch.float8_e4m3fn).view(torch.uint8).reshape(rows, cols)
    return q.numpy(), (e + 127).to(torch.int64).numpy()


@pytest.mark.parametrize("dist", ["normal", "student", "loguniform", "outliers"])
@pytest.mark.parametrize("floor", [False, True])
def test_quantize_mx_vs_torch_recipe(dist, floor):
    rng = np.random.default_rng(11)
    rows, cols = 160, 320  # a ragged 128-row tile and a ragged K tile
    if dist == "normal":
        v = rng.normal(size=(rows, cols))
    elif dist == "student":
        v = rng.standard_t(4, size=(rows, cols))
    elif dist == "loguniform":
        v = 10 ** rng.uniform(-8, -2, size=(rows, cols)) * rng.choice([-1, 1], size=(rows, cols))
    else:
        v = rng.normal(size=(rows, cols)) * 0.02
        v[:, rng.permutation(cols)[:4]] *= 50
    x = oracle.bf16_round(v)
    out = oracle.quantize_mx(x, oracle.ROWWISE | oracle.COLWISE | (oracle.SCALE_FLOOR if floor else 0))
    q_ref, byte_ref = _torch_mx_recipe(x, floor)
    assert np.array_equal(out["q_row"], q_ref)
    pos = _blocked_swizzle_index(rows, cols // 32)
    assert np.array_equal(out["s_row"][pos], byte_ref)
    # colwise = the same recipe on the transposed matrix
    qt_ref, bt_ref = _torch_mx_recipe(np.ascontiguousarray(x.T), floor)
    assert np.array_equal(out["q_col"], qt_ref)
    pos_t = _blocked_swizzle_index(cols, rows // 32)
    assert np.array_equal(out["s_col"][pos_t], bt_ref)
    # every byte not holding a logical scale is padding = 0
    mask = np.ones(out["s_row"].size, bool)
    mask[pos.reshape(-1)] = False
    assert not out["s_row"][mask].any()


def test_quantize_mx_error_bound():
    """|x - x^| <= half an E4M3 spacing at x/s, times s (no saturation: rceil)."""
    rng = np.random.default_rng(3)
    x = oracle.bf16_round(rng.standard_t(3, size=(64, 256)))
    out = oracle.quantize_mx(x)
    xv = oracle.bf16_decode(x)
    pos = _blocked_swizzle_index(64, 8)
    s = np.ldexp(1.0, out["s_row"][pos].astype(int) - 127)
    s_full = np.repeat(s, 32, axis=1)
    v = xv / s_full
    q = oracle.fp8_decode(out["q_row"])
    assert np.all(np.abs(v) <= 448)
    _, ex = np.frexp(np.abs(v))
    spacing = np.ldexp(1.0, np.maximum(ex - 1, -6) - 3)  # E4M3: 3 mantissa bits, min normal 2^-6
    assert np.all(np.abs(v - q) <= spacing / 2)


def test_swizzle_bijective_and_geometry():
    for rows, k in ((128, 128), (300, 96), (1, 32), (257, 4096)):
        kb = k // 32
        offs = np.array([[oracle.swizzle_offset(r, j, k) for j in range(kb)] for r in range(rows)])
        assert len(np.unique(offs)) == rows * kb
        assert offs.min() >= 0 and offs.max() < oracle.scale_bytes(rows, k)
        kt = math.ceil(k / 128)
        for r in range(0, rows, 37):
            for j in range(kb):
                assert offs[r, j] // 512 == (r // 128) * kt + j // 4  # its 128 x 4 tile
        # 32-row groups of one 4-column tile: the 4 K-blocks of a row are adjacent
        for r in range(0, rows, 29):
            for j in range(0, kb - kb % 4, 4):
                assert list(offs[r, j:j + 4] - offs[r, j]) == [0, 1, 2, 3]
        assert np.array_equal(offs, _blocked_swizzle_index(rows, kb))


def test_quantize_grouped_matches_per_group():
    rng = np.random.default_rng(5)
    counts = [0, 130, 1, 0, 255, 128]
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = oracle.bf16_round(rng.normal(size=(off[-1], 96)))
    q, s = oracle.quantize_mx_grouped(x, off)
    base = 0
    for g, m in enumerate(counts):
        if m == 0:
            continue
        sub = oracle.quantize_mx(x[off[g]:off[g + 1]])
        assert np.array_equal(q[off[g]:off[g + 1]], sub["q_row"])
        nb = sub["s_row"].size
        start = base // 128 * math.ceil(96 / 128) * 512
        assert np.array_equal(s[start:start + nb], sub["s_row"])
        base += (m + 127) // 128 * 128
    assert s.size == base // 128 * 512


# ------------------------------------------------------------ per-tensor --

def _page_recipe(x_bits, fmt):
    """The book's exercise-6 quantizer written with torch ops (fp32 tensors)."""
    fmax = 448.0 if fmt == E4M3 else 57344.0
    dt = torch.float8_e4m3fn if fmt == E4M3 else torch.float8_e5m2
    x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).float()
    amax = x.abs().amax().clamp_min(1e-12)
    # the quotient as one correctly rounded fp32 division (tensor / tensor);
    # torch's python-scalar / tensor form multiplies by a reciprocal instead
    scale = torch.tensor(fmax, dtype=torch.float32) / amax
    q = (x * scale).to(dt)
    return x.abs().amax().item(), scale.item(), q.view(torch.uint8).numpy()


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("case", ["outliers", "tiny", "zeros", "loguniform"])
def test_quantize_tensor_vs_page_recipe(fmt, case):
    rng = np.random.default_rng(2)
    if case == "outliers":
        v = rng.normal(size=(64, 512))
        v[:, rng.permutation(512)[:5]] *= 50
    elif case == "tiny":
        v = rng.normal(size=(37, 19)) * 1e-30
    elif case == "zeros":
        v = np.zeros((4, 8))
    else:
        v = 10 ** rng.uniform(-8, -2, size=(128, 64)) * rng.choice([-1, 1], size=(128, 64))
    x = oracle.bf16_round(v)
    amax, scale, q = oracle.quantize_tensor(x, fmt)
    r_amax, r_scale, r_q = _page_recipe(x, fmt)
    assert np.float32(amax) == np.float32(r_amax)
    assert np.float32(scale).view(np.uint32) == np.float32(r_scale).view(np.uint32)
    assert np.array_equal(q, r_q)
    if amax >= np.float32(1e-12):  # below the clamp everything is tiny
        top = 0x7E if fmt == E4M3 else 0x7B
        i = np.argmax(np.abs(oracle.bf16_decode(x)))
        assert q.reshape(-1)[i] & 0x7F == top  # amax * s rounds to the format max
    else:
        assert not np.any(q & 0x7F)


# ------------------------------------------------------------------ GEMMs --

def _deq_independent(q, s_bytes, rows, k):
    """Dequantize with torch's float8 decode and the reshape-built swizzle."""
    vals = torch_fp8_decode(q, E4M3).reshape(rows, k)
    pos = _blocked_swizzle_index(rows, k // 32)
    scales = np.ldexp(1.0, s_bytes[pos].astype(np.int64) - 127)
    return vals * np.repeat(scales, 32, axis=1)


def test_gemm_mx_vs_numpy():
    rng = np.random.default_rng(9)
    M, N, K = 130, 72, 160
    a = oracle.quantize_mx(oracle.bf16_round(rng.standard_t(4, size=(M, K))))
    b = oracle.quantize_mx(oracle.bf16_round(rng.normal(size=(N, K)) * 0.02))
    ref = _deq_independent(a["q_row"], a["s_row"], M, K) @ _deq_independent(b["q_row"], b["s_row"], N, K).T
    got = oracle.gemm_mx(a["q_row"], a["s_row"], b["q_row"], b["s_row"])
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    rows = np.array([129, 0, 64])
    got_r = oracle.gemm_mx(a["q_row"], a["s_row"], b["q_row"], b["s_row"], rows=rows)
    assert np.array_equal(got_r, got[rows])


def test_gemm_mx_special_cases_exact():
    rng = np.random.default_rng(4)
    N, K = 40, 64
    b = oracle.quantize_mx(oracle.bf16_round(rng.normal(size=(N, K))))
    bdeq = _deq_independent(b["q_row"], b["s_row"], N, K)
    # one-hot A rows (value 1.0 = code 0x38 with scale byte 127)
    M = K
    qa = np.zeros((M, K), np.uint8)
    qa[np.arange(M), np.arange(K)] = 0x38
    sa = np.zeros(oracle.scale_bytes(M, K), np.uint8)
    for r in range(M):
        for j in range(K // 32):
            sa[oracle.swizzle_offset(r, j, K)] = 127
    got = oracle.gemm_mx(qa, sa, b["q_row"], b["s_row"])
    assert np.array_equal(got, bdeq.T)  # C[m, n] = deq(B)[n, m], exactly
    # K = 32 of small powers of two: the FP64 sum is exact
    vals = 2.0 ** rng.integers(-3, 4, size=(8, 32)) * rng.choice([-1, 1], size=(8, 32))
    a2 = oracle.quantize_mx(oracle.bf16_round(vals))
    got2 = oracle.gemm_mx(a2["q_row"], a2["s_row"], a2["q_row"], a2["s_row"])
    assert np.array_equal(got2, vals @ vals.T)


@pytest.mark.parametrize("fa,fb", [(E4M3, E4M3), (E4M3, E5M2), (E5M2, E4M3)])
def test_gemm_tensor_vs_page_recipe(fa, fb):
    rng = np.random.default_rng(6)
    X = oracle.bf16_round(rng.normal(size=(33, 96)))
    W = oracle.bf16_round(rng.normal(size=(24, 96)) * 0.02)
    ax, sx, qx = oracle.quantize_tensor(X, fa)
    aw, sw, qw = oracle.quantize_tensor(W, fb)
    got = oracle.gemm_tensor(qx.reshape(33, 96), fa, sx, qw.reshape(24, 96), fb, sw)
    xf = torch_fp8_decode(qx, fa).reshape(33, 96)
    wf = torch_fp8_decode(qw, fb).reshape(24, 96)
    ref = (xf @ wf.T) / (float(sx) * float(sw))
    assert np.allclose(got, ref, rtol=1e-12, atol=0)


def test_gemm_grouped_vs_numpy():
    rng = np.random.default_rng(8)
    counts = [3, 0, 140, 1, 64]
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    G, N, K = len(counts), 48, 96
    x = oracle.bf16_round(rng.normal(size=(off[-1], K)))
    qa, sa = oracle.quantize_mx_grouped(x, off)
    w = oracle.bf16_round(rng.normal(size=(G * N, K)) * 0.02)
    wq = oracle.quantize_mx(w)
    qw = wq["q_row"].reshape(G, N, K)
    # N % 128 != 0 here, so build the per-expert scale arrays one by one
    sw = np.concatenate([oracle.quantize_mx(w[g * N:(g + 1) * N])["s_row"] for g in range(G)])
    got = oracle.gemm_grouped(qa, sa, qw, sw, off)
    base = 0
    for g, m in enumerate(counts):
        if m:
            # group g's A rows are rows 0..m-1 of a padded block starting at `base`
            start = base // 128 * math.ceil(K / 128) * 512
            nb = oracle.scale_bytes(m, K)
            adeq = _deq_independent(qa[off[g]:off[g + 1]], sa[start:start + nb], m, K)
            wdeq = _deq_independent(qw[g], sw[g * oracle.scale_bytes(N, K):(g + 1) * oracle.scale_bytes(N, K)], N, K)
            assert np.allclose(got[off[g]:off[g + 1]], adeq @ wdeq.T, rtol=1e-12, atol=1e-15)
        base += (m + 127) // 128 * 128
    want = [1, 150, 207]
    got_w = oracle.gemm_grouped(qa, sa, qw, sw, off, rows=want)
    assert np.array_equal(got_w, got[want])


# ----------------------------------------------------------- dequantize --

def test_dequantize_vs_torch_and_closed_form():
    """s q rounded once to BF16: against torch's float8 decode times the
    scale, rounded by torch (an independent path), and exact where the
    product is a BF16 value."""
    rng = np.random.default_rng(12)
    rows, cols = 160, 256
    q = rng.integers(0, 256, size=(rows, cols), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x38  # no NaN codes in this part
    bytes_ = rng.integers(90, 165, size=(rows, cols // 32))
    s = np.zeros(oracle.scale_bytes(rows, cols), np.uint8)
    pos = _blocked_swizzle_index(rows, cols // 32)
    s[pos] = bytes_
    got = oracle.dequantize_mx(q, s)
    vals = torch_fp8_decode(q, E4M3) * np.repeat(np.ldexp(1.0, bytes_ - 127), 32, axis=1)
    want = torch.from_numpy(vals.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)  # the products are exact in fp32 here
    # every value here is exactly representable: decoding gives the product back
    assert np.array_equal(oracle.bf16_decode(got), vals)


def test_dequantize_roundtrip_and_specials():
    rng = np.random.default_rng(13)
    x = oracle.bf16_round(rng.standard_t(4, size=(96, 128)))
    qd = oracle.quantize_mx(x)
    back = oracle.bf16_decode(oracle.dequantize_mx(qd["q_row"], qd["s_row"]))
    xv = oracle.bf16_decode(x)
    # |x - x^| bounded by half an E4M3 spacing at the block scale (rceil: no clipping)
    pos = _blocked_swizzle_index(96, 4)
    sc = np.repeat(np.ldexp(1.0, qd["s_row"][pos].astype(int) - 127), 32, axis=1)
    _, ex = np.frexp(np.abs(xv / sc))
    spacing = np.ldexp(1.0, np.maximum(ex - 1, -6) - 3) * sc
    assert np.all(np.abs(xv - back) <= spacing / 2)
    # NaN code, NaN scale, overflow to Inf, BF16-subnormal rounding
    q = np.array([[0x7F] + [0x38] * 31, [0x7E] * 32, [0x01] * 32], np.uint8)
    s = np.zeros(oracle.scale_bytes(3, 32), np.uint8)
    s[oracle.swizzle_offset(0, 0, 32)] = 127
    s[oracle.swizzle_offset(1, 0, 32)] = 254   # 448 * 2^127 overflows BF16
    s[oracle.swizzle_offset(2, 0, 32)] = 3     # 2^-9 * 2^-124 = 2^-133: smallest BF16 subnormal
    out = oracle.dequantize_mx(q, s)
    assert np.isnan(oracle.bf16_decode(out[0, :1]))[0]
    assert out[0, 1] == 0x3F80                  # 1.0
    assert np.all(out[1] == 0x7F80)             # +Inf
    assert np.all(out[2] == 0x0001)


def test_dequantize_grouped_is_plain_per_group():
    """Each group's scale rows are whole 128-row tiles of the grouped array,
    so the grouped dequantization of group g equals the plain one of its rows
    with that slice of tiles."""
    rng = np.random.default_rng(14)
    counts = np.array([0, 130, 5, 0, 256, 1])
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows, cols = int(off[-1]), 96
    x = oracle.bf16_round(rng.standard_normal((rows, cols)) * np.exp(rng.uniform(-8, 8, (rows, 1))))
    q, s = oracle.quantize_mx_grouped(x, off)
    got = oracle.dequantize_mx_grouped(q, s, off)
    nkc = (cols + 127) // 128
    padded = 0
    for g in range(counts.size):
        m = int(counts[g])
        if m:
            tiles = (m + 127) // 128
            sl = s[padded // 128 * nkc * 512:(padded // 128 + tiles) * nkc * 512]
            want = oracle.dequantize_mx(q[off[g]:off[g + 1]], sl)
            assert np.array_equal(got[off[g]:off[g + 1]], want)
        padded += (m + 127) // 128 * 128


# -------------------------------------------------------------- SwiGLU --

def test_swiglu_vs_torch_silu():
    """FP64 g sigma(g) u against torch's float64 SiLU times u, plus the
    identity silu(g) - silu(-g) = g and sigma(g) = 1 in FP64 for g >= 40."""
    rng = np.random.default_rng(15)
    rows, f = 64, 96
    h = oracle.bf16_round(rng.standard_normal((rows, 2 * f)) * 4)
    y = oracle.swiglu(h)
    hv = oracle.bf16_decode(h)
    g, u = torch.from_numpy(hv[:, :f]), torch.from_numpy(hv[:, f:])
    want = (torch.nn.functional.silu(g) * u).numpy()
    np.testing.assert_allclose(y, want, rtol=1e-15, atol=0)  # a few FP64 ulps
    # odd part of SiLU: silu(g) - silu(-g) = g
    gg = hv[:, :f]
    ones = oracle.bf16_round(np.ones_like(gg))
    pos = oracle.swiglu(np.concatenate([h[:, :f], ones], axis=1))
    neg = oracle.swiglu(np.concatenate([h[:, :f] ^ np.uint16(0x8000), ones], axis=1))
    np.testing.assert_allclose(pos - neg, gg, rtol=1e-15, atol=1e-300)
    # saturated gate: y = g u exactly; far negative gate: |y| below every BF16 value
    big = oracle.bf16_round(np.array([[40.0, -3.5], [100.0, 7.0], [-200.0, 1e30]]))
    hb = np.stack([big[:, 0], big[:, 1]], axis=1)
    yb = oracle.swiglu(hb)[:, 0]
    assert yb[0] == 40.0 * -3.5 and yb[1] == 700.0
    assert yb[2] < 0 and abs(yb[2]) < 2.0 ** -134


# ------------------------------------------------------- route weighting --

def _bf16_neighbours_table():
    bits = all_bf16_bits()
    vals = oracle.bf16_decode(bits)
    keep = np.isfinite(vals) & ~((bits == 0x8000))
    order = np.argsort(vals[keep], kind="stable")
    return vals[keep][order], bits[keep][order]


def _correctly_rounded_bf16(v: Fraction, table) -> int:
    """RNE of an exact rational to BF16 by comparing the two neighbours."""
    vals, bits = table
    top = Fraction(2) ** 128 - Fraction(2) ** 119  # halfway to the next binade: rounds to Inf
    if v >= top:
        return 0x7F80
    if v <= -top:
        return 0xFF80
    i = int(np.searchsorted(vals, float(v), side="left"))
    cands = [j for j in (i - 1, i, i + 1) if 0 <= j < vals.size]
    best = min(cands, key=lambda j: (abs(Fraction(vals[j]) - v), int(bits[j]) & 1))
    b = int(bits[best])
    if vals[best] == 0.0:
        b = 0x8000 if v < 0 else 0x0000
    return b


def test_route_weight_is_one_rounding_of_the_exact_product():
    rng = np.random.default_rng(16)
    table = _bf16_neighbours_table()
    tokens, cols, rows = 12, 64, 40
    dy = oracle.bf16_round(rng.standard_normal((tokens, cols)) * np.exp(rng.uniform(-30, 30, (tokens, 1))))
    # exact midpoints: 1 * (1 + 2^-8) and 1 * (1 + 3 * 2^-8) tie to the even neighbour
    dy[0, :4] = [0x3F80, 0x3F80, 0xBF80, 0x0001]
    tok = rng.integers(0, tokens, rows).astype(np.int32)
    tok[:3] = 0
    w = rng.uniform(0, 1, rows).astype(np.float32)
    w[:3] = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 2.0 ** -20], np.float32)
    tok[3] = -1  # out of range: zero row
    got = oracle.route_weight(dy, tok, w)
    assert list(got[0, :4]) == [0x3F80, 0x3F80, 0xBF80, 0x0001] and got[1, 0] == 0x3F82
    assert np.all(got[3] == 0)
    dyv = oracle.bf16_decode(dy)
    for i in range(rows):
        if tok[i] < 0:
            continue
        for c in range(0, cols, 7):
            v = Fraction(float(w[i])) * Fraction(float(dyv[tok[i], c]))
            assert got[i, c] == _correctly_rounded_bf16(v, table), (i, c)


# ------------------------------------------- delayed and automatic scaling --

def _torch_sat_cast(y32: torch.Tensor, fmt) -> np.ndarray:
    """torch's float8 cast after clamping to the largest finite value (torch
    itself does not saturate)."""
    fmax = 448.0 if fmt == E4M3 else 57344.0
    dt = torch.float8_e4m3fn if fmt == E4M3 else torch.float8_e5m2
    y = torch.where(torch.isnan(y32), y32, y32.clamp(-fmax, fmax))
    return y.to(dt).view(torch.uint8).numpy()


def _bf16_tensor(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_scaled_cast_vs_torch(fmt):
    """q = FP8(fp32(x s)) against torch's fp32 product and float8 cast, for
    scales that leave the tensor in range, saturate it or push it into the
    subnormals; the saturated count against torch's values at +-max."""
    rng = np.random.default_rng(40)
    bits = oracle.bf16_round(rng.standard_normal(5000) * np.exp(rng.uniform(-12, 12, 5000)))
    x = _bf16_tensor(bits)
    fmax = 448.0 if fmt == E4M3 else 57344.0
    for s in [1.0, 0.37, 1e3, 2.0 ** 20, 3e-5, 1e-12]:
        q, amax, sat = oracle.quantize_tensor_scaled(bits, fmt, s)
        y = x.float() * torch.tensor(s, dtype=torch.float32)
        want = _torch_sat_cast(y, fmt)
        assert np.array_equal(q, want), s
        dt = torch.float8_e4m3fn if fmt == E4M3 else torch.float8_e5m2
        assert sat == int((torch.from_numpy(want).view(dt).float().abs() == fmax).sum())
        assert amax == np.float32(np.abs(oracle.bf16_decode(bits)).max())


class _BookDelayedScale:
    """The book's delayed-scaling cast, restated with torch fp32 ops: scale
    from the max of the amax history (clamped at 1e-12) times the margin,
    cast, then record this tensor's amax at the ring pointer."""

    def __init__(self, history_len, margin, fmt):
        self.hist = torch.zeros(history_len, dtype=torch.float32)
        self.ptr = 0
        self.margin = margin
        self.fmt = fmt
        self.fmax = torch.tensor(448.0 if fmt == E4M3 else 57344.0, dtype=torch.float32)

    def cast(self, x):
        amax = self.hist.max().clamp_min(1e-12)
        scale = (self.fmax / amax) * self.margin
        q = _torch_sat_cast(x.float() * scale, self.fmt)
        self.hist[self.ptr] = x.float().abs().amax()
        self.ptr = (self.ptr + 1) % self.hist.numel()
        return q, scale


@pytest.mark.parametrize("fmt,margin", [(E4M3, 1.0), (E4M3, 0.9), (E5M2, 1.0)])
def test_delayed_scaling_vs_book_recipe(fmt, margin):
    """Seven steps with a 4-entry history: the zero history of the first step
    (scale 448e12, everything saturates), growth, a spike that saturates the
    next step's cast, and the ring wrapping."""
    rng = np.random.default_rng(41)
    book = _BookDelayedScale(4, margin, fmt)
    hist, pos = np.zeros(4, np.float32), 0
    for step, mag in enumerate([1.0, 1.0, 2.0, 50.0, 1.0, 0.01, 0.01]):
        bits = oracle.bf16_round(rng.standard_normal(3000) * mag)
        q, s, amax, sat, hist, pos = oracle.quantize_tensor_delayed(bits, fmt, margin, hist, pos)
        wq, ws = book.cast(_bf16_tensor(bits))
        assert np.float32(s) == np.float32(ws.item()), step
        assert np.array_equal(q, wq), step
        assert np.array_equal(hist, book.hist.numpy()) and pos == book.ptr, step
        if step == 0:
            assert sat == int((np.abs(oracle.bf16_decode(bits)) > 0).sum())  # all nonzero saturate


@pytest.mark.parametrize("fmt_in,fmt_out", [(E4M3, E4M3), (E5M2, E5M2), (E4M3, E5M2), (E5M2, E4M3)])
def test_requantize_vs_torch(fmt_in, fmt_out):
    """q'' = FP8(s_out (g' / s_in)) in fp32, against torch, for every code;
    and the identity for s_out = s_in, one format."""
    codes = np.arange(256, dtype=np.uint8)
    dt_in = torch.float8_e4m3fn if fmt_in == E4M3 else torch.float8_e5m2
    g = torch.from_numpy(codes).view(dt_in).float()
    for s_in, s_out in [(3.0, 1.5), (448.0 / 3.1, 448.0 / 7.9), (1.0, 2.0 ** -10), (0.75, 0.75 * 1.001)]:
        got, sat = oracle.requantize_tensor(codes, fmt_in, s_in, s_out, fmt_out)
        y = torch.tensor(s_out, dtype=torch.float32) * (g / torch.tensor(s_in, dtype=torch.float32))
        want = _torch_sat_cast(y, fmt_out)
        nan = torch.isnan(g).numpy()
        assert np.array_equal(got[~nan], want[~nan]), (s_in, s_out)
        assert np.all((got[nan] & 0x7F) == 0x7F)
    if fmt_in == fmt_out:
        same, _ = oracle.requantize_tensor(codes, fmt_in, 5.0, 5.0, fmt_out)
        finite = ~torch.isnan(g).numpy() & ~torch.isinf(g).numpy()
        assert np.array_equal(same[finite], codes[finite])


# ------------------------------------------- SwiGLU, correctly rounded --

def _mp_swiglu_bf16(gbits, ubits, table, digits=90):
    """BF16 RNE of g sigma(g) u from a 90-digit mpmath evaluation (exact
    rational rounding of the high-precision value)."""
    mpmath = pytest.importorskip("mpmath")
    out = []
    with mpmath.workdps(digits):
        for gb, ub in zip(gbits, ubits):
            g = Fraction(float(oracle.bf16_decode(np.array([gb], np.uint16))[0]))
            u = Fraction(float(oracle.bf16_decode(np.array([ub], np.uint16))[0]))
            gm = mpmath.mpf(g.numerator) / g.denominator
            um = mpmath.mpf(u.numerator) / u.denominator
            y = gm * um / (1 + mpmath.exp(-gm))
            man, exp = mpmath.mpf(y).man_exp if y != 0 else (0, 0)  # |mantissa|
            yf = Fraction(int(man)) * (Fraction(2) ** int(exp)) if y != 0 else Fraction(0)
            yf = -yf if y < 0 else yf
            b = _correctly_rounded_bf16(yf, table)
            if yf == 0:
                b = 0x8000 if (g < 0) != (u < 0) else 0x0000
            out.append(b)
    return np.array(out, np.uint16)


def _near_midpoint_pairs(n, rel, seed):
    """(g, u) BF16 pairs whose FP64 SwiGLU value lies within rel of a BF16
    rounding midpoint: the values a fast fp32 evaluation cannot round."""
    rng = np.random.default_rng(seed)
    found_g, found_u = [], []
    while len(found_g) < n:
        g = oracle.bf16_round(rng.standard_normal(1 << 20) * np.exp(rng.uniform(-3, 3, 1 << 20)))
        u = oracle.bf16_round(rng.standard_normal(1 << 20) * np.exp(rng.uniform(-20, 20, 1 << 20)))
        y = oracle.swiglu(np.stack([g, u], axis=1))[:, 0]
        a = np.abs(y)
        # the midpoint next to a: a's BF16 truncation plus half its unit
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
        unit = np.ldexp(1.0, (e - 7).astype(int))
        mid = np.floor(a / unit) * unit + unit / 2
        hit = (a > 2.0 ** -120) & (np.abs(a - mid) <= rel * a)
        found_g += list(g[hit])
        found_u += list(u[hit])
    return np.array(found_g[:n], np.uint16), np.array(found_u[:n], np.uint16)


def test_swiglu_bf16_vs_mpmath_random():
    """Correctly rounded SwiGLU against a 90-digit evaluation on random gates
    and ups spanning many binades (both signs, tiny and huge values)."""
    rng = np.random.default_rng(41)
    n = 3000
    g = oracle.bf16_round(rng.standard_normal(n) * np.exp(rng.uniform(-12, 5, n)))
    u = oracle.bf16_round(rng.standard_normal(n) * np.exp(rng.uniform(-60, 60, n)))
    g[:40] = oracle.bf16_round(-rng.uniform(60, 90, 40))  # e^g near fp32's normal limit
    got = oracle.swiglu_bf16(np.stack([g, u], axis=1))[:, 0]
    want = _mp_swiglu_bf16(g, u, _bf16_neighbours_table())
    assert np.array_equal(got, want), np.nonzero(got != want)[0][:8]


def test_swiglu_bf16_vs_mpmath_near_midpoints():
    """Values within 2^-24 of a BF16 rounding midpoint (where fp32 cannot
    tell the side): every one rounded as the 90-digit value says."""
    g, u = _near_midpoint_pairs(120, 2.0 ** -24, 42)
    got = oracle.swiglu_bf16(np.stack([g, u], axis=1))[:, 0]
    want = _mp_swiglu_bf16(g, u, _bf16_neighbours_table())
    assert np.array_equal(got, want), np.nonzero(got != want)[0][:8]
    # the plain FP64 rounding differs exactly where sigma(g) rounds to 1 in
    # FP64 (gates past ~37) and g u is itself a midpoint: it ties to even there
    h = np.stack([g, u], axis=1)
    plain = oracle.bf16_round(oracle.swiglu(h)[:, 0])
    d = plain != want
    gd, ud = oracle.bf16_decode(g), oracle.bf16_decode(u)
    assert np.all(gd[d] > 36) and np.all(oracle.swiglu(h)[d, 0] == gd[d] * ud[d])


def test_swiglu_bf16_saturated_gate_on_a_midpoint():
    """g u exactly a BF16 midpoint with a large positive gate: y = g u (1 -
    e^-g + ...) lies just below |g u| however small e^-g is, so it rounds
    toward zero; an FP64 evaluation lands on the midpoint itself and would
    take the even neighbour.  321 = 3 * 107, 259 = 7 * 37 and 265 = 5 * 53
    are odd 9-bit integers: (2k + 1) 2^e halves BF16 units."""
    cases = [(3.0 * 16, 107 / 128), (3.0 * 2 ** 20, -107 * 2.0 ** -30),
             (7.0 * 8, 37 / 64), (5.0 * 2 ** 100, 53 * 2.0 ** -120),
             (3.0 * 2 ** 120, -107.0 * 2 ** -10), (7.0 * 2 ** 60, 37.0 * 2 ** -90),
             (5.0 * 16, -53.0 * 2 ** 10)]
    g = oracle.bf16_round(np.array([c[0] for c in cases]))
    u = oracle.bf16_round(np.array([c[1] for c in cases]))
    assert np.array_equal(oracle.bf16_decode(g) * 1.0, [c[0] for c in cases])
    assert np.array_equal(oracle.bf16_decode(u) * 1.0, [c[1] for c in cases])
    p = oracle.bf16_decode(g) * oracle.bf16_decode(u)
    got = oracle.swiglu_bf16(np.stack([g, u], axis=1))[:, 0]
    for pv, b in zip(p, got):
        a = abs(pv)
        e = math.floor(math.log2(a))
        unit = 2.0 ** (e - 7)
        assert (a / unit) % 1 == 0.5  # a midpoint
        below = math.floor(a / unit) * unit
        assert float(oracle.bf16_decode(np.array([b], np.uint16))[0]) == math.copysign(below, pv)
    # the plain FP64 rounding ties to even instead, which differs for some
    plain = oracle.bf16_round(oracle.swiglu(np.stack([g, u], axis=1))[:, 0])
    assert (plain != got).any()
    # for gates small enough, a 90-digit evaluation agrees
    small = np.abs(oracle.bf16_decode(g)) < 100
    want = _mp_swiglu_bf16(g[small], u[small], _bf16_neighbours_table())
    assert np.array_equal(got[small], want)


def test_swiglu_bf16_equals_fp64_rounding_away_from_midpoints():
    rng = np.random.default_rng(43)
    h = oracle.bf16_round(rng.standard_normal((256, 512)) * 3)
    y = oracle.swiglu(h)
    assert np.array_equal(oracle.swiglu_bf16(h), oracle.bf16_round(y))


def test_swiglu_bf16_tiny_gate_half_product_on_a_midpoint():
    """|g| below 2^-54 with g u / 2 exactly a BF16 midpoint: sigma(g) = 1/2 +
    g/4 + ..., so |y| lies above the midpoint for g > 0 and below it for
    g < 0; in FP64 sigma(g) rounds to 1/2 exactly.  Gates near 1e-10 checked
    against the 90-digit evaluation too."""
    cases = [(7 * 2.0 ** -110, 37 * 2.0 ** 90), (-7 * 2.0 ** -110, 37 * 2.0 ** 90),
             (3 * 2.0 ** -120, 107 * 2.0 ** 100), (-3 * 2.0 ** -120, -107 * 2.0 ** 100),
             (5 * 2.0 ** -125, 53 * 2.0 ** 110), (-3 * 2.0 ** -60, 107.0)]
    g = oracle.bf16_round(np.array([c[0] for c in cases]))
    u = oracle.bf16_round(np.array([c[1] for c in cases]))
    gd, ud = oracle.bf16_decode(g), oracle.bf16_decode(u)
    assert np.array_equal(gd, [c[0] for c in cases]) and np.array_equal(ud, [c[1] for c in cases])
    got = oracle.swiglu_bf16(np.stack([g, u], axis=1))[:, 0]
    for gv, pv, b in zip(gd, gd * ud, got):
        m = abs(pv) / 2
        e = math.floor(math.log2(m))
        unit = 2.0 ** (e - 7)
        assert (m / unit) % 1 == 0.5  # the half product is a midpoint
        want = (math.floor(m / unit) + (1 if gv > 0 else 0)) * unit
        assert float(oracle.bf16_decode(np.array([b], np.uint16))[0]) == math.copysign(want, pv)
    rng = np.random.default_rng(44)
    gs = oracle.bf16_round(rng.standard_normal(400) * 1e-10)
    us = oracle.bf16_round(rng.standard_normal(400) * 1e20)
    want = _mp_swiglu_bf16(gs, us, _bf16_neighbours_table())
    assert np.array_equal(oracle.swiglu_bf16(np.stack([gs, us], axis=1))[:, 0], want)
