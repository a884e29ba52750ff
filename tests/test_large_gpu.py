"""Sizes past 2^31 elements or bytes, where any 32-bit index in a kernel
would wrap: the MX quantizer (both orientations) on a 65600 x 32768 BF16
tensor (2.15 G values), MX GEMMs whose A, B or C each hold more than 2^31
bytes, the per-tensor quantizer over 2.15 G values, a grouped GEMM over
65600 x 32768 expert rows, and the routed conversions (dequantize, SwiGLU +
quantize, route weighting + quantize) reading or writing past 2^31 values.  The outputs are too large for the oracle, so
sampled row tiles, rows and columns (the first, one in the middle and the
ragged last ones, where a wrapped index would land) are checked against it:
the MX rule is local to a 32-value block, so the oracle quantizing a sampled
slab or row on its own gives exactly that slab's bytes, and a sampled row of
C depends only on its row of A and on B."""
import numpy as np
import pytest
import torch

import mxfp8_precision_gemms_gb300 as m
import oracle
from gpu_util import assert_ok, device, gemm_tolerance_check, host

pytestmark = pytest.mark.gpu

ROWS, K = 65600, 32768          # 2,149,580,800 values; the last row tile holds 64 rows
SAMPLE_ROWS = [0, 1, 127, 32768, 65535, 65536, 65599]


def _bits(t: torch.Tensor) -> np.ndarray:
    return host(t.contiguous().view(torch.int16)).view(np.uint16)


def _randn_bf16(rows, cols, seed, scale=1.0):
    """Seeded N(0, scale^2) BF16 on the device, drawn in slabs of 8192 rows."""
    g = torch.Generator(device=device()).manual_seed(seed)
    x = torch.empty((rows, cols), dtype=torch.bfloat16, device=device())
    for r0 in range(0, rows, 8192):
        r1 = min(rows, r0 + 8192)
        x[r0:r1] = (torch.randn((r1 - r0, cols), generator=g, device=device()) * scale).to(torch.bfloat16)
    return x


@pytest.fixture(scope="module")
def big_x():
    x = _randn_bf16(ROWS, K, 11)
    yield x
    del x
    torch.cuda.empty_cache()


def test_quantize_mx_both_orientations_past_2g_values(big_x):
    got = m.fp8_quantize_mx(big_x, m.MX_ROWWISE | m.MX_COLWISE)
    assert_ok()
    nkr, nkc = K // 128, (ROWS + 127) // 128   # K tiles of the rowwise / colwise operand
    s_row, s_col = host(got["s_row"]), host(got["s_col"])
    for rt in (0, 256, nkc - 1):
        r0, r1 = rt * 128, min(ROWS, rt * 128 + 128)
        want = oracle.quantize_mx(_bits(big_x[r0:r1]), oracle.ROWWISE | oracle.COLWISE)
        assert np.array_equal(host(got["q_row"][r0:r1]), want["q_row"]), rt
        # row tile rt's scale tiles are contiguous: (rt * nkr + kt) * 512
        assert np.array_equal(s_row[rt * nkr * 512:(rt + 1) * nkr * 512], want["s_row"]), rt
        assert np.array_equal(host(got["q_col"][:, r0:r1]), want["q_col"]), rt
        # colwise tile (ct, rt) at (ct * nkc + rt) * 512; the slab alone has one K tile
        for ct in range(K // 128):
            o = (ct * nkc + rt) * 512
            assert np.array_equal(s_col[o:o + 512], want["s_col"][ct * 512:(ct + 1) * 512]), (rt, ct)
    del got


def _mx_rows(x: torch.Tensor, rows):
    return oracle.quantize_mx(_bits(x[rows]), oracle.ROWWISE)


def test_mx_gemm_a_and_b_past_2g_bytes(big_x):
    """A (65600 x 32768 bytes) as the left operand, then as the right one."""
    w = _randn_bf16(256, K, 12, 0.05)
    qx = m.fp8_quantize_mx(big_x, m.MX_ROWWISE)
    qw = m.fp8_quantize_mx(w, m.MX_ROWWISE)
    assert_ok()
    rows = torch.tensor(SAMPLE_ROWS, device=device())
    rx, rw = _mx_rows(big_x, rows), _mx_rows(w, slice(None))
    ref = oracle.gemm_mx(rx["q_row"], rx["s_row"], rw["q_row"], rw["s_row"])   # 7 x 256

    c = m.fp8_scaled_gemm(m.GEMM_MX, qx["q_row"], qx["s_row"], qw["q_row"], qw["s_row"])
    assert_ok()
    gemm_tolerance_check(c[rows], ref, "A past 2^31 bytes")
    del c
    ct = m.fp8_scaled_gemm(m.GEMM_MX, qw["q_row"], qw["s_row"], qx["q_row"], qx["s_row"])
    assert_ok()
    gemm_tolerance_check(ct[:, rows], ref.T.copy(), "B past 2^31 bytes")
    del ct, qx, qw


def test_mx_gemm_c_past_2g_bytes(big_x):
    """C = 65600 x 16400 BF16 (2.15 GB) from K = 128."""
    a = big_x[:, :128].contiguous()
    b = _randn_bf16(16400, 128, 13)
    qa, qb = m.fp8_quantize_mx_batch([a, b])
    c = m.fp8_scaled_gemm(m.GEMM_MX, qa["q_row"], qa["s_row"], qb["q_row"], qb["s_row"])
    assert_ok()
    rows = torch.tensor(SAMPLE_ROWS, device=device())
    ra, rb = _mx_rows(a, rows), _mx_rows(b, slice(None))
    ref = oracle.gemm_mx(ra["q_row"], ra["s_row"], rb["q_row"], rb["s_row"])
    gemm_tolerance_check(c[rows], ref, "C past 2^31 bytes")
    del c, qa, qb, a, b


@pytest.mark.parametrize("workspace", [False, True])
def test_quantize_tensor_past_2g_values(big_x, workspace):
    x = big_x.view(-1)
    ws = torch.zeros(m.mxfp8_tensor_workspace_bytes(), dtype=torch.uint8, device=device()) if workspace else None
    q, amax, scale = m.fp8_quantize_tensor(x, m.FP8_E4M3, workspace=ws)
    assert_ok()
    bits = _bits(x)
    # the amax is the largest BF16 magnitude; the oracle's rule gives the
    # scale from it (a tensor holding only that value has the same amax)
    top = bits[np.argmax(bits & 0x7FFF)]
    w_amax, w_scale, _ = oracle.quantize_tensor(np.array([top], np.uint16), m.FP8_E4M3)
    assert host(amax).view(np.uint32)[0] == np.float32(w_amax).view(np.uint32)
    assert host(scale).view(np.uint32)[0] == np.float32(w_scale).view(np.uint32)
    n = bits.size
    for lo in (0, n // 2, (1 << 31) - 2048, n - 4096):   # one straddles 2^31
        wq, _, _ = oracle.quantize_tensor_scaled(bits[lo:lo + 4096], m.FP8_E4M3, float(w_scale))
        assert np.array_equal(host(q[lo:lo + 4096]), wq), lo
    del q, bits


def test_grouped_gemm_past_2g_bytes(big_x):
    counts = [20000, 0, 32768, 12832]   # 65600 rows, an empty expert
    G, N = len(counts), 256
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    off_d = torch.from_numpy(off).to(device())
    w = _randn_bf16(G * N, K, 14, 0.05)
    qa, sa = m.fp8_quantize_mx_grouped(big_x, off_d)
    qw = m.fp8_quantize_mx(w, m.MX_ROWWISE)
    c = m.fp8_grouped_gemm(qa, sa, qw["q_row"].view(G, N, K), qw["s_row"], off_d)
    assert_ok()
    for g in range(G):
        lo, hi = int(off[g]), int(off[g + 1])
        if hi == lo:
            continue
        rows = sorted({lo, lo + 1, (lo + hi) // 2, hi - 1})
        rx = _mx_rows(big_x, torch.tensor(rows, device=device()))
        rw = _mx_rows(w[g * N:(g + 1) * N], slice(None))
        ref = oracle.gemm_mx(rx["q_row"], rx["s_row"], rw["q_row"], rw["s_row"])
        gemm_tolerance_check(c[torch.tensor(rows, device=device())], ref, f"expert {g}")
    del c, qa, sa, qw, w


def _row_tiles(rows):
    last = (rows + 127) // 128 - 1
    return [(rt, rt * 128, min(rows, rt * 128 + 128)) for rt in (0, last // 2, last)]


def test_dequantize_past_2g_values(big_x):
    qx = m.fp8_quantize_mx(big_x, m.MX_ROWWISE)
    out = m.fp8_dequantize_mx(qx["q_row"], qx["s_row"])
    assert_ok()
    for rt, r0, r1 in _row_tiles(ROWS):
        want = oracle.quantize_mx(_bits(big_x[r0:r1]), oracle.ROWWISE)
        assert np.array_equal(_bits(out[r0:r1]), oracle.dequantize_mx(want["q_row"], want["s_row"])), rt
    del qx, out


def test_swiglu_quantize_past_2g_values(big_x):
    """h = the 65600 x 32768 tensor as gate | up (f = 16384): input offsets
    past 2^31 values."""
    f = K // 2
    q, s = m.fp8_swiglu_quantize_mx(big_x)
    assert_ok()
    nkc = f // 128
    sh = host(s)
    for rt, r0, r1 in _row_tiles(ROWS):
        want = oracle.quantize_mx(oracle.swiglu_bf16(_bits(big_x[r0:r1])), oracle.ROWWISE)
        assert np.array_equal(host(q[r0:r1]), want["q_row"]), rt
        assert np.array_equal(sh[rt * nkc * 512:(rt + 1) * nkc * 512], want["s_row"]), rt
    del q, s


def test_route_weight_quantize_past_2g_values(big_x):
    """dY = the 65600 x 32768 tensor; 65600 dispatched rows gather scattered
    tokens with random fp32 weights."""
    rows = ROWS
    tok = torch.from_numpy((np.arange(rows, dtype=np.int64) * 7919 % ROWS).astype(np.int32)).to(device())
    g = torch.Generator(device=device()).manual_seed(15)
    wt = torch.rand(rows, generator=g, device=device(), dtype=torch.float32)
    q, s = m.fp8_route_weight_quantize_mx(big_x, tok, wt)
    assert_ok()
    nkc = K // 128
    sh = host(s)
    for rt, r0, r1 in _row_tiles(rows):
        gathered = _bits(big_x[tok[r0:r1].long()])
        bits = oracle.route_weight(gathered, np.arange(r1 - r0, dtype=np.int32), host(wt[r0:r1]))
        want = oracle.quantize_mx(bits, oracle.ROWWISE)
        assert np.array_equal(host(q[r0:r1]), want["q_row"]), rt
        assert np.array_equal(sh[rt * nkc * 512:(rt + 1) * nkc * 512], want["s_row"]), rt
    del q, s
