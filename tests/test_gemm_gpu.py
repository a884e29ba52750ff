"""GPU parity of the scaled GEMMs against the FP64 oracle.

Both sides quantize the same seeded BF16 inputs (the quantized bytes are
checked equal first), then the GPU GEMM output must satisfy
|gpu - ref| <= 1e-2 |ref| + 1e-3 rms(ref) elementwise; special cases whose
exact result is a BF16 value must match bit for bit."""
import numpy as np
import pytest
import torch

import mxfp8_precision_gemms_gb300 as m
import oracle
import workloads
from gpu_util import assert_ok, device, filled, gemm_tolerance_check, host, to_dev_bf16, to_dev_u8

pytestmark = pytest.mark.gpu


def quantize_both(bits, flags=m.MX_ROWWISE):
    got = m.fp8_quantize_mx(to_dev_bf16(bits), flags)
    want = oracle.quantize_mx(bits, flags)
    for k in want:
        assert np.array_equal(host(got[k]), want[k]), k
    return got, want


# K % 256 == 0 loads each slot pair with one copy per operand (3D K-chunk
# maps); other K (384, 640: odd numbers of 128-wide K steps) take the
# per-slot copies with a half-empty last pair
MX_SHAPES = [(128, 256, 128), (256, 256, 256), (200, 136, 96), (1, 8, 32), (384, 512, 1024),
             (130, 264, 4096), (1000, 1024, 160), (256, 768, 2048), (300, 512, 384),
             (512, 256, 640)]


@pytest.mark.parametrize("M,N,K", MX_SHAPES)
def test_mx_gemm_matches_oracle(M, N, K):
    a = workloads.bits(workloads.student_t((M, K), 4, 1, 0))
    b = workloads.bits(workloads.normal((N, K), 0.02, 1, 1))
    ga, wa = quantize_both(a)
    gb, wb = quantize_both(b)
    c = filled((M, N), 0x7FC0, torch.int16).view(torch.bfloat16)
    m.fp8_scaled_gemm(m.GEMM_MX, ga["q_row"], ga["s_row"], gb["q_row"], gb["s_row"], c=c)
    assert_ok()
    ref = oracle.gemm_mx(wa["q_row"], wa["s_row"], wb["q_row"], wb["s_row"])
    gemm_tolerance_check(c, ref, f"MX {M}x{N}x{K}")


@pytest.mark.parametrize("K", [128, 256])
def test_mx_gemm_short_last_wave(K):
    """4096 x 4032: 256 tiles leave 28 for the last wave of 76 CTA pairs,
    which run as 56 half tiles of 128 columns (the last tile's second half
    holds 64 valid columns); K = 128 takes the per-slot copies, K = 256 the
    slot-pair copies.  Every element against the oracle."""
    M, N = 4096, 4032
    a = workloads.bits(workloads.student_t((M, K), 4, 3, 0))
    b = workloads.bits(workloads.normal((N, K), 0.02, 3, 1))
    ga, wa = quantize_both(a)
    gb, wb = quantize_both(b)
    c = filled((M, N), 0x7FC0, torch.int16).view(torch.bfloat16)
    m.fp8_scaled_gemm(m.GEMM_MX, ga["q_row"], ga["s_row"], gb["q_row"], gb["s_row"], c=c)
    assert_ok()
    ref = oracle.gemm_mx(wa["q_row"], wa["s_row"], wb["q_row"], wb["s_row"])
    gemm_tolerance_check(c, ref, f"short last wave K={K}")


def test_mx_gemm_ldc_and_untouched_padding():
    M, N, K, ldc = 192, 264, 256, 280
    a = workloads.bits(workloads.normal((M, K), 1.0, 2, 0))
    b = workloads.bits(workloads.normal((N, K), 1.0, 2, 1))
    ga, wa = quantize_both(a)
    gb, wb = quantize_both(b)
    cbuf = filled((M, ldc), 0x1234, torch.int16)
    c = cbuf.view(torch.bfloat16)[:, :N]
    m.fp8_scaled_gemm(m.GEMM_MX, ga["q_row"], ga["s_row"], gb["q_row"], gb["s_row"], c=c)
    assert_ok()
    assert (host(cbuf)[:, N:] == 0x1234).all()
    ref = oracle.gemm_mx(wa["q_row"], wa["s_row"], wb["q_row"], wb["s_row"])
    gemm_tolerance_check(c, ref, "ldc")


def test_mx_gemm_one_hot_rows_exact():
    """A = identity (value 1.0 at scale 1): C = bf16(deq(B)^T) exactly."""
    N, K = 256, 256
    b = workloads.bits(workloads.normal((N, K), 1.0, 3, 1))
    gb, wb = quantize_both(b)
    M = K
    qa = np.zeros((M, K), np.uint8)
    qa[np.arange(M), np.arange(K)] = 0x38  # E4M3 1.0
    sa = np.zeros(oracle.scale_bytes(M, K), np.uint8)
    for r in range(M):
        for j in range(K // 32):
            sa[oracle.swizzle_offset(r, j, K)] = 127
    c = m.fp8_scaled_gemm(m.GEMM_MX, to_dev_u8(qa), to_dev_u8(sa), gb["q_row"], gb["s_row"])
    assert_ok()
    ref = oracle.gemm_mx(qa, sa, wb["q_row"], wb["s_row"])
    want = oracle.bf16_round(ref)
    assert np.array_equal(host(c.view(torch.int16)).view(np.uint16), want)


def test_mx_gemm_small_integers_exact():
    """K = 32 and 64 of small powers of two: FP32 sums are exact, outputs are BF16 values."""
    rng = np.random.default_rng(0)
    for K in (32, 64):
        v = 2.0 ** rng.integers(-2, 3, size=(128, K)) * rng.choice([-1, 1], size=(128, K))
        bits = oracle.bf16_round(v)
        ga, wa = quantize_both(bits)
        c = m.fp8_scaled_gemm(m.GEMM_MX, ga["q_row"], ga["s_row"], ga["q_row"], ga["s_row"])
        assert_ok()
        ref = oracle.gemm_mx(wa["q_row"], wa["s_row"], wa["q_row"], wa["s_row"])
        assert np.array_equal(ref, v @ v.T)
        assert np.array_equal(host(c.view(torch.int16)).view(np.uint16), oracle.bf16_round(ref))


def test_mx_gemm_scales_vary_per_block():
    """Blocks of wildly different magnitude along K: a wrong scale layout or
    scale id shows up at once."""
    M, N, K = 256, 256, 512
    g = torch.Generator().manual_seed(11)
    ka = torch.pow(2.0, torch.randint(-20, 20, (M, K // 32), generator=g).float()).repeat_interleave(32, 1)
    kb = torch.pow(2.0, torch.randint(-20, 20, (N, K // 32), generator=g).float()).repeat_interleave(32, 1)
    a = workloads.bits((torch.randn(M, K, generator=g) * ka).to(torch.bfloat16))
    b = workloads.bits((torch.randn(N, K, generator=g) * kb).to(torch.bfloat16))
    ga, wa = quantize_both(a)
    gb, wb = quantize_both(b)
    c = m.fp8_scaled_gemm(m.GEMM_MX, ga["q_row"], ga["s_row"], gb["q_row"], gb["s_row"])
    assert_ok()
    ref = oracle.gemm_mx(wa["q_row"], wa["s_row"], wb["q_row"], wb["s_row"])
    gemm_tolerance_check(c, ref, "per-block scales")


def test_mx_gemm_dgrad_wgrad_orientations():
    """dX = dY W and dW = dY^T X through colwise quantization (Eq. 60)."""
    T, din, dout = 256, 384, 512
    dy = workloads.bits(workloads.log_uniform_signed((T, dout), 1e-8, 1e-2, 4, 0))
    w = workloads.bits(workloads.normal((dout, din), 0.02, 4, 1))
    x = workloads.bits(workloads.normal((T, din), 1.0, 4, 2))
    gdy, wdy = quantize_both(dy, m.MX_ROWWISE | m.MX_COLWISE)
    gw, ww = quantize_both(w, m.MX_COLWISE)
    gx, wx = quantize_both(x, m.MX_COLWISE)
    dx = m.fp8_scaled_gemm(m.GEMM_MX, gdy["q_row"], gdy["s_row"], gw["q_col"], gw["s_col"])
    dw = m.fp8_scaled_gemm(m.GEMM_MX, gdy["q_col"], gdy["s_col"], gx["q_col"], gx["s_col"])
    assert_ok()
    gemm_tolerance_check(dx, oracle.gemm_mx(wdy["q_row"], wdy["s_row"], ww["q_col"], ww["s_col"]), "dgrad")
    gemm_tolerance_check(dw, oracle.gemm_mx(wdy["q_col"], wdy["s_col"], wx["q_col"], wx["s_col"]), "wgrad")


@pytest.mark.parametrize("fa,fb", [(m.FP8_E4M3, m.FP8_E4M3), (m.FP8_E4M3, m.FP8_E5M2),
                                   (m.FP8_E5M2, m.FP8_E4M3)])
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (300, 520, 4112), (64, 8, 16)])
def test_tensor_gemm_matches_oracle(fa, fb, M, N, K):
    w = workloads.tensor4096(seed=5, device="cpu", m=M, n=N, k=K)
    xb, wbits = workloads.bits(w["X"]), workloads.bits(w["W"])
    qx, ax, sx = m.fp8_quantize_tensor(to_dev_bf16(xb), fa)
    qw, aw, sw = m.fp8_quantize_tensor(to_dev_bf16(wbits), fb)
    c = m.fp8_scaled_gemm(m.GEMM_TENSOR, qx, sx, qw, sw, a_fmt=fa, b_fmt=fb)
    assert_ok()
    _, rsx, rqx = oracle.quantize_tensor(xb, fa)
    _, rsw, rqw = oracle.quantize_tensor(wbits, fb)
    assert np.array_equal(host(qx), rqx) and np.array_equal(host(qw), rqw)
    ref = oracle.gemm_tensor(rqx, fa, rsx, rqw, fb, rsw)
    gemm_tolerance_check(c, ref, "tensor")


def _grouped_case(counts, N, K, seed=0):
    off = workloads.offsets_from_counts(counts)
    total = int(off[-1])
    G = len(counts)
    x = workloads.bits(workloads.normal((total, K), 1.0, seed, 0))
    w = workloads.bits(workloads.normal((G * N, K), 0.02, seed, 1))
    off_d = torch.from_numpy(off).to(device())
    qa, sa = m.fp8_quantize_mx_grouped(to_dev_bf16(x), off_d)
    qw = torch.empty((G, N, K), dtype=torch.uint8, device=device())
    sb = m.mxfp8_scale_bytes(N, K)
    sw = torch.empty(G * sb, dtype=torch.uint8, device=device())
    wd = to_dev_bf16(w)
    for g in range(G):
        m.fp8_quantize_mx(wd[g * N:(g + 1) * N], m.MX_ROWWISE, q_row=qw[g], s_row=sw[g * sb:(g + 1) * sb])
    rqa, rsa = oracle.quantize_mx_grouped(x, off)
    assert np.array_equal(host(qa), rqa) and np.array_equal(host(sa)[: rsa.size], rsa)
    rw = [oracle.quantize_mx(w[g * N:(g + 1) * N]) for g in range(G)]
    rqw = np.stack([r["q_row"] for r in rw])
    rsw = np.concatenate([r["s_row"] for r in rw])
    assert np.array_equal(host(qw), rqw) and np.array_equal(host(sw), rsw)
    return off, off_d, qa, sa, qw, sw, rqa, rsa, rqw, rsw


@pytest.mark.parametrize("counts,N,K", [([0, 1, 127, 128, 129, 0, 300, 5], 256, 256),
                                        ([64] * 4, 136, 96), ([0, 0, 1000, 0], 512, 512),
                                        ([3, 700, 2, 90, 11, 256, 1, 0, 45], 1024, 2048),
                                        ([40, 0, 300, 129], 256, 384)])
def test_grouped_gemm_matches_oracle(counts, N, K):
    off, off_d, qa, sa, qw, sw, rqa, rsa, rqw, rsw = _grouped_case(counts, N, K)
    c = filled((int(off[-1]), N), 0x7FC0, torch.int16).view(torch.bfloat16)
    m.fp8_grouped_gemm(qa, sa, qw, sw, off_d, c=c)
    assert_ok()
    ref = oracle.gemm_grouped(rqa, rsa, rqw, rsw, off)
    gemm_tolerance_check(c, ref, f"grouped {counts}")


def test_grouped_gemm_bad_offsets_recorded():
    counts = [64, 64, 128]
    off, off_d, qa, sa, qw, sw, *_ = _grouped_case(counts, 128, 128)
    bad = torch.tensor([0, 100, 50, 256], dtype=torch.int32, device=device())
    c = filled((256, 128), 0x1111, torch.int16)
    m.fp8_grouped_gemm(qa, sa, qw, sw, bad, c=c.view(torch.bfloat16))
    assert m.mxfp8_last_device_status() == m.MXFP8_ERR_DEVICE_CHECK
    assert (host(c) == 0x1111).all()


def test_wait_timeout_is_reported_and_context_survives():
    a = workloads.bits(workloads.normal((256, 256), 1.0, 6, 0))
    ga, wa = quantize_both(a)
    m.mxfp8_set_wait_limit_ns(50_000_000)  # 50 ms
    try:
        m.mxfp8_debug_inject_wait_timeout(True)
        m.fp8_scaled_gemm(m.GEMM_MX, ga["q_row"], ga["s_row"], ga["q_row"], ga["s_row"])
        assert m.mxfp8_last_device_status() == m.MXFP8_ERR_TIMEOUT
    finally:
        m.mxfp8_debug_inject_wait_timeout(False)
        m.mxfp8_set_wait_limit_ns(0)
    c = m.fp8_scaled_gemm(m.GEMM_MX, ga["q_row"], ga["s_row"], ga["q_row"], ga["s_row"])
    assert_ok()
    gemm_tolerance_check(c, oracle.gemm_mx(wa["q_row"], wa["s_row"], wa["q_row"], wa["s_row"]), "after timeout")


def test_k_zero_and_empty():
    dev = device()
    c = filled((64, 64), 0x3F80, torch.int16)
    z = torch.empty(0, dtype=torch.uint8, device=dev)
    m.fp8_scaled_gemm(m.GEMM_MX, z.view(64, 0), z, z.view(64, 0), z, c=c.view(torch.bfloat16))
    assert_ok()
    assert (host(c) == 0).all()
    a0 = torch.empty((0, 32), dtype=torch.uint8, device=dev)
    b8 = torch.empty((8, 32), dtype=torch.uint8, device=dev)
    e = m.fp8_scaled_gemm(m.GEMM_MX, a0, z, b8, z)
    assert e.shape == (0, 8)
