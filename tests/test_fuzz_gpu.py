"""Seeded random shapes against the oracle: ragged M, N and K for the MX GEMM
(through both the slot-pair and the per-slot load paths), ragged expert
groups for the grouped GEMM, and random tensor shapes for the quantizers in
every orientation.  The shapes are drawn once from a fixed seed, so a
failure names a reproducible case."""
import numpy as np
import pytest
import torch

import mxfp8_precision_gemms_gb300 as m
import oracle
from gpu_util import assert_ok, device, gemm_tolerance_check, host, to_dev_bf16

pytestmark = pytest.mark.gpu

_rng = np.random.default_rng(2024)
GEMM_CASES = [(int(_rng.integers(1, 700)), int(_rng.integers(1, 90)) * 8, int(_rng.integers(1, 40)) * 32)
              for _ in range(24)]
QUANT_CASES = [(int(_rng.integers(1, 40)) * 32, int(_rng.integers(1, 60)) * 32) for _ in range(16)]
GROUP_CASES = [[int(c) for c in _rng.integers(0, 400, int(_rng.integers(1, 9)))] for _ in range(8)]
TENSOR_CASES = [(int(_rng.integers(1, 600)), int(_rng.integers(1, 70)) * 8, int(_rng.integers(1, 40)) * 16,
                 int(_rng.integers(0, 2)), int(_rng.integers(0, 2))) for _ in range(12)]


def _bits(shape, seed, scale=1.0):
    r = np.random.default_rng(seed)
    v = r.standard_normal(shape) * scale * np.exp(r.uniform(-3, 3, (shape[0], 1)))
    return oracle.bf16_round(v)


@pytest.mark.parametrize("M,N,K", GEMM_CASES)
def test_mx_gemm_random_shapes(M, N, K):
    a, b = _bits((M, K), M * 7 + K), _bits((N, K), N * 5 + K)
    qa, qb = m.fp8_quantize_mx_batch([to_dev_bf16(a), to_dev_bf16(b)])
    c = m.fp8_scaled_gemm(m.GEMM_MX, qa["q_row"], qa["s_row"], qb["q_row"], qb["s_row"])
    assert_ok()
    ra, rb = oracle.quantize_mx(a, oracle.ROWWISE), oracle.quantize_mx(b, oracle.ROWWISE)
    assert np.array_equal(host(qa["q_row"]), ra["q_row"]) and np.array_equal(host(qb["s_row"]), rb["s_row"])
    ref = oracle.gemm_mx(ra["q_row"], ra["s_row"], rb["q_row"], rb["s_row"])
    gemm_tolerance_check(c, ref, f"mx gemm {M}x{N}x{K}")


@pytest.mark.parametrize("rows,cols", QUANT_CASES)
def test_quantize_random_shapes_all_orientations(rows, cols):
    x = _bits((rows, cols), rows + 3 * cols, 4.0)
    for flags in (m.MX_ROWWISE, m.MX_COLWISE, m.MX_ROWWISE | m.MX_COLWISE,
                  m.MX_ROWWISE | m.MX_COLWISE | m.MX_SCALE_FLOOR):
        got = m.fp8_quantize_mx(to_dev_bf16(x), flags)
        assert_ok()
        want = oracle.quantize_mx(x, flags)
        for k in want:
            assert np.array_equal(host(got[k]), want[k]), (flags, k)


@pytest.mark.parametrize("counts", GROUP_CASES)
def test_grouped_gemm_random_groups(counts):
    G, N, K = len(counts), 256, 256
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    total = int(off[-1])
    x = _bits((max(total, 1), K), total + 11)[:total]
    w = _bits((G * N, K), G + 13, 0.05)
    off_d = torch.from_numpy(off).to(device())
    qa, sa = m.fp8_quantize_mx_grouped(to_dev_bf16(x), off_d)
    qw = m.fp8_quantize_mx(to_dev_bf16(w), m.MX_ROWWISE)
    c = m.fp8_grouped_gemm(qa, sa, qw["q_row"].view(G, N, K), qw["s_row"], off_d)
    assert_ok()
    if total == 0:
        return
    rqa, rsa = oracle.quantize_mx_grouped(x, off)
    assert np.array_equal(host(qa), rqa)
    rw = oracle.quantize_mx(w, oracle.ROWWISE)
    for g in range(G):
        lo, hi = int(off[g]), int(off[g + 1])
        if hi == lo:
            continue
        xa = oracle.quantize_mx(x[lo:hi], oracle.ROWWISE)
        ref = oracle.gemm_mx(xa["q_row"], xa["s_row"], rw["q_row"][g * N:(g + 1) * N],
                             oracle.quantize_mx(w[g * N:(g + 1) * N], oracle.ROWWISE)["s_row"])
        gemm_tolerance_check(c[lo:hi], ref, f"group {g} of {counts}")


@pytest.mark.parametrize("M,N,K,fa,fb", TENSOR_CASES)
def test_tensor_gemm_random_shapes(M, N, K, fa, fb):
    a, b = _bits((M, K), M + 5 * K), _bits((N, K), N + 7 * K)
    qa, _, sa = m.fp8_quantize_tensor(to_dev_bf16(a).reshape(-1), fa)
    qb, _, sb = m.fp8_quantize_tensor(to_dev_bf16(b).reshape(-1), fb)
    c = m.fp8_scaled_gemm(m.GEMM_TENSOR, qa.view(M, K), sa, qb.view(N, K), sb, a_fmt=fa, b_fmt=fb)
    assert_ok()
    wa, wsa, wqa = oracle.quantize_tensor(a.reshape(-1), fa)
    wb, wsb, wqb = oracle.quantize_tensor(b.reshape(-1), fb)
    assert np.array_equal(host(qa), wqa.reshape(-1)) and np.array_equal(host(qb), wqb.reshape(-1))
    ref = oracle.gemm_tensor(wqa.reshape(M, K), fa, wsa, wqb.reshape(N, K), fb, wsb)
    gemm_tolerance_check(c, ref, f"tensor gemm {M}x{N}x{K} fmts {fa}{fb}")
