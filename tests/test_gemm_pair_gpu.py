"""GPU parity of fp8_scaled_gemm_pair, two independent scaled GEMMs in one
launch with the CTA pairs split between them: each output is bit-identical
to fp8_scaled_gemm's (the same dot products in the same K order) and within
the GEMM tolerance of the FP64 oracle; shapes that split a last wave into
half tiles on one side, ragged and single-row problems, per-tensor mode with
mixed formats, degenerate problems, C with a wider row stride, and the
backward workload's dgrad and wgrad at full size."""
import numpy as np
import pytest
import torch

import mxfp8_precision_gemms_gb300 as m
import oracle
import workloads
from gpu_util import assert_ok, device, filled, gemm_tolerance_check, host, to_dev_bf16

pytestmark = pytest.mark.gpu


def _mx_problem(M, N, K, seed):
    a = workloads.bits(workloads.student_t((M, K), 4, seed, 0))
    b = workloads.bits(workloads.normal((N, K), 0.02, seed, 1))
    ga = m.fp8_quantize_mx(to_dev_bf16(a), m.MX_ROWWISE)
    gb = m.fp8_quantize_mx(to_dev_bf16(b), m.MX_ROWWISE)
    wa = oracle.quantize_mx(a, oracle.ROWWISE)
    wb = oracle.quantize_mx(b, oracle.ROWWISE)
    assert np.array_equal(host(ga["q_row"]), wa["q_row"]) and np.array_equal(host(gb["s_row"]), wb["s_row"])
    return (dict(a=ga["q_row"], a_scale=ga["s_row"], b=gb["q_row"], b_scale=gb["s_row"]),
            (wa["q_row"], wa["s_row"], wb["q_row"], wb["s_row"]))


def _same(x, y):
    return torch.equal(x.contiguous().view(torch.int16), y.contiguous().view(torch.int16))


PAIRS = [((384, 512, 1024), (256, 768, 2048)),    # different K, slot-pair copies
         ((1000, 1024, 160), (200, 136, 96)),     # ragged; per-slot copies
         ((4096, 4032, 256), (512, 256, 640)),    # a last wave split into half tiles
         ((1, 8, 32), (130, 264, 4096)),          # one row against a long K
         ((2048, 2048, 512), (2048, 2048, 512))]  # equal halves


@pytest.mark.parametrize("s0,s1", PAIRS)
def test_mx_pair_matches_single_calls_and_oracle(s0, s1):
    g0, w0 = _mx_problem(*s0, seed=11)
    g1, w1 = _mx_problem(*s1, seed=12)
    c0, c1 = m.fp8_scaled_gemm_pair(m.GEMM_MX, g0, g1)
    assert_ok()
    for g, c, w, shape in ((g0, c0, w0, s0), (g1, c1, w1, s1)):
        single = m.fp8_scaled_gemm(m.GEMM_MX, g["a"], g["a_scale"], g["b"], g["b_scale"])
        assert_ok()
        assert _same(c, single), shape
        gemm_tolerance_check(c, oracle.gemm_mx(*w), f"pair MX {shape}")


def test_tensor_pair_mixed_formats():
    """Per-tensor mode: E4M3 x E5M2 beside E5M2 x E4M3, scales from the
    per-tensor quantizer."""
    out, refs, singles = [], [], []
    for (M, N, K), (fa, fb), seed in (((640, 512, 768), (m.FP8_E4M3, m.FP8_E5M2), 21),
                                      ((256, 1024, 256), (m.FP8_E5M2, m.FP8_E4M3), 22)):
        a = workloads.normal((M, K), 1.0, seed, 0, device=device())
        b = workloads.normal((N, K), 0.05, seed, 1, device=device())
        qa, aa, sa = m.fp8_quantize_tensor(a, fa)
        qb, ab, sb = m.fp8_quantize_tensor(b, fb)
        g = dict(a=qa.view(M, K), a_scale=sa, b=qb.view(N, K), b_scale=sb, a_fmt=fa, b_fmt=fb)
        out.append(g)
        singles.append(m.fp8_scaled_gemm(m.GEMM_TENSOR, g["a"], sa, g["b"], sb, a_fmt=fa, b_fmt=fb))
        refs.append(oracle.gemm_tensor(host(g["a"]), fa, float(host(sa)[0]), host(g["b"]), fb,
                                       float(host(sb)[0])))
    c0, c1 = m.fp8_scaled_gemm_pair(m.GEMM_TENSOR, out[0], out[1])
    assert_ok()
    for c, single, ref in zip((c0, c1), singles, refs):
        assert _same(c, single)
        gemm_tolerance_check(c, ref, "pair per-tensor")


def test_pair_with_degenerate_problem_and_wide_ldc():
    """K = 0 (C zero-filled) or M = 0 (nothing written) beside a normal
    problem; C in buffers with a wider row stride keeps its padding."""
    g0, w0 = _mx_problem(300, 512, 384, seed=31)
    N, ldc = 512, 520
    for other in ("k0", "m0"):
        cbuf = filled((300, ldc), 0x1234, torch.int16)
        c = cbuf.view(torch.bfloat16)[:, :N]
        g0c = dict(g0, c=c)
        if other == "k0":
            e = torch.empty((0,), dtype=torch.uint8, device=device())
            cz = filled((64, 128), 0x5555, torch.int16).view(torch.bfloat16)
            g1 = dict(a=torch.empty((64, 0), dtype=torch.uint8, device=device()), a_scale=e,
                      b=torch.empty((128, 0), dtype=torch.uint8, device=device()), b_scale=e, c=cz)
        else:
            g1, _ = _mx_problem(8, 256, 256, seed=32)
            g1 = dict(g1, a=g1["a"][:0])
            cz = filled((0, 256), 0x5555, torch.int16).view(torch.bfloat16)
            g1["c"] = cz
        c0, c1 = m.fp8_scaled_gemm_pair(m.GEMM_MX, g0c, g1)
        assert_ok()
        assert (host(cbuf)[:, N:] == 0x1234).all()
        gemm_tolerance_check(c0, oracle.gemm_mx(*w0), f"pair beside {other}")
        if other == "k0":
            assert (host(cz.view(torch.int16)) == 0).all()


def test_backward_pair_full_size():
    """The backward workload's dgrad (8192 x 4096 x 4096) and wgrad (4096 x
    4096 x 8192) in one launch: bit-identical to the two separate GEMMs, and
    sampled rows against the oracle."""
    w = workloads.backward(seed=0, device=device())
    dy = m.fp8_quantize_mx(w["dY"], m.MX_ROWWISE | m.MX_COLWISE)
    wt = m.fp8_quantize_mx(w["W"], m.MX_COLWISE)
    xt = m.fp8_quantize_mx(w["X"], m.MX_COLWISE)
    gd = dict(a=dy["q_row"], a_scale=dy["s_row"], b=wt["q_col"], b_scale=wt["s_col"])
    gw = dict(a=dy["q_col"], a_scale=dy["s_col"], b=xt["q_col"], b_scale=xt["s_col"])
    dx, dw = m.fp8_scaled_gemm_pair(m.GEMM_MX, gd, gw)
    assert_ok()
    dx1 = m.fp8_scaled_gemm(m.GEMM_MX, gd["a"], gd["a_scale"], gd["b"], gd["b_scale"])
    dw1 = m.fp8_scaled_gemm(m.GEMM_MX, gw["a"], gw["a_scale"], gw["b"], gw["b_scale"])
    assert_ok()
    assert _same(dx, dx1) and _same(dw, dw1)
    rng = np.random.default_rng(7)
    for c, g, n_rows, what in ((dx, gd, 8192, "dgrad"), (dw, gw, 4096, "wgrad")):
        rows = np.sort(rng.choice(n_rows, 16, replace=False)).astype(np.int64)
        ref = oracle.gemm_mx(host(g["a"]), host(g["a_scale"]), host(g["b"]), host(g["b_scale"]), rows=rows)
        gemm_tolerance_check(c[torch.from_numpy(rows).to(c.device)], ref, what)
