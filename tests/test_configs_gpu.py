"""Parity at the benchmark workloads' full sizes.

Every quantized byte (payload and scale arrays) is compared with the oracle
in full; GEMM outputs are compared on sampled rows (all columns of each
sampled row), with |gpu - ref| <= 1e-2 |ref| + 1e-3 rms(ref), rms taken over
the sampled outputs.  Inputs are drawn on the GPU by the seeded generators
and copied to the host for the oracle."""
import numpy as np
import pytest
import torch

import mxfp8_precision_gemms_gb300 as m
import oracle
import workloads
from gpu_util import assert_ok, device, gemm_tolerance_check, host

pytestmark = pytest.mark.gpu

ROW, COL = m.MX_ROWWISE, m.MX_COLWISE


def sample_rows(n, k, seed):
    rng = np.random.default_rng(seed)
    rows = set([0, n - 1, n // 2]) | set(rng.choice(n, size=k, replace=False).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def check_mx(t, flags):
    """GPU and oracle MX quantization of one workload tensor; bytes must match."""
    got = m.fp8_quantize_mx(t, flags)
    assert_ok()
    want = oracle.quantize_mx(workloads.bits(t), flags)
    for k in want:
        g = host(got[k])
        assert np.array_equal(g, want[k]), f"{k}: {(g != want[k]).sum()} bytes differ"
    return got, want


def test_mx256():
    w = workloads.mx256(seed=0, device=device())
    ga, wa = check_mx(w["A"], ROW)
    gb, wb = check_mx(w["B"], ROW)
    c = m.fp8_scaled_gemm(m.GEMM_MX, ga["q_row"], ga["s_row"], gb["q_row"], gb["s_row"])
    assert_ok()
    gemm_tolerance_check(c, oracle.gemm_mx(wa["q_row"], wa["s_row"], wb["q_row"], wb["s_row"]), "mx256")


def test_tensor4096():
    w = workloads.tensor4096(seed=0, device=device())
    out = {}
    ws = torch.zeros(m.mxfp8_tensor_workspace_bytes(), dtype=torch.uint8, device=device())
    for name in ("X", "W"):
        q, amax, scale = m.fp8_quantize_tensor(w[name], m.FP8_E4M3, workspace=ws)
        assert_ok()
        ra, rs, rq = oracle.quantize_tensor(workloads.bits(w[name]), oracle.E4M3)
        assert np.array_equal(host(q), rq)
        assert host(amax).view(np.uint32)[0] == np.float32(ra).view(np.uint32)
        assert host(scale).view(np.uint32)[0] == np.float32(rs).view(np.uint32)
        out[name] = (q, scale, rq, rs)
    c = m.fp8_scaled_gemm(m.GEMM_TENSOR, out["X"][0], out["X"][1], out["W"][0], out["W"][1])
    assert_ok()
    rows = sample_rows(4096, 40, 1)
    ref = oracle.gemm_tensor(out["X"][2], oracle.E4M3, out["X"][3], out["W"][2], oracle.E4M3,
                             out["W"][3], rows=rows)
    gemm_tolerance_check(c[torch.from_numpy(rows).to(c.device)], ref, "tensor4096")


def test_mlp_up():
    w = workloads.mlp_up(seed=0, device=device())
    gx, wx = check_mx(w["X"], ROW)
    gw, ww = check_mx(w["W"], ROW)
    c = m.fp8_scaled_gemm(m.GEMM_MX, gx["q_row"], gx["s_row"], gw["q_row"], gw["s_row"])
    assert_ok()
    rows = sample_rows(8192, 24, 2)
    ref = oracle.gemm_mx(wx["q_row"], wx["s_row"], ww["q_row"], ww["s_row"], rows=rows)
    gemm_tolerance_check(c[torch.from_numpy(rows).to(c.device)], ref, "mlp_up")


def test_backward():
    w = workloads.backward(seed=0, device=device())
    gdy, wdy = check_mx(w["dY"], ROW | COL)
    gw, ww = check_mx(w["W"], COL)
    gx, wx = check_mx(w["X"], COL)
    dx = m.fp8_scaled_gemm(m.GEMM_MX, gdy["q_row"], gdy["s_row"], gw["q_col"], gw["s_col"])
    dw = m.fp8_scaled_gemm(m.GEMM_MX, gdy["q_col"], gdy["s_col"], gx["q_col"], gx["s_col"])
    assert_ok()
    rows = sample_rows(8192, 24, 3)
    ref = oracle.gemm_mx(wdy["q_row"], wdy["s_row"], ww["q_col"], ww["s_col"], rows=rows)
    gemm_tolerance_check(dx[torch.from_numpy(rows).to(dx.device)], ref, "dgrad")
    rows = sample_rows(4096, 24, 4)
    ref = oracle.gemm_mx(wdy["q_col"], wdy["s_col"], wx["q_col"], wx["s_col"], rows=rows)
    gemm_tolerance_check(dw[torch.from_numpy(rows).to(dw.device)], ref, "wgrad")


def test_grouped():
    w = workloads.grouped(seed=0, device=device())
    off = w["offsets"]
    G, N, K = 64, 1024, 2048
    total = int(off[-1])
    assert total == 32768 * 8 and w["counts"].sum() == total
    off_d = torch.from_numpy(off).to(device())
    qa, sa = m.fp8_quantize_mx_grouped(w["X"], off_d)
    Wst = w["W"].reshape(G * N, K)
    qw = m.fp8_quantize_mx(Wst, ROW)
    assert_ok()
    rqa, rsa = oracle.quantize_mx_grouped(workloads.bits(w["X"]), off)
    assert np.array_equal(host(qa), rqa)
    assert np.array_equal(host(sa)[: rsa.size], rsa)
    rw = oracle.quantize_mx(workloads.bits(Wst), oracle.ROWWISE)
    assert np.array_equal(host(qw["q_row"]), rw["q_row"])
    assert np.array_equal(host(qw["s_row"]), rw["s_row"])
    c = m.fp8_grouped_gemm(qa, sa, qw["q_row"].view(G, N, K), qw["s_row"], off_d)
    assert_ok()
    # rows: the first and last row of every non-empty group, plus random ones
    rng = np.random.default_rng(5)
    want = set(rng.choice(total, size=64, replace=False).tolist())
    for g in range(G):
        if off[g + 1] > off[g]:
            want |= {int(off[g]), int(off[g + 1]) - 1}
    rows = np.array(sorted(want), dtype=np.int64)
    ref = oracle.gemm_grouped(rqa, rsa, rw["q_row"].reshape(G, N, K), rw["s_row"], off, rows=rows)
    gemm_tolerance_check(c[torch.from_numpy(rows).to(c.device)], ref, "grouped")
