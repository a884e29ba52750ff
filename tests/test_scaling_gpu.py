"""GPU parity of the per-tensor scaling kernels: the cast with a given scale
(amax and saturated count included), the delayed-scaling cast over an amax
history ring, and FP8-LM's requantization to a shared scale — all bit-exact
against the oracle, plus the package's DelayedScaling state object."""
import numpy as np
import pytest
import torch

import mxfp8_precision_gemms_gb300 as m
import oracle
import workloads
from gpu_util import assert_ok, device, host, to_dev_bf16, to_dev_u8
from mxfp8_precision_gemms_gb300 import scaling

pytestmark = pytest.mark.gpu

FMTS = [(m.FP8_E4M3, oracle.E4M3), (m.FP8_E5M2, oracle.E5M2)]


def _f32(v):
    return torch.tensor([float(np.float32(v))], dtype=torch.float32, device=device())


def _bits(n, seed, spread=12.0):
    rng = np.random.default_rng(seed)
    return oracle.bf16_round(rng.standard_normal(n) * np.exp(rng.uniform(-spread, spread, n)))


@pytest.mark.parametrize("fmt,ofmt", FMTS)
@pytest.mark.parametrize("n", [0, 1, 7, 8, 4099, 1 << 20])
def test_scaled_cast(fmt, ofmt, n):
    bits = _bits(n, n + fmt)
    x = to_dev_bf16(bits) if n else torch.empty(0, dtype=torch.bfloat16, device=device())
    for s in [1.0, 0.37, 1e3, 2.0 ** 20, 3e-5]:
        q, amax, sat = m.fp8_quantize_tensor_scaled(x, _f32(s), fmt)
        assert_ok()
        rq, ra, rs = oracle.quantize_tensor_scaled(bits, ofmt, s)
        assert np.array_equal(host(q), rq), s
        assert host(amax)[0] == ra and int(host(sat)[0]) == rs, s


@pytest.mark.parametrize("fmt,ofmt", FMTS)
@pytest.mark.parametrize("margin", [1.0, 0.9])
def test_delayed_scaling_sequence(fmt, ofmt, margin):
    """Seven steps with a 4-entry ring: zero history (saturating first cast),
    growth, a spike, decay, wrap-around; every output and the state."""
    st = scaling.DelayedScaling(history_len=4, margin=margin, fmt=fmt, device=device())
    hist, pos = np.zeros(4, np.float32), 0
    for step, mag in enumerate([1.0, 1.0, 2.0, 50.0, 1.0, 0.01, 0.01]):
        bits = _bits(10007, 50 + step, spread=1.0) if step else _bits(10007, 50, spread=1.0)
        bits = oracle.bf16_round(oracle.bf16_decode(bits) * mag)
        q, s, amax, sat = st.cast(to_dev_bf16(bits))
        assert_ok()
        rq, rs, ra, rsat, hist, pos = oracle.quantize_tensor_delayed(bits, ofmt, margin, hist, pos)
        assert host(s)[0] == rs and host(amax)[0] == ra and int(host(sat)[0]) == rsat, step
        assert np.array_equal(host(q), rq), step
        assert np.array_equal(host(st.history), hist) and int(host(st.pos)[0]) == pos, step


def test_delayed_scaling_bad_position_recorded():
    st = scaling.DelayedScaling(history_len=3, device=device())
    st.pos.fill_(7)
    st.cast(to_dev_bf16(_bits(64, 1)))
    assert m.mxfp8_last_device_status() == m.MXFP8_ERR_DEVICE_CHECK
    assert int(host(st.pos)[0]) == 1  # restarted at 0, then advanced


@pytest.mark.parametrize("fin,ofin", FMTS)
@pytest.mark.parametrize("fout,ofout", FMTS)
def test_requantize_every_code(fin, ofin, fout, ofout):
    codes = np.tile(np.arange(256, dtype=np.uint8), 5)[:1100]
    for s_in, s_out in [(3.0, 1.5), (448.0 / 3.1, 448.0 / 7.9), (1.0, 2.0 ** -10), (0.75, 0.75 * 1.001), (1.0, 300.0)]:
        q, sat = m.fp8_requantize_tensor(to_dev_u8(codes), _f32(s_in), _f32(s_out), fin, fout)
        assert_ok()
        rq, rsat = oracle.requantize_tensor(codes, ofin, s_in, s_out, ofout)
        assert np.array_equal(host(q), rq), (s_in, s_out)
        assert int(host(sat)[0]) == rsat


def test_requantize_large_with_tail():
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 256, size=(1 << 22) + 13, dtype=np.uint8)
    q, sat = m.fp8_requantize_tensor(to_dev_u8(codes), _f32(17.0), _f32(5.0))
    assert_ok()
    rq, rsat = oracle.requantize_tensor(codes, oracle.E4M3, 17.0, 5.0, oracle.E4M3)
    assert np.array_equal(host(q), rq) and int(host(sat)[0]) == rsat


def test_delayed_full_size_tensor4096():
    """Three delayed-scaling steps over the 4096 x 4096 outlier-column
    activation (the per-tensor workload), E4M3."""
    x = workloads.tensor4096(seed=0, device=device())["X"].reshape(-1)
    bits = workloads.bits(x)
    st = scaling.DelayedScaling(history_len=16, device=device())
    hist, pos = np.zeros(16, np.float32), 0
    for step in range(3):
        q, s, amax, sat = st.cast(x)
        assert_ok()
        rq, rs, ra, rsat, hist, pos = oracle.quantize_tensor_delayed(bits, oracle.E4M3, 1.0, hist, pos)
        assert host(s)[0] == rs and host(amax)[0] == ra and int(host(sat)[0]) == rsat
        assert np.array_equal(host(q), rq)


def test_shared_scale_reduce_one_rank_on_gpu():
    """The reduction protocol with the library's requantization on one rank:
    the shared scale is this rank's, the payload comes back unchanged."""
    bits = _bits(5000, 3, spread=2.0)
    x = to_dev_bf16(bits)
    ws = torch.zeros(m.mxfp8_tensor_workspace_bytes(), dtype=torch.uint8, device=device())
    q, amax, s = m.fp8_quantize_tensor(x, m.FP8_E4M3, workspace=ws)
    sv = float(host(s)[0])

    def requant(qq, s_in, s_out):
        out, sat = m.fp8_requantize_tensor(qq, _f32(s_in), _f32(s_out))
        return out, int(host(sat)[0])

    def decode(qq):
        return torch.from_numpy(oracle.fp8_decode(host(qq), oracle.E4M3)).float()

    total, s_total, overflow = scaling.shared_scale_reduce(q, sv, m.FP8_E4M3, None, requant, decode)
    assert s_total == pytest.approx(sv) and overflow == 0
    assert np.array_equal(total.numpy(), oracle.fp8_decode(host(q), oracle.E4M3).astype(np.float32))


@pytest.mark.parametrize("orient", ["row", "col"])
def test_scale_rule_study_counts(orient):
    """The floor-vs-rceil study's clipped count equals the oracle's: values
    with |x| > 448 * 2^e for their block's floor exponent; rceil clips none."""
    import bench
    rng = np.random.default_rng(9)
    bits = oracle.bf16_round(rng.standard_t(4, size=(256, 512)))
    x = to_dev_bf16(bits)
    st_r, _ = bench._rule_stats(m, x, 0, orient)
    st_f, _ = bench._rule_stats(m, x, m.MX_SCALE_FLOOR, orient)
    assert st_r["clipped_frac"] == 0.0
    v = oracle.bf16_decode(bits)
    blocks = (v if orient == "row" else v.T).reshape(-1, 32)
    e = oracle.e8m0_scale_byte(np.abs(blocks).max(axis=1), floor=True).astype(np.int64) - 127
    want = int((np.abs(blocks) > 448.0 * np.ldexp(1.0, e)[:, None]).sum())
    assert st_f["clipped_frac"] == pytest.approx(want / v.size, abs=0)
    assert want > 0
