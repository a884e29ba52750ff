"""GPU parity of the quantizer kernels against the FP64 oracle: every payload
byte and every scale byte (padding included) must match exactly."""
import numpy as np
import pytest
import torch

import mxfp8_precision_gemms_gb300 as m
import oracle
import workloads
from gpu_util import assert_ok, device, filled, host, to_dev_bf16

pytestmark = pytest.mark.gpu

ROW, COL, FLOOR = m.MX_ROWWISE, m.MX_COLWISE, m.MX_SCALE_FLOOR


def random_bits(shape, dist, seed):
    g = torch.Generator().manual_seed(seed)
    if dist == "normal":
        x = torch.randn(*shape, generator=g)
    elif dist == "student":
        return workloads.bits(workloads.student_t(shape, 4, seed, 0))
    elif dist == "loguniform":
        return workloads.bits(workloads.log_uniform_signed(shape, 1e-8, 1e-2, seed, 0))
    elif dist == "wide":  # magnitudes over ~60 binades
        x = torch.randn(*shape, generator=g) * torch.pow(2.0, torch.randint(-40, 20, shape, generator=g).float())
    else:
        raise ValueError(dist)
    return workloads.bits(x.to(torch.bfloat16))


def run_mx(bits, flags, ld=None):
    rows, cols = bits.shape
    if ld is not None and ld != cols:
        wide = np.zeros((rows, ld), np.uint16)
        wide[:, :cols] = bits
        x = to_dev_bf16(wide)[:, :cols]
    else:
        x = to_dev_bf16(bits)
    out = {}
    if flags & ROW:
        out["q_row"] = filled((rows, cols), 0xA5)
        out["s_row"] = filled(m.mxfp8_scale_bytes(rows, cols), 0xA5)
    if flags & COL:
        out["q_col"] = filled((cols, rows), 0xA5)
        out["s_col"] = filled(m.mxfp8_scale_bytes(cols, rows), 0xA5)
    m.fp8_quantize_mx(x, flags, **out)
    assert_ok()
    return {k: host(v) for k, v in out.items()}


SHAPES = [(32, 32), (128, 128), (160, 320), (96, 4096), (1056, 96), (4128, 160), (64, 8192)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("flags", [ROW, COL, ROW | COL, ROW | FLOOR, ROW | COL | FLOOR])
def test_quantize_mx_matches_oracle(shape, flags):
    bits = random_bits(shape, "student", seed=shape[0] * 7 + shape[1])
    got = run_mx(bits, flags)
    want = oracle.quantize_mx(bits, flags)
    for k in want:
        assert np.array_equal(got[k], want[k]), k


@pytest.mark.parametrize("dist", ["normal", "loguniform", "wide"])
def test_quantize_mx_distributions(dist):
    bits = random_bits((256, 512), dist, seed=3)
    got = run_mx(bits, ROW | COL)
    want = oracle.quantize_mx(bits, ROW | COL)
    for k in want:
        assert np.array_equal(got[k], want[k]), k


def test_quantize_mx_leading_dimension():
    bits = random_bits((192, 256), "normal", seed=5)
    got = run_mx(bits, ROW | COL, ld=264)
    want = oracle.quantize_mx(bits, ROW | COL)
    for k in want:
        assert np.array_equal(got[k], want[k]), k


@pytest.mark.parametrize("flags", [ROW, ROW | FLOOR])
@pytest.mark.parametrize("ld,shift,qshift", [(264, 0, 0), (256, 8, 0), (256, 0, 16), (272, 8, 16)])
def test_quantize_mx_rowwise_16_byte_aligned(flags, ld, shift, qshift):
    """Rowwise outputs when only the documented 16-byte alignment holds (row
    stride, input start or payload start off a 32-byte boundary)."""
    rows, cols = 200, 224
    bits = random_bits((rows, cols), "student", seed=ld + shift + qshift)
    wide = np.zeros((rows + 1, ld), np.uint16)
    flat = wide.reshape(-1)
    view = np.lib.stride_tricks.as_strided(flat[shift:], shape=(rows, cols), strides=(ld * 2, 2))
    view[:] = bits
    xd = to_dev_bf16(flat)[shift:shift + rows * ld].view(rows, ld)[:, :cols]
    qbuf = filled(rows * cols + 32, 0xA5)
    q = qbuf[qshift:qshift + rows * cols].view(rows, cols)
    s = filled(m.mxfp8_scale_bytes(rows, cols), 0xA5)
    m.fp8_quantize_mx(xd, flags, q_row=q, s_row=s)
    assert_ok()
    want = oracle.quantize_mx(bits, flags)
    assert np.array_equal(host(q), want["q_row"])
    assert np.array_equal(host(s), want["s_row"])
    hb = host(qbuf)
    assert np.all(hb[:qshift] == 0xA5) and np.all(hb[qshift + rows * cols:] == 0xA5)


@pytest.mark.parametrize("flags", [ROW, ROW | FLOOR])
def test_quantize_mx_batch_matches_oracle(flags):
    """Several tensors in one launch: ragged rows, a wide row stride, an empty
    tensor, a 16- but not 32-byte aligned input; each equals the oracle."""
    shapes = [(300, 256), (1024, 4096), (0, 64), (96, 96), (200, 224), (128, 32)]
    bits = [random_bits(sh, "student", seed=11 + i) if sh[0] else np.zeros(sh, np.uint16)
            for i, sh in enumerate(shapes)]
    xs = []
    for i, b in enumerate(bits):
        if i == 1:  # row stride 4104 > cols
            wide = np.zeros((b.shape[0], 4104), np.uint16)
            wide[:, :b.shape[1]] = b
            xs.append(to_dev_bf16(wide)[:, :b.shape[1]])
        elif i == 4:  # input start 16 bytes past a 32-byte boundary
            flat = np.zeros(b.size + 8, np.uint16)
            flat[8:] = b.reshape(-1)
            xs.append(to_dev_bf16(flat)[8:].view(b.shape))
        else:
            xs.append(to_dev_bf16(b))
    outs = [{"q_row": filled(b.shape, 0xA5), "s_row": filled(m.mxfp8_scale_bytes(*b.shape), 0xA5)}
            for b in bits]
    m.fp8_quantize_mx_batch(xs, flags, outs=outs)
    assert_ok()
    for b, o in zip(bits, outs):
        if b.size == 0:
            continue
        want = oracle.quantize_mx(b, flags)
        assert np.array_equal(host(o["q_row"]), want["q_row"])
        assert np.array_equal(host(o["s_row"]), want["s_row"])


def test_quantize_mx_batch_of_sixteen_mlp_operands():
    """Sixteen tensors; the first two are the MLP up-projection's X and W rows
    (student-t activations, N(0, 0.02) weights) at a reduced size."""
    w = workloads.mlp_up(seed=2, device="cpu", tokens=512, d_in=1024, d_out=768)
    bits = [workloads.bits(w["X"]), workloads.bits(w["W"])]
    bits += [random_bits((32 * (t + 1), 64 * ((t % 3) + 1)), "wide", seed=40 + t) for t in range(14)]
    outs = m.fp8_quantize_mx_batch([to_dev_bf16(b) for b in bits])
    assert_ok()
    for b, o in zip(bits, outs):
        want = oracle.quantize_mx(b, ROW)
        assert np.array_equal(host(o["q_row"]), want["q_row"])
        assert np.array_equal(host(o["s_row"]), want["s_row"])


@pytest.mark.parametrize("floor", [0, FLOOR])
def test_quantize_mx_batch_mixed_orientations(floor):
    """The backward's operands in one call (dY both ways, W and X colwise) plus
    rowwise-only and empty tensors, and more colwise tensors than one launch
    takes (nine): every output equals the oracle's."""
    w = workloads.backward(seed=4, device="cpu", tokens=512, d_in=384, d_out=256)
    bits = [workloads.bits(w["dY"]), workloads.bits(w["W"]), workloads.bits(w["X"])]
    flags = [ROW | COL, COL, COL]
    bits += [random_bits((96, 160), "student", seed=60), np.zeros((0, 64), np.uint16)]
    flags += [ROW, COL]
    bits += [random_bits((32 * (t + 1), 32 * (t + 2)), "wide", seed=70 + t) for t in range(7)]
    flags += [COL if t % 2 else ROW | COL for t in range(7)]
    flags = [f | floor for f in flags]
    outs = m.fp8_quantize_mx_batch([to_dev_bf16(b) for b in bits], flags)
    assert_ok()
    for b, f, o in zip(bits, flags, outs):
        if b.size == 0:
            continue
        want = oracle.quantize_mx(b, f)
        for k in want:
            assert np.array_equal(host(o[k]), want[k]), k


@pytest.mark.parametrize("flags", [COL, ROW | COL, COL | FLOOR])
def test_quantize_mx_colwise_16_byte_aligned_outputs(flags):
    """Colwise (and both-orientation) outputs that start 16 bytes past a
    32-byte boundary (the tile kernel's 16-byte store path), alone and in a
    batch."""
    rows, cols = 224, 160
    bits = random_bits((rows, cols), "student", seed=90 + flags)
    want = oracle.quantize_mx(bits, flags)
    for batched in (False, True):
        bufs, out = [], {}
        for k, shape in (("q_row", (rows, cols)), ("q_col", (cols, rows))):
            if k in want:
                b = filled(rows * cols + 64, 0xA5)
                bufs.append(b)
                out[k] = b[16:16 + rows * cols].view(shape)
        for k, n in (("s_row", m.mxfp8_scale_bytes(rows, cols)), ("s_col", m.mxfp8_scale_bytes(cols, rows))):
            if k in want:
                out[k] = filled(n, 0xA5)
        x = to_dev_bf16(bits)
        if batched:
            m.fp8_quantize_mx_batch([x, x], [flags, flags], outs=[out, {k: torch.empty_like(v) for k, v in out.items()}])
        else:
            m.fp8_quantize_mx(x, flags, **out)
        assert_ok()
        for k in want:
            assert np.array_equal(host(out[k]).reshape(want[k].shape), want[k]), (k, batched)
        for b in bufs:
            hb = host(b)
            assert np.all(hb[:16] == 0xA5) and np.all(hb[16 + rows * cols:] == 0xA5)


def _anchor_blocks(floor):
    """Blocks whose scale byte is fixed by an anchor value, filled with every
    finite BF16 pattern at or below the anchor: all BF16 values x all scales."""
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_decode(allb)
    fin = np.isfinite(vals)
    b_fin, v_fin = allb[fin], np.abs(vals[fin])
    order = np.argsort(v_fin, kind="stable")
    b_sorted, v_sorted = b_fin[order], v_fin[order]
    blocks, bytes_expected = [], []
    top = 246 if floor else 247
    for byte in range(0, top + 1, 1):
        if floor:
            anchor_bits = np.uint16(((byte + 8) << 7) | 0x7F)
        else:
            anchor_bits = np.uint16(((byte + 8) << 7) | 0x60) if byte < 247 else np.uint16(0x7F7F)
        a = oracle.bf16_decode(np.array([anchor_bits]))[0]
        cand = b_sorted[v_sorted <= a]
        pad = (-cand.size) % 31
        cand = np.concatenate([cand, np.zeros(pad, np.uint16)]).reshape(-1, 31)
        anchors = np.full((cand.shape[0], 1), anchor_bits, np.uint16)
        anchors[1::2] |= 0x8000
        blocks.append(np.concatenate([anchors, cand], axis=1))
        bytes_expected.append(np.full(cand.shape[0], byte))
    blocks = np.concatenate(blocks)
    nb = blocks.shape[0]
    per_row = 128
    rows = -(-nb // per_row)
    full = np.zeros((rows * per_row, 32), np.uint16)
    full[:nb] = blocks
    return full.reshape(rows, per_row * 32), np.concatenate(bytes_expected), nb


@pytest.mark.parametrize("floor", [False, True])
def test_quantize_all_bf16_at_every_scale(floor):
    bits, want_bytes, nb = _anchor_blocks(floor)
    flags = ROW | (FLOOR if floor else 0)
    got = run_mx(bits, flags)
    want = oracle.quantize_mx(bits, flags)
    # the construction really pins each block's scale
    rows, cols = bits.shape
    r = np.arange(nb) // (cols // 32)
    j = np.arange(nb) % (cols // 32)
    offs = (r // 128) * ((cols + 127) // 128) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + j % 4 \
        + (j // 4) * 512
    assert np.array_equal(want["s_row"][offs], want_bytes)
    assert np.array_equal(got["s_row"], want["s_row"])
    assert np.array_equal(got["q_row"], want["q_row"])


def test_special_blocks():
    x = np.zeros((32, 128), np.uint16)
    x[0, 3] = 0x7FC0          # NaN -> whole block 0xFF / 0x7F
    x[1, 40] = 0x7F80         # +Inf
    x[2, 70] = 0xFF80         # -Inf
    x[3, :] = 0x8000          # all -0
    x[4, 0:32] = 0x0001       # smallest subnormal
    x[5, 32] = 0x43FA         # 500 -> floor saturates, rceil does not
    x[5, 33] = 0xB586         # a tiny negative value next to it
    for flags in (ROW | COL, ROW | COL | FLOOR):
        got = run_mx(x, flags)
        want = oracle.quantize_mx(x, flags)
        for k in want:
            assert np.array_equal(got[k], want[k]), (flags, k)


def test_quantize_grouped_matches_oracle():
    counts = [0, 1, 127, 128, 129, 0, 300, 5, 0]
    off = workloads.offsets_from_counts(counts)
    bits = random_bits((int(off[-1]), 256), "student", seed=9)
    x = to_dev_bf16(bits)
    G = len(counts)
    q = filled((int(off[-1]), 256), 0xA5)
    s = filled(m.mxfp8_grouped_scale_bytes(int(off[-1]), 256, G), 0xA5)
    m.fp8_quantize_mx_grouped(x, torch.from_numpy(off).to(device()), 0, q=q, s=s)
    assert_ok()
    wq, ws = oracle.quantize_mx_grouped(bits, off)
    assert np.array_equal(host(q), wq)
    assert np.array_equal(host(s)[: ws.size], ws)


@pytest.mark.parametrize("bad", ["decreasing", "last", "first"])
def test_quantize_grouped_bad_offsets_recorded(bad):
    off = np.array([0, 64, 128, 256], np.int32)
    if bad == "decreasing":
        off[2] = 32
    elif bad == "last":
        off[3] = 200
    else:
        off[0] = 4
    bits = random_bits((256, 64), "normal", seed=1)
    q = filled((256, 64), 0x5A)
    s = filled(m.mxfp8_grouped_scale_bytes(256, 64, 3), 0x5A)
    m.fp8_quantize_mx_grouped(to_dev_bf16(bits), torch.from_numpy(off).to(device()), 0, q=q, s=s)
    assert m.mxfp8_last_device_status() == m.MXFP8_ERR_DEVICE_CHECK
    assert m.mxfp8_last_device_status() == m.MXFP8_OK  # the word was cleared
    assert (host(q) == 0x5A).all() and (host(s) == 0x5A).all()


@pytest.mark.parametrize("fmt", [m.FP8_E4M3, m.FP8_E5M2])
def test_quantize_tensor_batch_matches_oracle(fmt):
    """Several tensors in one launch: each gets the amax, scale and payload
    the single-tensor rule gives it (including an empty and an odd-sized one)."""
    w = workloads.tensor4096(seed=3, device="cpu", m=512, n=384, k=1024)
    cases = [workloads.bits(w["X"]).reshape(-1), workloads.bits(w["W"]).reshape(-1),
             np.zeros((0,), np.uint16), random_bits((100003,), "loguniform", seed=5).reshape(-1),
             workloads.bits((torch.randn(4000) * 1e-30).to(torch.bfloat16)),
             np.zeros((4096,), np.uint16)]
    xs = [to_dev_bf16(b) for b in cases]
    qs = [filled(b.size, 0xA5) for b in cases]
    amax = filled(len(cases), -1.0, torch.float32)
    scale = filled(len(cases), -1.0, torch.float32)
    ws = filled(m.mxfp8_tensor_workspace_bytes(), 0x77)
    for _ in range(2):
        m.fp8_quantize_tensor_batch(xs, fmt, workspace=ws, qs=qs, amax=amax, scale=scale)
        assert_ok()
    ha, hs = host(amax).view(np.uint32), host(scale).view(np.uint32)
    for t, b in enumerate(cases):
        wa, wsc, wq = oracle.quantize_tensor(b, fmt)
        assert np.array_equal(host(qs[t]), wq.reshape(-1)), t
        assert ha[t] == np.float32(wa).view(np.uint32), t
        assert hs[t] == np.float32(wsc).view(np.uint32), t


@pytest.mark.parametrize("fmt", [m.FP8_E4M3, m.FP8_E5M2])
def test_quantize_tensor_16_byte_aligned(fmt):
    """Inputs that start 16 bytes past a 32-byte boundary (the 16-byte load
    path of the single-launch kernel), with odd sizes, alone and batched."""
    sizes = [1000003, 4097, 40]
    bits = [random_bits((n,), "student", seed=80 + n % 7).reshape(-1) for n in sizes]
    xs = []
    for b in bits:
        flat = np.zeros(b.size + 8, np.uint16)
        flat[8:] = b
        xs.append(to_dev_bf16(flat)[8:])
    ws = torch.zeros(m.mxfp8_tensor_workspace_bytes(), dtype=torch.uint8, device=device())
    qs, amax, scale = m.fp8_quantize_tensor_batch(xs, fmt, workspace=ws)
    assert_ok()
    for t, b in enumerate(bits):
        wa, wsc, wq = oracle.quantize_tensor(b, fmt)
        assert np.array_equal(host(qs[t]), wq.reshape(-1)), t
        assert host(amax).view(np.uint32)[t] == np.float32(wa).view(np.uint32)
        assert host(scale).view(np.uint32)[t] == np.float32(wsc).view(np.uint32)
        q1, a1, s1 = m.fp8_quantize_tensor(xs[t], fmt, workspace=ws)
        assert_ok()
        assert np.array_equal(host(q1), wq.reshape(-1)), t


def test_quantize_tensor_batch_of_sixteen():
    """The largest batch: sixteen tensors of different sizes."""
    cases = [random_bits((1 + 997 * t,), "normal", seed=10 + t).reshape(-1) for t in range(16)]
    xs = [to_dev_bf16(b) for b in cases]
    qs, amax, scale = m.fp8_quantize_tensor_batch(xs, m.FP8_E4M3)
    assert_ok()
    for t, b in enumerate(cases):
        wa, wsc, wq = oracle.quantize_tensor(b, m.FP8_E4M3)
        assert np.array_equal(host(qs[t]), wq.reshape(-1)), t
        assert float(host(scale)[t]) == np.float32(wsc), t


@pytest.mark.parametrize("fused", [False, True], ids=["two_kernels", "single_launch"])
@pytest.mark.parametrize("fmt", [m.FP8_E4M3, m.FP8_E5M2])
@pytest.mark.parametrize("case", ["outliers", "loguniform", "tiny", "zeros", "odd", "empty"])
def test_quantize_tensor_matches_oracle(fmt, case, fused):
    if case == "outliers":
        w = workloads.tensor4096(seed=1, device="cpu", m=512, n=8, k=1024)
        bits = workloads.bits(w["X"])
    elif case == "loguniform":
        bits = random_bits((1024, 777 * 8 // 8), "loguniform", seed=2)
    elif case == "tiny":
        bits = workloads.bits((torch.randn(300, 40) * 1e-30).to(torch.bfloat16))
    elif case == "zeros":
        bits = np.zeros((64, 64), np.uint16)
    elif case == "odd":
        bits = random_bits((1000003,), "normal", seed=4)
    else:
        bits = np.zeros((0,), np.uint16)
    x = to_dev_bf16(bits.reshape(-1))
    q = filled(bits.size, 0xA5)
    amax = filled(1, -1.0, torch.float32)
    scale = filled(1, -1.0, torch.float32)
    ws = filled(m.mxfp8_tensor_workspace_bytes(), 0x77) if fused else None
    for _ in range(2):  # twice: the workspace keeps the last call's contents
        m.fp8_quantize_tensor(x, fmt, q=q, amax=amax, scale=scale, workspace=ws)
        assert_ok()
    wa, ws, wq = oracle.quantize_tensor(bits.reshape(-1), fmt)
    assert np.array_equal(host(q), wq.reshape(-1))
    assert host(amax).view(np.uint32)[0] == np.float32(wa).view(np.uint32)
    assert host(scale).view(np.uint32)[0] == np.float32(ws).view(np.uint32)
