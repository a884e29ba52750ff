"""FP8-LM's gradient reduction with per-rank scales and its automatic scaling
factor ("FP8-LM: Training FP8 Large Language Models", Section 2.1, Eq. 3-6),
run as two gloo ranks on the CPU.  The protocol is the package's
(`scaling.shared_scale_reduce`, `scaling.AutoScale`); the per-rank arithmetic
(casts, requantization, decoding) is the oracle's, passed in as callables."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from mxfp8_precision_gemms_gb300 import scaling

E4M3 = oracle.E4M3


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _grad_bits(rank, step, n=4096):
    rng = np.random.default_rng(100 * step + rank)
    mag = [1e-3, 5e-3][rank]
    if step == 2 and rank == 1:
        mag *= 2000.0  # a gradient spike on one rank
    return oracle.bf16_round(rng.standard_normal(n) * mag)


def _requant(q, s_in, s_out):
    out, sat = oracle.requantize_tensor(q.numpy(), E4M3, s_in, s_out, E4M3)
    return torch.from_numpy(out), sat


def _decode(q):
    return torch.from_numpy(oracle.fp8_decode(q.numpy(), E4M3))


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    g = dist.group.WORLD
    # (1) per-rank current scaling, then the shared-scale reduction
    amax, s, q = oracle.quantize_tensor(_grad_bits(rank, 0), E4M3)
    total, s_total, overflow = scaling.shared_scale_reduce(torch.from_numpy(q), float(s), E4M3, g,
                                                           _requant, _decode)
    out[(rank, "current")] = (float(s), total.numpy().copy(), s_total, overflow)
    # (2) FP8-LM's mu: cast g' = mu g directly (scale = mu), reduce, adapt mu
    auto = scaling.AutoScale(mu=2.0 ** 10)
    mus = []
    for step in range(4):
        mu = np.float32(auto.mu)
        qm, _, _ = oracle.quantize_tensor_scaled(_grad_bits(rank, step), E4M3, mu)
        total, s_total, overflow = scaling.shared_scale_reduce(torch.from_numpy(qm), float(mu), E4M3, g,
                                                               _requant, _decode)
        mus.append((float(mu), overflow, auto.update(overflow, total.numel())))
    out[(rank, "mu")] = mus
    dist.barrier()
    dist.destroy_process_group()


@pytest.fixture(scope="module")
def two_ranks():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    return dict(out)


def test_shared_min_scale_and_sum(two_ranks):
    s0, t0, st0, o0 = two_ranks[(0, "current")]
    s1, t1, st1, o1 = two_ranks[(1, "current")]
    s_g = min(s0, s1)
    assert st0 == st1 == pytest.approx(2 * s_g)
    # every rank gets the same sum: each rank's payload requantized to s_g, decoded, added in fp32
    want = np.zeros(4096, np.float32)
    for r in range(2):
        amax, s, q = oracle.quantize_tensor(_grad_bits(r, 0), E4M3)
        q2, _ = oracle.requantize_tensor(q, E4M3, s, s_g, E4M3)
        want += oracle.fp8_decode(q2, E4M3).astype(np.float32)
    assert np.array_equal(t0, want) and np.array_equal(t1, want)
    # the mean gradient comes back within the FP8 rounding of both steps
    mean = sum(oracle.bf16_decode(_grad_bits(r, 0)) for r in range(2)) / 2
    err = np.abs(t0 / st0 - mean)
    assert np.max(err) <= 2 * 2 * (448 / s_g) * 2.0 ** -4 / st0 * s_g + 1e-12
    assert o0 == o1 == int((np.abs(want) > 448).sum())


def test_auto_scale_reacts_to_the_spike(two_ranks):
    seq0, seq1 = two_ranks[(0, "mu")], two_ranks[(1, "mu")]
    assert seq0 == seq1  # mu is shared: both ranks see the same overflow
    growth = 2.0 ** (1 / 1000)
    mu = 2.0 ** 10
    for step, (mu_used, overflow, mu_next) in enumerate(seq0):
        assert mu_used == pytest.approx(mu, rel=1e-6)
        if step == 2:
            assert overflow > 0 and mu_next == pytest.approx(mu / 2, rel=1e-12)
        else:
            assert overflow == 0 and mu_next == pytest.approx(mu * growth, rel=1e-12)
        mu = mu_next


def test_auto_scale_rule():
    a = scaling.AutoScale(mu=8.0)
    assert a.update(0, 10 ** 6) == pytest.approx(8.0 * 2 ** 0.001)
    assert a.update(10, 10 ** 6) == pytest.approx(8.0 * 2 ** 0.002)       # 1e-5 is not above 0.001 %
    assert a.update(11, 10 ** 6) == pytest.approx(4.0 * 2 ** 0.002)       # above: halve
    b = scaling.AutoScale(mu=1.0)
    for _ in range(1000):
        b.update(0, 100)
    assert b.mu == pytest.approx(2.0, rel=1e-9)                           # doubles over 1000 steps
