"""Seeded synthetic inputs for the MXFP8 quantize + scaled-GEMM workloads.

This module holds no arithmetic of the method: it only draws random BF16
tensors (and expert token counts) with the shapes and value distributions of
the five benchmark workloads.  Both the CUDA path and the CPU oracle consume
what it returns; neither is imported here.

Seeds: every operand has its own stream, ``seed * 1000 + operand_index``.
Values are drawn in fp32 by torch's generator on the requested device and
rounded to BF16 by torch's conversion (round to nearest even).  The same seed
gives different numbers on CPU and CUDA (different generators); a test always
feeds the one tensor it drew to both sides.

Workloads (one GB300; shapes from the benchmark definition):
  mx256      A, B 256 x 256, N(0, 1)
  tensor4096 X 4096 x 4096 N(0, 1) with round(1% of 4096) = 41 seeded columns
             scaled by 50 (outlier channels); W 4096 x 4096 N(0, 0.02)
  mlp_up     X 8192 x 4096 Student-t(4); W 16384 x 4096 N(0, 0.02)
  backward   dY 8192 x 4096 with |v| = 10^U(-8, -2) and a random sign;
             W 4096 x 4096 N(0, 0.02); X 8192 x 4096 N(0, 1)
  grouped    64 experts, counts ~ Multinomial(32768 * 8, p_e ~ e^-1.1);
             dispatched X (262144 x 2048) N(0, 1); W 64 x 1024 x 2048 N(0, 0.02)

Routed-path conversions (the grouped workload's surroundings):
  swiglu_hidden     the up/gate output of the grouped workload, H 262144 x 1024
                    N(0, 1) read as gate | up halves of 512, with the grouped
                    workload's expert offsets
  combine_backward  dY 32768 x 2048 with |v| = 10^U(-8, -2) and a random sign;
                    every token routed to 8 distinct experts of 64 drawn with
                    p_e ~ e^-1.1 (Gumbel top-k, without replacement), rows
                    sorted by expert then token; route weights = softmax of
                    8 N(0, 1) logits per token, fp32
"""
from __future__ import annotations

import numpy as np
import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def _stream(seed: int, operand: int) -> int:
    return int(seed) * 1000 + int(operand)


def normal(shape, std: float, seed: int, operand: int, device="cpu") -> torch.Tensor:
    g = _gen(_stream(seed, operand), device)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def student_t(shape, df: int, seed: int, operand: int, device="cpu") -> torch.Tensor:
    """Student-t with integer df: Z / sqrt(chi2_df / df), chi2 from df squared normals."""
    g = _gen(_stream(seed, operand), device)
    z = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    chi2 = torch.zeros_like(z)
    for _ in range(df):
        n = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
        chi2.addcmul_(n, n)
    return (z / torch.sqrt(chi2 / df)).to(torch.bfloat16)


def log_uniform_signed(shape, lo: float, hi: float, seed: int, operand: int,
                       device="cpu") -> torch.Tensor:
    """|v| = 10^U(log10 lo, log10 hi), sign +-1 with probability 1/2."""
    g = _gen(_stream(seed, operand), device)
    u = torch.rand(*shape, generator=g, device=device, dtype=torch.float32)
    s = torch.rand(*shape, generator=g, device=device, dtype=torch.float32)
    a, b = np.log10(lo), np.log10(hi)
    mag = torch.pow(10.0, a + (b - a) * u)
    return torch.where(s < 0.5, -mag, mag).to(torch.bfloat16)


def outlier_columns(x_f32_shape, frac: float, seed: int, operand: int) -> np.ndarray:
    """Indices of round(frac * cols) columns chosen by a seeded permutation."""
    cols = x_f32_shape[-1]
    k = int(round(frac * cols))
    rng = np.random.Generator(np.random.PCG64(_stream(seed, operand)))
    return np.sort(rng.permutation(cols)[:k])


def zipf_counts(total: int, experts: int, s: float, seed: int, operand: int) -> np.ndarray:
    """Expert token counts ~ Multinomial(total, p_e ~ e^-s, e = 1..experts)."""
    p = np.arange(1, experts + 1, dtype=np.float64) ** (-s)
    p /= p.sum()
    rng = np.random.Generator(np.random.PCG64(_stream(seed, operand)))
    return rng.multinomial(total, p).astype(np.int64)


def offsets_from_counts(counts) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(counts, dtype=np.int64))]).astype(np.int32)


def bits(t: torch.Tensor) -> np.ndarray:
    """BF16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- workloads --

def mx256(seed=0, device="cpu", m=256, n=256, k=256):
    return {"A": normal((m, k), 1.0, seed, 0, device),
            "B": normal((n, k), 1.0, seed, 1, device)}


def tensor4096(seed=0, device="cpu", m=4096, n=4096, k=4096):
    g = _gen(_stream(seed, 0), device)
    x = torch.randn(m, k, generator=g, device=device, dtype=torch.float32)
    cols = torch.as_tensor(outlier_columns((m, k), 0.01, seed, 2), device=device)
    x[:, cols] *= 50.0
    return {"X": x.to(torch.bfloat16),
            "W": normal((n, k), 0.02, seed, 1, device),
            "outlier_cols": cols.cpu().numpy()}


def mlp_up(seed=0, device="cpu", tokens=8192, d_in=4096, d_out=16384):
    return {"X": student_t((tokens, d_in), 4, seed, 0, device),
            "W": normal((d_out, d_in), 0.02, seed, 1, device)}


def backward(seed=0, device="cpu", tokens=8192, d_in=4096, d_out=4096):
    return {"dY": log_uniform_signed((tokens, d_out), 1e-8, 1e-2, seed, 0, device),
            "W": normal((d_out, d_in), 0.02, seed, 1, device),
            "X": normal((tokens, d_in), 1.0, seed, 2, device)}


def grouped(seed=0, device="cpu", tokens=32768, top_k=8, experts=64, hidden=2048,
            ffn=1024, zipf_s=1.1):
    counts = zipf_counts(tokens * top_k, experts, zipf_s, seed, 3)
    total = int(counts.sum())
    return {"X": normal((total, hidden), 1.0, seed, 0, device),
            "W": normal((experts, ffn, hidden), 0.02, seed, 1, device),
            "counts": counts,
            "offsets": offsets_from_counts(counts)}


def swiglu_hidden(seed=0, device="cpu", tokens=32768, top_k=8, experts=64, ffn=1024,
                  zipf_s=1.1):
    counts = zipf_counts(tokens * top_k, experts, zipf_s, seed, 3)  # the grouped workload's
    total = int(counts.sum())
    return {"H": normal((total, ffn), 1.0, seed, 4, device),
            "counts": counts, "offsets": offsets_from_counts(counts)}


def routing(seed=0, tokens=32768, top_k=8, experts=64, zipf_s=1.1):
    """Token -> expert assignments (top_k distinct experts per token, Gumbel
    top-k on log p_e) sorted by expert then token, with softmax route weights;
    token_rows / token_weights give the same routing per token (the
    dispatched row and weight of each of its top_k slots)."""
    rng = np.random.Generator(np.random.PCG64(_stream(seed, 5)))
    logp = -zipf_s * np.log(np.arange(1, experts + 1, dtype=np.float64))
    keys = logp[None, :] + rng.gumbel(size=(tokens, experts))
    chosen = np.argpartition(-keys, top_k - 1, axis=1)[:, :top_k]
    logits = rng.standard_normal((tokens, top_k))
    w = np.exp(logits - logits.max(axis=1, keepdims=True))
    w /= w.sum(axis=1, keepdims=True)
    tok = np.repeat(np.arange(tokens, dtype=np.int64), top_k)
    exp_ = chosen.reshape(-1)
    order = np.lexsort((tok, exp_))
    counts = np.bincount(exp_, minlength=experts).astype(np.int64)
    # the same routing from the token side: dispatched row of (token, slot)
    inv = np.empty(order.size, np.int64)
    inv[order] = np.arange(order.size)
    return {"row_token": tok[order].astype(np.int32),
            "row_weight": w.reshape(-1)[order].astype(np.float32),
            "token_rows": inv.reshape(tokens, top_k).astype(np.int32),
            "token_weights": w.astype(np.float32),
            "counts": counts, "offsets": offsets_from_counts(counts)}


def combine_backward(seed=0, device="cpu", tokens=32768, d_model=2048, **kw):
    r = routing(seed=seed, tokens=tokens, **kw)
    r["dY"] = log_uniform_signed((tokens, d_model), 1e-8, 1e-2, seed, 6, device)
    return r


WORKLOADS = {
    "mx256": (mx256, "MXFP8 quantize+GEMM M=N=K=256"),
    "tensor4096": (tensor4096, "per-tensor FP8 forward GEMM M=N=K=4096, 1% outlier columns"),
    "mlp_up": (mlp_up, "MXFP8 MLP up-projection X[8192x4096] . W[16384x4096]^T"),
    "backward": (backward, "MXFP8 dgrad + wgrad of a 4096->4096 linear over 8192 tokens"),
    "grouped": (grouped, "MXFP8 grouped expert GEMM, 64 experts top-8 Zipf(1.1), 2048->1024"),
    "swiglu_hidden": (swiglu_hidden, "fused SwiGLU + MX quantize of the grouped up/gate output"),
    "combine_backward": (combine_backward, "fused route weighting + MX gradient quantize"),
}
