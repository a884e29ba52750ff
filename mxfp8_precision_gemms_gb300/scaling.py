"""Host-side state and protocols around the per-tensor FP8 kernels.

* DelayedScaling — the amax-history state of one tensor ("3.8 Mixed
  Precision, bf16 & FP8 Training", "Per-tensor scaling and the
  delayed-scaling recipe"), kept on the device and advanced by
  ``fp8_quantize_tensor_delayed``.
* AutoScale — FP8-LM's automatic gradient scaling factor mu ("FP8-LM:
  Training FP8 Large Language Models", Section 2.1, Eq. 3): halved when the
  overflow ratio exceeds 0.001 %, otherwise multiplied by 2^(1/1000) per step.
* shared_scale_reduce — FP8-LM's reduction of per-rank FP8 gradients with
  per-rank scales (Section 2.1, Eq. 4-6): the group's scale is the minimum
  of the ranks' scales, every rank requantizes to it, the payloads are summed
  and the sum carries the scale N * s_g.

The per-tensor casts and the requantization run in the library's kernels
(fp8_quantize_tensor_delayed, fp8_requantize_tensor) when the caller passes
them; in shared_scale_reduce the decode of the requantized payload is the
caller's callable, while the fp32 sum over ranks and the overflow count are
torch operations over the process group (the protocol is exercised on CPU
ranks with gloo: every box here has one GPU).
"""
from __future__ import annotations

import math
from typing import Callable

import torch

from . import FP8_E4M3, FP8_E5M2, fp8_quantize_tensor_delayed

FP8_MAX = {FP8_E4M3: 448.0, FP8_E5M2: 57344.0}


class DelayedScaling:
    """Amax history (fp32[history_len]) and ring position (int32[1]) of one
    tensor on one device; ``cast`` runs one delayed-scaling cast."""

    def __init__(self, history_len: int = 16, margin: float = 1.0, fmt: int = FP8_E4M3,
                 device=None):
        device = torch.device(device) if device is not None else torch.device("cuda")
        self.history = torch.zeros(history_len, dtype=torch.float32, device=device)
        self.pos = torch.zeros(1, dtype=torch.int32, device=device)
        self.margin = float(margin)
        self.fmt = fmt

    def cast(self, x: torch.Tensor, q=None, stream=None):
        """Returns (q, scale, amax, saturated count) as device tensors."""
        return fp8_quantize_tensor_delayed(x, self.history, self.pos, fmt=self.fmt,
                                           margin=self.margin, q=q, stream=stream)

    def state_dict(self) -> dict:
        return {"history": self.history.detach().cpu().clone(), "pos": self.pos.detach().cpu().clone(),
                "margin": self.margin, "fmt": self.fmt}

    def load_state_dict(self, sd: dict) -> None:
        self.history.copy_(sd["history"])
        self.pos.copy_(sd["pos"])
        self.margin = float(sd["margin"])
        self.fmt = int(sd["fmt"])


class AutoScale:
    """FP8-LM's automatic scaling factor mu for one gradient tensor: after
    each step's reduction, mu is halved if the overflow ratio (saturated
    payloads / values) is above ``threshold`` (0.001 %), else multiplied by
    2^(1/growth_steps) (doubling over 1000 steps)."""

    def __init__(self, mu: float = 1.0, threshold: float = 1e-5, growth_steps: int = 1000):
        self.mu = float(mu)
        self.threshold = float(threshold)
        self.growth = 2.0 ** (1.0 / growth_steps)

    def update(self, saturated: int, n: int) -> float:
        ratio = saturated / n if n else 0.0
        if ratio > self.threshold:
            self.mu *= 0.5
        else:
            self.mu *= self.growth
        return self.mu


def shared_scale_reduce(q, scale: float, fmt: int, group,
                        requantize: Callable, decode: Callable,
                        all_reduce_min: Callable | None = None,
                        all_reduce_sum: Callable | None = None):
    """Reduce per-rank FP8 tensors that carry per-rank scales.

    q, scale  this rank's payload and its scale (x ~ decode(q) / scale).
    requantize(q, s_in, s_out) -> (q_out, saturated_count)
    decode(q) -> fp32 tensor of the payload's values (no scale).
    group     a torch.distributed process group (or None for one rank);
              the two all-reduce callables default to torch.distributed's.

    Returns (total, s_total, overflow) where total is the fp32 sum over ranks
    of the requantized payloads (every value carries the shared scale s_g),
    s_total = N * s_g (so the mean gradient is total / s_total) and overflow
    is the number of summed values beyond the format's largest finite value,
    i.e. those an FP8 sum would saturate: the count AutoScale reacts to.
    """
    import torch.distributed as dist

    world = dist.get_world_size(group) if group is not None else 1

    def _min(t):
        if group is not None:
            dist.all_reduce(t, op=dist.ReduceOp.MIN, group=group)
        return t

    def _sum(t):
        if group is not None:
            dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
        return t

    all_reduce_min = all_reduce_min or _min
    all_reduce_sum = all_reduce_sum or _sum
    s = torch.tensor([float(scale)], dtype=torch.float32)
    s_g = float(all_reduce_min(s)[0])
    if not math.isfinite(s_g) or s_g <= 0.0:
        raise ValueError(f"shared scale {s_g} is not a positive finite number")
    q2, _ = requantize(q, float(scale), s_g)
    total = all_reduce_sum(decode(q2).to(torch.float32))
    overflow = int((total.abs() > FP8_MAX[fmt]).sum())
    return total, world * s_g, overflow
