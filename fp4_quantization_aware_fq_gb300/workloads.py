"""Seeded synthetic inputs for the fake-quantization workloads.

This module only draws random tensors; it holds none of the quantization
arithmetic.  The same tensors feed the CUDA library and the CPU oracle, so
both sides see identical bits.  All draws use torch's CPU generator (or a
CUDA generator where noted, for benchmark-sized inputs that are never handed
to the oracle); bfloat16 tensors are made with torch's nearest-even cast.

Workloads (shapes and distributions of the pages' QAT / TetraJet-v2 use):
  nvfp4_small   fp32 [256, 1024] ~ N(0, 1)                                seed 0
  mxfp4_weight  bf16 [4096, 4096] ~ N(0, 0.02), 0.1% of entries x100        seed 1
  nvfp4_act     bf16 [8192, 8192] ~ N(0, 1), 8 outlier columns x50          seed 2
  grad_2level   bf16 [16384, 4096] ~ Laplace(0, 1e-3)                       seed 3
  moe_qat       32 experts x (bf16 [2880, 5760] + [5760, 2880]) ~ N(0, .02) seed 4,
                master updates delta_t ~ N(0, 1e-4)                        seed 1000 + t
  channel_act   bf16 [8192, 8192] ~ N(0, 1), 64 outlier channels x50 shared by every
                batch of a calibration window (channel seed 5; batch seed 500 + t)
  qad_logits    bf16 teacher / student logits [4096, 201088] (gpt-oss's vocabulary
                size): teacher ~ N(0, 3^2), student = teacher + N(0, 0.3^2)      seed 6
Each generator takes the shape as an argument so that tests can draw smaller
tensors with the same recipe.
"""
from __future__ import annotations

import torch

WORKLOADS = {
    "nvfp4_small": dict(shape=(256, 1024), seed=0),
    "mxfp4_weight": dict(shape=(4096, 4096), seed=1),
    "nvfp4_act": dict(shape=(8192, 8192), seed=2),
    "grad_2level": dict(shape=(16384, 4096), seed=3),
    "moe_qat": dict(experts=32, up_shape=(2880, 5760), down_shape=(5760, 2880), seed=4),
    "channel_act": dict(shape=(8192, 8192), seed=500, channel_seed=5, n_outlier_cols=64),
    "qad_logits": dict(shape=(4096, 201088), seed=6),
}


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, std=1.0, seed=0, dtype=torch.float32, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    x = torch.randn(shape, generator=g, dtype=torch.float32, device=device) * std
    return x.to(dtype)


def nvfp4_small(shape=(256, 1024), seed=0, device="cpu") -> torch.Tensor:
    """FP32 activations ~ N(0, 1)."""
    return normal(shape, 1.0, seed, torch.float32, device)


def mxfp4_weight(shape=(4096, 4096), seed=1, device="cpu") -> torch.Tensor:
    """BF16 weight ~ N(0, 0.02) with 0.1% of entries (uniform random positions)
    multiplied by 100."""
    g = _gen(seed, device)
    x = torch.randn(shape, generator=g, dtype=torch.float32, device=device) * 0.02
    n = x.numel()
    k = max(1, n // 1000) if n >= 1000 else max(1, n // 100)
    idx = torch.randperm(n, generator=g, device=device)[:k]
    x.view(-1)[idx] *= 100.0
    return x.to(torch.bfloat16)


def nvfp4_act(shape=(8192, 8192), seed=2, n_outlier_cols=8, device="cpu") -> torch.Tensor:
    """BF16 activations ~ N(0, 1) with a few outlier channels (columns) x50."""
    g = _gen(seed, device)
    x = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
    cols = torch.randperm(shape[1], generator=g, device=device)[:n_outlier_cols]
    x[:, cols] *= 50.0
    return x.to(torch.bfloat16)


def outlier_channels(cols: int, n: int, channel_seed: int) -> torch.Tensor:
    """The n outlier channels of an activation recipe (uniform random)."""
    return torch.randperm(cols, generator=_gen(channel_seed))[:n]


def channel_act(shape=(8192, 8192), seed=500, channel_seed=5, n_outlier_cols=64, factor=50.0,
                device="cpu") -> torch.Tensor:
    """BF16 activations ~ N(0, 1) whose outlier channels -- fixed by
    channel_seed, so that every batch of a calibration window shares them --
    are multiplied by factor; seed draws the batch."""
    g = _gen(seed, device)
    x = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
    x[:, outlier_channels(shape[1], n_outlier_cols, channel_seed).to(device)] *= factor
    return x.to(torch.bfloat16)


def qad_logits(shape=(4096, 201088), seed=6, teacher_std=3.0, student_noise=0.3,
               dtype=torch.bfloat16, device="cpu"):
    """Teacher and student logits of a distillation step: the teacher ~ N(0,
    teacher_std^2); the student (a quantized copy of the teacher) adds
    N(0, student_noise^2).  Both rounded to dtype."""
    g = _gen(seed, device)
    zt = torch.randn(shape, generator=g, dtype=torch.float32, device=device) * teacher_std
    zs = zt + torch.randn(shape, generator=g, dtype=torch.float32, device=device) * student_noise
    return zt.to(dtype), zs.to(dtype)


def grad_2level(shape=(16384, 4096), seed=3, scale=1e-3, device="cpu") -> torch.Tensor:
    """BF16 gradient ~ Laplace(0, scale), by the inverse CDF of a uniform draw."""
    g = _gen(seed, device)
    u = torch.rand(shape, generator=g, dtype=torch.float64, device=device) - 0.5
    u = u.clamp(-0.5 + 1e-12, 0.5 - 1e-12)
    x = -scale * torch.sign(u) * torch.log1p(-2.0 * u.abs())
    return x.to(torch.bfloat16)


def moe_weights(experts=32, up_shape=(2880, 5760), down_shape=(5760, 2880), seed=4,
                device="cpu"):
    """List of BF16 expert weights: per expert the fused up/gate matrix and the
    down matrix, ~ N(0, 0.02)."""
    g = _gen(seed, device)
    out = []
    for _ in range(experts):
        for shp in (up_shape, down_shape):
            out.append((torch.randn(shp, generator=g, dtype=torch.float32, device=device)
                        * 0.02).to(torch.bfloat16))
    return out


def master_update(shape, step: int, std=1e-4, device="cpu", seed_base=1000) -> torch.Tensor:
    """Synthetic optimizer update for one step ~ N(0, std), FP32."""
    return normal(shape, std, seed_base + step, torch.float32, device)


def bf16_bits(t: torch.Tensor):
    """numpy uint16 view of a bfloat16 tensor's bits (no arithmetic)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
