"""Seeded synthetic inputs for the skinny GEMM and its epilogues.

This module holds no arithmetic of the method: it only draws random tensors
with the shapes and distributions of the decode workloads, from fixed seeds, so
that the CUDA path and the CPU oracle are fed identical bytes.

Workloads (shapes follow the pages: HIDDEN = 8192, POOLED = 4096; the
o_proj K at TP8 is 128 * 64 / 8 = 1024):

* ``unpooler_shard``: x BF16 [1, 4096] ~ N(0, 1), W BF16 [1024, 4096] ~ N(0, 0.02).
* ``gemm_sweep``: x BF16 [M, K] ~ N(0, 1), W BF16 [N, K] ~ N(0, 0.02), with
  ``copies`` distinct weights (seed 100 + i) so that the rotated set exceeds L2.
* ``pooler``: x BF16 [b, 8192] ~ N(0, 1), W BF16 [4096, 8192] ~ N(0, 0.02)
  (seed 200 + i), norm weight BF16 [4096] ~ N(0, 0.1) (seed 300), gain_center
  1.0, eps 1e-6; calibration batch x_cal ~ N(0, 1) [16, 8192] (seed 1000).
* ``oproj_boundary``: x BF16 [b, 1024] ~ N(0, 1), W BF16 [8192, 1024] ~ N(0, 0.02)
  (seed 400 + i), post/pre norm weights BF16 [8192] ~ 1 + N(0, 0.1) (seeds 500,
  501), beta BF16 [8192] ~ U(0.5, 1.5) (seed 502), alpha 1.0, stream FP32
  [b, 8192] ~ N(0, 1) (seed 503).
* ``chain`` weights: drawn on the device with torch's CUDA generator, seed
  10000 + 16 * layer + role.
"""
from __future__ import annotations

import torch

HIDDEN = 8192
POOLED = 4096
OPROJ_K = 1024
UNPOOLER_K = 4096
EPS = 1e-6
GAIN_CENTER = 1.0


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, std: float, seed: int, mean: float = 0.0, device="cpu") -> torch.Tensor:
    """BF16 tensor of N(mean, std^2) draws (drawn in FP32, then cast)."""
    t = torch.randn(*shape, generator=_gen(seed, device), dtype=torch.float32, device=device)
    return (t * std + mean).to(torch.bfloat16)


def uniform_bf16(shape, lo: float, hi: float, seed: int, device="cpu") -> torch.Tensor:
    t = torch.rand(*shape, generator=_gen(seed, device), dtype=torch.float32, device=device)
    return (t * (hi - lo) + lo).to(torch.bfloat16)


def normal_f32(shape, seed: int, std: float = 1.0, device="cpu") -> torch.Tensor:
    t = torch.randn(*shape, generator=_gen(seed, device), dtype=torch.float32, device=device)
    return t * std


# ------------------------------------------------------------ workloads ----
def unpooler_shard():
    """(x [1, 4096], W [1024, 4096]) BF16: the M = 1 unpooler shard."""
    return normal_bf16((1, 4096), 1.0, 0), normal_bf16((1024, 4096), 0.02, 1)


def gemm_x(m: int, k: int, seed: int = 0) -> torch.Tensor:
    return normal_bf16((m, k), 1.0, seed)


def gemm_weight(n: int, k: int, copy: int = 0, base_seed: int = 100, device="cpu") -> torch.Tensor:
    return normal_bf16((n, k), 0.02, base_seed + copy, device=device)


def pooler(b: int, copy: int = 0):
    """dict with x, w, norm_w, x_cal, eps, gain_center for the pooler workload."""
    return dict(
        x=normal_bf16((b, HIDDEN), 1.0, 0),
        w=normal_bf16((POOLED, HIDDEN), 0.02, 200 + copy),
        norm_w=normal_bf16((POOLED,), 0.1, 300),
        x_cal=normal_bf16((16, HIDDEN), 1.0, 1000),
        eps=EPS,
        gain_center=GAIN_CENTER,
    )


def oproj_boundary(b: int, copy: int = 0):
    """dict with x, w, post_w, pre_w, beta, alpha, stream, eps for the o_proj +
    dual-norm workload."""
    return dict(
        x=normal_bf16((b, OPROJ_K), 1.0, 0),
        w=normal_bf16((HIDDEN, OPROJ_K), 0.02, 400 + copy),
        post_w=normal_bf16((HIDDEN,), 0.1, 500, mean=1.0),
        pre_w=normal_bf16((HIDDEN,), 0.1, 501, mean=1.0),
        beta=uniform_bf16((HIDDEN,), 0.5, 1.5, 502),
        alpha=1.0,
        stream=normal_f32((b, HIDDEN), 503),
        eps=EPS,
    )


def chain_weight(layer: int, role: int, shape, std: float = 0.02, mean: float = 0.0,
                 device="cuda") -> torch.Tensor:
    """Per-layer weight of the 48-layer decode chain, drawn on ``device``.
    Roles: 0 o_proj [8192, 8192], 1 pooler [4096, 8192], 2 unpooler
    [8192, 4096], 3 post-norm weight, 4 pre-norm weight, 5 beta, 6 pooler norm
    weight."""
    seed = 10000 + 16 * layer + role
    return normal_bf16(shape, std, seed, mean=mean, device=device)


def chain_beta(layer: int, device="cuda") -> torch.Tensor:
    return uniform_bf16((HIDDEN,), 0.5, 1.5, 10000 + 16 * layer + 5, device=device)


def bits(t: torch.Tensor):
    """Raw bit pattern of a BF16 tensor as a numpy uint16 array (CPU copy)."""
    import numpy as np

    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a, device="cpu") -> torch.Tensor:
    """BF16 tensor whose bit pattern is the numpy uint16 array ``a``."""
    import numpy as np

    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(
        torch.bfloat16).to(device)
