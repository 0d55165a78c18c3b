"""Small-batch dense GEMV on NVFP4 (or BF16) weights. float64 CPU definition.

TEST INFRASTRUCTURE ONLY (see the package docstring).

"Day-0 Support for Flint on vLLM", section "Optimisation": besides the MoE
kernels, small-batch dense GEMVs serve the dense MLPs of the first layers and
the projections, with the same weight-only NVFP4 weights and BF16
activations. The pages print no formula; the plain reading, with the MoE
layer's rounding points, is for every token row x (bf16 values) and output n:

    y_n = bf16(float32(G * sum_k c[n, k] * x_k))      (sum in float64)

with c = E2M1(code) * E4M3(scale) the dequantised weight and G the FP32 tensor
scale (c the bf16 weight and G = 1 for a BF16 matrix). With a norm weight the
rows are first normalised as in the pre-norm block (moe.rmsnorm).
"""
from __future__ import annotations

import numpy as np

from .moe import bf16_round, f32, rmsnorm


def gemv(x: np.ndarray, w, norm_weight: np.ndarray | None = None, eps: float = 0.0) -> np.ndarray:
    """y [B, N] (float64 bf16 values) for x [B, K] and a matrix w [N, K]
    (moe.NVFP4Matrix or moe.BF16Matrix)."""
    x = np.asarray(x, dtype=np.float64)
    if norm_weight is not None:
        x = rmsnorm(x, norm_weight, eps)
    return bf16_round(f32(np.float64(w.G) * (x @ w.c().T)))
