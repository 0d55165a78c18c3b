"""Device-resident synthetic layers built through the library's own entry points.

Weights are drawn on the GPU by flint_synth_normal (stream (seed, layer,
tensor, expert), N(0, 0.02)), quantised by flint_moe_quantize_nvfp4 (NVFP4
layers) or rounded to bf16 (BF16 layers), and repacked by flint_moe_pack.
PyTorch only allocates the buffers.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

from . import binding as fb

WEIGHT_SIGMA = 0.02
ROUTER_SIGMA = 0.02
NORM_SIGMA = 0.1
NORM_EPS = 1e-6


@dataclass
class DeviceLayer:
    cfg: fb.flint_moe_config
    packed: torch.Tensor
    router: torch.Tensor
    bias: torch.Tensor | None
    handle: fb.flint_moe_layer
    canonical: dict = field(default_factory=dict)
    norm: torch.Tensor | None = None


def _fill_normal(out: torch.Tensor, seed: int, layer: int, tensor: int, expert: int, sigma: float, bf16: bool,
                 stream=None) -> None:
    key = fb.flint_synth_stream_key(seed, layer, tensor, expert)
    fb.flint_synth_normal(key, 0, out.numel(), sigma, bf16, out, stream)


def synth_router(cfg, seed: int, layer: int, device) -> torch.Tensor:
    r = torch.empty(cfg.num_experts, cfg.hidden, dtype=torch.int16, device=device)
    for e in range(cfg.num_experts):
        _fill_normal(r[e], seed, layer, fb.ROUTER, e, ROUTER_SIGMA, True)
    return r


def synth_x(B: int, hidden: int, seed: int, layer: int, device) -> torch.Tensor:
    x = torch.empty(B, hidden, dtype=torch.int16, device=device)
    for t in range(B):
        _fill_normal(x[t], seed, layer, fb.X, t, 1.0, True)
    return x


def synth_norm(hidden: int, seed: int, layer: int, device) -> torch.Tensor:
    """RMSNorm weight: bf16 bits of float32(1 + 0.1 * N(0, 1))."""
    n = torch.empty(hidden, dtype=torch.float32, device=device)
    _fill_normal(n, seed, layer, fb.NORM, 0, NORM_SIGMA, False)
    return (1.0 + n).to(torch.bfloat16).view(torch.int16)


def synth_canonical(cfg, seed: int, layer: int, device) -> dict:
    """Canonical weights of all E + S experts (shared experts last)."""
    E_all = cfg.num_experts + cfg.n_shared
    H, I = cfg.hidden, cfg.inter
    shapes = {"gate": (I, H), "up": (I, H), "down": (H, I)}
    tags = {"gate": fb.GATE, "up": fb.UP, "down": fb.DOWN}
    out = {}
    for m, (rows, cols) in shapes.items():
        if cfg.weight_fmt == fb.NVFP4:
            w = torch.empty(E_all, rows, cols, dtype=torch.float32, device=device)
            for e in range(E_all):
                _fill_normal(w[e], seed, layer, tags[m], e, WEIGHT_SIGMA, False)
            codes = torch.empty(E_all, rows, cols // 2, dtype=torch.uint8, device=device)
            scales = torch.empty(E_all, rows, cols // 16, dtype=torch.uint8, device=device)
            glob = torch.empty(E_all, dtype=torch.float32, device=device)
            fb.flint_moe_quantize_nvfp4(w, E_all, rows, cols, codes, scales, glob)
            del w
            out[m + "_codes"], out[m + "_scales"], out[m + "_global"] = codes, scales, glob
        else:
            w = torch.empty(E_all, rows, cols, dtype=torch.int16, device=device)
            for e in range(E_all):
                _fill_normal(w[e], seed, layer, tags[m], e, WEIGHT_SIGMA, True)
            out[m + "_bf16"] = w
    return out


def synth_layer(cfg, seed: int, layer: int = 0, device="cuda", bias: torch.Tensor | None = None,
                keep_canonical: bool = False, norm_eps: float | None = None) -> DeviceLayer:
    """A packed layer; with norm_eps it also gets a pre-norm RMSNorm weight."""
    canon = synth_canonical(cfg, seed, layer, device)
    packed = torch.empty(fb.flint_moe_packed_bytes(cfg), dtype=torch.uint8, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    fb.flint_moe_pack(cfg, canon, packed, status)
    if int(status.item()) != 0:
        raise RuntimeError(f"flint_moe_pack reported device status {int(status.item())}")
    router = synth_router(cfg, seed, layer, device)
    handle = fb.flint_moe_layer_init(cfg, packed, router, bias)
    norm = None
    if norm_eps is not None:
        norm = synth_norm(cfg.hidden, seed, layer, device)
        fb.flint_moe_layer_set_norm(handle, norm, norm_eps)
    return DeviceLayer(cfg=cfg, packed=packed, router=router, bias=bias, handle=handle,
                       canonical=canon if keep_canonical else {}, norm=norm)


def synth_dense(N: int, K: int, seed: int, layer: int = 0, fmt: int = fb.NVFP4, device="cuda"):
    """A packed dense matrix W [N][K] (stream (seed, layer, DOWN, 0), N(0, 0.02)),
    quantised (NVFP4) or rounded (BF16) on the GPU. Returns (packed, canonical)."""
    if fmt == fb.NVFP4:
        w = torch.empty(N, K, dtype=torch.float32, device=device)
        _fill_normal(w, seed, layer, fb.DOWN, 0, WEIGHT_SIGMA, False)
        canon = {"codes": torch.empty(N, K // 2, dtype=torch.uint8, device=device),
                 "scales": torch.empty(N, K // 16, dtype=torch.uint8, device=device),
                 "global": torch.empty(1, dtype=torch.float32, device=device)}
        fb.flint_moe_quantize_nvfp4(w, 1, N, K, canon["codes"], canon["scales"], canon["global"])
        del w
    else:
        canon = {"bf16": torch.empty(N, K, dtype=torch.int16, device=device)}
        _fill_normal(canon["bf16"], seed, layer, fb.DOWN, 0, WEIGHT_SIGMA, True)
    packed = torch.empty(fb.flint_gemv_packed_bytes(N, K, fmt), dtype=torch.uint8, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    fb.flint_gemv_pack(canon, N, K, fmt, packed, status)
    if int(status.item()) != 0:
        raise RuntimeError(f"flint_gemv_pack reported device status {int(status.item())}")
    return packed, canon


def workspace(cfg, max_batch: int, device="cuda") -> torch.Tensor:
    ws = torch.empty(fb.flint_moe_workspace_bytes(cfg, max_batch), dtype=torch.uint8, device=device)
    fb.flint_moe_workspace_init(cfg, max_batch, ws)
    return ws


def prefill_workspace(cfg, max_tokens: int, device="cuda") -> torch.Tensor:
    nbytes = fb.flint_moe_prefill_workspace_bytes(cfg, max_tokens)
    if nbytes == 0:
        raise ValueError("configuration or token count not supported by the prefill path")
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    fb.flint_moe_prefill_workspace_init(cfg, max_tokens, ws)
    return ws
