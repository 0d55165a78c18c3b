"""The MoE decode layer: router, experts, combine. float64 CPU definition.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Layer (pages: "Day-0 Support for Flint on vLLM", section "Model
architecture": 256 experts, sigmoid top-6, plus one shared expert; section
"Optimisation": router and expert GEMVs, SiLU with the reference rounding,
routing and combine fused into the GEMVs). For one token x (bf16 values):

    logit_e = sum_h x_h * Wr[e, h]                (float64, rounded once to float32)
    s_e     = float32(1 / (1 + exp(-logit_e)))
    key_e   = float32(s_e + bias_e)               (bias only selects; zero if absent)
    top-k   = first k of (key desc, e asc)        (full sort; ties to the lower index)
    w_j     = float32(s_j / sum_top s) * routed_scale   (renormalised; else s_j * routed_scale)
    g_i     = float32(G_g * sum_h c_g[i, h] x_h)  (likewise u_i)
    h_i     = bf16(float32(silu(g_i) * u_i)),     silu(z) = z / (1 + exp(-z))
    y_j     = G_d * sum_i c_d[j, i] h_i           (float64)
    out_j   = bf16(float32(sum_k w_k y_{e_k, j} + sum_shared y_{S, j}))

Readings where the pages are silent: renormalisation, the selection bias, the
intermediate size and the rounding points come from the workload definition; the shared expert is unweighted and has the routed
experts' intermediate size; there is no residual add inside the layer (the
pre-norm block below adds it around the layer); tokens are routed
independently. For BF16 expert weights c is the bf16 weight and G = 1.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import nvfp4


# ------------------------------------------------------------ rounding points

def f32(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64).astype(np.float32)


def bf16_round(a) -> np.ndarray:
    """Round to bf16 (nearest even) through float32; returns float64 values.
    float64 -> float32 is numpy's IEEE round-to-nearest-even."""
    b = f32(a).view(np.uint32).astype(np.uint64)
    b = ((b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)) << np.uint64(16)
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def bf16_bits_to_f64(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(a) -> np.ndarray:
    return (bf16_round(a).astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# ------------------------------------------------------------ config

@dataclass
class Config:
    hidden: int
    num_experts: int
    top_k: int
    inter: int
    n_shared: int = 1
    renormalize: bool = True
    routed_scale: float = 1.0


@dataclass
class Routing:
    idx: np.ndarray      # int64 [B, k]
    w: np.ndarray        # float32 [B, k]
    s: np.ndarray        # float32 [B, E] sigmoid scores
    key: np.ndarray      # float32 [B, E] selection keys
    gap: np.ndarray      # float64 [B]: key of k-th minus key of (k+1)-th (inf if k == E)
    logits: np.ndarray   # float32 [B, E]


# ------------------------------------------------------------ router

def sigmoid_f32(logit) -> np.ndarray:
    l = np.asarray(logit, dtype=np.float32).astype(np.float64)
    return f32(1.0 / (1.0 + np.exp(-l)))


def route(x: np.ndarray, router: np.ndarray, cfg: Config, bias: np.ndarray | None = None) -> Routing:
    """Sigmoid top-k routing of every token (rows of x, float64 bf16 values)."""
    x = np.asarray(x, dtype=np.float64)
    wr = np.asarray(router, dtype=np.float64)
    logits = f32(x @ wr.T)
    s = sigmoid_f32(logits)
    b = np.zeros(cfg.num_experts, np.float32) if bias is None else np.asarray(bias, np.float32)
    key = (s + b[None, :]).astype(np.float32)
    B, E, k = x.shape[0], cfg.num_experts, cfg.top_k
    idx = np.zeros((B, k), np.int64)
    w = np.zeros((B, k), np.float32)
    gap = np.full(B, np.inf)
    experts = np.arange(E)
    for t in range(B):
        order = np.lexsort((experts, -key[t].astype(np.float64)))   # key desc, then e asc
        top = order[:k]
        idx[t] = top
        if k < E:
            gap[t] = float(key[t, order[k - 1]]) - float(key[t, order[k]])
        st = s[t, top].astype(np.float64)
        if cfg.renormalize:
            wt = f32(st / st.sum())
        else:
            wt = f32(st)
        w[t] = (wt * np.float32(cfg.routed_scale)).astype(np.float32)
    return Routing(idx=idx, w=w, s=s, key=key, gap=gap, logits=logits)


# ------------------------------------------------------------ experts

@dataclass
class NVFP4Matrix:
    codes: np.ndarray    # uint8 [rows, cols/2]
    scales: np.ndarray   # uint8 [rows, cols/16]
    G: np.float32

    def c(self) -> np.ndarray:
        return nvfp4.dequant_c(self.codes, self.scales)


@dataclass
class BF16Matrix:
    bits: np.ndarray     # uint16 [rows, cols]
    G: np.float32 = np.float32(1.0)

    def c(self) -> np.ndarray:
        return bf16_bits_to_f64(self.bits)


def silu(z) -> np.ndarray:
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def expert_hidden(x: np.ndarray, gate, up) -> np.ndarray:
    """h = bf16(float32(silu(g) * u)) for rows of x; g, u rounded to float32."""
    g = f32(np.float64(gate.G) * (np.asarray(x, np.float64) @ gate.c().T))
    u = f32(np.float64(up.G) * (np.asarray(x, np.float64) @ up.c().T))
    return bf16_round(f32(silu(g.astype(np.float64)) * u.astype(np.float64)))


def expert_out(h: np.ndarray, down) -> np.ndarray:
    """y = G_d * (c_d h), float64, for rows of h."""
    return np.float64(down.G) * (np.asarray(h, np.float64) @ down.c().T)


def expert(x: np.ndarray, weights) -> np.ndarray:
    gate, up, down = weights
    return expert_out(expert_hidden(x, gate, up), down)


# ------------------------------------------------------------ layer

def moe_layer(x: np.ndarray, router: np.ndarray, get_expert, cfg: Config,
              bias: np.ndarray | None = None, tokens=None):
    """Decode one batch. ``get_expert(e)`` returns (gate, up, down) matrices of
    expert e; shared experts are e = E .. E + n_shared - 1. Only the experts the
    routing selects are requested. ``tokens`` restricts the output rows that are
    computed (routing is always computed for every token).

    Returns (out float64 bf16 values [len(tokens), H], Routing)."""
    x = np.asarray(x, dtype=np.float64)
    routing = route(x, router, cfg, bias)
    B = x.shape[0]
    tokens = list(range(B)) if tokens is None else list(tokens)
    cache: dict[int, tuple] = {}

    def weights(e):
        if e not in cache:
            cache[e] = get_expert(e)
        return cache[e]

    out = np.zeros((len(tokens), cfg.hidden), np.float64)
    for row, t in enumerate(tokens):
        acc = np.zeros(cfg.hidden, np.float64)
        for j in range(cfg.top_k):
            e = int(routing.idx[t, j])
            acc += np.float64(routing.w[t, j]) * expert(x[t:t + 1], weights(e))[0]
        for s in range(cfg.n_shared):
            acc += expert(x[t:t + 1], weights(cfg.num_experts + s))[0]
        out[row] = bf16_round(f32(acc))
    return out, routing


# ------------------------------------------------------------ pre-norm block

def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm of every row of x (bf16 values) with weight gamma (bf16 values),
    rounded to bf16: y = bf16(x * gamma / sqrt(mean(x^2) + eps)), float64 inside.

    The pages describe Flint as a pre-norm MoE ("Day-0 Support for Flint on
    vLLM", section "Model architecture") whose norm kernels follow the reference
    rounding (section "Optimisation") without printing the norm; the plain RMS
    normalisation with a learned per-channel weight is the reading, its output
    rounded to bf16 because it is the layer's bf16 activation."""
    x = np.asarray(x, dtype=np.float64)
    g = np.asarray(gamma, dtype=np.float64)
    ms = np.mean(x * x, axis=1, keepdims=True)
    return bf16_round(x / np.sqrt(ms + np.float64(eps)) * g[None, :])


def moe_block(r: np.ndarray, router: np.ndarray, get_expert, cfg: Config, gamma: np.ndarray, eps: float,
              bias: np.ndarray | None = None, tokens=None):
    """One pre-norm MoE sublayer on the residual stream r (bf16 values):
    r' = bf16(r + moe_layer(rmsnorm(r))), the layer output being bf16 already.

    Returns (r' float64 bf16 values [len(tokens), H], Routing)."""
    r = np.asarray(r, dtype=np.float64)
    tokens = list(range(r.shape[0])) if tokens is None else list(tokens)
    out, routing = moe_layer(rmsnorm(r, gamma, eps), router, get_expert, cfg, bias, tokens)
    return bf16_round(r[tokens] + out), routing


def distinct_experts(routing: Routing) -> int:
    return int(np.unique(routing.idx).size)


def unique_weight_bytes(cfg: Config, distinct: int, batch: int, nvfp4_weights: bool = True) -> int:
    """Algorithmic bytes of one decode: bf16 router, the touched experts (routed
    distinct plus shared; NVFP4 codes + E4M3 scales + float32 G, or bf16) and
    the bf16 x and out."""
    H, I = cfg.hidden, cfg.inter
    if nvfp4_weights:
        per_matrix = I * H // 2 + I * H // 16 + 4
    else:
        per_matrix = I * H * 2
    return (cfg.num_experts * H * 2 + (distinct + cfg.n_shared) * 3 * per_matrix
            + 2 * batch * H * 2)


def expected_distinct(E: int, k: int, B: int) -> float:
    """Expected distinct experts among B tokens' uniform top-k picks."""
    return E * (1.0 - (1.0 - k / E) ** B)
