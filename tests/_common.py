"""Helpers shared by the GPU tests: oracle-side inputs and the pass rules.

The oracle's inputs come from the CPU generator (synth) and the oracle's own
quantiser; nothing here reads a value produced by the CUDA path into the oracle.
"""
import numpy as np

import synth
from oracle import moe, nvfp4

TINY = dict(hidden=256, num_experts=16, top_k=2, inter=64, n_shared=1)
FLINT = dict(hidden=2048, num_experts=256, top_k=6, inter=512, n_shared=1)

GAP_MIN = 1e-6          # tokens whose k-th / (k+1)-th key gap is below this are excluded
W_TOL = 1e-6            # routing weights
OUT_REL = 2.0 ** -7     # |d| <= 2^-7 * max(1, |ref|)


def oracle_config(d, renormalize=True, routed_scale=1.0):
    return moe.Config(hidden=d["hidden"], num_experts=d["num_experts"], top_k=d["top_k"], inter=d["inter"],
                      n_shared=d["n_shared"], renormalize=renormalize, routed_scale=routed_scale)


def oracle_experts(d, seed, layer, bf16=False):
    cache = {}

    def get(e):
        if e not in cache:
            mats = synth.expert_f32(seed, layer, e, d["hidden"], d["inter"])
            if bf16:
                cache[e] = tuple(moe.BF16Matrix(synth.f32_to_bf16_bits(m)) for m in mats)
            else:
                cache[e] = tuple(moe.NVFP4Matrix(*nvfp4.quantize(m)) for m in mats)
        return cache[e]
    return get


def oracle_inputs(d, seed, layer, B):
    x = moe.bf16_bits_to_f64(synth.x_bf16(seed, layer, B, d["hidden"]))
    router = moe.bf16_bits_to_f64(synth.router_bf16(seed, layer, d["num_experts"], d["hidden"]))
    return x, router


def bits_to_f64(t):
    """int16 torch tensor of bf16 bit patterns -> float64 numpy."""
    return moe.bf16_bits_to_f64(t.cpu().numpy().view(np.uint16))


def check_routing(routing, idx_gpu, w_gpu, tokens=None):
    """Indices bit-exact and weights within W_TOL for tokens whose gap allows a
    decision; returns the list of excluded tokens."""
    B = routing.idx.shape[0]
    tokens = range(B) if tokens is None else tokens
    excluded = []
    for t in tokens:
        if routing.gap[t] < GAP_MIN:
            excluded.append(t)
            continue
        assert idx_gpu[t].tolist() == routing.idx[t].tolist(), (t, idx_gpu[t], routing.idx[t])
        assert np.all(np.abs(w_gpu[t].astype(np.float64) - routing.w[t].astype(np.float64)) <= W_TOL), t
    return excluded


def check_out(ref, got, label=""):
    ref = np.asarray(ref, np.float64)
    got = np.asarray(got, np.float64)
    assert ref.shape == got.shape
    assert np.all(np.isfinite(got)), label
    err = np.abs(got - ref)
    tol = OUT_REL * np.maximum(1.0, np.abs(ref))
    bad = err > tol
    assert not bad.any(), f"{label}: {int(bad.sum())} of {bad.size} beyond tolerance, worst {float((err / tol).max()):.3f}x"
    return float((err / tol).max())
