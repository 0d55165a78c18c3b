"""Helpers shared by the GPU tests: oracle-side inputs and the pass rules.

The oracle's inputs come from the CPU generator (synth) and the oracle's own
quantiser; nothing here reads a value produced by the CUDA path into the oracle.
Expert weights for the oracle are generated on the host, several experts at a
time in a pool of worker processes started with `spawn` (a process forked
after the first CUDA call can hang), and each matrix's dequantised weights are
computed once and reused across tokens (the values are the oracle's own
``c()``; keeping them as float32 is exact, since every NVFP4 product E2M1 x
E4M3 and every bf16 value is a float32 number).
"""
import atexit
import os

import numpy as np

import synth
from oracle import moe, nvfp4

TINY = dict(hidden=256, num_experts=16, top_k=2, inter=64, n_shared=1)
FLINT = dict(hidden=2048, num_experts=256, top_k=6, inter=512, n_shared=1)

GAP_MIN = 1e-6          # tokens whose k-th / (k+1)-th key gap is below this are excluded
W_TOL = 1e-6            # routing weights
OUT_REL = 2.0 ** -7     # |d| <= 2^-7 * max(1, |ref|)

# Worst errors of every output comparison of the session, printed at its end
# (label, elements, worst err / tol, worst and median error in bf16 ulps of ref).
RESULTS = []


def oracle_config(d, renormalize=True, routed_scale=1.0):
    return moe.Config(hidden=d["hidden"], num_experts=d["num_experts"], top_k=d["top_k"], inter=d["inter"],
                      n_shared=d["n_shared"], renormalize=renormalize, routed_scale=routed_scale)


class CachedMatrix:
    """An oracle matrix whose dequantised weights c() are computed once."""

    def __init__(self, m):
        self.m = m
        self.G = m.G
        self._c = None

    def c(self):
        if self._c is None:
            c = self.m.c()
            c32 = c.astype(np.float32)
            assert np.array_equal(c32.astype(np.float64), c)  # exact: see the module docstring
            self._c = c32
        return self._c.astype(np.float64)


def _make_expert(args):
    """Worker: (gate, up, down) of one expert as plain arrays."""
    hidden, inter, seed, layer, e, bf16 = args
    mats = synth.expert_f32(seed, layer, e, hidden, inter)
    if bf16:
        return [("bf16", synth.f32_to_bf16_bits(m)) for m in mats]
    return [("nvfp4",) + tuple(nvfp4.quantize(m)) for m in mats]


def _wrap(parts):
    out = []
    for p in parts:
        m = moe.BF16Matrix(p[1]) if p[0] == "bf16" else moe.NVFP4Matrix(p[1], p[2], p[3])
        out.append(CachedMatrix(m))
    return tuple(out)


_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        import multiprocessing as mp
        from concurrent.futures import ProcessPoolExecutor
        n = max(1, min(16, (os.cpu_count() or 2) - 1))
        _POOL = ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn"))
        atexit.register(_POOL.shutdown)
    return _POOL


def oracle_experts(d, seed, layer, bf16=False, prefetch=()):
    """get(e) -> (gate, up, down) oracle matrices of expert e (shared experts
    are e >= E). Experts listed in `prefetch` are generated up front in
    parallel; any other is generated on first use."""
    cache = {}
    todo = sorted(set(int(e) for e in prefetch))
    if len(todo) > 2:
        args = [(d["hidden"], d["inter"], seed, layer, e, bf16) for e in todo]
        for e, parts in zip(todo, _pool().map(_make_expert, args)):
            cache[e] = _wrap(parts)

    def get(e):
        if e not in cache:
            cache[e] = _wrap(_make_expert((d["hidden"], d["inter"], seed, layer, e, bf16)))
        return cache[e]
    return get


def needed_experts(d, routing, tokens):
    """The experts whose weights the oracle reads for these tokens."""
    sel = set(routing.idx[list(tokens)].ravel().tolist()) if len(tokens) else set()
    return sorted(sel | {d["num_experts"] + s for s in range(d["n_shared"])})


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


# The GPU computes the pre-norm RMSNorm r * w / sqrt(mean(r^2) + eps) in FP32
# before rounding it to bf16: each lane sums the squares of 64 of a 2048-wide
# row's elements, a 5-level butterfly adds the lanes, then a division, a square
# root, a reciprocal and two products. All terms positive, that is at most
# (64 + 5) rounding errors of 2^-24 relative in the sum, half of it after the
# root, a few more after: below 2^-18 relative. Where the float64 value lies
# within that of a bf16 rounding boundary, the GPU may round it to the other
# neighbour.
NORM_REL = 2.0 ** -18
NORM_MAX_UNDECIDED = 12  # at most 2^12 rounding combinations tried per token


def prenorm_undecided(r, gamma, eps):
    """The oracle's normalised rows xn (bf16 values) and, per element, the other
    bf16 value the GPU's FP32 normalisation may round to (equal to xn where
    the rounding is decided)."""
    x = np.asarray(r, np.float64)
    g = np.asarray(gamma, np.float64)
    v = x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + np.float64(eps)) * g[None, :]
    xn = moe.bf16_round(v)
    lo, hi = moe.bf16_round(v * (1 - NORM_REL)), moe.bf16_round(v * (1 + NORM_REL))
    alt = np.where(lo != xn, lo, hi)
    return xn, alt


def check_routing_prenorm(r, gamma, eps, router, cfg, bias, idx_gpu, w_gpu, tokens=None):
    """check_routing for the pre-norm block. The oracle's routing of the
    normalised rows must match, or, for a token whose normalisation has
    elements within NORM_REL of a bf16 rounding boundary, the routing of one
    of the rows those elements' two roundings give (the rounding is the one
    step where FP32 and float64 may decide differently). Returns (excluded
    tokens, tokens matched through another rounding)."""
    xn, alt = prenorm_undecided(r, gamma, eps)
    routing = moe.route(xn, router, cfg, bias)
    B = routing.idx.shape[0]
    tokens = range(B) if tokens is None else tokens
    excluded, rerounded = [], []
    for t in tokens:
        if routing.gap[t] < GAP_MIN:
            excluded.append(t)
            continue
        def same(rt, row=0):
            return (idx_gpu[t].tolist() == rt.idx[row].tolist() and
                    np.all(np.abs(w_gpu[t].astype(np.float64) - rt.w[row].astype(np.float64)) <= W_TOL))
        if same(routing, t):
            continue
        und = np.nonzero(alt[t] != xn[t])[0]
        assert 0 < len(und) <= NORM_MAX_UNDECIDED, (t, len(und), idx_gpu[t], routing.idx[t], w_gpu[t], routing.w[t])
        rows = np.repeat(xn[t][None, :], 2 ** len(und), axis=0)
        for m in range(1, 2 ** len(und)):
            flip = [und[j] for j in range(len(und)) if (m >> j) & 1]
            rows[m, flip] = alt[t, flip]
        rt = moe.route(rows, router, cfg, bias)
        assert any(same(rt, m) for m in range(1, rows.shape[0])), (t, idx_gpu[t], routing.idx[t], w_gpu[t],
                                                                  routing.w[t])
        rerounded.append(t)
    return excluded, rerounded


def bf16_ulp(ref):
    """Spacing of bf16 numbers at |ref| (8 significant bits; the subnormal
    spacing 2^-133 below 2^-126)."""
    a = np.abs(np.asarray(ref, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def check_out(ref, got, label=""):
    """The output rule |got - ref| <= 2^-7 max(1, |ref|), element by element.
    The error is also measured in bf16 ulps of ref (recorded for the session
    summary): the fixed rule is loose where |ref| << 1, the ulp count is not."""
    ref = np.asarray(ref, np.float64)
    got = np.asarray(got, np.float64)
    assert ref.shape == got.shape
    assert np.all(np.isfinite(got)), label
    err = np.abs(got - ref)
    tol = OUT_REL * np.maximum(1.0, np.abs(ref))
    bad = err > tol
    ulps = err / bf16_ulp(ref)
    worst_ulp = float(ulps.max()) if ulps.size else 0.0
    med_ulp = float(np.median(ulps)) if ulps.size else 0.0
    ratio = float((err / tol).max()) if err.size else 0.0
    RESULTS.append((label, int(ref.size), ratio, worst_ulp, med_ulp))
    assert not bad.any(), (f"{label}: {int(bad.sum())} of {bad.size} beyond tolerance, worst {ratio:.3f}x, "
                           f"worst {worst_ulp:.1f} bf16 ulps of ref")
    return ratio
