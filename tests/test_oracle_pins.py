"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test ties one oracle function to a table, a library routine, a brute
force search, an invariant or a textbook special case, so that a dropped term,
a wrong sign, index or operand order in the oracle fails at least one of them.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import synth
from oracle import moe, nvfp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a, b = line.split()
            rows.append((a, b))
    return rows


# ------------------------------------------------------------------ NVFP4 codes

def test_e2m1_decode_table():
    rows = _read_table("e2m1_table.txt")
    assert len(rows) == 16
    for code, value in rows:
        got = float(nvfp4.e2m1_decode(int(code)))
        want = float(value)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), (code, got, want)


def test_e4m3_decode_table():
    for code, value in _read_table("e4m3_table.txt"):
        got = float(nvfp4.e4m3_decode(int(code, 16)))
        if value == "nan":
            assert math.isnan(got)
        else:
            assert got == float(value) and math.copysign(1, got) == math.copysign(1, float(value)), code


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256)
    ours = nvfp4.e4m3_decode(codes)
    theirs = torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(theirs)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], theirs[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(theirs[~nan]))


def _e4m3_midpoints():
    grid = nvfp4.e4m3_decode(np.arange(0x7F))
    mids = (grid[:-1] + grid[1:]) / 2
    return np.concatenate([grid, mids]).astype(np.float32)


def test_e4m3_encode_matches_torch():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        _e4m3_midpoints(), -_e4m3_midpoints(),
        rng.uniform(-448, 448, 20000).astype(np.float32),
        (rng.standard_normal(20000) * np.exp2(rng.integers(-12, 9, 20000))).astype(np.float32),
    ]).astype(np.float32)
    vals = vals[np.abs(vals) <= 448]
    ours = nvfp4.e4m3_encode(vals)
    theirs = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # torch keeps the sign of values that round to zero, as we do
    assert np.array_equal(ours, theirs)


def test_e4m3_encode_saturates():
    assert int(nvfp4.e4m3_encode(np.float32(449.0))) == 0x7E
    assert int(nvfp4.e4m3_encode(np.float32(1e30))) == 0x7E
    assert int(nvfp4.e4m3_encode(np.float32(-500.0))) == 0xFE


def _e2m1_brute(x):
    """Nearest of the 16 codes by exhaustive search; tie -> even code; keep sign."""
    out = []
    for v in np.asarray(x, np.float64):
        best = None
        for code in range(8):
            mag = float(nvfp4.e2m1_decode(code))
            d = abs(abs(v) - mag)
            key = (d, code & 1)
            if best is None or key < best[0]:
                best = (key, code)
        code = best[1] if abs(v) <= 6 else 7
        out.append(code | (8 if math.copysign(1, v) < 0 else 0))
    return np.array(out, np.uint8)


def test_e2m1_encode_bruteforce():
    rng = np.random.default_rng(2)
    grid = nvfp4.e2m1_decode(np.arange(8))
    mids = (grid[:-1] + grid[1:]) / 2
    vals = np.concatenate([grid, mids, -grid, -mids, rng.uniform(-8, 8, 3000),
                           np.nextafter(mids, 0), np.nextafter(mids, 10)]).astype(np.float32)
    assert np.array_equal(nvfp4.e2m1_encode(vals), _e2m1_brute(vals))


def test_e2m1_ties_golden():
    for value, code in _read_table("e2m1_ties.txt"):
        assert int(nvfp4.e2m1_encode(np.float32(float(value)))) == int(code), value


def test_nibble_order():
    # element 2j is the low nibble of byte j
    b = np.array([[0x21, 0x43]], np.uint8)
    assert nvfp4.unpack_codes(b).tolist() == [[1, 2, 3, 4]]
    assert np.array_equal(nvfp4.pack_codes(nvfp4.unpack_codes(b)), b)


# ------------------------------------------------------------------ quantiser

def _quant_error_bound(w, codes, scales, G):
    """Per element: half the E2M1 gap around the chosen code, times the block
    scale, plus the saturation excess when |w| exceeds 6 * scale * G, plus a few
    float32 roundings of the intermediate steps."""
    q = np.abs(nvfp4.e2m1_decode(nvfp4.unpack_codes(codes)))
    s = np.repeat(nvfp4.e4m3_decode(scales), nvfp4.BLOCK, axis=1) * np.float64(G)
    grid = nvfp4.e2m1_decode(np.arange(8))
    gaps = np.diff(grid)
    idx = np.searchsorted(grid, q)
    gap_up = np.where(idx < 7, gaps[np.minimum(idx, 6)], 0.0)
    gap_dn = np.where(idx > 0, gaps[np.maximum(idx - 1, 0)], 0.0)
    half = 0.5 * np.maximum(gap_up, gap_dn) * s
    sat = np.maximum(np.abs(w) - 6 * s, 0)
    return half + sat + 4 * np.finfo(np.float32).eps * np.abs(w).astype(np.float64) + 1e-30


def test_quantize_roundtrip_bound():
    w = synth.matrix_f32(0, 0, synth.GATE, 3, 64, 512, 0.02)
    codes, scales, G = nvfp4.quantize(w)
    d = nvfp4.dequantize(codes, scales, G)
    err = np.abs(d - w.astype(np.float64))
    assert np.all(err <= _quant_error_bound(w, codes, scales, G))
    # the largest element of the tensor lands on a full-scale code
    assert np.max(np.abs(d)) == pytest.approx(float(np.max(np.abs(w))), rel=0.07)


def test_quantize_idempotent_on_exact_grid():
    """Weights that are already E2M1 * E4M3 * G, with G a power of two, every
    block holding a +-6 and one block at scale 448, quantise back to the same
    codes and scales (sign of zero included)."""
    rng = np.random.default_rng(3)
    rows, cols = 8, 64
    elems = rng.integers(0, 16, (rows, cols)).astype(np.uint8)
    for r in range(rows):
        for b in range(cols // 16):
            elems[r, b * 16 + rng.integers(0, 16)] = rng.choice([7, 15])
    scales = rng.integers(0x08, 0x7E, (rows, cols // 16)).astype(np.uint8)
    scales[0, 0] = 0x7E
    G = np.float32(2.0 ** -14)
    codes = nvfp4.pack_codes(elems)
    w = nvfp4.dequantize(codes, scales, G).astype(np.float32)
    c2, s2, G2 = nvfp4.quantize(w)
    assert G2 == G
    assert np.array_equal(s2, scales)
    assert np.array_equal(c2, codes)


def test_quantize_zero_tensor_and_zero_block():
    codes, scales, G = nvfp4.quantize(np.zeros((4, 32), np.float32))
    assert G == 0 and not codes.any() and not scales.any()
    w = synth.matrix_f32(0, 0, synth.UP, 0, 4, 32, 0.02)
    w[1, 16:] = 0
    codes, scales, G = nvfp4.quantize(w)
    assert scales[1, 1] == 0 and not codes[1, 8:].any()


# ------------------------------------------------------------------ rounding

def test_bf16_round_matches_torch():
    rng = np.random.default_rng(4)
    v = np.concatenate([rng.standard_normal(50000) * np.exp2(rng.integers(-40, 40, 50000)),
                        [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 65504.0]])
    ours = moe.bf16_round(v)
    theirs = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(ours, theirs)


def test_synth_bf16_matches_torch():
    v = synth.normal_f32(12345, 0, 4096)
    bits = synth.f32_to_bf16_bits(v)
    theirs = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits, theirs)


def test_synth_normal_moments():
    z = synth.normal_f32(synth.stream_key(0, 0, synth.X, 0), 0, 200000).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    assert np.abs(z).max() <= 6.0
    # counter-based: any window equals the matching slice of a longer draw
    key = synth.stream_key(7, 3, synth.GATE, 11)
    assert np.array_equal(synth.normal_f32(key, 1000, 50), synth.normal_f32(key, 0, 1050)[1000:])


# ------------------------------------------------------------------ router

def _tiny_cfg(**kw):
    base = dict(hidden=256, num_experts=16, top_k=2, inter=64, n_shared=1)
    base.update(kw)
    return moe.Config(**base)


def _inputs(cfg, B, seed=0):
    router = moe.bf16_bits_to_f64(synth.router_bf16(seed, 0, cfg.num_experts, cfg.hidden))
    x = moe.bf16_bits_to_f64(synth.x_bf16(seed, 0, B, cfg.hidden))
    return x, router


def test_topk_matches_bruteforce_subsets():
    cfg = _tiny_cfg()
    x, router = _inputs(cfg, 8)
    r = moe.route(x, router, cfg)
    for t in range(8):
        best = max(itertools.combinations(range(cfg.num_experts), cfg.top_k),
                   key=lambda c: (sum(float(r.key[t, e]) for e in c), [-e for e in c]))
        assert sorted(r.idx[t].tolist()) == sorted(best)
        # ordered by key descending
        assert all(r.key[t, r.idx[t, j]] >= r.key[t, r.idx[t, j + 1]] for j in range(cfg.top_k - 1))


def test_sigmoid_and_logits_against_direct_sum():
    cfg = _tiny_cfg()
    x, router = _inputs(cfg, 2)
    r = moe.route(x, router, cfg)
    for t in range(2):
        for e in (0, 5, 15):
            dot = math.fsum(float(a) * float(b) for a, b in zip(x[t], router[e]))
            assert r.logits[t, e] == np.float32(dot)
            assert abs(float(r.s[t, e]) - 1 / (1 + math.exp(-float(np.float32(dot))))) < 1e-7


def test_routing_weights_sum_to_one():
    cfg = moe.Config(hidden=2048, num_experts=256, top_k=6, inter=512)
    x, router = _inputs(cfg, 8)
    r = moe.route(x, router, cfg)
    assert np.all(r.w >= 0)
    assert np.all(np.abs(r.w.astype(np.float64).sum(1) - 1) <= 2 ** -20)
    assert r.idx.shape == (8, 6) and all(len(set(row)) == 6 for row in r.idx.tolist())


def test_routed_scale_with_and_without_renormalisation():
    """The routed scale multiplies the final weights: after renormalisation a
    token's weights sum to the scale (a scale applied before renormalising would
    cancel); without renormalisation each weight is the scale times the sigmoid
    of its logit, here recomputed from an exact sum, and the experts are the k
    largest sigmoids found by brute force."""
    scale = 2.5
    cfg = _tiny_cfg(top_k=3, routed_scale=scale)
    x, router = _inputs(cfg, 4, seed=3)
    r = moe.route(x, router, cfg)
    assert np.all(np.abs(r.w.astype(np.float64).sum(1) - scale) <= scale * 2 ** -20)
    cfg_raw = _tiny_cfg(top_k=3, routed_scale=scale, renormalize=False)
    r_raw = moe.route(x, router, cfg_raw)
    for t in range(4):
        sig = [1 / (1 + math.exp(-float(np.float32(math.fsum(float(a) * float(b) for a, b in zip(x[t], router[e]))))))
               for e in range(cfg.num_experts)]
        best = sorted(range(cfg.num_experts), key=lambda e: (-sig[e], e))[:3]
        assert r_raw.idx[t].tolist() == best
        for j, e in enumerate(best):
            assert abs(float(r_raw.w[t, j]) - scale * sig[e]) <= scale * 2 ** -21


def test_ties_go_to_lower_index():
    cfg = _tiny_cfg(top_k=3)
    x = np.zeros((1, cfg.hidden))            # all logits 0, all scores 0.5
    router = np.ones((cfg.num_experts, cfg.hidden))
    r = moe.route(x, router, cfg)
    assert r.idx[0].tolist() == [0, 1, 2]
    assert r.gap[0] == 0.0
    assert np.allclose(r.w, 1 / 3)


def test_bias_selects_but_does_not_weight():
    cfg = _tiny_cfg()
    x, router = _inputs(cfg, 1)
    bias = np.zeros(16, np.float32)
    bias[[13, 14]] = 10.0
    r = moe.route(x, router, cfg, bias)
    assert sorted(r.idx[0].tolist()) == [13, 14]
    s = r.s[0, [r.idx[0, 0], r.idx[0, 1]]].astype(np.float64)
    assert np.allclose(r.w[0], s / s.sum(), rtol=1e-6)


# ------------------------------------------------------------------ layer

def _tiny_experts(cfg, seed=0):
    cache = {}

    def get(e):
        if e not in cache:
            g, u, d = synth.expert_f32(seed, 0, e, cfg.hidden, cfg.inter)
            cache[e] = tuple(moe.NVFP4Matrix(*nvfp4.quantize(m)) for m in (g, u, d))
        return cache[e]
    return get


def test_layer_matches_dense_all_experts_formulation():
    """Second formulation: every expert computed densely for every token, then
    multiplied by a routing mask built from the top-k indices."""
    cfg = _tiny_cfg()
    B = 4
    x, router = _inputs(cfg, B)
    get = _tiny_experts(cfg)
    out, r = moe.moe_layer(x, router, get, cfg)
    E = cfg.num_experts
    Y = np.stack([moe.expert(x, get(e)) for e in range(E + 1)])       # [E+1, B, H]
    mask = np.zeros((B, E + 1))
    for t in range(B):
        for j in range(cfg.top_k):
            mask[t, r.idx[t, j]] = r.w[t, j]
        mask[t, E] = 1.0
    dense = moe.bf16_round(moe.f32(np.einsum("tb,tbh->bh", mask.T, Y)))
    assert np.array_equal(out, dense)


def test_expert_applies_each_matrix_scale_to_its_own_product():
    """One expert with real block scales and three different per-tensor scales
    (gate 0.75, up 1.25, down 0.5), against torch on the full weights
    E2M1 * E4M3 * G built here from the codes (E4M3 through torch's float8
    type): a dropped G_d moves y by its own size, and the gate and up scales
    swapped move most elements of h by far more than their bf16 rounding."""
    rng = np.random.default_rng(11)
    H, I, B = 64, 32, 3
    # x / 8 (exact) puts g around |g| ~ 2, where SiLU is far from linear, so
    # silu(G_g g) * G_u u is not symmetric in the two scales
    x = moe.bf16_bits_to_f64(synth.x_bf16(4, 0, B, H)) / 8

    def rand_matrix(rows, cols, G):
        elems = rng.integers(0, 16, (rows, cols)).astype(np.uint8)
        scales = rng.integers(0x28, 0x48, (rows, cols // 16)).astype(np.uint8)
        return moe.NVFP4Matrix(nvfp4.pack_codes(elems), scales, np.float32(G))

    g, u, d = rand_matrix(I, H, 0.75), rand_matrix(I, H, 1.25), rand_matrix(H, I, 0.5)
    y = moe.expert(x, (g, u, d))

    E2M1 = torch.tensor([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6], dtype=torch.float64)

    def W(m):
        q = E2M1[torch.from_numpy(nvfp4.unpack_codes(m.codes).astype(np.int64))]
        sc = torch.from_numpy(m.scales).view(torch.float8_e4m3fn).double().repeat_interleave(16, dim=1)
        return q * sc * float(m.G)

    xt = torch.from_numpy(x)
    gg = (xt @ W(g).T).float().double()
    uu = (xt @ W(u).T).float().double()
    h_ref = (torch.nn.functional.silu(gg) * uu).float().to(torch.bfloat16).double()
    ref = (h_ref @ W(d).T).numpy()
    h_ref = h_ref.numpy()

    def h_ok(h):  # within one bf16 rounding of the reference, element by element
        return np.abs(h - h_ref) <= 2 ** -7 * np.abs(h_ref) + 2 ** -40

    assert np.all(h_ok(moe.expert_hidden(x, g, u)))
    assert np.max(np.abs(y - ref)) <= 2 ** -7 * np.max(np.abs(ref))
    swapped = moe.expert_hidden(x, moe.NVFP4Matrix(g.codes, g.scales, u.G), moe.NVFP4Matrix(u.codes, u.scales, g.G))
    assert np.mean(h_ok(swapped)) < 0.5


def test_layer_reduces_to_textbook_swiglu():
    """All block scales 1.0 (E4M3 0x38) and G = 1: every weight is an E2M1
    value and the layer is a dense SwiGLU MoE, computed here with torch in
    float64 from the weight values directly, with all experts routed (k = E)."""
    cfg = _tiny_cfg(num_experts=4, top_k=4, hidden=64, inter=32)
    rng = np.random.default_rng(5)
    B = 3
    x = moe.bf16_bits_to_f64(synth.x_bf16(9, 0, B, cfg.hidden))
    router = moe.bf16_bits_to_f64(synth.router_bf16(9, 0, cfg.num_experts, cfg.hidden))
    mats = {}

    def rand_matrix(rows, cols):
        elems = rng.integers(0, 16, (rows, cols)).astype(np.uint8)
        return moe.NVFP4Matrix(nvfp4.pack_codes(elems), np.full((rows, cols // 16), 0x38, np.uint8),
                               np.float32(1.0))

    for e in range(cfg.num_experts + 1):
        mats[e] = (rand_matrix(cfg.inter, cfg.hidden), rand_matrix(cfg.inter, cfg.hidden),
                   rand_matrix(cfg.hidden, cfg.inter))
    out, r = moe.moe_layer(x, router, lambda e: mats[e], cfg)

    E2M1 = torch.tensor([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6], dtype=torch.float64)

    def W(m):
        return E2M1[torch.from_numpy(nvfp4.unpack_codes(m.codes).astype(np.int64))]

    xt = torch.from_numpy(x)
    logits = (xt @ torch.from_numpy(router).T).float()
    s = torch.sigmoid(logits.double()).float().double()
    wts = (s / s.sum(1, keepdim=True)).float().double()
    acc = torch.zeros(B, cfg.hidden, dtype=torch.float64)
    for e in range(cfg.num_experts + 1):
        g, u, d = mats[e]
        gg = (xt @ W(g).T).float().double()
        uu = (xt @ W(u).T).float().double()
        h = (torch.nn.functional.silu(gg) * uu).float().to(torch.bfloat16).double()
        y = h @ W(d).T
        acc += (wts[:, e:e + 1] if e < cfg.num_experts else 1.0) * y
    ref = acc.float().to(torch.bfloat16).double().numpy()
    ulp = np.abs(ref) * 2 ** -7 + 1e-30
    assert np.all(np.abs(out - ref) <= ulp)
    assert np.mean(out == ref) > 0.98


def test_expected_distinct():
    assert moe.expected_distinct(256, 6, 1) == pytest.approx(6.0)
    assert moe.expected_distinct(256, 6, 8) == pytest.approx(44.2, abs=0.1)


def test_unique_bytes_flint_batch1():
    cfg = moe.Config(hidden=2048, num_experts=256, top_k=6, inter=512)
    assert moe.unique_weight_bytes(cfg, 6, 1) == 1048576 + 7 * 3 * (524288 + 65536 + 4) + 8192


def test_tiny_layer_regression_record():
    """The oracle still reproduces its committed decode of the tiny layer."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_tiny_golden", os.path.join(GOLDEN, "make_tiny_golden.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    x, router, get = mod.tiny_inputs()
    out, r = moe.moe_layer(x, router, get, mod.CFG)
    rec = {}
    with open(os.path.join(GOLDEN, "tiny_layer_seed0.txt")) as f:
        for line in f:
            if line.startswith("#"):
                continue
            k, *v = line.split()
            rec[k] = v
    assert r.idx[0].tolist() == [int(v) for v in rec["idx"]]
    assert r.w[0].tolist() == [float(v) for v in rec["w"]]
    assert moe.f64_to_bf16_bits(out[0]).tolist() == [int(v, 16) for v in rec["out_bf16_hex"]]


# ------------------------------------------------------------------ pre-norm block

def test_rmsnorm_matches_torch_rms_norm():
    """The normalisation against torch's rms_norm in float64 (a library
    routine), both rounded by the same bf16 rounding."""
    H = 256
    x = moe.bf16_bits_to_f64(synth.x_bf16(3, 0, 5, H))
    g = moe.bf16_bits_to_f64(synth.norm_bf16(3, 0, H))
    for eps in (1e-6, 0.5):
        ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (H,), weight=torch.from_numpy(g), eps=eps).numpy()
        assert np.array_equal(moe.rmsnorm(x, g, eps), moe.bf16_round(ref))


def test_rmsnorm_closed_forms():
    H = 256
    g = np.ones(H)
    # a constant row normalises to its sign (eps = 0)
    assert np.array_equal(moe.rmsnorm(np.full((1, H), -3.0), g, 0.0), np.full((1, H), -1.0))
    # one nonzero element v: mean square v^2 / H, so it becomes sign(v) * sqrt(H) = 16
    x = np.zeros((1, H))
    x[0, 7] = 0.375
    y = moe.rmsnorm(x, g, 0.0)
    assert y[0, 7] == 16.0 and np.count_nonzero(y) == 1
    # the weight multiplies channel by channel
    gw = moe.bf16_bits_to_f64(synth.norm_bf16(1, 0, H))
    assert np.array_equal(moe.rmsnorm(np.full((1, H), 2.0), gw, 0.0)[0], moe.bf16_round(gw))


def test_rmsnorm_is_scale_invariant():
    """Scaling a row by a power of two changes nothing when eps = 0 (exact)."""
    H = 512
    x = moe.bf16_bits_to_f64(synth.x_bf16(4, 0, 3, H))
    g = moe.bf16_bits_to_f64(synth.norm_bf16(4, 0, H))
    for k in (-6, 5):
        assert np.array_equal(moe.rmsnorm(x * 2.0 ** k, g, 0.0), moe.rmsnorm(x, g, 0.0))


def test_moe_block_with_zero_experts_is_the_identity():
    """With every expert weight zero the layer adds exactly zero, so the block
    returns the residual stream unchanged; the routing still happens on the
    normalised input (the same selection as routing rmsnorm(r) directly)."""
    cfg = moe.Config(hidden=256, num_experts=16, top_k=2, inter=64, n_shared=1)
    zero = nvfp4.quantize(np.zeros((64, 256), np.float32))
    zero_d = nvfp4.quantize(np.zeros((256, 64), np.float32))
    get = lambda e: (moe.NVFP4Matrix(*zero), moe.NVFP4Matrix(*zero), moe.NVFP4Matrix(*zero_d))  # noqa: E731
    r = moe.bf16_bits_to_f64(synth.x_bf16(5, 0, 3, 256)) * 8.0  # still bf16 values
    router = moe.bf16_bits_to_f64(synth.router_bf16(5, 0, 16, 256))
    g = moe.bf16_bits_to_f64(synth.norm_bf16(5, 0, 256))
    out, routing = moe.moe_block(r, router, get, cfg, g, 1e-6)
    assert np.array_equal(out, r)
    assert np.array_equal(routing.idx, moe.route(moe.rmsnorm(r, g, 1e-6), router, cfg).idx)


def test_moe_block_adds_the_rounded_layer_output_to_the_residual():
    """The pre-norm block with non-zero experts, computed independently with
    torch in float64: RMSNorm by torch's rms_norm, the layer as a textbook
    dense SwiGLU MoE with every expert routed (k = E, block scales 2^-4, G = 1,
    so every weight is an E2M1 value / 16), and r' = bf16(r + bf16(layer)).
    The two agree element by element except where the two float64 sums round
    differently (a few percent of elements, by one bf16 ulp). Rounding r + acc
    only once, or subtracting the layer output, would differ from the torch
    block in far more elements; the test checks that it can tell."""
    H, I, E = 64, 32, 4
    cfg = moe.Config(hidden=H, num_experts=E, top_k=E, inter=I, n_shared=1)
    rng = np.random.default_rng(17)
    B = 6
    r = moe.bf16_bits_to_f64(synth.x_bf16(13, 0, B, H))
    router = moe.bf16_bits_to_f64(synth.router_bf16(13, 0, E, H))
    gamma = moe.bf16_bits_to_f64(synth.norm_bf16(13, 0, H))
    eps = 1e-6

    def rand_matrix(rows, cols):
        elems = rng.integers(0, 16, (rows, cols)).astype(np.uint8)
        return moe.NVFP4Matrix(nvfp4.pack_codes(elems), np.full((rows, cols // 16), 0x18, np.uint8), np.float32(1.0))

    mats = {e: (rand_matrix(I, H), rand_matrix(I, H), rand_matrix(H, I)) for e in range(E + 1)}
    out_o, _ = moe.moe_block(r, router, lambda e: mats[e], cfg, gamma, eps)

    E2M1 = torch.tensor([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6], dtype=torch.float64)

    def W(m):
        return E2M1[torch.from_numpy(nvfp4.unpack_codes(m.codes).astype(np.int64))] / 16.0

    def bf16(t):
        return t.float().to(torch.bfloat16).double()

    rt = torch.from_numpy(r)
    xt = bf16(torch.nn.functional.rms_norm(rt, (H,), weight=torch.from_numpy(gamma), eps=eps))
    s = torch.sigmoid((xt @ torch.from_numpy(router).T).float().double()).float().double()
    wts = (s / s.sum(1, keepdim=True)).float().double()
    acc = torch.zeros(B, H, dtype=torch.float64)
    for e in range(E + 1):
        g, u, d = mats[e]
        gg = (xt @ W(g).T).float().double()
        uu = (xt @ W(u).T).float().double()
        h = bf16(torch.nn.functional.silu(gg) * uu)
        acc += (wts[:, e:e + 1] if e < E else 1.0) * (h @ W(d).T)
    block = bf16(rt + bf16(acc)).numpy()
    once = bf16(rt + acc).numpy()          # the residual add without rounding the layer output first
    minus = bf16(rt - bf16(acc)).numpy()   # the layer output subtracted

    assert np.abs(bf16(acc).numpy()).max() > 0.5      # the layer output is of the residual's size
    ulp = np.abs(block) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(out_o - block) <= ulp)
    agree = np.mean(out_o == block)
    assert agree > 0.97
    assert np.mean(once == block) < agree - 0.05       # a single rounding would be seen
    assert np.mean(minus == block) < 0.2


# ------------------------------------------------------------------ dense GEMV

def _dense_matrix(seed, N, K):
    w = synth.matrix_f32(seed, 0, synth.DOWN, 0, N, K, 0.02)
    return moe.NVFP4Matrix(*nvfp4.quantize(w))


def test_gemv_matches_torch_matmul_of_the_dequantised_matrix():
    from oracle import dense
    W = _dense_matrix(11, 48, 256)
    x = moe.bf16_bits_to_f64(synth.x_bf16(11, 0, 3, 256))
    ref = torch.from_numpy(x) @ torch.from_numpy(nvfp4.dequantize(W.codes, W.scales, W.G)).T
    assert np.array_equal(dense.gemv(x, W), moe.bf16_round(ref.numpy()))


def test_gemv_one_hot_input_selects_a_column():
    """x = e_j gives y = bf16(G * c[:, j]) exactly."""
    from oracle import dense
    W = _dense_matrix(12, 32, 128)
    for j in (0, 17, 127):
        x = np.zeros((1, 128))
        x[0, j] = 1.0
        assert np.array_equal(dense.gemv(x, W)[0], moe.bf16_round(np.float64(W.G) * W.c()[:, j]))


def test_gemv_commutes_with_power_of_two_scaling():
    from oracle import dense
    W = _dense_matrix(13, 64, 256)
    x = moe.bf16_bits_to_f64(synth.x_bf16(13, 0, 2, 256))
    for k in (-5, 4):
        assert np.array_equal(dense.gemv(x * 2.0 ** k, W), dense.gemv(x, W) * 2.0 ** k)


def test_gemv_with_norm_weight_is_gemv_of_the_normalised_rows():
    from oracle import dense
    W = _dense_matrix(14, 32, 256)
    x = moe.bf16_bits_to_f64(synth.x_bf16(14, 0, 2, 256)) * 4.0
    g = moe.bf16_bits_to_f64(synth.norm_bf16(14, 0, 256))
    assert np.array_equal(dense.gemv(x, W, g, 1e-6), dense.gemv(moe.rmsnorm(x, g, 1e-6), W))
    # and normalisation makes the result independent of the row scale (eps = 0)
    assert np.array_equal(dense.gemv(x, W, g, 0.0), dense.gemv(x * 0.125, W, g, 0.0))
