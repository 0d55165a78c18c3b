"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Pass rules, fixed in advance: expert indices and dequantised weights
bit-exact (ties to the lower index); tokens whose top-k / top-(k+1) key gap
is below 1e-6 are reported and excluded; routing weights within 1e-6;
outputs within 2^-7 * max(1, |ref|) per element.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import moe, nvfp4
from w4a16_moe_decode_gb300 import binding as fb
from w4a16_moe_decode_gb300 import layers
from w4a16_moe_decode_gb300.build import build

from _common import (FLINT, TINY, bits_to_f64, check_out, check_routing, check_routing_prenorm, needed_experts,
                     oracle_config, oracle_experts, oracle_inputs)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    fb.lib()


def cfg_of(d, fmt=fb.NVFP4, **kw):
    return fb.make_config(hidden=d["hidden"], num_experts=d["num_experts"], top_k=d["top_k"], inter=d["inter"],
                          n_shared=d["n_shared"], weight_fmt=fmt, **kw)


def gpu_decode(cfg, dl, B, seed, layer, ws=None):
    x = layers.synth_x(B, cfg.hidden, seed, layer, DEV)
    out = torch.full_like(x, 0x7FC0)  # bf16 NaN pattern: every element must be written
    ws = layers.workspace(cfg, B, DEV) if ws is None else ws
    fb.flint_moe_decode(dl.handle, x, B, out, ws)
    idx = torch.empty(B, cfg.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(B, cfg.top_k, dtype=torch.float32, device=DEV)
    fb.flint_moe_debug_routing(cfg, ws, B, idx, w)
    st, bits = fb.flint_moe_read_status(ws)
    assert st == fb.OK and bits == 0
    return x, out, idx.cpu().numpy(), w.cpu().numpy()


def run_parity(d, B, seed=0, layer=0, fmt=fb.NVFP4, tokens=None, bias=None, renormalize=True, routed_scale=1.0):
    """Decode B tokens on the GPU and compare with the oracle: the routing of
    every token (indices bit-exact, weights within 1e-6, tokens whose key gap is
    below 1e-6 excluded), and the outputs of `tokens` (default: all)."""
    cfg = cfg_of(d, fmt, renormalize=renormalize, routed_scale=routed_scale)
    bias_t = None if bias is None else torch.from_numpy(np.asarray(bias, np.float32)).to(DEV)
    dl = layers.synth_layer(cfg, seed, layer, DEV, bias=bias_t)
    x, out, idx, w = gpu_decode(cfg, dl, B, seed, layer)
    xo, router = oracle_inputs(d, seed, layer, B)
    assert np.array_equal(bits_to_f64(x), xo)  # both generators drew the same activations
    oc = oracle_config(d, renormalize, routed_scale)
    tokens = list(range(B)) if tokens is None else tokens
    routing = moe.route(xo, router, oc, bias)
    excluded = check_routing(routing, idx, w)  # every token
    get = oracle_experts(d, seed, layer, fmt == fb.BF16, prefetch=needed_experts(d, routing, tokens))
    ref, routing2 = moe.moe_layer(xo, router, get, oc, bias, tokens)
    assert np.array_equal(routing2.idx, routing.idx)
    keep = [i for i, t in enumerate(tokens) if t not in excluded]
    got = bits_to_f64(out)[tokens]
    worst = check_out(ref[keep], got[keep], f"decode {d['hidden']}x{d['num_experts']} B={B} seed={seed}")
    return worst, excluded, routing


def tile_samples(B):
    """Output tokens checked at batch B: all of them up to 8; beyond, two of
    every 8-token tile (its first and last column) and the batch's last token."""
    if B <= 8:
        return list(range(B))
    return sorted({t for base in range(0, B, 8) for t in (base, min(base + 7, B - 1))} | {B - 1})


# ---------------------------------------------------------------- inputs and formats

def test_synth_gpu_matches_cpu_generator():
    for key, start, n, sigma in [(synth.stream_key(0, 0, synth.GATE, 3), 0, 4099, 0.02),
                                 (synth.stream_key(7, 46, synth.X, 31), 123456789, 1000, 1.0)]:
        f = torch.empty(n, dtype=torch.float32, device=DEV)
        fb.flint_synth_normal(key, start, n, sigma, False, f)
        assert np.array_equal(f.cpu().numpy(), synth.normal_scaled_f32(key, start, n, sigma))
        b = torch.empty(n, dtype=torch.int16, device=DEV)
        fb.flint_synth_normal(key, start, n, sigma, True, b)
        assert np.array_equal(b.cpu().numpy().view(np.uint16),
                              synth.f32_to_bf16_bits(synth.normal_scaled_f32(key, start, n, sigma)))


def _gpu_quantize(w):
    n_mat, rows, cols = w.shape
    wd = torch.from_numpy(np.ascontiguousarray(w)).to(DEV)
    codes = torch.empty(n_mat, rows, cols // 2, dtype=torch.uint8, device=DEV)
    scales = torch.empty(n_mat, rows, cols // 16, dtype=torch.uint8, device=DEV)
    g = torch.empty(n_mat, dtype=torch.float32, device=DEV)
    fb.flint_moe_quantize_nvfp4(wd, n_mat, rows, cols, codes, scales, g)
    return codes.cpu().numpy(), scales.cpu().numpy(), g.cpu().numpy()


def test_quantizer_gpu_matches_oracle():
    mats = [synth.matrix_f32(0, 0, synth.GATE, e, 512, 2048, 0.02) for e in (0, 255)]
    special = synth.matrix_f32(1, 0, synth.UP, 0, 32, 256, 0.02)
    special[0] = 0.0                                   # an all-zero row: zero scales and codes
    special[1, :16] = 0.0                              # one zero block
    grid = np.array([0, .25, .5, .75, 1, 1.25, 1.5, 1.75, 2, 2.5, 3, 3.5, 4, 5, 6, 7], np.float32)
    special[2, :16] = grid * np.float32(special.__abs__().max() / 6)   # values near E2M1 midpoints
    special[3, :16] = -special[2, :16]
    for w in mats + [special]:
        c, s, g = _gpu_quantize(w[None])
        oc, os_, og = nvfp4.quantize(w)
        assert np.array_equal(s[0], os_)
        assert np.array_equal(c[0], oc)
        assert g[0] == og
    zero = np.zeros((1, 16, 32), np.float32)
    c, s, g = _gpu_quantize(zero)
    assert not c.any() and not s.any() and g[0] == 0


@pytest.mark.parametrize("d,fmt", [(TINY, fb.NVFP4), (TINY, fb.BF16), (FLINT, fb.NVFP4)])
def test_pack_is_a_bijection(d, fmt):
    cfg = cfg_of(d, fmt)
    canon = layers.synth_canonical(cfg, 3, 0, DEV)
    packed = torch.empty(fb.flint_moe_packed_bytes(cfg), dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    fb.flint_moe_pack(cfg, canon, packed, status)
    back = {k: torch.full_like(v, 0x5A if v.dtype != torch.float32 else 7.0) for k, v in canon.items()}
    fb.flint_moe_unpack_debug(cfg, packed, back)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for k in canon:
        assert torch.equal(canon[k], back[k]), k


def test_pack_flags_nan_scales():
    cfg = cfg_of(TINY)
    canon = layers.synth_canonical(cfg, 0, 0, DEV)
    canon["down_scales"][3, 5, 1] = 0x7F
    packed = torch.empty(fb.flint_moe_packed_bytes(cfg), dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    fb.flint_moe_pack(cfg, canon, packed, status)
    assert int(status.item()) & fb.DEV_ERR_NAN_SCALE


@pytest.mark.parametrize("d,experts", [(TINY, range(17)), (FLINT, (0, 77, 256))])
def test_dequantised_weights_bit_exact(d, experts):
    cfg = cfg_of(d)
    dl = layers.synth_layer(cfg, 0, 0, DEV)
    shapes = [(d["inter"], d["hidden"]), (d["inter"], d["hidden"]), (d["hidden"], d["inter"])]
    get = oracle_experts(d, 0, 0)
    for e in experts:
        mats = get(e)
        for m in range(3):
            out = torch.empty(shapes[m], dtype=torch.float32, device=DEV)
            fb.flint_moe_debug_dequant(cfg, dl.packed, e, m, out)
            ref = (mats[m].c().astype(np.float32) * np.float32(mats[m].G)).astype(np.float32)
            assert np.array_equal(out.cpu().numpy(), ref), (e, m)


# ---------------------------------------------------------------- the decode layer

@pytest.mark.parametrize("B,seed", [(1, 0), (1, 1), (3, 2), (8, 3), (9, 4), (32, 5)])
def test_decode_tiny(B, seed):
    run_parity(TINY, B, seed)


def test_decode_flint_batch1():
    worst, excluded, routing = run_parity(FLINT, 1, seed=0)
    assert not excluded


@pytest.mark.parametrize("B,seed", [(2, 1), (4, 2), (8, 0)])
def test_decode_flint_every_token(B, seed):
    """Flint shape at 2, 4 and 8 tokens: every token's routing and output."""
    run_parity(FLINT, B, seed=seed)


def test_decode_flint_batch32_routing_of_every_token():
    """32 tokens: every token's routing; outputs of two tokens per 8-token tile."""
    run_parity(FLINT, 32, seed=5, tokens=tile_samples(32))


def test_decode_bf16_weights():
    run_parity(FLINT, 1, seed=0, fmt=fb.BF16)
    run_parity(FLINT, 2, seed=3, fmt=fb.BF16)
    run_parity(FLINT, 8, seed=0, fmt=fb.BF16)
    run_parity(TINY, 5, seed=1, fmt=fb.BF16)


def test_decode_all_experts_routed_no_renorm_scaled():
    d = dict(TINY, top_k=16)
    run_parity(d, 4, seed=6, renormalize=False, routed_scale=2.5)


def test_decode_without_shared_expert():
    run_parity(dict(TINY, n_shared=0), 3, seed=7)
    run_parity(dict(TINY, n_shared=2), 2, seed=8)


def test_decode_selection_bias():
    bias = np.zeros(16, np.float32)
    bias[[2, 9]] = 1.0
    _, _, routing = run_parity(TINY, 4, seed=9, bias=bias)
    assert all(set(routing.idx[t]) == {2, 9} for t in range(4))


@pytest.mark.parametrize("E,k,B,seed", [(512, 4, 12, 12), (300, 3, 10, 13), (100, 5, 9, 14)])
def test_decode_expert_counts_off_the_flint_shape(E, k, B, seed):
    """More experts than one warp's 8-per-lane top-k holds (E > 256: the
    16-per-lane path), a count that is not a multiple of 32, and one that leaves
    the last lanes partly empty; B > 8 puts tokens on every warp of a block."""
    run_parity(dict(TINY, num_experts=E, top_k=k), B, seed)


def test_decode_exact_key_ties_go_to_the_lower_index():
    """A selection bias of 2^24 makes the keys of experts 3, 5, 9, 12 exactly
    equal in FP32 (2^24 + s rounds to 2^24 for every score s in (0, 1)), so the
    top-2 is decided by the index alone: experts 3 and 5, in that order, for
    every token. The pass rules exclude such tokens from the oracle comparison
    (their gap is 0), so the choice is checked here against the definition."""
    bias = np.zeros(16, np.float32)
    bias[[12, 5, 9, 3]] = 2.0 ** 24
    cfg = cfg_of(TINY)
    dl = layers.synth_layer(cfg, 15, 0, DEV, bias=torch.from_numpy(bias).to(DEV))
    x, out, idx, w = gpu_decode(cfg, dl, 6, 15, 0)
    assert (idx == np.array([3, 5], np.int32)[None, :]).all()
    xo, router = oracle_inputs(TINY, 15, 0, 6)
    routing = moe.route(xo, router, oracle_config(TINY), bias)
    assert (routing.idx == np.array([3, 5])[None, :]).all()
    np.testing.assert_allclose(w, routing.w, rtol=0, atol=1e-6)


def test_routing_reciprocal_is_the_ieee_quotient():
    """The sigmoid's reciprocal (hardware approximation plus one Newton-Raphson
    step) equals the IEEE quotient 1.0f / y for every FP32 y in [1, 2^125)."""
    assert fb.flint_moe_debug_rcp_check(0x3F800000, (127 + 125) << 23) == 0


def _stack_bias_vector(E=256):
    import os
    import sys
    sys.path.insert(0, os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden"))
    import make_stack_bias as msb
    b = np.zeros(E, np.float32)
    b[:msb.N_BIASED] = np.float32(msb.read_beta())
    return b


@pytest.mark.parametrize("B,L", [(1, 0), (2, 1), (4, 2), (8, 3), (32, 46)])
def test_decode_flint_stack_layers_with_selection_bias(B, L):
    """Layers of the skewed 47-layer stack workload (generator seed 1000 + L,
    selection bias on experts 0..25): every token's routing; outputs of every
    token up to 8, of two tokens per 8-token tile at 32."""
    bias = _stack_bias_vector()
    _, _, routing = run_parity(FLINT, B, seed=1000 + L, layer=L, bias=bias, tokens=tile_samples(B))
    if B >= 4:
        assert (routing.idx < 26).any()


def test_flint_stack_chain_graph_equals_serial():
    """Three chained Flint-shape layers with the stack's selection bias, batch
    4: a CUDA-graph replay (PDL between all kernels) is bit-identical to the
    same decodes run one at a time with a full synchronisation between them."""
    cfg = cfg_of(FLINT)
    bias = torch.from_numpy(_stack_bias_vector()).to(DEV)
    B = 4
    dls = [layers.synth_layer(cfg, 1000 + L, L, DEV, bias=bias) for L in range(3)]
    ws = layers.workspace(cfg, 32, DEV)
    x0 = layers.synth_x(B, cfg.hidden, 1000, 0, DEV)
    serial = [x0] + [torch.empty_like(x0) for _ in range(3)]
    for L in range(3):
        fb.flint_moe_decode(dls[L].handle, serial[L], B, serial[L + 1], ws)
        torch.cuda.synchronize()
    bufs = [x0] + [torch.zeros_like(x0) for _ in range(3)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for L in range(3):
                fb.flint_moe_decode(dls[L].handle, bufs[L], B, bufs[L + 1], ws, s)
    s.synchronize()
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(serial[1:], bufs[1:]):
            assert torch.equal(a, b)
    st, bits = fb.flint_moe_read_status(ws)
    assert st == fb.OK and bits == 0


def run_parity_prenorm(d, B, seed=0, layer=0, tokens=None, bias=None, inplace=False, scale=8.0):
    """The pre-norm block r' = r + layer(rmsnorm(r)) against the oracle; the
    residual stream is the seeded x times a power of two (still bf16)."""
    cfg = cfg_of(d)
    bias_t = None if bias is None else torch.from_numpy(np.asarray(bias, np.float32)).to(DEV)
    dl = layers.synth_layer(cfg, seed, layer, DEV, bias=bias_t, norm_eps=1e-6)
    r = (layers.synth_x(B, cfg.hidden, seed, layer, DEV).view(torch.bfloat16) * scale).view(torch.int16)
    r_in = r.clone()
    out = r if inplace else torch.full_like(r, 0x7FC0)
    ws = layers.workspace(cfg, B, DEV)
    fb.flint_moe_decode_prenorm(dl.handle, r, B, out, ws)
    idx = torch.empty(B, cfg.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(B, cfg.top_k, dtype=torch.float32, device=DEV)
    fb.flint_moe_debug_routing(cfg, ws, B, idx, w)
    st, bits = fb.flint_moe_read_status(ws)
    assert st == fb.OK and bits == 0
    xo, router = oracle_inputs(d, seed, layer, B)
    ro = xo * scale
    assert np.array_equal(bits_to_f64(r_in), ro)  # both generators drew the same residual stream
    gamma = moe.bf16_bits_to_f64(synth.norm_bf16(seed, layer, d["hidden"]))
    assert np.array_equal(bits_to_f64(dl.norm), gamma)
    tokens = list(range(B)) if tokens is None else tokens
    oc = oracle_config(d)
    routing = moe.route(moe.rmsnorm(ro, gamma, 1e-6), router, oc, bias)
    excluded, _ = check_routing_prenorm(ro, gamma, 1e-6, router, oc, bias, idx.cpu().numpy(), w.cpu().numpy())
    get = oracle_experts(d, seed, layer, prefetch=needed_experts(d, routing, tokens))
    ref, routing2 = moe.moe_block(ro, router, get, oc, gamma, 1e-6, bias, tokens)
    assert np.array_equal(routing2.idx, routing.idx)
    keep = [i for i, t in enumerate(tokens) if t not in excluded]
    check_out(ref[keep], bits_to_f64(out)[tokens][keep], f"decode prenorm {d['hidden']} B={B} seed={seed}")
    return routing


@pytest.mark.parametrize("B,seed,inplace", [(1, 20, False), (3, 21, True), (32, 22, False)])
def test_decode_prenorm_tiny(B, seed, inplace):
    run_parity_prenorm(TINY, B, seed, inplace=inplace)


def test_decode_prenorm_flint():
    """Pre-norm block at the Flint shape: 1 token (the router normalises in
    shared memory), 2 (each router warp normalises inside its dot product),
    8 and 16 (the rows arrive normalised by the normalisation kernel)."""
    run_parity_prenorm(FLINT, 1, seed=23)
    run_parity_prenorm(FLINT, 2, seed=24)
    run_parity_prenorm(FLINT, 8, seed=1004, layer=4, bias=_stack_bias_vector(), inplace=True)
    run_parity_prenorm(FLINT, 16, seed=25, layer=2, tokens=[0, 9, 15])


def test_decode_batch0_is_a_noop():
    cfg = cfg_of(TINY)
    dl = layers.synth_layer(cfg, 0, 0, DEV)
    out = torch.full((1, cfg.hidden), 123, dtype=torch.int16, device=DEV)
    ws = layers.workspace(cfg, 1, DEV)
    fb.flint_moe_decode(dl.handle, out, 0, out, ws)
    torch.cuda.synchronize()
    assert int(out[0, 0]) == 123


def test_decode_deterministic_and_chained_through_a_graph():
    """Three layers chained (out of one is x of the next), launched with PDL,
    captured in a CUDA graph and replayed twice: both replays are bit-identical
    to the same decodes run one at a time with a full synchronisation between
    them, and the first layer matches the oracle."""
    d = TINY
    cfg = cfg_of(d)
    B = 2
    dls = [layers.synth_layer(cfg, 11, L, DEV) for L in range(3)]
    ws = layers.workspace(cfg, B, DEV)
    x0 = layers.synth_x(B, cfg.hidden, 11, 0, DEV)
    bufs = [x0] + [torch.empty_like(x0) for _ in range(3)]
    serial = [x0] + [torch.empty_like(x0) for _ in range(3)]
    for L in range(3):
        fb.flint_moe_decode(dls[L].handle, serial[L], B, serial[L + 1], ws)
        torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for L in range(3):
                fb.flint_moe_decode(dls[L].handle, bufs[L], B, bufs[L + 1], ws, s)
    s.synchronize()
    for _ in range(2):
        for b in bufs[1:]:
            b.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(serial[1:], bufs[1:]):
            assert torch.equal(a, b)
    xo, router = oracle_inputs(d, 11, 0, B)
    ref, routing = moe.moe_layer(xo, router, oracle_experts(d, 11, 0), oracle_config(d))
    keep = [t for t in range(B) if routing.gap[t] >= 1e-6]
    check_out(ref[keep], bits_to_f64(serial[1])[keep], "layer 0")
    st, bits = fb.flint_moe_read_status(ws)
    assert st == fb.OK and bits == 0


def test_bounded_wait_gives_up_and_reports():
    """The failure path of every kernel wait, without a fault: a wait that
    nothing completes times out (about 200 ms), sets the timeout bit and
    returns; the context stays usable for the next decode."""
    import time
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    t0 = time.time()
    fb.flint_moe_debug_wait_timeout(status)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x1  # FLINT_MOE_DEV_ERR_TIMEOUT
    assert time.time() - t0 < 10.0
    worst, excluded, _ = run_parity(TINY, 3, seed=5)  # the GPU still decodes correctly


@pytest.mark.parametrize("d,B,prenorm", [(TINY, 3, False), (FLINT, 1, False), (FLINT, 8, False), (FLINT, 2, True),
                                           (FLINT, 4, True), (FLINT, 8, True)])
def test_decode_with_x_and_out_in_pinned_host_memory(d, B, prenorm):
    """x and out in pinned host memory (the kernels read and write them across
    the host link): bit-identical to the same decode on device buffers, with
    the pre-norm block updating the residual stream in host memory in place."""
    cfg = cfg_of(d)
    dl = layers.synth_layer(cfg, 41, 0, DEV, norm_eps=1e-6 if prenorm else None)
    ws = layers.workspace(cfg, B, DEV)
    x = layers.synth_x(B, cfg.hidden, 41, 0, DEV)
    ref = torch.empty_like(x)
    call = fb.flint_moe_decode_prenorm if prenorm else fb.flint_moe_decode
    call(dl.handle, x, B, ref, ws)
    xh = x.cpu().pin_memory()
    oh = xh if prenorm else torch.full((B, cfg.hidden), 0x7FC0, dtype=torch.int16).pin_memory()
    call(dl.handle, xh, B, oh, ws)
    torch.cuda.synchronize()
    assert torch.equal(oh, ref.cpu())
    st, bits = fb.flint_moe_read_status(ws)
    assert st == fb.OK and bits == 0
    unpinned = torch.zeros(B, cfg.hidden, dtype=torch.int16)  # ordinary host memory: refused before any launch
    with pytest.raises(fb.FlintMoeError):
        call(dl.handle, unpinned, B, ref, ws)


@pytest.mark.parametrize("prefill", [False, True])
def test_prenorm_rounding_decision_at_32_tokens(prefill):
    """Seed 61, 32 tokens: the FP32 normalisation of token 31 rounds an element
    to the other bf16 neighbour than the float64 oracle does (it lies within
    FP32 error of the rounding boundary), which moves that token's routing
    weights by about 4e-6 with the same experts. The pre-norm check accepts it
    through that rounding, on the small-batch kernels and on the
    expert-grouped path alike."""
    d, seed, B = FLINT, 61, 32
    cfg = cfg_of(d)
    dl = layers.synth_layer(cfg, seed, 0, DEV, norm_eps=1e-6)
    r = layers.synth_x(B, cfg.hidden, seed, 0, DEV)
    out = torch.full_like(r, 0x7FC0)
    idx = torch.empty(B, cfg.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(B, cfg.top_k, dtype=torch.float32, device=DEV)
    if prefill:
        ws = layers.prefill_workspace(cfg, B, DEV)
        fb.flint_moe_prefill_prenorm(dl.handle, r, B, out, ws)
        fb.flint_moe_prefill_debug_routing(cfg, ws, B, idx, w)
    else:
        ws = layers.workspace(cfg, B, DEV)
        fb.flint_moe_decode_prenorm(dl.handle, r, B, out, ws)
        fb.flint_moe_debug_routing(cfg, ws, B, idx, w)
    st, bits = fb.flint_moe_read_status(ws)
    assert st == fb.OK and bits == 0
    ro, router = oracle_inputs(d, seed, 0, B)
    gamma = moe.bf16_bits_to_f64(synth.norm_bf16(seed, 0, d["hidden"]))
    oc = oracle_config(d)
    excluded, rerounded = check_routing_prenorm(ro, gamma, 1e-6, router, oc, None, idx.cpu().numpy(),
                                                w.cpu().numpy())
    assert excluded == [] and rerounded == [31]
    tokens = [0, 16, 31]
    routing = moe.route(moe.rmsnorm(ro, gamma, 1e-6), router, oc)
    get = oracle_experts(d, seed, 0, prefetch=needed_experts(d, routing, tokens))
    ref, _ = moe.moe_block(ro, router, get, oc, gamma, 1e-6, None, tokens)
    check_out(ref, bits_to_f64(out)[tokens], f"prenorm B=32 seed=61, {'prefill' if prefill else 'decode'}")
