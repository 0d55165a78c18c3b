"""Parity of the expert-grouped tensor-core path (flint_moe_prefill) with the
CPU oracle, through the C ABI.

Same pass rules as the decode path, fixed in advance: expert indices
bit-exact with ties to the lower index (tokens whose top-k / top-(k+1) key gap
is below 1e-6 are reported and excluded), routing weights within 1e-6, outputs
within 2^-7 * max(1, |ref|) per element. Router logits: the tensor cores
accumulate the bf16 products in FP32, so each logit is compared with the
oracle's float64 sum within 2^-16 of the sum of |x_h w_h| (a few FP32
rounding steps of that magnitude).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import moe
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


def cfg_of(d, **kw):
    return fb.make_config(hidden=d["hidden"], num_experts=d["num_experts"], top_k=d["top_k"], inter=d["inter"],
                          n_shared=d["n_shared"], weight_fmt=fb.NVFP4, **kw)


def gpu_prefill(cfg, dl, B, seed, layer, ws=None, want_logits=False):
    x = layers.synth_x(B, cfg.hidden, seed, layer, DEV)
    out = torch.full_like(x, 0x7FC0)  # bf16 NaN pattern: every element must be written
    ws = layers.prefill_workspace(cfg, B, DEV) if ws is None else ws
    fb.flint_moe_prefill(dl.handle, x, B, out, ws)
    idx = torch.empty(B, cfg.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(B, cfg.top_k, dtype=torch.float32, device=DEV)
    logits = torch.empty(B, cfg.num_experts, dtype=torch.float32, device=DEV) if want_logits else None
    fb.flint_moe_prefill_debug_routing(cfg, ws, B, idx, w, logits)
    st, bits = fb.flint_moe_read_status(ws)
    assert st == fb.OK and bits == 0, (st, bits)
    return x, out, idx.cpu().numpy(), w.cpu().numpy(), (None if logits is None else logits.cpu().numpy())


def run_parity(d, B, seed=0, layer=0, tokens=None, bias=None):
    cfg = cfg_of(d)
    bias_t = None if bias is None else torch.from_numpy(np.asarray(bias, np.float32)).to(DEV)
    dl = layers.synth_layer(cfg, seed, layer, DEV, bias=bias_t)
    x, out, idx, w, _ = gpu_prefill(cfg, dl, B, seed, layer)
    xo, router = oracle_inputs(d, seed, layer, B)
    assert np.array_equal(bits_to_f64(x), xo)
    tokens = list(range(B)) if tokens is None else tokens
    routing = moe.route(xo, router, oracle_config(d), bias)
    excluded = check_routing(routing, idx, w)  # every token
    get = oracle_experts(d, seed, layer, prefetch=needed_experts(d, routing, tokens))
    ref, _ = moe.moe_layer(xo, router, get, oracle_config(d), bias, tokens)
    keep = [i for i, t in enumerate(tokens) if t not in excluded]
    worst = check_out(ref[keep], bits_to_f64(out)[tokens][keep], f"prefill {d['hidden']} B={B} seed={seed}")
    return worst, excluded, routing


@pytest.mark.parametrize("d,B", [(TINY, 37), (FLINT, 130)])
def test_router_logits_on_the_tensor_cores(d, B):
    cfg = cfg_of(d)
    dl = layers.synth_layer(cfg, 2, 0, DEV)
    _, _, _, _, logits = gpu_prefill(cfg, dl, B, 2, 0, want_logits=True)
    xo, router = oracle_inputs(d, 2, 0, B)
    ref = xo @ router.T
    mag = np.abs(xo) @ np.abs(router).T
    err = np.abs(logits.astype(np.float64) - ref)
    assert np.all(err <= 2.0 ** -16 * mag + 1e-30), float((err / (mag + 1e-30)).max())


@pytest.mark.parametrize("B", [1, 2, 16, 37, 129, 300])
def test_prefill_parity_tiny_all_tokens(B):
    worst, excluded, _ = run_parity(TINY, B, seed=B)
    assert len(excluded) <= max(1, B // 20)


# The batch sizes straddle the path's tile choices: up to 256 tokens the shared
# expert takes 16-token mma.sync tiles, beyond it tensor-core tiles; up to 512
# tokens routed experts with at most 16 tokens take small tiles, from 513 on
# every slot takes tensor-core tiles.
@pytest.mark.parametrize("B,tokens", [(1, [0]), (16, [0, 7, 15]), (64, [0, 1, 33, 63]), (256, [0, 100, 255]),
                                      (257, [0, 128, 256]), (300, [0, 128, 299]), (512, [0, 255, 511]),
                                      (513, [0, 256, 512])])
def test_prefill_parity_flint_sampled(B, tokens):
    worst, excluded, routing = run_parity(FLINT, B, seed=11, tokens=tokens)
    assert not set(excluded) & set(tokens) and len(excluded) <= max(1, B // 50)


def test_prefill_routing_exact_for_every_token_flint():
    """All 512 tokens' top-6 indices and weights (the full routing, not a sample)."""
    d, B = FLINT, 512
    cfg = cfg_of(d)
    dl = layers.synth_layer(cfg, 5, 0, DEV)
    _, _, idx, w, _ = gpu_prefill(cfg, dl, B, 5, 0)
    xo, router = oracle_inputs(d, 5, 0, B)
    routing = moe.route(xo, router, oracle_config(d))
    excluded = check_routing(routing, idx, w)
    assert len(excluded) <= 5


def test_prefill_with_selection_bias():
    """Skewed routing (bias on experts 0..25): the bias decides selection only."""
    bias = np.zeros(256, np.float32)
    bias[:26] = np.float32(0.134765625)
    worst, excluded, routing = run_parity(FLINT, 96, seed=21, tokens=[0, 50, 95], bias=bias)
    assert (routing.idx < 26).mean() > 0.3


def test_prefill_reuses_its_workspace_and_is_deterministic():
    d, B = TINY, 200
    cfg = cfg_of(d)
    dl = layers.synth_layer(cfg, 4, 0, DEV)
    ws = layers.prefill_workspace(cfg, B, DEV)
    _, out1, idx1, _, _ = gpu_prefill(cfg, dl, B, 4, 0, ws=ws)
    _, out2, idx2, _, _ = gpu_prefill(cfg, dl, B, 4, 0, ws=ws)
    assert torch.equal(out1, out2)
    assert np.array_equal(idx1, idx2)
    # a smaller call on the same workspace (counters were reset by the plan kernel)
    x, out3, _, _, _ = gpu_prefill(cfg, dl, 17, 4, 0, ws=ws)
    xo, router = oracle_inputs(d, 4, 0, 17)
    ref, routing = moe.moe_layer(xo, router, oracle_experts(d, 4, 0), oracle_config(d))
    keep = [t for t in range(17) if routing.gap[t] >= 1e-6]
    check_out(ref[keep], bits_to_f64(out3)[keep], "reuse B=17")


def test_prefill_and_decode_agree_at_32_tokens():
    """The two paths at the low-latency path's largest batch, both against the oracle."""
    d, B, tokens = FLINT, 32, [0, 13, 31]
    cfg = cfg_of(d)
    dl = layers.synth_layer(cfg, 8, 0, DEV)
    x, out_p, idx_p, _, _ = gpu_prefill(cfg, dl, B, 8, 0)
    out_d = torch.full_like(x, 0x7FC0)
    ws = layers.workspace(cfg, B, DEV)
    fb.flint_moe_decode(dl.handle, x, B, out_d, ws)
    idx_d = torch.empty(B, cfg.top_k, dtype=torch.int32, device=DEV)
    w_d = torch.empty(B, cfg.top_k, dtype=torch.float32, device=DEV)
    fb.flint_moe_debug_routing(cfg, ws, B, idx_d, w_d)
    xo, router = oracle_inputs(d, 8, 0, B)
    routing = moe.route(xo, router, oracle_config(d))
    get = oracle_experts(d, 8, 0, prefetch=needed_experts(d, routing, tokens))
    ref, _ = moe.moe_layer(xo, router, get, oracle_config(d), None, tokens)
    keep = [i for i, t in enumerate(tokens) if routing.gap[t] >= 1e-6]
    check_out(ref[keep], bits_to_f64(out_p)[tokens][keep], "prefill B=32")
    check_out(ref[keep], bits_to_f64(out_d)[tokens][keep], "decode B=32")
    decided = [t for t in range(B) if routing.gap[t] >= 1e-6]
    assert np.array_equal(idx_p[decided], idx_d.cpu().numpy()[decided])


def test_prefill_parity_at_the_largest_bench_size():
    """4096 tokens, the bench's largest prefill point: the routing of every
    token against the oracle, and the outputs of sampled tokens spread over
    the batch (first, last, and tokens in different token tiles)."""
    d, B = FLINT, 4096
    tokens = [0, 127, 128, 2047, 4095]
    cfg = cfg_of(d)
    dl = layers.synth_layer(cfg, 13, 0, DEV)
    x, out, idx, w, _ = gpu_prefill(cfg, dl, B, 13, 0)
    xo, router = oracle_inputs(d, 13, 0, B)
    routing = moe.route(xo, router, oracle_config(d))
    get = oracle_experts(d, 13, 0, prefetch=needed_experts(d, routing, tokens))
    ref, _ = moe.moe_layer(xo, router, get, oracle_config(d), None, tokens)
    excluded = check_routing(routing, idx, w)  # every token
    assert len(excluded) <= B // 100
    keep = [i for i, t in enumerate(tokens) if t not in excluded]
    check_out(ref[keep], bits_to_f64(out)[tokens][keep], "prefill B=4096")


def run_prefill_prenorm(d, B, seed, tokens=None, bias=None, inplace=False, scale=8.0, layer=0):
    """The pre-norm block r' = r + layer(rmsnorm(r)) on the tensor-core path
    against the oracle; the residual stream is the seeded x times a power of two."""
    cfg = cfg_of(d)
    bias_t = None if bias is None else torch.from_numpy(np.asarray(bias, np.float32)).to(DEV)
    dl = layers.synth_layer(cfg, seed, layer, DEV, bias=bias_t, norm_eps=1e-6)
    r = (layers.synth_x(B, cfg.hidden, seed, layer, DEV).view(torch.bfloat16) * scale).view(torch.int16)
    r_in = r.clone()
    out = r if inplace else torch.full_like(r, 0x7FC0)
    ws = layers.prefill_workspace(cfg, B, DEV)
    fb.flint_moe_prefill_prenorm(dl.handle, r, B, out, ws)
    idx = torch.empty(B, cfg.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(B, cfg.top_k, dtype=torch.float32, device=DEV)
    fb.flint_moe_prefill_debug_routing(cfg, ws, B, idx, w)
    st, bits = fb.flint_moe_read_status(ws)
    assert st == fb.OK and bits == 0
    xo, router = oracle_inputs(d, seed, layer, B)
    ro = xo * scale
    assert np.array_equal(bits_to_f64(r_in), ro)
    gamma = moe.bf16_bits_to_f64(synth.norm_bf16(seed, layer, d["hidden"]))
    tokens = list(range(B)) if tokens is None else tokens
    routing = moe.route(moe.rmsnorm(ro, gamma, 1e-6), router, oracle_config(d), bias)
    excluded, _ = check_routing_prenorm(ro, gamma, 1e-6, router, oracle_config(d), bias, idx.cpu().numpy(),
                                        w.cpu().numpy())  # every token
    get = oracle_experts(d, seed, layer, prefetch=needed_experts(d, routing, tokens))
    ref, _ = moe.moe_block(ro, router, get, oracle_config(d), gamma, 1e-6, bias, tokens)
    keep = [i for i, t in enumerate(tokens) if t not in excluded]
    check_out(ref[keep], bits_to_f64(out)[tokens][keep], f"prefill prenorm B={B} seed={seed}")
    return excluded


@pytest.mark.parametrize("B,inplace", [(1, False), (37, True), (200, False)])
def test_prefill_prenorm_tiny(B, inplace):
    excluded = run_prefill_prenorm(TINY, B, seed=40 + B, inplace=inplace)
    assert len(excluded) <= max(1, B // 20)


def test_prefill_prenorm_flint_with_stack_bias():
    bias = np.zeros(256, np.float32)
    bias[:26] = np.float32(0.134765625)
    excluded = run_prefill_prenorm(FLINT, 64, seed=1005, layer=5, tokens=[0, 31, 63], bias=bias, inplace=True)
    assert not set(excluded) & {0, 31, 63} and len(excluded) <= 1
