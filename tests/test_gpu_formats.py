"""The CUDA path on inputs that reach the ends of its number formats, against
the CPU oracle, through the C ABI.

* The whole NVFP4 code space: hand-made canonical matrices in which every
  16-element block holds all 16 E2M1 codes once and the blocks' E4M3 scale
  codes run through every finite code of both signs (0x00, the subnormals
  0x01..0x07, the normals up to 0x7E, and 0x80..0xFE), so every (E2M1 code,
  E4M3 scale) pair occurs in every matrix. The decode kernels' dequantisation
  must give c * G bit for bit, and the decode and tensor-core paths built from
  these matrices must match the oracle. NVIDIA's NVFP4 format is named on the
  page "Day-0 Support for Flint on vLLM", section "Model architecture".
* Activation rows over a wide range: elements 2^-30 .. 2^-40 of their row's
  maximum, rows scaled up to 2^56 (the largest for which silu(g) * u stays
  in FP32 range: the layer's own definition overflows beyond), rows near
  bf16's smallest normal, and, for the pre-norm block (whose RMSNorm brings any
  row back to unit scale), rows near bf16's largest normal. These reach the
  per-token power-of-two prescale of the gate/up products (decode and
  tensor-core paths) and the RMSNorm's range handling.

Pass rules as everywhere: indices bit-exact (tokens whose key gap is below
1e-6 excluded, except exact ties, where the definition's lower-index rule
decides and is checked), weights within 1e-6, outputs within
2^-7 * max(1, |ref|), dequantised weights bit-exact.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import moe, nvfp4
from w4a16_moe_decode_gb300 import binding as fb
from w4a16_moe_decode_gb300 import layers
from w4a16_moe_decode_gb300.build import build

from _common import (FLINT, TINY, bits_to_f64, check_out, check_routing, check_routing_prenorm, oracle_config,
                     oracle_experts, oracle_inputs)

pytestmark = pytest.mark.gpu
DEV = "cuda"
FINITE_E4M3 = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)  # 254 codes


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    fb.lib()


def cfg_of(d, **kw):
    return fb.make_config(hidden=d["hidden"], num_experts=d["num_experts"], top_k=d["top_k"], inter=d["inter"],
                          n_shared=d["n_shared"], weight_fmt=fb.NVFP4, **kw)


# ---------------------------------------------------------------- the NVFP4 code space

def code_space_matrix(rng, rows, cols, G):
    """Every block: the 16 E2M1 codes in a random order; block scales: the 254
    finite E4M3 codes, repeated in fresh random orders to fill the matrix."""
    nblk = rows * cols // 16
    reps = -(-nblk // FINITE_E4M3.size)
    scales = np.concatenate([rng.permutation(FINITE_E4M3) for _ in range(reps)])[:nblk]
    elems = np.argsort(rng.random((nblk, 16)), axis=1).astype(np.uint8)
    return moe.NVFP4Matrix(nvfp4.pack_codes(elems.reshape(rows, cols)), scales.reshape(rows, cols // 16),
                           np.float32(G))


def code_space_layer(d, seed):
    """Oracle matrices of all E + S experts. The tensor scales are arbitrary
    FP32 values of a size that keeps g, u, h and y finite."""
    rng = np.random.default_rng(seed)
    H, I = d["hidden"], d["inter"]
    mats = {}
    for e in range(d["num_experts"] + d["n_shared"]):
        Gg = np.float32(rng.uniform(1.0, 2.0) * 2.0 ** -12)
        Gu = np.float32(rng.uniform(1.0, 2.0) * 2.0 ** -12)
        Gd = np.float32(rng.uniform(1.0, 2.0) * 2.0 ** -13)
        mats[e] = (code_space_matrix(rng, I, H, Gg), code_space_matrix(rng, I, H, Gu), code_space_matrix(rng, H, I, Gd))
    return mats


def device_layer(cfg, mats, seed, layer, bias=None, norm_eps=None):
    """Packs the oracle's canonical matrices with flint_moe_pack (the bytes go
    to the device as they are) and draws the router like every other test."""
    E_all = cfg.num_experts + cfg.n_shared
    canon = {}
    for mi, m in enumerate(("gate", "up", "down")):
        canon[m + "_codes"] = torch.from_numpy(np.stack([mats[e][mi].codes for e in range(E_all)])).to(DEV)
        canon[m + "_scales"] = torch.from_numpy(np.stack([mats[e][mi].scales for e in range(E_all)])).to(DEV)
        canon[m + "_global"] = torch.tensor([float(mats[e][mi].G) for e in range(E_all)], dtype=torch.float32,
                                            device=DEV)
    packed = torch.empty(fb.flint_moe_packed_bytes(cfg), dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    fb.flint_moe_pack(cfg, canon, packed, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    router = layers.synth_router(cfg, seed, layer, DEV)
    handle = fb.flint_moe_layer_init(cfg, packed, router, bias)
    norm = None
    if norm_eps is not None:
        norm = layers.synth_norm(cfg.hidden, seed, layer, DEV)
        fb.flint_moe_layer_set_norm(handle, norm, norm_eps)
    return layers.DeviceLayer(cfg=cfg, packed=packed, router=router, bias=bias, handle=handle, norm=norm)


def test_code_space_covers_every_pair():
    """The hand-made matrices really hold every (E2M1 code, finite E4M3 scale) pair."""
    m = code_space_matrix(np.random.default_rng(0), 64, 256, 1.0)
    elems = nvfp4.unpack_codes(m.codes).reshape(-1, 16)
    sc = m.scales.reshape(-1)
    pairs = {(int(s), int(c)) for s, blk in zip(sc, elems) for c in blk}
    assert len(pairs) == 254 * 16


@pytest.mark.parametrize("d", [TINY, FLINT])
def test_dequant_is_exact_over_the_code_space(d):
    """flint_moe_debug_dequant (the decode kernels' own dequantisation) gives
    fp32(c) * G rounded once in FP32, bit for bit, for every pair."""
    dd = dict(d, num_experts=2, top_k=2) if d is FLINT else d
    cfg = cfg_of(dd)
    mats = code_space_layer(dd, 7)
    dl = device_layer(cfg, mats, 7, 0)
    for e in range(dd["num_experts"] + dd["n_shared"]):
        for mi in range(3):
            m = mats[e][mi]
            out = torch.empty(m.codes.shape[0], m.codes.shape[1] * 2, dtype=torch.float32, device=DEV)
            fb.flint_moe_debug_dequant(cfg, dl.packed, e, mi, out)
            ref = (m.c().astype(np.float32) * np.float32(m.G)).astype(np.float32)
            got = out.cpu().numpy()
            assert np.array_equal(got.view(np.uint32) & 0x7FFFFFFF, ref.view(np.uint32) & 0x7FFFFFFF), (e, mi)
            nz = ref != 0
            assert np.array_equal(np.signbit(got[nz]), np.signbit(ref[nz])), (e, mi)


def _gpu_run(cfg, dl, x, B, prefill=False, prenorm=False):
    out = torch.full_like(x, 0x7FC0)  # bf16 NaN pattern: every element must be written
    idx = torch.empty(B, cfg.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(B, cfg.top_k, dtype=torch.float32, device=DEV)
    if prefill:
        ws = layers.prefill_workspace(cfg, B, DEV)
        (fb.flint_moe_prefill_prenorm if prenorm else fb.flint_moe_prefill)(dl.handle, x, B, out, ws)
        fb.flint_moe_prefill_debug_routing(cfg, ws, B, idx, w)
    else:
        ws = layers.workspace(cfg, B, DEV)
        (fb.flint_moe_decode_prenorm if prenorm else fb.flint_moe_decode)(dl.handle, x, B, out, ws)
        fb.flint_moe_debug_routing(cfg, ws, B, idx, w)
    st, bits = fb.flint_moe_read_status(ws)
    assert st == fb.OK and bits == 0, (st, bits)
    return out, idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("B,prefill", [(1, False), (5, False), (12, False), (40, True)])
def test_layer_on_the_code_space(B, prefill):
    """The layer built from the code-space matrices (tiny shape): every token's
    routing and output, on the small-batch kernels (1 and 5 tokens: the
    work-item down kernel; 12: the staged down kernel) and the tensor-core path."""
    d = TINY
    cfg = cfg_of(d)
    mats = code_space_layer(d, 11)
    dl = device_layer(cfg, mats, 11, 0)
    x = layers.synth_x(B, cfg.hidden, 11, 0, DEV)
    out, idx, w = _gpu_run(cfg, dl, x, B, prefill)
    xo, router = oracle_inputs(d, 11, 0, B)
    ref, routing = moe.moe_layer(xo, router, lambda e: mats[e], oracle_config(d))
    excluded = check_routing(routing, idx, w)
    keep = [t for t in range(B) if t not in excluded]
    got = bits_to_f64(out)
    check_out(ref[keep], got[keep], f"code space {'prefill' if prefill else 'decode'} B={B}")
    assert np.abs(ref).max() > 1.0  # large weights really reached the output


# ---------------------------------------------------------------- wide-range activations

def wide_rows(H, seed):
    """bf16 bit patterns of 8 activation rows (see the module docstring):
    0 the seeded N(0, 1) row; 1 64 'anchor' elements N(0, 1), every other
    element N(0, 1) times 2^-(30..40); 2 the same with the anchors times 2^24;
    3 anchors times 2^50; 4 the row times 2^-100; 5 the row times 2^-118 (near
    bf16's smallest normal); 6 the row times 2^56; 7 anchors times 2^-60 with
    the other elements 2^-(30..40) below them (down to about 2^-100)."""
    rng = np.random.default_rng(seed)
    base = moe.bf16_bits_to_f64(synth.x_bf16(seed, 0, 8, H))
    rows = np.empty((8, H))
    for t in range(8):
        v = base[t].copy()
        anchors = np.zeros(H, bool)
        anchors[rng.choice(H, 64, replace=False)] = True
        small = np.exp2(-rng.integers(30, 41, H).astype(np.float64))
        aniso = np.where(anchors, v, v * small)
        rows[t] = {0: v, 1: aniso, 2: aniso * 2.0 ** 24, 3: aniso * 2.0 ** 50, 4: v * 2.0 ** -100,
                   5: v * 2.0 ** -118, 6: v * 2.0 ** 56, 7: aniso * 2.0 ** -60}[t]
    return moe.f64_to_bf16_bits(rows)


def run_wide(d, prefill):
    """Routing forced by a selection bias of +2 on k experts (every scale of
    row decides nothing then: a saturated sigmoid would tie many experts) and
    weights w = sigmoid (no renormalisation, so a zero score gives a zero
    weight rather than 0 / 0); the outputs of every token are compared."""
    cfg = cfg_of(d, renormalize=False)
    k, E = d["top_k"], d["num_experts"]
    bias = np.zeros(E, np.float32)
    chosen = np.arange(1, E, max(1, E // k))[:k]
    bias[chosen] = 2.0
    bias_t = torch.from_numpy(bias).to(DEV)
    seed = 31
    dl = layers.synth_layer(cfg, seed, 0, DEV, bias=bias_t)
    bits = wide_rows(d["hidden"], seed)
    B = bits.shape[0]
    x = torch.from_numpy(bits.view(np.int16)).to(DEV)
    out, idx, w = _gpu_run(cfg, dl, x, B, prefill)
    xo = moe.bf16_bits_to_f64(bits)
    _, router = oracle_inputs(d, seed, 0, 1)
    oc = oracle_config(d, renormalize=False)
    get = oracle_experts(d, seed, 0, prefetch=sorted(set(chosen.tolist()) | {E + s for s in range(d["n_shared"])}))
    ref, routing = moe.moe_layer(xo, router, get, oc, bias)
    assert all(set(routing.idx[t].tolist()) == set(chosen.tolist()) for t in range(B))
    excluded = check_routing(routing, idx, w)
    assert not excluded
    check_out(ref, bits_to_f64(out), f"wide range {'prefill' if prefill else 'decode'} H={d['hidden']}")
    return ref


@pytest.mark.parametrize("d,prefill", [(TINY, False), (FLINT, False), (TINY, True), (FLINT, True)])
def test_wide_range_activations(d, prefill):
    ref = run_wide(d, prefill)
    assert np.abs(ref[6]).max() > 2.0 ** 100 and np.abs(ref[0]).max() < 2.0 ** 10  # the range was reached


def test_wide_range_routing_without_bias():
    """The same rows routed by their own scores (no bias), on both paths:
    rows of moderate size are decided by the gap rule; rows of tiny size give
    every expert the score 1/2 exactly (ties), which the lower-index rule
    decides; rows of huge size saturate and are excluded."""
    d = TINY
    cfg = cfg_of(d)
    seed = 31
    dl = layers.synth_layer(cfg, seed, 0, DEV)
    bits = wide_rows(d["hidden"], seed)
    B = bits.shape[0]
    x = torch.from_numpy(bits.view(np.int16)).to(DEV)
    xo = moe.bf16_bits_to_f64(bits)
    _, router = oracle_inputs(d, seed, 0, 1)
    for prefill in (False, True):
        out, idx, w = _gpu_run(cfg, dl, x, B, prefill)
        routing = moe.route(xo, router, oracle_config(d))
        excluded = check_routing(routing, idx, w)
        assert 0 not in excluded and 1 not in excluded
        ties = [t for t in range(B) if np.all(routing.s[t] == np.float32(0.5))]
        assert {4, 5, 7} <= set(ties)
        for t in ties:  # every score exactly 1/2: the top-k are experts 0 .. k-1
            assert routing.idx[t].tolist() == list(range(d["top_k"]))
            assert idx[t].tolist() == list(range(d["top_k"])), (prefill, t, idx[t])
        get = oracle_experts(d, seed, 0)
        decided = [t for t in range(B) if t not in excluded or t in ties]
        ref, _ = moe.moe_layer(xo, router, get, oracle_config(d), None, decided)
        check_out(ref, bits_to_f64(out)[decided], f"wide range, own routing, {'prefill' if prefill else 'decode'}")


@pytest.mark.parametrize("prefill,B", [(False, 1), (False, 2), (False, 4), (True, 4)])
def test_prenorm_rows_near_the_ends_of_bf16(prefill, B):
    """Pre-norm block on residual rows near bf16's largest normal (the sum of
    squares of such a row overflows FP32: the RMSNorm must still normalise it)
    and near its smallest normal, with the rows' own routing checked against
    the oracle's and every output compared. 1 and 2 rows take the router's
    path in which several warps share a row's normalisation."""
    d = TINY
    seed = 37
    base = moe.bf16_bits_to_f64(synth.x_bf16(seed, 0, 4, d["hidden"]))
    scales = np.array([2.0 ** 124, 2.0 ** 100, 2.0 ** -120, 1.0])[:, None]
    bits = moe.f64_to_bf16_bits(base * scales)[:B]
    cfg = cfg_of(d)
    dl = layers.synth_layer(cfg, seed, 0, DEV, norm_eps=1e-6)
    x = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV)
    out, idx, w = _gpu_run(cfg, dl, x, B, prefill, prenorm=True)
    ro = moe.bf16_bits_to_f64(bits)
    assert np.abs(ro[0]).max() > 2.0 ** 125  # near bf16's largest normal
    _, router = oracle_inputs(d, seed, 0, 1)
    gamma = moe.bf16_bits_to_f64(synth.norm_bf16(seed, 0, d["hidden"]))
    ref, routing = moe.moe_block(ro, router, oracle_experts(d, seed, 0), oracle_config(d), gamma, 1e-6)
    excluded, _ = check_routing_prenorm(ro, gamma, 1e-6, router, oracle_config(d), None, idx, w)
    assert not ({0, 1, 3} & set(t for t in excluded))
    check_out(ref, bits_to_f64(out), f"prenorm near the ends of bf16, B={B}, {'prefill' if prefill else 'decode'}")
