"""The C-ABI library builds, loads and validates arguments on the host (no GPU)."""
import ctypes
import glob
import os
import re

import pytest

from w4a16_moe_decode_gb300 import binding as fb
from w4a16_moe_decode_gb300.build import INCLUDE, build

DECL = re.compile(r"^[A-Za-z_][\w\s\*]*?\b(flint_\w+)\s*\(", re.M)


@pytest.fixture(scope="module")
def lib():
    build()
    return fb.lib()


def _declared():
    names = set()
    for h in glob.glob(os.path.join(INCLUDE, "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"typedef struct.*?\}\s*\w+;", "", src, flags=re.S)
        names.update(DECL.findall(src))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert {"flint_moe_decode", "flint_moe_pack", "flint_synth_normal", "flint_gemv", "flint_gemv_pack"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), n


def test_no_oracle_in_product_path():
    root = os.path.dirname(INCLUDE)
    pkg = os.path.join(root, "w4a16_moe_decode_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*.*"), recursive=True):
        if path.endswith((".py", ".cu", ".cuh", ".h")):
            text = open(path).read()
            assert "import oracle" not in text and "from oracle" not in text, path


def test_binding_fails_loudly_without_the_library(monkeypatch):
    """No fallback: without the compiled library every call path stops with an
    error that says how to build it."""
    monkeypatch.setattr(fb, "LIB", os.path.join(os.path.dirname(fb.LIB), "missing", "libflint_moe.so"))
    monkeypatch.setattr(fb, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        fb.lib()


def flint_cfg(**kw):
    return fb.make_config(**kw)


def test_config_checks(lib):
    assert fb.flint_moe_check_config(flint_cfg()) == fb.OK
    assert fb.flint_moe_check_config(flint_cfg(hidden=256, num_experts=16, top_k=2, inter=64)) == fb.OK
    assert fb.flint_moe_check_config(flint_cfg(hidden=300)) == fb.EUNSUPPORTED
    assert fb.flint_moe_check_config(flint_cfg(hidden=2304)) == fb.EUNSUPPORTED
    assert fb.flint_moe_check_config(flint_cfg(inter=100)) == fb.EUNSUPPORTED
    assert fb.flint_moe_check_config(flint_cfg(top_k=0)) == fb.EUNSUPPORTED
    assert fb.flint_moe_check_config(flint_cfg(top_k=17)) == fb.EUNSUPPORTED
    assert fb.flint_moe_check_config(flint_cfg(num_experts=4, top_k=5)) == fb.EUNSUPPORTED
    assert fb.flint_moe_check_config(flint_cfg(num_experts=513)) == fb.EUNSUPPORTED
    assert fb.flint_moe_check_config(flint_cfg(n_shared=5)) == fb.EUNSUPPORTED
    assert fb.flint_moe_check_config(flint_cfg(weight_fmt=2)) == fb.EUNSUPPORTED


def test_packed_bytes_is_the_nvfp4_and_bf16_byte_count(lib):
    # NVFP4: per [rows, cols] matrix rows*cols/2 code bytes + rows*cols/16 scale
    # bytes; per expert 3 matrices; float32 tensor scales after the experts.
    c = flint_cfg()
    per_expert = 3 * (512 * 2048 // 2 + 512 * 2048 // 16)
    assert per_expert == 1769472
    n = fb.flint_moe_packed_bytes(c)
    assert n >= 257 * per_expert + 257 * 12 and n < 257 * per_expert + 257 * 16 + 256
    b = fb.flint_moe_packed_bytes(flint_cfg(weight_fmt=fb.BF16))
    assert b >= 257 * 3 * 512 * 2048 * 2
    assert fb.flint_moe_packed_bytes(flint_cfg(hidden=300)) == 0


def test_workspace_bytes(lib):
    c = flint_cfg()
    assert fb.flint_moe_workspace_bytes(c, 0) == 0
    assert fb.flint_moe_workspace_bytes(c, 33) == 0
    w1, w8, w32 = (fb.flint_moe_workspace_bytes(c, b) for b in (1, 8, 32))
    assert 0 < w1 < w8 < w32
    # the bf16 h rows dominate: every slot (the shared expert and up to B * k
    # distinct selected experts) owns one row per token
    assert w32 >= (1 + min(256, 32 * 6)) * 32 * 512 * 2
    assert w32 <= fb.lib().flint_moe_workspace_bytes(ctypes.byref(c), 32)  # same call through ctypes


def test_decode_rejects_bad_arguments_on_the_host(lib):
    c = flint_cfg()
    layer = fb.flint_moe_layer()
    layer.cfg = c
    layer.packed = 0x10000
    layer.router = 0x20000
    x, out, ws = 0x30000, 0x40000, 0x50000
    L = fb.lib()
    assert L.flint_moe_decode(ctypes.byref(layer), x, 0, out, ws, None) == fb.OK      # B = 0: nothing to do
    assert L.flint_moe_decode(ctypes.byref(layer), x, 33, out, ws, None) == fb.EINVAL
    assert L.flint_moe_decode(ctypes.byref(layer), x, -1, out, ws, None) == fb.EINVAL
    assert L.flint_moe_decode(ctypes.byref(layer), None, 1, out, ws, None) == fb.EINVAL
    assert L.flint_moe_decode(ctypes.byref(layer), x + 2, 1, out, ws, None) == fb.EALIGN
    assert L.flint_moe_decode(ctypes.byref(layer), x, 1, out + 8, ws, None) == fb.EALIGN
    assert L.flint_moe_decode(None, x, 1, out, ws, None) == fb.EINVAL
    layer.cfg.hidden = 300
    assert L.flint_moe_decode(ctypes.byref(layer), x, 1, out, ws, None) == fb.EUNSUPPORTED


def test_rcp_check_rejects_ranges_outside_its_domain(lib):
    n = ctypes.c_uint64(7)
    L = fb.lib()
    assert L.flint_moe_debug_rcp_check(0x3F7FFFFF, 0x3F800010, ctypes.byref(n), None) == fb.EINVAL  # below 1.0
    assert L.flint_moe_debug_rcp_check(0x3F800000, ((127 + 125) << 23) + 1, ctypes.byref(n), None) == fb.EINVAL
    assert L.flint_moe_debug_rcp_check(0x3F800010, 0x3F800000, ctypes.byref(n), None) == fb.EINVAL
    assert L.flint_moe_debug_rcp_check(0x3F800000, 0x3F800010, None, None) == fb.EINVAL


def test_prenorm_needs_a_norm_weight(lib):
    c = flint_cfg()
    L = fb.lib()
    layer = fb.flint_moe_layer()
    assert L.flint_moe_layer_init(ctypes.byref(c), 0x10000, 0x20000, None, ctypes.byref(layer)) == fb.OK
    assert layer.norm_weight is None
    assert L.flint_moe_decode_prenorm(ctypes.byref(layer), 0x30000, 1, 0x30000, 0x50000, None) == fb.EINVAL
    assert L.flint_moe_layer_set_norm(ctypes.byref(layer), 0x60008, ctypes.c_float(1e-6)) == fb.EALIGN
    assert L.flint_moe_layer_set_norm(ctypes.byref(layer), 0x60000, ctypes.c_float(float("nan"))) == fb.EINVAL
    assert L.flint_moe_layer_set_norm(ctypes.byref(layer), 0x60000, ctypes.c_float(-1.0)) == fb.EINVAL
    assert L.flint_moe_layer_set_norm(ctypes.byref(layer), 0x60000, ctypes.c_float(1e-6)) == fb.OK
    assert layer.norm_weight == 0x60000 and abs(layer.norm_eps - 1e-6) < 1e-12
    assert L.flint_moe_decode_prenorm(ctypes.byref(layer), 0x30000, 0, 0x30000, 0x50000, None) == fb.OK  # B = 0


def test_gemv_host_validation(lib):
    L = fb.lib()
    assert fb.flint_gemv_packed_bytes(2048, 2048, fb.NVFP4) == 128 * 32 * 576 + 256
    assert fb.flint_gemv_packed_bytes(2048, 2048, fb.BF16) == 128 * 32 * 2048 + 256
    for N, K in ((2040, 2048), (2048, 200), (2048, 3072), (2048, 16384), (0, 256)):
        assert fb.flint_gemv_packed_bytes(N, K, fb.NVFP4) == 0
    args = lambda N, K, B, x=0x30000, y=0x40000, w=None, eps=0.0: (0x10000, N, K, fb.NVFP4, x, B, y, w,  # noqa: E731
                                                                  ctypes.c_float(eps), None, None)
    assert L.flint_gemv(*args(2048, 2048, 0)) == fb.OK                    # B = 0: nothing to do
    assert L.flint_gemv(*args(2040, 2048, 1)) == fb.EUNSUPPORTED
    assert L.flint_gemv(*args(2048, 2048, 33)) == fb.EINVAL
    assert L.flint_gemv(*args(2048, 2048, 1, x=0x30008)) == fb.EALIGN
    assert L.flint_gemv(*args(2048, 2048, 1, w=0x50004)) == fb.EALIGN
    assert L.flint_gemv(*args(2048, 2048, 1, eps=float("nan"))) == fb.EINVAL


def test_layer_init_and_pack_validate(lib):
    c = flint_cfg()
    layer = fb.flint_moe_layer()
    L = fb.lib()
    assert L.flint_moe_layer_init(ctypes.byref(c), 0x10000, 0x20000, None, ctypes.byref(layer)) == fb.OK
    assert layer.cfg.hidden == 2048 and layer.packed == 0x10000
    assert L.flint_moe_layer_init(ctypes.byref(c), 0x10004, 0x20000, None, ctypes.byref(layer)) == fb.EALIGN
    assert L.flint_moe_layer_init(ctypes.byref(c), None, 0x20000, None, ctypes.byref(layer)) == fb.EINVAL
    src = fb.flint_moe_src()
    assert L.flint_moe_pack(ctypes.byref(c), ctypes.byref(src), 0x10000, 10, None, None) == fb.EINVAL
    assert L.flint_moe_quantize_nvfp4(0x1000, 1, 4, 24, 0x2000, 0x3000, 0x4000, None) == fb.EINVAL


def test_synth_stream_key_matches_cpu_generator(lib):
    import synth
    for args in [(0, 0, 1, 0), (12345, 3, 4, 200), (2**63 + 5, 46, 2, 256)]:
        assert fb.flint_synth_stream_key(*args) == synth.stream_key(*args)


def test_prefill_workspace_bytes(lib):
    c = flint_cfg()
    assert fb.flint_moe_prefill_workspace_bytes(c, 0) == 0
    assert fb.flint_moe_prefill_workspace_bytes(c, 65537) == 0
    assert fb.flint_moe_prefill_workspace_bytes(flint_cfg(weight_fmt=fb.BF16), 64) == 0  # NVFP4 only
    w16, w512, w4096 = (fb.flint_moe_prefill_workspace_bytes(c, t) for t in (16, 512, 4096))
    assert 0 < w16 < w512 < w4096
    # the FP32 expert outputs y [T][S + k][H], h [T (S + k)][I] bf16, the
    # routed pairs' grouped activation rows [T k][H] f16 and the normalised and
    # f16 token rows [T][H] (two of them) dominate
    big = 4096 * (7 * (2048 * 4 + 512 * 2) + 6 * 2048 * 2 + 2 * 2048 * 2)
    assert big <= w4096 < big * 1.05


def test_prefill_rejects_bad_arguments_on_the_host(lib):
    c = flint_cfg()
    layer = fb.flint_moe_layer()
    layer.cfg = c
    layer.packed = 0x10000
    layer.router = 0x20000
    x, out, ws = 0x100000, 0x200000, 0x300000
    need = fb.flint_moe_prefill_workspace_bytes(c, 64)
    L = fb.lib()
    P = L.flint_moe_prefill
    assert P(ctypes.byref(layer), x, 0, out, ws, need, None) == fb.OK  # B = 0: nothing to do
    assert P(ctypes.byref(layer), x, -1, out, ws, need, None) == fb.EINVAL
    assert P(ctypes.byref(layer), x, 65537, out, ws, need, None) == fb.EINVAL
    assert P(ctypes.byref(layer), None, 64, out, ws, need, None) == fb.EINVAL
    assert P(ctypes.byref(layer), x, 64, out, None, need, None) == fb.EINVAL
    assert P(ctypes.byref(layer), x + 2, 64, out, ws, need, None) == fb.EALIGN
    assert P(ctypes.byref(layer), x, 64, out, ws + 16, need, None) == fb.EALIGN
    assert P(ctypes.byref(layer), x, 64, out, ws, need - 1, None) == fb.EINVAL   # workspace too small
    assert P(ctypes.byref(layer), x, 64, x + 4096, ws, need, None) == fb.EINVAL  # out overlaps x
    assert P(None, x, 64, out, ws, need, None) == fb.EINVAL
    PN = L.flint_moe_prefill_prenorm
    assert PN(ctypes.byref(layer), x, 64, out, ws, need, None) == fb.EINVAL  # no norm weight set
    layer.norm_weight = 0x400000
    layer.norm_eps = 1e-6
    assert PN(ctypes.byref(layer), x, 64, x + 4096, ws, need, None) == fb.EINVAL  # partial overlap
    layer.norm_weight = 0x400008
    assert PN(ctypes.byref(layer), x, 64, out, ws, need, None) == fb.EINVAL  # misaligned norm weight
    layer.cfg.weight_fmt = fb.BF16
    assert P(ctypes.byref(layer), x, 64, out, ws, need, None) == fb.EUNSUPPORTED


def test_wait_timeout_check_validates_on_the_host(lib):
    assert fb.lib().flint_moe_debug_wait_timeout(None, None) == fb.EINVAL


def test_noalloc_rejects_a_workspace_beyond_its_scratch(lib):
    """flint_moe_decode_noalloc checks the workspace a shape needs against its
    8 MiB scratch array before anything touches the device, so this runs
    without a GPU (and null tensor pointers are never used)."""
    big = fb.make_config(hidden=8192, num_experts=512, top_k=16, inter=4096)
    assert fb.flint_moe_workspace_bytes(big, 32) > (8 << 20)
    layer = fb.flint_moe_layer()
    layer.cfg = big
    st = lib.flint_moe_decode_noalloc(ctypes.byref(layer), None, 32, None, None, None)
    assert st == fb.EUNSUPPORTED
    # the Flint shape fits at every batch up to 32, so only null pointers stop it
    flint = fb.make_config()
    assert fb.flint_moe_workspace_bytes(flint, 32) <= (8 << 20)
    layer.cfg = flint
    assert lib.flint_moe_decode_noalloc(ctypes.byref(layer), None, 32, None, None, None) == fb.EINVAL
