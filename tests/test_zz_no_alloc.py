"""flint_moe_decode_noalloc: the decode for callers that cannot allocate device
memory (for example a plugin whose host application owns every device
allocation, or a latency-critical loop where cudaMalloc could synchronise the
device). It uses the library's own static scratch array instead of a caller
workspace; its results must match flint_moe_decode's, call after call.
"""
import ctypes

import numpy as np
import pytest
import torch

from w4a16_moe_decode_gb300 import binding as fb
from w4a16_moe_decode_gb300 import layers
from w4a16_moe_decode_gb300.build import build

from _common import FLINT, TINY, bits_to_f64, check_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    fb.lib()


@pytest.mark.parametrize("d,B", [(FLINT, 1), (FLINT, 8), (TINY, 5)])
def test_noalloc_matches_workspace_decode_on_consecutive_calls(d, B):
    cfg = fb.make_config(**d)
    dl = layers.synth_layer(cfg, 21, 0, "cuda")
    ws = layers.workspace(cfg, B, "cuda")
    for call, seed in enumerate((31, 32)):  # two calls in a row, different tokens each time
        x = layers.synth_x(B, cfg.hidden, seed, 0, "cuda")
        ref = torch.empty_like(x)
        fb.flint_moe_decode(dl.handle, x, B, ref, ws)
        out = torch.full_like(x, 0x7FC0)  # bf16 NaN pattern: every element must be overwritten
        fb.flint_moe_decode_noalloc(dl.handle, x, B, out)
        torch.cuda.synchronize()
        check_out(bits_to_f64(ref), bits_to_f64(out), f"call {call}")
    st, bits = fb.flint_moe_read_status(ws)
    assert st == fb.OK and bits == 0


def test_noalloc_rejects_a_workspace_beyond_its_scratch():
    cfg = fb.make_config(hidden=8192, num_experts=512, top_k=16, inter=4096)
    assert fb.flint_moe_workspace_bytes(cfg, 32) > (1 << 20)
    layer = fb.flint_moe_layer()
    layer.cfg = cfg
    layer.packed = 0x10000
    layer.router = 0x20000
    st = fb.lib().flint_moe_decode_noalloc(ctypes.byref(layer), 0x30000, 32, 0x40000, None)
    assert st == fb.EUNSUPPORTED
