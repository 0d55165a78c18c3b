"""flint_moe_decode_noalloc: the decode for callers that cannot allocate device
memory (for example a plugin whose host application owns every device
allocation, or a latency-critical loop where cudaMalloc could synchronise the
device). It uses the library's own static scratch array instead of a caller
workspace; it runs the same kernels on the same inputs, and the combine is
added in a fixed order, so its outputs must equal flint_moe_decode's bit for
bit, call after call. (The shape check that rejects workspaces beyond the
scratch array is a CPU test in test_library_cpu.py.)
"""
import ctypes

import pytest
import torch

from w4a16_moe_decode_gb300 import binding as fb
from w4a16_moe_decode_gb300 import layers
from w4a16_moe_decode_gb300.build import build

from _common import FLINT, TINY

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    fb.lib()


def test_noalloc_first_call_inside_a_stream_capture_is_refused():
    """The first call on a device looks up the scratch array's address, which
    is not a stream operation: inside a capture it is refused with EINVAL (and
    nothing is captured). Every other test of this process runs after this one
    and makes the first real call outside any capture."""
    cfg = fb.make_config(**TINY)
    dl = layers.synth_layer(cfg, 21, 0, "cuda")
    x = layers.synth_x(2, cfg.hidden, 31, 0, "cuda")
    out = torch.empty_like(x)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            st = fb.lib().flint_moe_decode_noalloc(ctypes.byref(dl.handle), x.data_ptr(), 2, out.data_ptr(), None,
                                                   s.cuda_stream)
    assert st == fb.EINVAL
    del g


@pytest.mark.parametrize("d,B", [(FLINT, 1), (FLINT, 8), (TINY, 5)])
def test_noalloc_matches_workspace_decode_on_consecutive_calls(d, B):
    cfg = fb.make_config(**d)
    dl = layers.synth_layer(cfg, 21, 0, "cuda")
    ws = layers.workspace(cfg, B, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for seed in (31, 32):  # two calls in a row, different tokens each time
        x = layers.synth_x(B, cfg.hidden, seed, 0, "cuda")
        ref = torch.empty_like(x)
        fb.flint_moe_decode(dl.handle, x, B, ref, ws)
        out = torch.full_like(x, 0x7FC0)  # bf16 NaN pattern: every element must be overwritten
        fb.flint_moe_decode_noalloc(dl.handle, x, B, out, status)
        torch.cuda.synchronize()
        assert torch.equal(ref, out), seed
    assert int(status.item()) == 0  # no device-side error in either call
    st, bits = fb.flint_moe_read_status(ws)
    assert st == fb.OK and bits == 0
