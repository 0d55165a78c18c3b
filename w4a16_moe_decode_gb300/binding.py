"""ctypes binding of libflint_moe.so: the C entry points under the same names.

Argument marshalling only: tensors become device pointers, streams become
cudaStream_t handles, and a non-OK status becomes a FlintMoeError. Every step
of the computation runs in the library's CUDA kernels. If the library has not
been built the first call raises; nothing falls back to another
implementation.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB

c_int32 = ctypes.c_int32
c_void_p = ctypes.c_void_p
c_size_t = ctypes.c_size_t

STATUS_NAMES = {0: "FLINT_MOE_OK", 1: "FLINT_MOE_EINVAL", 2: "FLINT_MOE_EALIGN", 3: "FLINT_MOE_ECUDA",
                4: "FLINT_MOE_ETIMEOUT", 5: "FLINT_MOE_EUNSUPPORTED"}
OK, EINVAL, EALIGN, ECUDA, ETIMEOUT, EUNSUPPORTED = range(6)
NVFP4, BF16 = 0, 1
DEV_ERR_TIMEOUT, DEV_ERR_NAN_SCALE, DEV_ERR_SLOTS = 1, 2, 4

# synth tensor tags (same numbering as the CPU generator)
ROUTER, GATE, UP, DOWN, X, BIAS, NORM = 1, 2, 3, 4, 5, 6, 7


class FlintMoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}")
        self.status = status


class flint_moe_config(ctypes.Structure):
    _fields_ = [("hidden", c_int32), ("num_experts", c_int32), ("top_k", c_int32), ("inter", c_int32),
                ("n_shared", c_int32), ("weight_fmt", c_int32), ("renormalize", c_int32),
                ("routed_scale", ctypes.c_float)]


class flint_moe_nvfp4_src(ctypes.Structure):
    _fields_ = [("codes", c_void_p), ("scales", c_void_p), ("global_", c_void_p)]


class flint_moe_src(ctypes.Structure):
    _fields_ = [("gate", flint_moe_nvfp4_src), ("up", flint_moe_nvfp4_src), ("down", flint_moe_nvfp4_src),
                ("gate_bf16", c_void_p), ("up_bf16", c_void_p), ("down_bf16", c_void_p)]


class flint_gemv_src(ctypes.Structure):
    _fields_ = [("codes", c_void_p), ("scales", c_void_p), ("global_", c_void_p), ("bf16", c_void_p)]


class flint_moe_layer(ctypes.Structure):
    _fields_ = [("cfg", flint_moe_config), ("packed", c_void_p), ("router", c_void_p), ("sel_bias", c_void_p),
                ("norm_weight", c_void_p), ("norm_eps", ctypes.c_float)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it was never built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB)
        P = ctypes.POINTER
        sig = {
            "flint_moe_check_config": (c_int32, [P(flint_moe_config)]),
            "flint_moe_packed_bytes": (c_size_t, [P(flint_moe_config)]),
            "flint_moe_workspace_bytes": (c_size_t, [P(flint_moe_config), c_int32]),
            "flint_moe_workspace_init": (c_int32, [P(flint_moe_config), c_int32, c_void_p, c_void_p]),
            "flint_moe_pack": (c_int32, [P(flint_moe_config), P(flint_moe_src), c_void_p, c_size_t, c_void_p, c_void_p]),
            "flint_moe_unpack_debug": (c_int32, [P(flint_moe_config), c_void_p, P(flint_moe_src), c_void_p]),
            "flint_moe_layer_init": (c_int32, [P(flint_moe_config), c_void_p, c_void_p, c_void_p, P(flint_moe_layer)]),
            "flint_moe_decode": (c_int32, [P(flint_moe_layer), c_void_p, c_int32, c_void_p, c_void_p, c_void_p]),
            "flint_moe_layer_set_norm": (c_int32, [P(flint_moe_layer), c_void_p, ctypes.c_float]),
            "flint_moe_decode_prenorm": (c_int32, [P(flint_moe_layer), c_void_p, c_int32, c_void_p, c_void_p,
                                                   c_void_p]),
            "flint_moe_decode_noalloc": (c_int32, [P(flint_moe_layer), c_void_p, c_int32, c_void_p, c_void_p,
                                                   c_void_p]),
            "flint_moe_debug_routing": (c_int32, [P(flint_moe_config), c_void_p, c_int32, c_void_p, c_void_p, c_void_p]),
            "flint_moe_debug_dequant": (c_int32, [P(flint_moe_config), c_void_p, c_int32, c_int32, c_void_p, c_void_p]),
            "flint_moe_read_status": (c_int32, [c_void_p, P(c_int32), c_void_p]),
            "flint_moe_trace": (c_int32, [c_int32, c_void_p, c_void_p]),
            "flint_moe_debug_rcp_check": (c_int32, [ctypes.c_uint32, ctypes.c_uint32, P(ctypes.c_uint64), c_void_p]),
            "flint_moe_debug_wait_timeout": (c_int32, [c_void_p, c_void_p]),
            "flint_moe_quantize_nvfp4": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                                   c_void_p]),
            "flint_gemv_packed_bytes": (c_size_t, [c_int32, c_int32, c_int32]),
            "flint_gemv_pack": (c_int32, [P(flint_gemv_src), c_int32, c_int32, c_int32, c_void_p, c_size_t, c_void_p,
                                          c_void_p]),
            "flint_gemv_unpack_debug": (c_int32, [c_void_p, c_int32, c_int32, c_int32, P(flint_gemv_src), c_void_p]),
            "flint_gemv": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_int32, c_void_p, c_void_p,
                                     ctypes.c_float, c_void_p, c_void_p]),
            "flint_moe_prefill_workspace_bytes": (c_size_t, [P(flint_moe_config), c_int32]),
            "flint_moe_prefill_workspace_init": (c_int32, [P(flint_moe_config), c_int32, c_void_p, c_void_p]),
            "flint_moe_prefill": (c_int32, [P(flint_moe_layer), c_void_p, c_int32, c_void_p, c_void_p, c_size_t,
                                            c_void_p]),
            "flint_moe_prefill_prenorm": (c_int32, [P(flint_moe_layer), c_void_p, c_int32, c_void_p, c_void_p,
                                                    c_size_t, c_void_p]),
            "flint_moe_prefill_debug_routing": (c_int32, [P(flint_moe_config), c_void_p, c_int32, c_void_p, c_void_p,
                                                          c_void_p, c_void_p]),
            "flint_synth_stream_key": (ctypes.c_uint64, [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                                                         ctypes.c_uint32]),
            "flint_synth_normal": (ctypes.c_int, [ctypes.c_uint64, ctypes.c_uint64, c_size_t, ctypes.c_float, c_int32,
                                                  c_void_p, c_void_p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, st: int) -> None:
    if st != OK:
        raise FlintMoeError(fn, st)


def make_config(hidden=2048, num_experts=256, top_k=6, inter=512, n_shared=1, weight_fmt=NVFP4, renormalize=True,
                routed_scale=1.0) -> flint_moe_config:
    return flint_moe_config(hidden, num_experts, top_k, inter, n_shared, weight_fmt, int(bool(renormalize)),
                            float(routed_scale))


def flint_moe_check_config(cfg: flint_moe_config) -> int:
    return lib().flint_moe_check_config(ctypes.byref(cfg))


def flint_moe_packed_bytes(cfg: flint_moe_config) -> int:
    return lib().flint_moe_packed_bytes(ctypes.byref(cfg))


def flint_moe_workspace_bytes(cfg: flint_moe_config, max_batch: int) -> int:
    return lib().flint_moe_workspace_bytes(ctypes.byref(cfg), max_batch)


def flint_moe_workspace_init(cfg, max_batch, workspace, stream=None) -> None:
    _check("flint_moe_workspace_init",
           lib().flint_moe_workspace_init(ctypes.byref(cfg), max_batch, _ptr(workspace), _stream(stream)))


def _src_struct(src: dict) -> flint_moe_src:
    s = flint_moe_src()
    for m in ("gate", "up", "down"):
        part = getattr(s, m)
        part.codes = _ptr(src.get(m + "_codes"))
        part.scales = _ptr(src.get(m + "_scales"))
        part.global_ = _ptr(src.get(m + "_global"))
        setattr(s, m, part)
        setattr(s, m + "_bf16", _ptr(src.get(m + "_bf16")))
    return s


def flint_moe_pack(cfg, src: dict, dst, dev_status=None, stream=None, dst_bytes=None) -> None:
    """src: dict with keys {gate,up,down}_{codes,scales,global} or {gate,up,down}_bf16 (tensors)."""
    s = _src_struct(src)
    nbytes = dst.numel() * dst.element_size() if dst_bytes is None else dst_bytes
    _check("flint_moe_pack", lib().flint_moe_pack(ctypes.byref(cfg), ctypes.byref(s), _ptr(dst), nbytes,
                                                  _ptr(dev_status), _stream(stream)))


def flint_moe_unpack_debug(cfg, packed, dst: dict, stream=None) -> None:
    s = _src_struct(dst)
    _check("flint_moe_unpack_debug", lib().flint_moe_unpack_debug(ctypes.byref(cfg), _ptr(packed), ctypes.byref(s),
                                                                  _stream(stream)))


def flint_moe_layer_init(cfg, packed, router, sel_bias=None) -> flint_moe_layer:
    layer = flint_moe_layer()
    _check("flint_moe_layer_init", lib().flint_moe_layer_init(ctypes.byref(cfg), _ptr(packed), _ptr(router),
                                                              _ptr(sel_bias), ctypes.byref(layer)))
    return layer


def flint_moe_decode(layer: flint_moe_layer, x, B: int, out, workspace, stream=None) -> None:
    _check("flint_moe_decode", lib().flint_moe_decode(ctypes.byref(layer), _ptr(x), B, _ptr(out), _ptr(workspace),
                                                      _stream(stream)))


def flint_moe_layer_set_norm(layer: flint_moe_layer, norm_weight, eps: float) -> None:
    _check("flint_moe_layer_set_norm", lib().flint_moe_layer_set_norm(ctypes.byref(layer), _ptr(norm_weight),
                                                                      float(eps)))


def flint_moe_decode_prenorm(layer: flint_moe_layer, residual_in, B: int, residual_out, workspace,
                             stream=None) -> None:
    _check("flint_moe_decode_prenorm", lib().flint_moe_decode_prenorm(ctypes.byref(layer), _ptr(residual_in), B,
                                                                      _ptr(residual_out), _ptr(workspace),
                                                                      _stream(stream)))


def flint_moe_decode_noalloc(layer: flint_moe_layer, x, B: int, out, dev_status=None, stream=None) -> None:
    """flint_moe_decode with the library's own 8 MiB device scratch array in
    place of a workspace, for callers that cannot allocate device memory.
    dev_status (int32 device tensor, optional) receives the device status bits."""
    _check("flint_moe_decode_noalloc", lib().flint_moe_decode_noalloc(ctypes.byref(layer), _ptr(x), B, _ptr(out),
                                                                      _ptr(dev_status), _stream(stream)))


def flint_moe_prefill_workspace_bytes(cfg: flint_moe_config, max_tokens: int) -> int:
    return lib().flint_moe_prefill_workspace_bytes(ctypes.byref(cfg), max_tokens)


def flint_moe_prefill_workspace_init(cfg, max_tokens, workspace, stream=None) -> None:
    _check("flint_moe_prefill_workspace_init",
           lib().flint_moe_prefill_workspace_init(ctypes.byref(cfg), max_tokens, _ptr(workspace), _stream(stream)))


def flint_moe_prefill(layer: flint_moe_layer, x, B: int, out, workspace, workspace_bytes=None, stream=None) -> None:
    """The expert-grouped tensor-core path for B tokens (include/flint_moe_prefill.h)."""
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    _check("flint_moe_prefill", lib().flint_moe_prefill(ctypes.byref(layer), _ptr(x), B, _ptr(out), _ptr(workspace),
                                                        nbytes, _stream(stream)))


def flint_moe_prefill_prenorm(layer: flint_moe_layer, residual_in, B: int, residual_out, workspace,
                              workspace_bytes=None, stream=None) -> None:
    nbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    _check("flint_moe_prefill_prenorm",
           lib().flint_moe_prefill_prenorm(ctypes.byref(layer), _ptr(residual_in), B, _ptr(residual_out),
                                           _ptr(workspace), nbytes, _stream(stream)))


def flint_moe_prefill_debug_routing(cfg, workspace, B, idx, w, logits=None, stream=None) -> None:
    _check("flint_moe_prefill_debug_routing",
           lib().flint_moe_prefill_debug_routing(ctypes.byref(cfg), _ptr(workspace), B, _ptr(idx), _ptr(w),
                                                 _ptr(logits), _stream(stream)))


def flint_moe_debug_routing(cfg, workspace, B, idx, w, stream=None) -> None:
    _check("flint_moe_debug_routing", lib().flint_moe_debug_routing(ctypes.byref(cfg), _ptr(workspace), B, _ptr(idx),
                                                                    _ptr(w), _stream(stream)))


def flint_moe_debug_dequant(cfg, packed, expert, mat, out, stream=None) -> None:
    _check("flint_moe_debug_dequant", lib().flint_moe_debug_dequant(ctypes.byref(cfg), _ptr(packed), expert, mat,
                                                                    _ptr(out), _stream(stream)))


def flint_moe_read_status(workspace, stream=None) -> tuple[int, int]:
    """(status code, device status bits); synchronises the stream."""
    v = c_int32(0)
    st = lib().flint_moe_read_status(_ptr(workspace), ctypes.byref(v), _stream(stream))
    if st not in (OK, ETIMEOUT):
        raise FlintMoeError("flint_moe_read_status", st)
    return st, v.value


def flint_moe_trace(op: int, stream=None):
    """op 0 clears the phase trace; op 1 returns it as a numpy uint64 array
    [64 calls][24 events][2] (earliest, latest ns over blocks). Needs the trace
    build of the library (FLINT_MOE_LIB pointing at it)."""
    import numpy as np
    buf = np.zeros((64, 24, 2), dtype=np.uint64) if op == 1 else None
    st = lib().flint_moe_trace(op, None if buf is None else buf.ctypes.data, _stream(stream))
    _check("flint_moe_trace", st)
    return buf


def flint_moe_debug_rcp_check(lo_bits: int, hi_bits: int, stream=None) -> int:
    """Mismatches between the routing reciprocal and IEEE 1.0f / y over the FP32
    bit patterns [lo_bits, hi_bits) (within [1, 2^125)); synchronises."""
    n = ctypes.c_uint64(0)
    _check("flint_moe_debug_rcp_check", lib().flint_moe_debug_rcp_check(lo_bits, hi_bits, ctypes.byref(n),
                                                                        _stream(stream)))
    return n.value


def flint_moe_debug_wait_timeout(dev_status, stream=None) -> None:
    _check("flint_moe_debug_wait_timeout", lib().flint_moe_debug_wait_timeout(_ptr(dev_status), _stream(stream)))


def flint_moe_quantize_nvfp4(w, n_mat, rows, cols, codes, scales, global_, stream=None) -> None:
    _check("flint_moe_quantize_nvfp4", lib().flint_moe_quantize_nvfp4(_ptr(w), n_mat, rows, cols, _ptr(codes),
                                                                      _ptr(scales), _ptr(global_), _stream(stream)))


def _gemv_src(d: dict) -> flint_gemv_src:
    return flint_gemv_src(_ptr(d.get("codes")), _ptr(d.get("scales")), _ptr(d.get("global")), _ptr(d.get("bf16")))


def flint_gemv_packed_bytes(N: int, K: int, fmt: int = NVFP4) -> int:
    return lib().flint_gemv_packed_bytes(N, K, fmt)


def flint_gemv_pack(src: dict, N: int, K: int, fmt, dst, dev_status=None, stream=None) -> None:
    """src: {codes, scales, global} (NVFP4) or {bf16} tensors of W [N][K]."""
    s = _gemv_src(src)
    _check("flint_gemv_pack", lib().flint_gemv_pack(ctypes.byref(s), N, K, fmt, _ptr(dst),
                                                    dst.numel() * dst.element_size(), _ptr(dev_status),
                                                    _stream(stream)))


def flint_gemv_unpack_debug(packed, N: int, K: int, fmt, dst: dict, stream=None) -> None:
    s = _gemv_src(dst)
    _check("flint_gemv_unpack_debug", lib().flint_gemv_unpack_debug(_ptr(packed), N, K, fmt, ctypes.byref(s),
                                                                    _stream(stream)))


def flint_gemv(packed, N: int, K: int, fmt, x, B: int, y, norm_weight=None, eps: float = 0.0, dev_status=None,
               stream=None) -> None:
    _check("flint_gemv", lib().flint_gemv(_ptr(packed), N, K, fmt, _ptr(x), B, _ptr(y), _ptr(norm_weight),
                                          float(eps), _ptr(dev_status), _stream(stream)))


def flint_synth_stream_key(seed, layer, tensor, expert) -> int:
    return lib().flint_synth_stream_key(seed, layer, tensor, expert)


def flint_synth_normal(key, start, n, sigma, out_bf16, out, stream=None) -> None:
    st = lib().flint_synth_normal(key, start, n, sigma, int(bool(out_bf16)), _ptr(out), _stream(stream))
    if st != 0:
        raise FlintMoeError("flint_synth_normal", st)
