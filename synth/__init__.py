"""Seeded synthetic inputs for the Flint-style MoE decode layer (CPU side).

This module only draws random numbers. It holds none of the layer's arithmetic:
no NVFP4 encoding or decoding, no routing, no GEMV. Both the CPU oracle's tests
and the GPU path's tests take their inputs from here; the GPU library carries its
own implementation of the same generator (``flint_synth_normal``), written from
the same published definitions, so that full-size weights can be drawn on the
device and still be reproduced here expert by expert.

Generator definition (the GPU side implements exactly this):

* ``mix(z)`` is the SplitMix64 output function (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014, as used by
  Vigna's ``splitmix64.c``)::

      z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
      z = (z ^ (z >> 27)) * 0x94D049BB133111EB
      z =  z ^ (z >> 31)                         (all mod 2**64)

* ``u(key, i) = mix(key + (i + 1) * 0x9E3779B97F4A7C15)`` is output ``i`` of
  SplitMix64 started at state ``key``; a counter-based stream, so any element
  can be regenerated on its own.
* ``stream_key(seed, layer, tensor, expert) =
  mix(seed ^ mix((layer << 48) | (tensor << 32) | expert))``.
* Normal number ``n`` of a stream takes ``u(key, 3n) .. u(key, 3n + 2)``, splits
  them into twelve 16-bit fields ``f_j`` (least significant first) and forms
  the Irwin-Hall sum of twelve uniforms ``(f_j + 1/2) / 65536`` minus 6:
  ``z = (sum_j (2 f_j + 1) - 12 * 65536) * 2**-17``. ``z`` is exact in float32.
* A scaled draw is ``float32(z) * float32(sigma)``, one float32 multiply
  rounded to nearest even; a bf16 draw rounds that float32 to bf16, nearest even.

Workload recipe of the decode layer (sizes are the caller's): router weights
bf16 N(0, 0.02); expert weights float32 N(0, 0.02), quantised to NVFP4 by the
caller; activations x bf16 N(0, 1). Element ``(r, c)`` of a ``[rows, cols]``
tensor is normal number ``r * cols + c`` of its stream.
"""
from __future__ import annotations

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK64 = (1 << 64) - 1

# tensor tags of the stream key
ROUTER = 1
GATE = 2
UP = 3
DOWN = 4
X = 5
BIAS = 6
NORM = 7


def _mix_scalar(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def _mix(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * _M1
    z = z ^ (z >> np.uint64(27))
    z = z * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, layer: int, tensor: int, expert: int) -> int:
    """64-bit key of one tensor's stream (see module docstring)."""
    packed = ((layer & 0xFFFF) << 48) | ((tensor & 0xFFFF) << 32) | (expert & 0xFFFFFFFF)
    return _mix_scalar((seed & _MASK64) ^ _mix_scalar(packed))


def uniform_u64(key: int, start: int, n: int) -> np.ndarray:
    """Outputs ``start .. start + n - 1`` of the SplitMix64 stream at ``key``."""
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key & _MASK64) + i * np.uint64(GOLDEN)
        return _mix(z)


def normal_f32(key: int, start: int, n: int) -> np.ndarray:
    """Normals ``start .. start + n - 1`` of the stream, float32, exact."""
    u = uniform_u64(key, 3 * start, 3 * n).reshape(n, 3)
    acc = np.zeros(n, dtype=np.int64)
    for w in range(3):
        col = u[:, w]
        for f in range(4):
            acc += 2 * ((col >> np.uint64(16 * f)) & np.uint64(0xFFFF)).astype(np.int64) + 1
    acc -= 12 * 65536
    return (acc.astype(np.float32) * np.float32(2.0 ** -17)).astype(np.float32)


def normal_scaled_f32(key: int, start: int, n: int, sigma: float) -> np.ndarray:
    """``float32(z) * float32(sigma)``, rounded once to float32."""
    return (normal_f32(key, start, n) * np.float32(sigma)).astype(np.float32)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest even); returns the uint16 patterns."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def matrix_f32(seed: int, layer: int, tensor: int, expert: int, rows: int, cols: int,
               sigma: float) -> np.ndarray:
    """A [rows, cols] float32 tensor of N(0, sigma) draws."""
    key = stream_key(seed, layer, tensor, expert)
    return normal_scaled_f32(key, 0, rows * cols, sigma).reshape(rows, cols)


def router_bf16(seed: int, layer: int, num_experts: int, hidden: int, sigma: float = 0.02) -> np.ndarray:
    """Router weights [E, H] as bf16 bit patterns; row e is the stream (ROUTER, e)."""
    out = np.empty((num_experts, hidden), dtype=np.uint16)
    for e in range(num_experts):
        key = stream_key(seed, layer, ROUTER, e)
        out[e] = f32_to_bf16_bits(normal_scaled_f32(key, 0, hidden, sigma))
    return out


def x_bf16(seed: int, layer: int, batch: int, hidden: int, sigma: float = 1.0) -> np.ndarray:
    """Activations [B, H] as bf16 bit patterns; row t is the stream (X, t)."""
    out = np.empty((batch, hidden), dtype=np.uint16)
    for t in range(batch):
        key = stream_key(seed, layer, X, t)
        out[t] = f32_to_bf16_bits(normal_scaled_f32(key, 0, hidden, sigma))
    return out


def expert_f32(seed: int, layer: int, expert: int, hidden: int, inter: int, sigma: float = 0.02):
    """Float32 gate [I, H], up [I, H] and down [H, I] weights of one expert."""
    gate = matrix_f32(seed, layer, GATE, expert, inter, hidden, sigma)
    up = matrix_f32(seed, layer, UP, expert, inter, hidden, sigma)
    down = matrix_f32(seed, layer, DOWN, expert, hidden, inter, sigma)
    return gate, up, down


def bias_f32(seed: int, layer: int, num_experts: int, sigma: float) -> np.ndarray:
    key = stream_key(seed, layer, BIAS, 0)
    return normal_scaled_f32(key, 0, num_experts, sigma)


def norm_bf16(seed: int, layer: int, hidden: int, sigma: float = 0.1) -> np.ndarray:
    """RMSNorm weight of a layer: bf16 bits of float32(1 + sigma * N(0, 1))."""
    key = stream_key(seed, layer, NORM, 0)
    return f32_to_bf16_bits(np.float32(1.0) + normal_scaled_f32(key, 0, hidden, sigma))
