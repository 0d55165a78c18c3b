"""NVFP4 weight format: decode, encode (quantise) and dequantise, float64 CPU.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages ("Day-0 Support for Flint on vLLM", section "Model architecture")
name the format only as NVIDIA's NVFP4, stored weight-only beside BF16
activations. Its public definition, used here:

* element: E2M1 (OCP Microscaling Formats v1.0, FP4 E2M1): bit 3 sign,
  bits 2..1 exponent (bias 1), bit 0 mantissa; exponent 0 is subnormal with
  value mantissa * 0.5. Magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}; code 8 is -0.
* block scale: one FP8 E4M3 ("fn" variant) per 16 consecutive elements of a
  row: bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0 mantissa; exponent 0
  subnormal (mantissa * 2**-9); 0x7F and 0xFF are NaN; no infinities; max 448.
* tensor scale: one float32 G per matrix.

A weight is ``E2M1(code) * E4M3(scale) * G``; ``c = E2M1 * E4M3`` is exact in
float32 (at most 6 significant bits, range 2**-10 .. 2688).

The quantiser only produces test weights; the pages do not describe one. It
follows the public two-level NVFP4 recipe:
``G = amax / (6 * 448)``; per block ``s = E4M3_rn(amax_blk / (6 * G))``;
``code = E2M1_rn(w / (E4M3(s) * G))``; every step float32, round to nearest
even, saturating to the largest finite value; an all-zero tensor (G = 0) or a
block whose scale decodes to 0 gets all codes 0. The sign of a value that
rounds to zero is kept (code 8), as IEEE rounding keeps it.
"""
from __future__ import annotations

import numpy as np

E2M1_MAX = 6.0
E4M3_MAX = 448.0
BLOCK = 16


# ---------------------------------------------------------------- decode

def e2m1_decode(code) -> np.ndarray:
    """E2M1 code (0..15) -> float64 value, from the bit fields."""
    code = np.asarray(code, dtype=np.int64)
    sign = np.where(code & 8, -1.0, 1.0)
    exp = (code >> 1) & 3
    man = code & 1
    mag = np.where(exp == 0, man * 0.5, (1.0 + man * 0.5) * np.exp2(exp - 1.0))
    return sign * mag


def e4m3_decode(code) -> np.ndarray:
    """E4M3 ("fn") code (0..255) -> float64 value, NaN for 0x7F / 0xFF."""
    code = np.asarray(code, dtype=np.int64)
    sign = np.where(code & 0x80, -1.0, 1.0)
    exp = (code >> 3) & 0xF
    man = code & 7
    mag = np.where(exp == 0, man * 2.0 ** -9, (1.0 + man / 8.0) * np.exp2(exp - 7.0))
    mag = np.where((code & 0x7F) == 0x7F, np.nan, mag)
    return sign * mag


# ---------------------------------------------------------------- encode

def _round_to_grid(mag: np.ndarray, grid: np.ndarray, grid_codes: np.ndarray) -> np.ndarray:
    """Nearest grid value to each non-negative ``mag``; ties go to the code
    whose lowest bit is 0 (the even mantissa); above the grid saturates."""
    mag = np.asarray(mag, dtype=np.float64)
    top = len(grid) - 1
    hi = np.searchsorted(grid, mag, side="left")           # grid[hi] >= mag
    hi = np.minimum(hi, top)
    lo = np.maximum(hi - 1, 0)
    exact = grid[hi] == mag
    d_lo = mag - grid[lo]
    d_hi = grid[hi] - mag
    pick_hi = np.where(d_hi < d_lo, True,
                       np.where(d_hi > d_lo, False, (grid_codes[hi] & 1) == 0))
    out = np.where(pick_hi, grid_codes[hi], grid_codes[lo])
    out = np.where(exact, grid_codes[hi], out)
    out = np.where(mag >= grid[top], grid_codes[top], out)
    return out


_E2M1_CODES = np.arange(8, dtype=np.int64)
_E2M1_GRID = e2m1_decode(_E2M1_CODES)                       # 0, .5, 1, 1.5, 2, 3, 4, 6
_E4M3_CODES = np.arange(0x7F, dtype=np.int64)               # non-negative finite codes
_E4M3_GRID = e4m3_decode(_E4M3_CODES)                       # increasing, 0 .. 448


def e2m1_encode(x) -> np.ndarray:
    """Round float32 values to E2M1 codes: nearest, ties to even, saturating at 6."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    mag = _round_to_grid(np.abs(x), _E2M1_GRID, _E2M1_CODES)
    return (mag | np.where(np.signbit(x), 8, 0)).astype(np.uint8)


def e4m3_encode(x) -> np.ndarray:
    """Round float32 values to E4M3 codes: nearest, ties to even, saturating at 448."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    mag = _round_to_grid(np.abs(x), _E4M3_GRID, _E4M3_CODES)
    return (mag | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


# ---------------------------------------------------------------- layout

def unpack_codes(codes: np.ndarray) -> np.ndarray:
    """[rows, cols/2] bytes -> [rows, cols] codes; element 2j is the low nibble."""
    codes = np.asarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = codes & 0x0F
    out[..., 1::2] = codes >> 4
    return out


def pack_codes(elems: np.ndarray) -> np.ndarray:
    """[rows, cols] codes -> [rows, cols/2] bytes (inverse of unpack_codes)."""
    elems = np.asarray(elems, dtype=np.uint8)
    return (elems[..., 0::2] | (elems[..., 1::2] << 4)).astype(np.uint8)


# ---------------------------------------------------------------- quantise

def quantize(w: np.ndarray):
    """float32 [rows, cols] -> (codes uint8 [rows, cols/2], scales uint8
    [rows, cols/16], G float32): the two-level recipe of the module docstring."""
    w = np.asarray(w, dtype=np.float32)
    rows, cols = w.shape
    assert cols % BLOCK == 0
    amax = np.float32(np.max(np.abs(w))) if w.size else np.float32(0)
    G = np.float32(amax / np.float32(E2M1_MAX * E4M3_MAX))
    blocks = w.reshape(rows, cols // BLOCK, BLOCK)
    if G == 0:
        return (np.zeros((rows, cols // 2), np.uint8),
                np.zeros((rows, cols // BLOCK), np.uint8), np.float32(0))
    amax_blk = np.max(np.abs(blocks), axis=2).astype(np.float32)
    six_g = np.float32(np.float32(E2M1_MAX) * G)
    scales = e4m3_encode((amax_blk / six_g).astype(np.float32))
    dec = e4m3_decode(scales).astype(np.float32)               # exact
    t = (dec * G).astype(np.float32)                           # float32 RN
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (blocks / t[:, :, None]).astype(np.float32)
    codes = e2m1_encode(r)
    codes = np.where((t == 0)[:, :, None], np.uint8(0), codes).reshape(rows, cols)
    return pack_codes(codes), scales.astype(np.uint8), G


def dequant_c(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """c[r, col] = E2M1(code) * E4M3(scale[r, col // 16]), float64 (exact)."""
    q = e2m1_decode(unpack_codes(codes))
    s = e4m3_decode(np.asarray(scales))
    return q * np.repeat(s, BLOCK, axis=-1)


def dequantize(codes: np.ndarray, scales: np.ndarray, G) -> np.ndarray:
    """Full weight c * G in float64."""
    return dequant_c(codes, scales) * np.float64(np.float32(G))
