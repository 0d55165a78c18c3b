"""Parity of the dense GEMV (through the C ABI) with the CPU oracle.

Pass rules, fixed in advance: the repack is a bijection (byte for byte); outputs
within 2^-7 * max(1, |ref|) per element.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import dense, moe, nvfp4
from w4a16_moe_decode_gb300 import binding as fb
from w4a16_moe_decode_gb300 import layers
from w4a16_moe_decode_gb300.build import build

from _common import bits_to_f64, check_out

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    fb.lib()


def oracle_matrix(N, K, seed, fmt):
    w = synth.matrix_f32(seed, 0, synth.DOWN, 0, N, K, 0.02)
    if fmt == fb.NVFP4:
        return moe.NVFP4Matrix(*nvfp4.quantize(w))
    return moe.BF16Matrix(synth.f32_to_bf16_bits(w))


def run_gemv(N, K, B, seed, fmt=fb.NVFP4, norm=False, rows=None):
    packed, _ = layers.synth_dense(N, K, seed, 0, fmt, DEV)
    x = layers.synth_x(B, K, seed, 0, DEV)
    y = torch.full((B, N), 0x7FC0, dtype=torch.int16, device=DEV)
    g = layers.synth_norm(K, seed, 0, DEV) if norm else None
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    fb.flint_gemv(packed, N, K, fmt, x, B, y, g, 1e-6, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    xo = moe.bf16_bits_to_f64(synth.x_bf16(seed, 0, B, K))
    assert np.array_equal(bits_to_f64(x), xo)
    go = moe.bf16_bits_to_f64(synth.norm_bf16(seed, 0, K)) if norm else None
    rows = list(range(B)) if rows is None else rows
    ref = dense.gemv(xo[rows], oracle_matrix(N, K, seed, fmt), go, 1e-6)
    check_out(ref, bits_to_f64(y)[rows], f"gemv N={N} K={K} B={B}")


@pytest.mark.parametrize("fmt", [fb.NVFP4, fb.BF16])
def test_gemv_pack_is_a_bijection(fmt):
    N, K = 48, 512
    packed, canon = layers.synth_dense(N, K, 31, 0, fmt, DEV)
    back = {k: torch.zeros_like(v) for k, v in canon.items()}
    fb.flint_gemv_unpack_debug(packed, N, K, fmt, back)
    torch.cuda.synchronize()
    for k in canon:
        assert torch.equal(canon[k], back[k]), k


@pytest.mark.parametrize("B,seed", [(1, 40), (5, 41), (8, 42), (9, 43), (32, 44)])
def test_gemv_small_shapes(B, seed):
    run_gemv(64, 256, B, seed)


def test_gemv_projection_shape():
    run_gemv(2048, 2048, 1, 45)
    run_gemv(2048, 2048, 8, 46, rows=[0, 7])


def test_gemv_wide_and_tall():
    run_gemv(256, 4096, 2, 47)
    run_gemv(4096, 512, 3, 48, rows=[2])


def test_gemv_bf16_weights_and_norm_prologue():
    run_gemv(128, 1024, 4, 49, fmt=fb.BF16)
    run_gemv(128, 1024, 4, 50, norm=True)
    run_gemv(96, 768, 17, 51, fmt=fb.BF16, norm=True)


@pytest.mark.parametrize("K,B,fmt,norm", [(8192, 1, fb.NVFP4, False), (8192, 9, fb.NVFP4, True),
                                          (4096, 32, fb.NVFP4, True), (8192, 3, fb.BF16, True),
                                          (4096, 17, fb.BF16, False)])
def test_gemv_split_over_a_cluster(K, B, fmt, norm):
    """K > 2048: the column slices of a tile are taken by the CTAs of a
    cluster and added in distributed shared memory (and, with a norm weight,
    the rows' sums of squares are shared the same way)."""
    run_gemv(64, K, B, 52 + B, fmt=fmt, norm=norm)


def test_gemv_split_norm_of_rows_beyond_the_fp32_square_range():
    """Rows whose sum of squares overflows FP32 (times 2^100), normalised on the
    split path: the scaled sum over the whole row."""
    N, K, B, seed = 32, 4096, 3, 60
    packed, _ = layers.synth_dense(N, K, seed, 0, fb.NVFP4, DEV)
    xo = moe.bf16_bits_to_f64(synth.x_bf16(seed, 0, B, K)) * np.array([2.0 ** 100, 1.0, 2.0 ** -100])[:, None]
    x = torch.from_numpy(moe.f64_to_bf16_bits(xo).view(np.int16)).to(DEV)
    y = torch.full((B, N), 0x7FC0, dtype=torch.int16, device=DEV)
    g = layers.synth_norm(K, seed, 0, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    fb.flint_gemv(packed, N, K, fb.NVFP4, x, B, y, g, 1e-6, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    go = moe.bf16_bits_to_f64(synth.norm_bf16(seed, 0, K))
    ref = dense.gemv(moe.bf16_bits_to_f64(moe.f64_to_bf16_bits(xo)), oracle_matrix(N, K, seed, fb.NVFP4), go, 1e-6)
    check_out(ref, bits_to_f64(y), "gemv split, rows beyond the FP32 square range")
