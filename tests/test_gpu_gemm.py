"""The grouped GEMM engine in isolation (tcgen05 for 16-bit, FFMA for fp32),
through the C ABI's test hook, against numpy float64 contractions of the
same rounded operands."""

import numpy as np
import pytest
import torch

from ffn_block_gb300 import binding as B
from ffn_block_gb300.device import TORCH_DTYPES
from ffn_block_gb300.inputs import round_to_storage

pytestmark = pytest.mark.gpu

# Output is rounded to the storage type once: ~2^-9 (bf16) / 2^-12 (fp16)
# relative, far below these bounds; fp32 accumulates in a different order.
TOL = {"f32": 1e-5, "bf16": 6e-3, "f16": 2e-3,
       # TF32 operands: at most 2^-9 relative error per product; random-sign
       # sums keep the norm-relative error near 2^-10.
       "tf32": 3e-3}


def _run(kind, dtype, M, N, K, G, seed=0):
    rng = np.random.default_rng(seed)
    if kind == 0:
        a_shape, b_shape, c_shape = (M, G, K), (G, K, N), (M, G, N)
    elif kind == 1:
        a_shape, b_shape, c_shape = (M, G, K), (G, N, K), (M, G, N)
    else:
        a_shape, b_shape, c_shape = (K, G, M), (K, G, N), (G, M, N)
    A = round_to_storage(rng.standard_normal(a_shape, dtype=np.float32), dtype)
    Bm = round_to_storage(rng.standard_normal(b_shape, dtype=np.float32), dtype)
    dt = TORCH_DTYPES[dtype]
    tA = torch.from_numpy(A).cuda().to(dt)
    tB = torch.from_numpy(Bm).cuda().to(dt)
    tC = torch.full(c_shape, float("nan"), device="cuda", dtype=dt)
    B.check(B.rmx_test_gemm(kind, dtype, M, N, K, G, tA, tB, tC), "rmx_test_gemm")
    B.check(B.rmx_check(), "rmx_check")
    A64, B64 = A.astype(np.float64), Bm.astype(np.float64)
    if kind == 0:
        ref = np.einsum("mgk,gkn->mgn", A64, B64)
    elif kind == 1:
        ref = np.einsum("mgk,gnk->mgn", A64, B64)
    else:
        ref = np.einsum("kgm,kgn->gmn", A64, B64)
    return tC.float().cpu().numpy().astype(np.float64), ref


SHAPES = [
    (128, 256, 64, 1),     # exactly one tile, one k-block
    (256, 512, 320, 2),    # several tiles and k-blocks
    (200, 264, 136, 3),    # ragged M, N, K
    (64, 64, 64, 2),       # smaller than one tile
    (8, 8, 8, 1),          # tiny
    (1000, 1200, 200, 2),  # ragged, wide
]


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("kind", [0, 1, 2])
@pytest.mark.parametrize("shape", SHAPES)
def test_grouped_gemm(kind, dtype, shape):
    M, N, K, G = shape
    got, ref = _run(kind, dtype, M, N, K, G)
    assert np.all(np.isfinite(got))
    err = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err < TOL[dtype], err


# Paired-CTA mode (a cluster of two CTAs shares each B tile) engages when M
# spans two or more 128-row tiles; an odd tile count leaves the second CTA of
# the last pair with rows wholly past M.
PAIR_SHAPES = [
    (300, 136, 72, 2),     # 3 M-tiles: last pair half empty; N < 256
    (384, 640, 1000, 1),   # 3 M-tiles, long ragged K
    (129, 264, 64, 2),     # 2 M-tiles, second one holds a single row
    (520, 200, 88, 3),     # M-major and N-major tails together
    (512, 384, 264, 2),    # MN extents multiples of 64: interleaved MN-major stages, ragged K
    (640, 1000, 136, 2),   # 5 M-tiles (an odd number of pairs), ragged N
    (1024, 2560, 256, 8),  # 320 pair tiles: the persistent grid wraps several times
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("kind", [0, 1, 2])
@pytest.mark.parametrize("shape", PAIR_SHAPES)
def test_grouped_gemm_paired_tiles(kind, dtype, shape):
    M, N, K, G = shape
    got, ref = _run(kind, dtype, M, N, K, G, seed=3)
    assert np.all(np.isfinite(got))
    err = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err < TOL[dtype], err


# TF32 (fp32 storage): the dgrad form (both operands K-major) runs on the
# tensor cores; the forward and weight-gradient forms read an operand
# MN-major and run in strict fp32 (the block stages transposed copies so
# that all of its contractions take the dgrad form).
@pytest.mark.parametrize("shape", SHAPES + PAIR_SHAPES)
def test_tf32_dgrad_form_on_tensor_cores(shape):
    M, N, K, G = shape
    B.rmx_profile_read()
    B.rmx_profile_enable(True)
    try:
        got, ref = _run(1, "tf32", M, N, K, G, seed=5)
    finally:
        B.rmx_profile_enable(False)
    assert set(B.rmx_profile_read()) == {"test_gemm"}
    assert np.all(np.isfinite(got))
    err = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err < TOL["tf32"], err
    assert err > 1e-7   # the operands really were read at TF32 precision
