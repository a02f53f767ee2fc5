"""The TF32 contract (page "Subgraph-fusion-based Mega-kernel Generation",
section "Run the benchmark": the float32 run with TF32 contractions): float32
storage and row passes, the four per-token contractions on the tensor cores
with TF32 operands.  Compared with the float64 oracle on y, dx and all 14
gradients at the TF32 tolerance, and checked to run no contraction on the CUDA
cores."""

import numpy as np
import pytest

from ffn_block_gb300 import binding as B
from ffn_block_gb300 import inputs as I
from ffn_block_gb300.device import RankMixerDevice

from parity_util import NAMES, TOL, compare, oracle_outputs

pytestmark = pytest.mark.gpu

SHAPES = [
    dict(B=2, T=8, D=64, H=128),       # the tiny oracle shape
    dict(B=64, T=16, D=256, H=512),    # the small fp32 shape
    dict(B=130, T=4, D=128, H=384),    # M spans two tiles with a tail, k = 3
    dict(B=7, T=8, D=64, H=192),       # batch (the weight gradients' K) not a multiple of 4
    dict(B=5, T=9, D=81, H=243),       # padded rows, odd C
]


@pytest.mark.parametrize("ln", ["init", "random"])
@pytest.mark.parametrize("dims", SHAPES, ids=lambda d: "B{B}_T{T}_D{D}_H{H}".format(**d))
def test_tf32_block(dims, ln):
    shape = I.Shape(dtype="tf32", **dims)
    arrays = I.make_inputs(shape, ln_params=ln)
    blk = RankMixerDevice(shape, arrays)
    B.rmx_profile_read()
    B.rmx_profile_enable(True)
    try:
        blk.step()
    finally:
        B.rmx_profile_enable(False)
    B.check(B.rmx_check(), "rmx_check")
    names = set(B.rmx_profile_read())
    assert not [n for n in names if n.endswith(".ffma")], names
    assert {"gemm1_fwd", "gemm2_fwd", "gemm1_dgrad", "gemm2_dgrad", "gemm1_wgrad", "gemm2_wgrad"} <= names
    errs = compare(blk.results(), oracle_outputs(arrays), TOL["tf32"], names=NAMES)
    # TF32 is less exact than the strict contract: the errors must show it.
    assert max(errs.values()) > TOL["f32"] * 1e-2
