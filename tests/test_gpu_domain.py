"""The held-out shape domain of the page "Subgraph-fusion-based Mega-kernel
Generation", section "Public checks and instructor coverage": any batch
1 <= B <= 1024, tokens 8 <= T <= 64, width 64 <= D <= 1280 with D divisible by
T, and H = k * D with k in {2, 3}, in each of the three storage types.

A seeded random draw of that domain (most of its widths are not a multiple of
8, so those blocks run on zero-padded rows) plus hand-picked corners, each
compared with the float64 oracle on y, dx and all 14 gradients (same
tolerances as the other parity tests).  16-bit blocks must run every
contraction on the tensor cores: no GEMM launch may fall back to the CUDA
cores (those launches are profiled under a name ending in ".ffma")."""

import numpy as np
import pytest

from ffn_block_gb300 import binding as B
from ffn_block_gb300 import inputs as I
from ffn_block_gb300.device import RankMixerDevice

from parity_util import TOL, compare, oracle_outputs

pytestmark = pytest.mark.gpu


def domain_shapes(n=30, seed=83):
    """n shapes drawn from the domain; B log-uniform, shrunk (halved) until
    the oracle's work B*T*D*H is at most 1.5e9; storage types in turn."""
    rng = np.random.default_rng(seed)
    dtypes = ["bf16", "f16", "f32"]
    out = []
    while len(out) < n:
        T = int(rng.integers(8, 65))
        C = int(rng.integers(-(-64 // T), 1280 // T + 1))
        D = T * C
        k = int(rng.integers(2, 4))
        B_ = max(1, min(1024, int(np.exp(rng.uniform(0.0, np.log(1024.0))))))
        while B_ > 1 and B_ * T * D * k * D > 1.5e9:
            B_ //= 2
        out.append((B_, T, D, k * D, dtypes[len(out) % 3]))
    return out


CORNERS = [
    (1024, 8, 72, 144, "bf16"),    # largest batch, D = 72 (aligned), B % 8 == 0
    (1000, 10, 90, 270, "f16"),    # large ragged batch, D and H not multiples of 8
    (13, 8, 128, 256, "bf16"),     # weight gradients reduce over K = B = 13
    (777, 12, 84, 168, "bf16"),    # B % 8 != 0 and D % 8 != 0
    (3, 64, 1280, 2560, "f32"),    # widest fp32 rows with k = 2 (H > 2048)
    (2, 64, 1280, 3840, "f32"),    # widest fp32 rows with k = 3
    (2, 64, 1280, 3840, "bf16"),   # widest 16-bit rows with k = 3
    (1, 8, 64, 192, "f16"),        # smallest of everything, k = 3
    (5, 9, 81, 243, "bf16"),       # odd C (= 9), odd H
]


def _case(B_, T, D, H, dtype):
    shape = I.Shape(B=B_, T=T, D=D, H=H, dtype=dtype)
    arrays = I.make_inputs(shape, ln_params="random")
    blk = RankMixerDevice(shape, arrays)
    B.rmx_profile_read()
    B.rmx_profile_enable(True)
    try:
        blk.step()
    finally:
        B.rmx_profile_enable(False)
    B.check(B.rmx_check(), "rmx_check")
    names = set(B.rmx_profile_read())
    got = blk.results()
    compare(got, oracle_outputs(arrays), TOL[dtype])
    if dtype != "f32":
        assert not [n for n in names if n.endswith(".ffma")], names


@pytest.mark.parametrize("dims", domain_shapes(), ids=lambda d: "B%d_T%d_D%d_H%d_%s" % d)
def test_domain_sweep(dims):
    _case(*dims)


@pytest.mark.parametrize("dims", CORNERS, ids=lambda d: "B%d_T%d_D%d_H%d_%s" % d)
def test_domain_corners(dims):
    _case(*dims)
