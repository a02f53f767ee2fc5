"""The unfused comparison arm of bench.py (a plain PyTorch composition of
the block, measured beside the fused path) computes the same block as the
oracle: checked in float64 on the CPU."""

import numpy as np
import torch

import bench
from ffn_block_gb300 import inputs as I
from oracle import rmx_oracle as O


def test_unfused_arm_matches_oracle():
    shape = I.Shape(B=2, T=8, D=64, H=128, dtype="f32")
    arrays = I.make_inputs(shape, ln_params="random")
    a = I.to_float64(arrays)
    p = {k: a[k] for k in I.PARAM_NAMES}
    y, dx, grads = O.forward_backward(a["x"], a["dy"], p)
    t = lambda v: torch.from_numpy(np.ascontiguousarray(v))
    ty, tdx, tg = bench.unfused_forward_backward(t(a["x"]), t(a["dy"]), {k: t(v) for k, v in p.items()})
    assert np.allclose(ty.numpy(), y, rtol=1e-9, atol=1e-9)
    assert np.allclose(tdx.numpy(), dx, rtol=1e-8, atol=1e-9)
    for k in I.PARAM_NAMES:
        g = tg[k].numpy()
        assert np.linalg.norm(g - grads[k]) <= 1e-8 * max(np.linalg.norm(grads[k]), 1e-30), k
