"""The no-allocation norm2 backward (rmx_ln2_backward_noalloc).

Callers that cannot hand the library scratch memory -- a framework that owns
all device memory and gives a plugin only its inputs and outputs, or a
deployment with a fixed footprint -- use this entry point; its partial sums
live in a fixed device array inside the library.  The test calls it twice in
a row through the C ABI and checks each result against what rmx_backward
produces for the same tensors, within the parity tolerance.  It is kept in a
file of its own that pytest collects last.
"""

import numpy as np
import pytest
import torch

from ffn_block_gb300 import binding as B
from ffn_block_gb300 import inputs as I
from ffn_block_gb300.device import RankMixerDevice
from oracle import rmx_oracle as O

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2, "f16": 2e-2}


def _saved_views(blk):
    """s2 and norm2's statistics inside rmx_forward's saved buffer: the
    tensors out1, Z, hidden, s2, then ten float32 [B*T] statistic vectors,
    each segment starting on a 256-byte boundary."""
    s = blk.shape
    e = 4 if s.dtype == "f32" else 2
    N = s.B * s.T
    up = lambda v: (v + 255) // 256 * 256
    off = 0
    offs = []
    for nbytes in (N * s.D * e, N * 2 * s.H * e, N * s.H * e, N * s.D * e):
        offs.append(off)
        off = up(off + nbytes)
    stats = blk.saved[off:off + 10 * N * 4].view(torch.float32)
    s2 = blk.saved[offs[3]:offs[3] + N * s.D * e].view(blk.dtype)
    return s2, stats[4 * N:5 * N], stats[5 * N:6 * N]


def _rel(a, ref):
    a, ref = np.asarray(a, np.float64), np.asarray(ref, np.float64)
    return np.linalg.norm(a - ref) / np.linalg.norm(ref)


@pytest.mark.parametrize("dims,dtype", [
    (dict(B=1024, T=64, D=1280, H=256), "bf16"),   # production B, T, D
    (dict(B=256, T=32, D=512, H=1536), "bf16"),
    (dict(B=37, T=8, D=240, H=360), "f16"),
    (dict(B=64, T=16, D=256, H=512), "f32"),
])
def test_noalloc_norm2_backward_matches_rmx_backward(dims, dtype):
    shape = I.Shape(dtype=dtype, **dims)
    arrays = I.make_inputs(shape, ln_params="random")
    blk = RankMixerDevice(shape, arrays)
    blk.step()
    B.check(B.rmx_check())
    s2, mean2, rstd2 = _saved_views(blk)

    # ds2 is internal to rmx_backward, so it is checked against the oracle.
    a = I.to_float64(arrays)
    _, cache = O.forward(a["x"], {k: a[k] for k in I.PARAM_NAMES})
    ds2_ref, _, _ = O.layer_norm_backward(a["dy"], a["gamma2"], cache["st2"])

    for call in range(2):
        ds2 = torch.full_like(blk.x, float("nan"))
        dg2 = torch.full_like(blk.grads["gamma2"], float("nan"))
        db2 = torch.full_like(blk.grads["beta2"], float("nan"))
        dbo = torch.full_like(blk.grads["bout"], float("nan"))
        B.check(B.rmx_ln2_backward_noalloc(blk.cfg, blk.dy, s2, mean2, rstd2, blk.params["gamma2"],
                                           ds2, dg2, db2, dbo), f"no-alloc call {call}")
        B.check(B.rmx_check(), f"no-alloc call {call}")
        for got, ref in ((dg2, blk.grads["gamma2"]), (db2, blk.grads["beta2"]), (dbo, blk.grads["bout"])):
            g = got.float().cpu().numpy()
            assert np.all(np.isfinite(g))
            assert _rel(g, ref.float().cpu().numpy()) <= TOL[dtype]
        g = ds2.float().cpu().numpy()
        assert np.all(np.isfinite(g))
        assert _rel(g, ds2_ref) <= TOL[dtype]


def test_noalloc_rejects_oversized_and_bad_arguments():
    big = B.make_config(4, 1024, 2048, 128, "bf16")      # 3*T*D floats > the 16 MiB array
    p = 0x1000
    assert B.rmx_ln2_backward_noalloc(big, p, p, p, p, p, p, p, p, p) == B.RMX_ERR_UNSUPPORTED
    cfg = B.make_config(4, 8, 64, 128, "bf16")
    assert B.rmx_ln2_backward_noalloc(cfg, p, p, p, p, p, None, p, p, p) == B.RMX_ERR_INVALID_ARG
    assert B.rmx_ln2_backward_noalloc(cfg, p, p, p, p, p, p + 8, p, p, p) == B.RMX_ERR_ALIGNMENT
    empty = B.make_config(0, 8, 64, 128, "bf16")
    assert B.rmx_ln2_backward_noalloc(empty, p, p, p, p, p, p, p, p, p) == B.RMX_ERR_INVALID_ARG
