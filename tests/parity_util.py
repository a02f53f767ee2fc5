"""Helpers shared by the GPU parity tests: run the oracle and the CUDA path on
the same seeded inputs and compare them tensor by tensor."""

import numpy as np

from ffn_block_gb300 import inputs as I
from oracle import rmx_oracle as O

# Norm-relative tolerance per storage contract: strict fp32 1e-4, 16-bit 2e-2.
TOL = {"f32": 1e-4, "bf16": 2e-2, "f16": 2e-2}
NAMES = ("y", "dx") + I.PARAM_NAMES


def rel_err(a, ref):
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(a - ref)
    if den == 0.0:
        return num
    return num / den


def oracle_outputs(arrays: dict, samples=None) -> dict:
    """Oracle y, dx and gradients, optionally on a sub-batch of samples."""
    a = I.to_float64(arrays)
    x, dy = a["x"], a["dy"]
    if samples is not None:
        x, dy = x[samples], dy[samples]
    p = {k: a[k] for k in I.PARAM_NAMES}
    y, dx, grads = O.forward_backward(x, dy, p)
    out = {"y": y, "dx": dx}
    out.update(grads)
    return out


def compare(gpu: dict, ref: dict, tol: float, names=NAMES) -> dict:
    errs = {}
    for n in names:
        g = gpu[n]
        assert np.all(np.isfinite(g)), f"{n}: non-finite values"
        assert g.shape == ref[n].shape, (n, g.shape, ref[n].shape)
        errs[n] = rel_err(g, ref[n])
    bad = {n: e for n, e in errs.items() if not e <= tol}
    assert not bad, f"norm-relative error above {tol}: {bad} (all: {errs})"
    return errs
