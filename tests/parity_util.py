"""Helpers shared by the GPU parity tests: run the oracle and the CUDA path on
the same seeded inputs and compare them tensor by tensor."""

import numpy as np

from ffn_block_gb300 import inputs as I
from oracle import rmx_oracle as O

# Norm-relative tolerance per storage contract: strict fp32 1e-4, 16-bit 2e-2.
# TF32 contractions (fp32 storage): the tensor cores read each fp32 operand
# with a 10-bit mantissa, a relative error of at most 2^-10 per operand and
# 2^-9 per product.  Summed over K with random signs, a contraction's result
# is off by about 2^-10 of its norm; a gradient passes through up to three
# contractions and the LayerNorm backwards between them, which can each
# amplify it a few times: 5e-3 bounds that chain.
TOL = {"f32": 1e-4, "bf16": 2e-2, "f16": 2e-2, "tf32": 5e-3}
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


def oracle_outputs_chunked(arrays: dict, chunk: int = 128) -> dict:
    """Oracle y, dx and gradients of the whole batch, run on consecutive
    chunks of samples to bound host memory.  Exact decomposition: y and dx of
    a sample depend only on that sample, and every parameter gradient is a
    sum over samples, so the chunks' gradients are summed (in float64)."""
    a = I.to_float64(arrays)
    p = {k: a[k] for k in I.PARAM_NAMES}
    B = a["x"].shape[0]
    ys, dxs, tot = [], [], None
    for b0 in range(0, B, chunk):
        y, dx, grads = O.forward_backward(a["x"][b0:b0 + chunk], a["dy"][b0:b0 + chunk], p)
        ys.append(y)
        dxs.append(dx)
        if tot is None:
            tot = {k: v.copy() for k, v in grads.items()}
        else:
            for k, v in grads.items():
                tot[k] += v
    out = {"y": np.concatenate(ys), "dx": np.concatenate(dxs)}
    out.update(tot)
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
