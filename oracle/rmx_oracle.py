"""Float64 CPU oracle of the RankMixer block, forward and backward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import or call
this module; only the tests, the smoke check and the benchmark's CPU-baseline
leg use it.  It shares no code with the CUDA path.

Everything below follows the page "Subgraph-fusion-based Mega-kernel
Generation", section "Exact computation", written out as plainly as possible
in numpy float64 (numpy's ``@`` is the only library primitive used for the
per-token contractions).  The backward is the chain rule applied by hand to
the same steps; there is no fusion, blocking or reordering beyond what the
definitions state.

Readings taken where the page leaves a step open (each the plainest one that
the rest of the page supports):
  R1  (U, G) = split of Z into two H-wide halves, U the first half (the
      order in which a split along the last axis returns its pieces).
  R2  the outer LayerNorms use the same biased-variance formula as the
      page's LN(z), with epsilon inside the square root (the page names only
      their epsilon, 1e-3).
  R3  norm1's residual is the raw block input (the page writes
      norm1(out1 + inputs)); norm2's residual is out1 (norm2(out1 + out2)).
  R4  H = k * D (the page's shape line pairs D=1280 and k=2 with H=2560).
  R5  silu(g) = g * sigmoid(g), exact (no approximation is named).
  R6  parameter gradients are summed over every row that used the parameter:
      w1, b1, wout, bout over the batch b for their own token t; every
      gamma/beta and inner weight/bias over all B*T rows (each token has its
      own w1[t], b1[t], wout[t], bout[t]; the LayerNorm parameters are one
      vector shared by all rows).
  R7  the token-mixing backward is the same permutation (swapping the two T
      axes twice gives the identity, so the swap is its own inverse and its
      transpose).

Parity pins (tests/test_oracle.py): the page's token-mixing worked example,
the involution, the D == T transpose special case, LayerNorm invariants,
brute-force loops on tiny inputs, a zero-weight closed form, central finite
differences of every gradient, and an independent torch float64 autograd
composition.
"""

from __future__ import annotations

import numpy as np

EPS_OUTER = 1e-3   # norm0, norm1, norm2: the outer LayerNorms' epsilon on the page
EPS_INNER = 1e-5   # norm_x, norm_gate: the inner LayerNorms' epsilon on the page


# ---------------------------------------------------------------------------
# Building blocks, each a definition from the page.
# ---------------------------------------------------------------------------

def layer_norm(z, gamma, beta, eps):
    """LN(z) = ((z - mean(z)) / sqrt(mean((z - mean(z))^2) + eps)) * gamma + beta.

    Page "Subgraph-fusion-based Mega-kernel Generation", section "Exact
    computation", the LN(z) line; the mean runs over the last axis.
    Returns the output and (mean, rstd, xhat) for the backward.
    """
    mean = z.mean(axis=-1, keepdims=True)
    var = ((z - mean) ** 2).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (z - mean) * rstd
    return xhat * gamma + beta, (mean, rstd, xhat)


def layer_norm_backward(dout, gamma, stats):
    """Chain rule through layer_norm for one row-normalised tensor.

    With g = gamma * dout and n the row length:
      dz     = rstd * (g - mean(g) - xhat * mean(g * xhat))
      dgamma = sum over rows of dout * xhat
      dbeta  = sum over rows of dout
    """
    _, rstd, xhat = stats
    g = gamma * dout
    dz = rstd * (g - g.mean(axis=-1, keepdims=True)
                 - xhat * (g * xhat).mean(axis=-1, keepdims=True))
    lead = tuple(range(dout.ndim - 1))
    return dz, (dout * xhat).sum(axis=lead), dout.sum(axis=lead)


def token_mixer(a):
    """reshape(B, T, T, D/T), swap the two T axes, reshape back to [B, T, D].

    Section "Exact computation": on [1,2,4] rows [[0,1,2,3],[4,5,6,7]]
    become [[0,1,4,5],[2,3,6,7]].
    """
    B, T, D = a.shape
    if D % T:
        raise ValueError("token mixing needs D % T == 0")
    return a.reshape(B, T, T, D // T).swapaxes(1, 2).reshape(B, T, D)


def sigmoid(g):
    return 1.0 / (1.0 + np.exp(-g))


def silu(g):
    return g * sigmoid(g)


def silu_grad(g):
    """d/dg [g * sigmoid(g)] = sigmoid(g) * (1 + g * (1 - sigmoid(g)))."""
    s = sigmoid(g)
    return s * (1.0 + g * (1.0 - s))


# ---------------------------------------------------------------------------
# Forward.
# ---------------------------------------------------------------------------

def dense_ffn_v2_forward(inp, p):
    """The dense subgraph of section "Exact computation".

    Z[b,t,:] = inp[b,t,:] @ w1[t] + b1[t]; (U, G) = split(Z) (reading R1);
    hidden = LN_x(U) * silu(LN_gate(G));
    out[b,t,:] = hidden[b,t,:] @ wout[t] + bout[t].
    """
    B, T, D = inp.shape
    H = p["wout"].shape[1]
    Z = np.empty((B, T, 2 * H))
    for t in range(T):
        Z[:, t, :] = inp[:, t, :] @ p["w1"][t] + p["b1"][t]
    U, G = Z[..., :H], Z[..., H:]
    u, st_u = layer_norm(U, p["lnx_w"], p["lnx_b"], EPS_INNER)
    g, st_g = layer_norm(G, p["lng_w"], p["lng_b"], EPS_INNER)
    hidden = u * silu(g)
    out = np.empty((B, T, D))
    for t in range(T):
        out[:, t, :] = hidden[:, t, :] @ p["wout"][t] + p["bout"][t]
    cache = dict(Z=Z, u=u, g=g, st_u=st_u, st_g=st_g, hidden=hidden)
    return out, cache


def forward(x, p):
    """RankMixerBlock forward, section "Exact computation":

      out1   = token_mixer(norm0(inputs))
      out1   = norm1(out1 + inputs)
      out2   = dense_ffn_v2_compute(out1, ...)
      output = norm2(out1 + out2)

    Returns (y, cache); cache keeps what the backward needs.
    """
    a0, st0 = layer_norm(x, p["gamma0"], p["beta0"], EPS_OUTER)
    m = token_mixer(a0)
    s1 = m + x                                              # reading R3
    out1, st1 = layer_norm(s1, p["gamma1"], p["beta1"], EPS_OUTER)
    out2, ffn = dense_ffn_v2_forward(out1, p)
    s2 = out1 + out2
    y, st2 = layer_norm(s2, p["gamma2"], p["beta2"], EPS_OUTER)
    cache = dict(x=x, st0=st0, st1=st1, out1=out1, s2=s2, st2=st2, **ffn)
    return y, cache


# ---------------------------------------------------------------------------
# Backward (chain rule through the steps above, in reverse order).
# ---------------------------------------------------------------------------

def backward(dy, cache, p, intermediates=None):
    """Gradients of sum(dy * y) w.r.t. x and every parameter.

    Returns (dx, grads) where grads has one entry per parameter name, each
    with the parameter's shape (reading R6 for the reductions).  If
    `intermediates` is a dict, the gradients w.r.t. s2, Z and s1 are stored
    in it under "ds2", "dZ" and "ds1".
    """
    B, T, D = dy.shape
    H = p["wout"].shape[1]
    grads = {}

    # output = norm2(s2), s2 = out1 + out2
    ds2, grads["gamma2"], grads["beta2"] = layer_norm_backward(dy, p["gamma2"], cache["st2"])

    # out2[b,t] = hidden[b,t] @ wout[t] + bout[t]
    dhidden = np.empty((B, T, H))
    grads["wout"] = np.empty_like(p["wout"])
    for t in range(T):
        dhidden[:, t, :] = ds2[:, t, :] @ p["wout"][t].T
        grads["wout"][t] = cache["hidden"][:, t, :].T @ ds2[:, t, :]
    grads["bout"] = ds2.sum(axis=0)

    # hidden = u * silu(g), u = LN_x(U), g = LN_gate(G)
    g = cache["g"]
    du = dhidden * silu(g)
    dg = dhidden * cache["u"] * silu_grad(g)
    dU, grads["lnx_w"], grads["lnx_b"] = layer_norm_backward(du, p["lnx_w"], cache["st_u"])
    dG, grads["lng_w"], grads["lng_b"] = layer_norm_backward(dg, p["lng_w"], cache["st_g"])
    dZ = np.concatenate([dU, dG], axis=-1)

    # Z[b,t] = out1[b,t] @ w1[t] + b1[t]
    dout1 = ds2.copy()                                   # residual into norm2
    grads["w1"] = np.empty_like(p["w1"])
    for t in range(T):
        dout1[:, t, :] += dZ[:, t, :] @ p["w1"][t].T
        grads["w1"][t] = cache["out1"][:, t, :].T @ dZ[:, t, :]
    grads["b1"] = dZ.sum(axis=0)

    # out1 = norm1(s1), s1 = token_mixer(a0) + x
    ds1, grads["gamma1"], grads["beta1"] = layer_norm_backward(dout1, p["gamma1"], cache["st1"])
    dx = ds1.copy()                                      # residual path
    da0 = token_mixer(ds1)                               # reading R7

    # a0 = norm0(x)
    dx0, grads["gamma0"], grads["beta0"] = layer_norm_backward(da0, p["gamma0"], cache["st0"])
    dx += dx0
    if intermediates is not None:
        intermediates.update(ds2=ds2, dZ=dZ, ds1=ds1)
    return dx, grads


def forward_backward(x, dy, p):
    """One full step: y = block(x), then the gradients for upstream dy."""
    y, cache = forward(x, p)
    dx, grads = backward(dy, cache, p)
    return y, dx, grads
