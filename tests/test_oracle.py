"""Pins for the float64 oracle (CPU only).

Each test fixes the oracle against something other than itself: the page's
worked example, library routines it must reduce to, closed forms, invariants,
brute-force loops, central finite differences and an independent torch
float64 autograd composition.  The last test plants mistakes in the oracle and
checks that a pin catches each one.
"""

import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import rmx_oracle as O
from ffn_block_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _inputs(shape, ln="random", seed=7101):
    return I.to_float64(I.make_inputs(shape, seed=seed, ln_params=ln))


def _params(inp):
    return {k: inp[k] for k in I.PARAM_NAMES}


# --------------------------------------------------------------- token mixing

def test_token_mix_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "token_mix_example.json")))
    a = np.array(g["input"], dtype=np.float64)
    assert list(a.shape) == g["shape"]
    np.testing.assert_array_equal(O.token_mixer(a), np.array(g["output"], dtype=np.float64))


@pytest.mark.parametrize("B,T,D", [(2, 8, 64), (3, 4, 12), (1, 16, 16), (2, 40, 1200)])
def test_token_mix_involution(B, T, D):
    a = np.random.default_rng(1).standard_normal((B, T, D))
    np.testing.assert_array_equal(O.token_mixer(O.token_mixer(a)), a)


def test_token_mix_D_equals_T_is_a_transpose():
    a = np.random.default_rng(2).standard_normal((3, 8, 8))
    np.testing.assert_array_equal(O.token_mixer(a), np.transpose(a, (0, 2, 1)))


def test_token_mix_single_token_is_identity():
    a = np.random.default_rng(3).standard_normal((2, 1, 24))
    np.testing.assert_array_equal(O.token_mixer(a), a)


def test_token_mix_bruteforce_index_form():
    # m[b, i, j*C + c] = a[b, j, i*C + c]: the T axes of [B,T,T,C] swapped.
    B, T, D = 2, 4, 12
    C = D // T
    a = np.arange(B * T * D, dtype=np.float64).reshape(B, T, D)
    m = O.token_mixer(a)
    for b in range(B):
        for i in range(T):
            for j in range(T):
                for c in range(C):
                    assert m[b, i, j * C + c] == a[b, j, i * C + c]


def test_token_mix_rejects_indivisible():
    with pytest.raises(ValueError):
        O.token_mixer(np.zeros((1, 3, 8)))


# --------------------------------------------------------------- layer norm

@pytest.mark.parametrize("eps", [1e-3, 1e-5])
def test_layer_norm_invariants(eps):
    z = np.random.default_rng(4).standard_normal((7, 5, 96)) * 3.0 + 1.5
    y, (mean, rstd, xhat) = O.layer_norm(z, np.ones(96), np.zeros(96), eps)
    np.testing.assert_allclose(y.mean(-1), 0.0, atol=1e-12)
    var = np.var(z, axis=-1)                       # library routine, biased
    np.testing.assert_allclose((y ** 2).mean(-1), var / (var + eps), rtol=1e-12)
    np.testing.assert_allclose(mean[..., 0], z.mean(-1), rtol=1e-13)
    np.testing.assert_allclose(rstd[..., 0], 1.0 / np.sqrt(var + eps), rtol=1e-12)


@pytest.mark.parametrize("eps", [1e-3, 1e-5])
def test_layer_norm_is_torch_layer_norm(eps):
    rng = np.random.default_rng(5)
    z = rng.standard_normal((6, 33))
    w, b = rng.uniform(0.5, 1.5, 33), rng.standard_normal(33)
    y, _ = O.layer_norm(z, w, b, eps)
    yt = F.layer_norm(torch.from_numpy(z), (33,), torch.from_numpy(w), torch.from_numpy(b), eps)
    np.testing.assert_allclose(y, yt.numpy(), rtol=1e-12, atol=1e-12)


def test_layer_norm_constant_row_is_beta():
    z = np.full((2, 16), 3.25)
    b = np.linspace(-1, 1, 16)
    y, (_, rstd, xhat) = O.layer_norm(z, np.full(16, 2.0), b, 1e-3)
    np.testing.assert_array_equal(xhat, 0.0)
    np.testing.assert_allclose(rstd, 1.0 / np.sqrt(1e-3))
    np.testing.assert_array_equal(y, np.broadcast_to(b, y.shape))


def test_layer_norm_backward_rows_sum_to_zero():
    rng = np.random.default_rng(6)
    z = rng.standard_normal((4, 3, 50))
    gam = rng.uniform(0.5, 1.5, 50)
    _, st = O.layer_norm(z, gam, np.zeros(50), 1e-3)
    dz, _, _ = O.layer_norm_backward(rng.standard_normal(z.shape), gam, st)
    np.testing.assert_allclose(dz.sum(-1), 0.0, atol=1e-12)


def test_silu_grad_matches_torch():
    g = torch.linspace(-12, 12, 301, dtype=torch.float64, requires_grad=True)
    F.silu(g).sum().backward()
    np.testing.assert_allclose(O.silu(g.detach().numpy()), F.silu(g).detach().numpy(), rtol=1e-14)
    np.testing.assert_allclose(O.silu_grad(g.detach().numpy()), g.grad.numpy(), rtol=1e-12, atol=1e-15)


# --------------------------------------------------------------- forward

def _bruteforce_forward(x, p):
    """Whole forward with explicit Python loops, from the page's equations."""
    B, T, D = x.shape
    H = p["wout"].shape[1]
    C = D // T

    def ln_row(v, gam, bet, eps):
        n = len(v)
        mu = sum(v) / n
        var = sum((vi - mu) ** 2 for vi in v) / n
        r = 1.0 / np.sqrt(var + eps)
        return [(v[k] - mu) * r * gam[k] + bet[k] for k in range(n)]

    def silu1(z):
        return z / (1.0 + np.exp(-z))

    a0 = [[ln_row(list(x[b, t]), p["gamma0"], p["beta0"], 1e-3) for t in range(T)] for b in range(B)]
    y = np.zeros((B, T, D))
    for b in range(B):
        out1 = []
        for i in range(T):
            s1 = [a0[b][k // C][i * C + k % C] + x[b, i, k] for k in range(D)]
            out1.append(ln_row(s1, p["gamma1"], p["beta1"], 1e-3))
        for t in range(T):
            z = [sum(out1[t][d] * p["w1"][t, d, n] for d in range(D)) + p["b1"][t, n] for n in range(2 * H)]
            u = ln_row(z[:H], p["lnx_w"], p["lnx_b"], 1e-5)
            gg = ln_row(z[H:], p["lng_w"], p["lng_b"], 1e-5)
            hid = [u[h] * silu1(gg[h]) for h in range(H)]
            o2 = [sum(hid[h] * p["wout"][t, h, d] for h in range(H)) + p["bout"][t, d] for d in range(D)]
            y[b, t] = ln_row([out1[t][d] + o2[d] for d in range(D)], p["gamma2"], p["beta2"], 1e-3)
    return y


def test_forward_matches_bruteforce_loops():
    inp = _inputs(I.shape_of(I.EXTRA_SHAPES["preflight"]))
    y, _ = O.forward(inp["x"], _params(inp))
    np.testing.assert_allclose(y, _bruteforce_forward(inp["x"], _params(inp)), rtol=1e-11, atol=1e-12)


def test_zero_w1_closed_form():
    # w1 = 0, b1 = 0 => Z = 0 => LN of a constant row is its bias (0) =>
    # hidden = 0 => output = norm2(out1 + bout); and dwout = 0.
    inp = _inputs(I.shape_of("c0"), ln="init")
    p = _params(inp)
    p["w1"] = np.zeros_like(p["w1"])
    p["b1"] = np.zeros_like(p["b1"])
    y, cache = O.forward(inp["x"], p)
    a0, _ = O.layer_norm(inp["x"], p["gamma0"], p["beta0"], 1e-3)
    out1, _ = O.layer_norm(O.token_mixer(a0) + inp["x"], p["gamma1"], p["beta1"], 1e-3)
    ref, _ = O.layer_norm(out1 + p["bout"][None], p["gamma2"], p["beta2"], 1e-3)
    np.testing.assert_array_equal(cache["hidden"], 0.0)
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-13)
    _, grads = O.backward(inp["dy"], cache, p)
    np.testing.assert_array_equal(grads["wout"], 0.0)


def test_beta0_gradient_vanishes_when_D_equals_T():
    # With D == T each token chunk is one column, so dbeta0[d] = sum over b, j
    # of ds1[b, d, j]: row sums of a LayerNorm backward, which are zero.
    inp = _inputs(I.Shape(B=3, T=8, D=8, H=16))
    _, _, grads = O.forward_backward(inp["x"], inp["dy"], _params(inp))
    assert np.abs(grads["beta0"]).max() <= 1e-13 * np.abs(grads["gamma0"]).max()
    inp = _inputs(I.Shape(B=3, T=4, D=8, H=16))           # C = 2: no longer zero
    _, _, grads = O.forward_backward(inp["x"], inp["dy"], _params(inp))
    assert np.abs(grads["beta0"]).max() > 1e-3 * np.abs(grads["gamma0"]).max()


def test_per_token_gemm_is_textbook_matmul():
    rng = np.random.default_rng(7)
    inp = rng.standard_normal((3, 2, 5))
    p = {"w1": rng.standard_normal((2, 5, 8)), "b1": rng.standard_normal((2, 8)),
         "wout": rng.standard_normal((2, 4, 5)), "bout": rng.standard_normal((2, 5)),
         "lnx_w": np.ones(4), "lnx_b": np.zeros(4), "lng_w": np.ones(4), "lng_b": np.zeros(4)}
    _, cache = O.dense_ffn_v2_forward(inp, p)
    for b in range(3):
        for t in range(2):
            for n in range(8):
                ref = sum(inp[b, t, d] * p["w1"][t, d, n] for d in range(5)) + p["b1"][t, n]
                assert abs(cache["Z"][b, t, n] - ref) < 1e-12


# --------------------------------------------------------------- torch autograd

def _torch_block(x, p):
    """Independent composition with torch float64 ops (test-only)."""
    B, T, D = x.shape
    H = p["wout"].shape[1]
    a0 = F.layer_norm(x, (D,), p["gamma0"], p["beta0"], 1e-3)
    m = a0.view(B, T, T, D // T).transpose(1, 2).reshape(B, T, D)
    out1 = F.layer_norm(m + x, (D,), p["gamma1"], p["beta1"], 1e-3)
    z = torch.bmm(out1.transpose(0, 1), p["w1"]) + p["b1"][:, None, :]       # [T,B,2H]
    u, g = torch.chunk(z, 2, dim=-1)
    hid = F.layer_norm(u, (H,), p["lnx_w"], p["lnx_b"], 1e-5) * F.silu(F.layer_norm(g, (H,), p["lng_w"], p["lng_b"], 1e-5))
    out2 = (torch.bmm(hid, p["wout"]) + p["bout"][:, None, :]).transpose(0, 1)
    return F.layer_norm(out1 + out2, (D,), p["gamma2"], p["beta2"], 1e-3)


@pytest.mark.parametrize("cfg", ["c0", "preflight", "public", "c1"])
def test_matches_torch_float64_autograd(cfg):
    shape = I.shape_of(I.EXTRA_SHAPES[cfg] if cfg in I.EXTRA_SHAPES else cfg)
    inp = _inputs(shape)
    p = _params(inp)
    y, dx, grads = O.forward_backward(inp["x"], inp["dy"], p)
    tp = {k: torch.from_numpy(v.copy()).requires_grad_(True) for k, v in p.items()}
    tx = torch.from_numpy(inp["x"].copy()).requires_grad_(True)
    ty = _torch_block(tx, tp)
    ty.backward(torch.from_numpy(inp["dy"]))
    np.testing.assert_allclose(y, ty.detach().numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dx, tx.grad.numpy(), rtol=1e-9, atol=1e-10)
    for k in I.PARAM_NAMES:
        ref = tp[k].grad.numpy()
        assert grads[k].shape == ref.shape, k
        err = np.linalg.norm(grads[k] - ref) / max(np.linalg.norm(ref), 1e-300)
        assert err < 1e-10, (k, err)


# --------------------------------------------------------------- finite differences

def _loss(x, dy, p):
    y, _ = O.forward(x, p)
    return float((dy * y).sum())


def test_central_finite_differences_c0():
    shape = I.shape_of("c0")
    inp = _inputs(shape)
    p = _params(inp)
    x, dy = inp["x"], inp["dy"]
    _, dx, grads = O.forward_backward(x, dy, p)
    grads = dict(grads, x=dx)
    rng = np.random.default_rng(11)
    h = 1e-6

    def perturbed(name, delta):
        if name == "x":
            return _loss(x + delta, dy, p)
        q = dict(p)
        q[name] = p[name] + delta
        return _loss(x, dy, q)

    for name in ("x",) + I.PARAM_NAMES:
        base = x if name == "x" else p[name]
        an = grads[name]
        scale = np.abs(an).max()
        # Directional derivative along one random direction.
        v = rng.standard_normal(base.shape)
        fd = (perturbed(name, h * v) - perturbed(name, -h * v)) / (2 * h)
        ad = float((an * v).sum())
        assert abs(fd - ad) <= 1e-7 * max(abs(ad), np.linalg.norm(an)), (name, fd, ad)
        # A few single entries.
        flat = rng.choice(base.size, size=min(8, base.size), replace=False)
        for f in flat:
            e = np.zeros(base.size)
            e[f] = 1.0
            e = e.reshape(base.shape)
            fd = (perturbed(name, h * e) - perturbed(name, -h * e)) / (2 * h)
            assert abs(fd - an.reshape(-1)[f]) <= 2e-7 * scale + 1e-9, (name, f, fd, an.reshape(-1)[f])


# --------------------------------------------------------------- planted mistakes

def _mutants():
    def ln_bwd_no_gamma(dout, gamma, stats):
        return O.__dict__["_orig_lnb"](dout, np.ones_like(gamma), stats)

    def ln_bwd_sign(dout, gamma, stats):
        _, rstd, xhat = stats
        g = gamma * dout
        dz = rstd * (g - g.mean(axis=-1, keepdims=True) + xhat * (g * xhat).mean(axis=-1, keepdims=True))
        lead = tuple(range(dout.ndim - 1))
        return dz, (dout * xhat).sum(axis=lead), dout.sum(axis=lead)

    def tm_wrong(a):
        B, T, D = a.shape
        return a.reshape(B, T, D // T, T).swapaxes(2, 3).reshape(B, T, D) if T > 1 else a

    def silu_grad_dropped(g):
        return O.sigmoid(g)

    def ln_eps_outside(z, gamma, beta, eps):
        mean = z.mean(axis=-1, keepdims=True)
        var = ((z - mean) ** 2).mean(axis=-1, keepdims=True)
        rstd = 1.0 / (np.sqrt(var) + eps)
        xhat = (z - mean) * rstd
        return xhat * gamma + beta, (mean, rstd, xhat)

    return {
        "layer_norm_backward": ln_bwd_no_gamma,
        "layer_norm_backward ": ln_bwd_sign,
        "token_mixer": tm_wrong,
        "silu_grad": silu_grad_dropped,
        "layer_norm": ln_eps_outside,
    }


@pytest.mark.parametrize("target", list(_mutants().keys()))
def test_pins_catch_planted_mistakes(target, monkeypatch):
    name = target.strip()
    monkeypatch.setitem(O.__dict__, "_orig_lnb", O.layer_norm_backward)
    monkeypatch.setattr(O, name, _mutants()[target])
    pins = [test_token_mix_worked_example,
            lambda: test_layer_norm_is_torch_layer_norm(1e-3),
            test_central_finite_differences_c0,
            lambda: test_matches_torch_float64_autograd("c0")]
    caught = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught > 0, f"no pin caught the planted mistake in {name}"


def test_chunked_oracle_equals_whole_batch():
    # The full-batch parity test runs the oracle on chunks of samples and sums
    # the parameter gradients; that must equal one call on the whole batch.
    import sys, os
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    from parity_util import oracle_outputs, oracle_outputs_chunked
    shape = I.Shape(B=5, T=4, D=16, H=32, dtype="f32")
    arrays = I.make_inputs(shape, ln_params="random")
    whole = oracle_outputs(arrays)
    parts = oracle_outputs_chunked(arrays, chunk=2)
    for k, v in whole.items():
        np.testing.assert_allclose(parts[k], v, rtol=1e-12, atol=1e-12 * max(1.0, np.abs(v).max()))
