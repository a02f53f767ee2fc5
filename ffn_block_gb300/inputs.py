"""Seeded synthetic inputs for the RankMixer block.

This module only draws numbers: it holds none of the block's arithmetic, so
both the CUDA path (through the binding) and the float64 oracle can be fed
from it.

Recipe (page "Subgraph-fusion-based Mega-kernel Generation", section
"Weights and biases use the included he-uniform initializer"):

* parameters are drawn first, in the order w1, b1, wout, bout, each
  he-uniform: fan_in = product of every dimension but the last, values
  uniform in [-sqrt(6/fan_in), +sqrt(6/fan_in)];
* the input x is drawn after the parameters from the same stream
  (standard normal, seed 7101 by default, the public check's seed);
* the upstream gradient dy comes from a separate stream seeded seed+1000;
* outer LayerNorm gamma=1, beta=0; inner LayerNorm weight=1, bias=0
  ("init" mode).  Tests also use "random" mode, where every gamma/beta and
  inner weight/bias is drawn as well, so that a dropped or misplaced affine
  term cannot hide behind the identity initialisation;
* values are drawn in float32 and then rounded (round to nearest even) to the
  storage dtype.  The oracle receives exactly those rounded values.

Numbers come from numpy's PCG64 generator, not torch's CUDA generator.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

# Workloads.  c0/c1: strict fp32 contract; c2/c3: bf16 storage; c4: fp16
# storage with ragged sizes (B, D, H not multiples of 64, D/T = 30).
CONFIGS = {
    "c0": dict(B=2, T=8, D=64, H=128, dtype="f32"),
    "c1": dict(B=64, T=16, D=256, H=512, dtype="f32"),
    "c2": dict(B=256, T=32, D=512, H=1536, dtype="bf16"),
    "c3": dict(B=1024, T=64, D=1280, H=2560, dtype="bf16"),
    "c4": dict(B=1000, T=40, D=1200, H=3600, dtype="f16"),
}

# Small shapes from the page's public checks: (B,T,D,k) = (4,16,128,2) with
# seed 7101 and the CPU preflight shape (2,4,16,2).
EXTRA_SHAPES = {
    "public": dict(B=4, T=16, D=128, H=256),
    "preflight": dict(B=2, T=4, D=16, H=32),
}

PARAM_NAMES = (
    "w1", "b1", "wout", "bout",
    "gamma0", "beta0", "gamma1", "beta1", "gamma2", "beta2",
    "lnx_w", "lnx_b", "lng_w", "lng_b",
)

DEFAULT_SEED = 7101


@dataclass(frozen=True)
class Shape:
    B: int
    T: int
    D: int
    H: int
    dtype: str = "f32"

    @property
    def C(self) -> int:
        return self.D // self.T

    def param_shapes(self) -> dict:
        T, D, H = self.T, self.D, self.H
        return {
            "w1": (T, D, 2 * H), "b1": (T, 2 * H),
            "wout": (T, H, D), "bout": (T, D),
            "gamma0": (D,), "beta0": (D,), "gamma1": (D,), "beta1": (D,),
            "gamma2": (D,), "beta2": (D,),
            "lnx_w": (H,), "lnx_b": (H,), "lng_w": (H,), "lng_b": (H,),
        }


def shape_of(name_or_dict, dtype: str | None = None) -> Shape:
    d = dict(CONFIGS[name_or_dict]) if isinstance(name_or_dict, str) else dict(name_or_dict)
    if dtype is not None:
        d["dtype"] = dtype
    return Shape(**d)


def he_uniform(rng: np.random.Generator, shape) -> np.ndarray:
    fan_in = int(np.prod(shape[:-1])) if len(shape) > 1 else 1
    bound = np.float32(math.sqrt(6.0 / fan_in))
    u = rng.random(size=shape, dtype=np.float32)          # [0, 1)
    return (u * np.float32(2.0) - np.float32(1.0)) * bound


def round_to_storage(a: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to the storage dtype; returns float32 holding them."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    if dtype in ("f32", "tf32"):   # tf32: float32 storage (only the contractions differ)
        return a
    if dtype == "f16":
        return a.astype(np.float16).astype(np.float32)
    if dtype == "bf16":
        import torch
        return torch.from_numpy(a).to(torch.bfloat16).to(torch.float32).numpy()
    raise ValueError(f"unknown dtype {dtype}")


def make_inputs(shape: Shape, seed: int = DEFAULT_SEED, ln_params: str = "init",
                dy_rows=None) -> dict:
    """Return float32 numpy arrays already rounded to ``shape.dtype``.

    Keys: x, dy and every name in PARAM_NAMES.
    ``dy_rows``: if given, a list of sample indices b; dy is zeroed on every
    other sample (used to check full-size gradients on a few samples).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    ps = shape.param_shapes()
    out = {}
    for name in ("w1", "b1", "wout", "bout"):
        out[name] = he_uniform(rng, ps[name])
    if ln_params == "init":
        for name in ("gamma0", "gamma1", "gamma2", "lnx_w", "lng_w"):
            out[name] = np.ones(ps[name], np.float32)
        for name in ("beta0", "beta1", "beta2", "lnx_b", "lng_b"):
            out[name] = np.zeros(ps[name], np.float32)
    elif ln_params == "random":
        rng_ln = np.random.Generator(np.random.PCG64(seed + 2000))
        for name in ("gamma0", "gamma1", "gamma2", "lnx_w", "lng_w"):
            out[name] = rng_ln.uniform(0.5, 1.5, size=ps[name]).astype(np.float32)
        for name in ("beta0", "beta1", "beta2", "lnx_b", "lng_b"):
            out[name] = (0.2 * rng_ln.standard_normal(ps[name])).astype(np.float32)
    else:
        raise ValueError(ln_params)
    B, T, D = shape.B, shape.T, shape.D
    out["x"] = rng.standard_normal((B, T, D), dtype=np.float32)
    rng_dy = np.random.Generator(np.random.PCG64(seed + 1000))
    dy = rng_dy.standard_normal((B, T, D), dtype=np.float32)
    if dy_rows is not None:
        mask = np.zeros((B, 1, 1), np.float32)
        mask[list(dy_rows)] = 1.0
        dy = dy * mask
    out["dy"] = dy
    return {k: round_to_storage(v, shape.dtype) for k, v in out.items()}


def to_float64(inputs: dict) -> dict:
    return {k: np.asarray(v, dtype=np.float64) for k, v in inputs.items()}
