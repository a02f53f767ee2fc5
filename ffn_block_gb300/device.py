"""Device buffers of one RankMixer block, kept in torch CUDA memory.

torch provides the memory and the streams; every step of the block runs in
librmx.so through the C ABI (``binding``).
"""

from __future__ import annotations

import numpy as np
import torch

from . import binding as B
from .inputs import PARAM_NAMES, Shape

TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16, "tf32": torch.float32}


def _upload(a: np.ndarray, dt: torch.dtype, device) -> torch.Tensor:
    # Values are already rounded to the storage type, so the cast is exact.
    return torch.from_numpy(np.ascontiguousarray(a)).to(device).to(dt).contiguous()


def _ptr_or_none(t: torch.Tensor):
    return t if t.numel() > 0 else None


class RankMixerDevice:
    """Parameters, input, upstream gradient and every output of one block."""

    def __init__(self, shape: Shape, arrays: dict, device="cuda"):
        self.shape = shape
        self.device = torch.device(device)
        self.cfg = B.make_config(shape.B, shape.T, shape.D, shape.H, shape.dtype)
        dt = TORCH_DTYPES[shape.dtype]
        self.dtype = dt
        self.params = {n: _upload(arrays[n], dt, self.device) for n in PARAM_NAMES}
        self.x = _upload(arrays["x"], dt, self.device)
        self.dy = _upload(arrays["dy"], dt, self.device)
        self.y = torch.empty_like(self.x)
        self.dx = torch.empty_like(self.x)
        self.grads = {n: torch.empty_like(self.params[n]) for n in PARAM_NAMES}
        self.saved_bytes = B.rmx_saved_bytes(self.cfg)
        self.ws_bytes = B.rmx_workspace_bytes(self.cfg)
        self.saved = torch.empty(max(self.saved_bytes, 1), dtype=torch.uint8, device=self.device)
        self.ws = torch.empty(max(self.ws_bytes, 1), dtype=torch.uint8, device=self.device)
        self.c_params = B.make_params(self.params)
        self.c_grads = B.make_grads(self.grads)

    def forward(self, stream=None) -> None:
        B.check(B.rmx_forward(self.cfg, _ptr_or_none(self.x), self.c_params, self.saved, self.saved_bytes,
                              _ptr_or_none(self.y), stream), "rmx_forward")

    def backward(self, stream=None) -> None:
        B.check(B.rmx_backward(self.cfg, _ptr_or_none(self.x), _ptr_or_none(self.dy), self.saved,
                               self.saved_bytes, self.c_params, _ptr_or_none(self.dx), self.c_grads,
                               self.ws, self.ws_bytes, stream), "rmx_backward")

    def step(self, stream=None) -> None:
        self.forward(stream)
        self.backward(stream)

    def results(self) -> dict:
        """y, dx and every gradient as float64 numpy arrays (synchronises)."""
        torch.cuda.synchronize(self.device)
        out = {"y": self.y, "dx": self.dx}
        out.update({n: self.grads[n] for n in PARAM_NAMES})
        return {k: v.detach().float().cpu().numpy().astype(np.float64) for k, v in out.items()}
