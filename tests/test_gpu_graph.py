"""CUDA-graph replay of a whole step (rmx_graph_*): the replay computes
bitwise what rmx_forward + rmx_backward compute on the same buffers, also
after the inputs' values change between replays."""

import numpy as np
import pytest
import torch

from ffn_block_gb300 import binding as B
from ffn_block_gb300 import inputs as I
from ffn_block_gb300.device import RankMixerDevice

pytestmark = pytest.mark.gpu


def _outputs(blk):
    torch.cuda.synchronize()
    out = {"y": blk.y.clone(), "dx": blk.dx.clone()}
    out.update({n: g.clone() for n, g in blk.grads.items()})
    return out


@pytest.mark.parametrize("dims", [
    dict(B=64, T=16, D=256, H=512, dtype="bf16"),
    dict(B=130, T=8, D=128, H=384, dtype="f16"),
    dict(B=5, T=9, D=81, H=243, dtype="bf16"),     # padded rows
    dict(B=16, T=8, D=64, H=128, dtype="f32"),
    dict(B=16, T=8, D=64, H=128, dtype="tf32"),
], ids=lambda d: "B{B}_T{T}_D{D}_H{H}_{dtype}".format(**d))
def test_graph_replay_matches_direct_calls(dims):
    shape = I.Shape(**dims)
    blk = RankMixerDevice(shape, I.make_inputs(shape, ln_params="random"))
    blk.step()
    B.check(B.rmx_check())
    direct = _outputs(blk)
    for t in [blk.y, blk.dx, *blk.grads.values()]:
        t.fill_(float("nan"))
    g = B.rmx_graph_create(blk.cfg, blk.x, blk.dy, blk.c_params, blk.saved, blk.saved_bytes, blk.y, blk.dx,
                           blk.c_grads, blk.ws, blk.ws_bytes)
    try:
        stream = torch.cuda.Stream()
        before = B.rmx_launch_count()
        B.check(B.rmx_graph_launch(g, stream), "rmx_graph_launch")
        B.check(B.rmx_check(stream))
        assert B.rmx_launch_count() > before
        replay = _outputs(blk)
        for k in direct:
            assert torch.equal(replay[k], direct[k]), k
        # New input values in the same buffers: the replay follows them.
        x2 = I.make_inputs(shape, seed=I.DEFAULT_SEED + 5)["x"]
        blk.x.copy_(torch.from_numpy(np.ascontiguousarray(x2)).to(blk.x.device, blk.dtype))
        B.check(B.rmx_graph_launch(g, stream), "rmx_graph_launch")
        B.check(B.rmx_check(stream))
        replay2 = _outputs(blk)
        blk.step()
        B.check(B.rmx_check())
        direct2 = _outputs(blk)
        for k in direct2:
            assert torch.equal(replay2[k], direct2[k]), k
        assert not torch.equal(direct2["y"], direct["y"])
    finally:
        assert B.rmx_graph_destroy(g) == B.RMX_OK
