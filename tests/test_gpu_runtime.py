"""Runtime behaviour of the CUDA path: bitwise determinism, no writes outside
the buffers it is given, the bounded-wait error path, the host-memory
end-to-end entry point and the per-kernel profiler."""

import numpy as np
import pytest
import torch

from ffn_block_gb300 import binding as B
from ffn_block_gb300 import inputs as I
from ffn_block_gb300.device import RankMixerDevice

from parity_util import TOL, compare, oracle_outputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dims,dtype", [
    (dict(B=64, T=16, D=256, H=512), "f32"),
    (dict(B=96, T=8, D=240, H=360), "f16"),
    (dict(B=256, T=32, D=512, H=1536), "bf16"),
])
def test_repeated_steps_are_bitwise_identical(dims, dtype):
    shape = I.Shape(dtype=dtype, **dims)
    blk = RankMixerDevice(shape, I.make_inputs(shape, ln_params="random"))
    blk.step()
    first = {k: v.clone() for k, v in [("y", blk.y), ("dx", blk.dx)] + list(blk.grads.items())}
    for _ in range(2):
        blk.step()
    B.check(B.rmx_check())
    for k, v in [("y", blk.y), ("dx", blk.dx)] + list(blk.grads.items()):
        assert torch.equal(v, first[k]), k


GUARD = 4096  # bytes of canary on each side of every buffer the library writes
PATTERN = 0xA5


def _guarded_like(t: torch.Tensor):
    nbytes = t.numel() * t.element_size()
    raw = torch.full((nbytes + 2 * GUARD,), PATTERN, dtype=torch.uint8, device=t.device)
    view = raw[GUARD:GUARD + nbytes].view(t.dtype).view(t.shape)
    return raw, view


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_no_writes_outside_given_buffers(dtype):
    shape = I.Shape(B=37, T=8, D=240, H=360, dtype=dtype)   # ragged tails everywhere
    arrays = I.make_inputs(shape, ln_params="random")
    blk = RankMixerDevice(shape, arrays)
    raws = []
    for name in ("y", "dx"):
        raw, view = _guarded_like(blk.x)
        raws.append(raw)
        setattr(blk, name, view)
    for n in list(blk.grads):
        raw, view = _guarded_like(blk.grads[n])
        raws.append(raw)
        blk.grads[n] = view
    raw, view = _guarded_like(blk.saved)
    raws.append(raw)
    blk.saved = view
    raw, view = _guarded_like(blk.ws)
    raws.append(raw)
    blk.ws = view
    blk.c_grads = B.make_grads(blk.grads)
    blk.step()
    B.check(B.rmx_check())
    for raw in raws:
        head, tail = raw[:GUARD], raw[-GUARD:]
        assert torch.all(head == PATTERN).item() and torch.all(tail == PATTERN).item()
    compare(blk.results(), oracle_outputs(arrays), TOL[dtype])


def test_bounded_wait_reports_timeout_and_context_survives():
    assert B.rmx_check() == B.RMX_OK
    assert B.rmx_test_bounded_wait(20_000) == B.RMX_OK      # 20 ms limit
    assert B.rmx_check() == B.RMX_ERR_TIMEOUT
    assert B.rmx_check() == B.RMX_OK                        # the word is cleared
    shape = I.shape_of("c0")
    arrays = I.make_inputs(shape)
    blk = RankMixerDevice(shape, arrays)
    blk.step()
    assert B.rmx_check() == B.RMX_OK
    compare(blk.results(), oracle_outputs(arrays), TOL["f32"])


# x is uploaded in four chunks of samples (uneven or empty chunks when B is
# not a multiple of four); padded rows take the whole-batch path.
@pytest.mark.parametrize("dims", [
    dict(B=16, T=8, D=128, H=256, dtype="f32"),
    dict(B=16, T=8, D=128, H=256, dtype="bf16"),
    dict(B=3, T=8, D=128, H=256, dtype="bf16"),
    dict(B=7, T=16, D=64, H=192, dtype="f16"),
    dict(B=6, T=9, D=81, H=243, dtype="bf16"),
    dict(B=5, T=8, D=64, H=128, dtype="tf32"),
], ids=lambda d: "B{B}_T{T}_D{D}_H{H}_{dtype}".format(**d))
def test_host_memory_step_matches_device_step(dims):
    shape = I.Shape(**dims)
    arrays = I.make_inputs(shape, ln_params="random")
    blk = RankMixerDevice(shape, arrays)
    blk.step()
    ref = blk.results()
    hx = blk.x.cpu().pin_memory()
    hdy = blk.dy.cpu().pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    hdx = torch.empty_like(hx).pin_memory()
    staging = [torch.empty_like(blk.x) for _ in range(4)]   # device x, dy, y, dx
    dev = B.rmx_device_io(*[t.data_ptr() for t in staging])
    host = B.rmx_host_io(hx.data_ptr(), hdy.data_ptr(), hy.data_ptr(), hdx.data_ptr())
    stream = torch.cuda.Stream()
    B.check(B.rmx_step_host(blk.cfg, host, dev, blk.c_params, blk.c_grads, blk.saved, blk.saved_bytes,
                            blk.ws, blk.ws_bytes, stream), "rmx_step_host")
    B.check(B.rmx_check(stream))
    assert np.array_equal(hy.float().numpy(), ref["y"])
    assert np.array_equal(hdx.float().numpy(), ref["dx"])


def test_profiler_counts_every_launch():
    shape = I.shape_of("c1")
    blk = RankMixerDevice(shape, I.make_inputs(shape))
    B.rmx_profile_read()                     # drop anything recorded earlier
    before = B.rmx_launch_count()
    B.rmx_profile_enable(True)
    try:
        blk.step()
    finally:
        B.rmx_profile_enable(False)
    prof = B.rmx_profile_read()
    launched = B.rmx_launch_count() - before
    assert sum(n for n, _ in prof.values()) == launched
    # c1 is the strict fp32 contract: its contractions run on the CUDA cores.
    assert {"gemm1_fwd.ffma", "gemm2_fwd.ffma", "gemm1_wgrad.ffma", "gemm2_dgrad.ffma", "ln01_fwd", "ln1_bwd",
            "gate_bwd", "ln0_bwd_gather"} <= set(prof)
    assert all(ms >= 0.0 for _, ms in prof.values())


def test_profiler_select_times_one_kernel():
    shape = I.shape_of("c1")
    blk = RankMixerDevice(shape, I.make_inputs(shape))
    B.rmx_profile_read()
    before = B.rmx_launch_count()
    B.rmx_profile_select("gate_bwd")
    B.rmx_profile_enable(True)
    try:
        blk.step()
    finally:
        B.rmx_profile_enable(False)
        B.rmx_profile_select(None)
    prof = B.rmx_profile_read()
    assert set(prof) == {"gate_bwd"} and prof["gate_bwd"][0] == 1
    assert B.rmx_launch_count() - before > 1  # every launch is still counted
