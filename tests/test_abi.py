"""C-ABI checks that need no GPU: the library loads, exports every function
include/rmx.h declares, and rejects bad arguments on the host before any CUDA
call."""

import ctypes
import os

import pytest

from ffn_block_gb300 import binding as B
from ffn_block_gb300 import inputs as I


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.LIB_PATH):
        from ffn_block_gb300 import build
        build.build()
    return B.lib()


def test_exports_every_declared_function(lib):
    names = B.header_functions()
    assert "rmx_forward" in names and "rmx_backward" in names
    for n in names:
        assert hasattr(lib, n), f"librmx.so does not export {n}"


def test_status_strings_and_version(lib):
    assert B.status_str(B.RMX_OK) == "RMX_OK"
    assert B.status_str(B.RMX_ERR_TIMEOUT) == "RMX_ERR_TIMEOUT"
    assert B.rmx_version() >= 100


def _expected_saved(s):
    e = 4 if s.dtype == "f32" else 2
    N = s.B * s.T
    up = lambda v: (v + 255) // 256 * 256
    total = 0
    tiles = (2 * s.H + 127) // 128     # Z statistics per 128-column group
    for n in (N * s.D * e, N * 2 * s.H * e, N * s.H * e, N * s.D * e, 10 * N * 4, N * tiles * 4 * 4, N * s.D * e):
        total = up(total + n)
    return total


@pytest.mark.parametrize("name", ["c0", "c1", "c2", "c3", "c4"])
def test_saved_bytes_layout(lib, name):
    s = I.shape_of(name)
    cfg = B.make_config(s.B, s.T, s.D, s.H, s.dtype)
    assert B.rmx_saved_bytes(cfg) == _expected_saved(s)
    assert B.rmx_workspace_bytes(cfg) > 0


@pytest.mark.parametrize("bad", [
    dict(B=-1, T=8, D=64, H=128), dict(B=2, T=0, D=64, H=128), dict(B=2, T=8, D=60, H=128),
    dict(B=2, T=8, D=64, H=0), dict(B=2, T=8, D=0, H=128)])
def test_invalid_config_rejected(lib, bad):
    cfg = B.make_config(dtype="f32", **bad)
    assert B.rmx_saved_bytes(cfg) == 0
    assert B.rmx_workspace_bytes(cfg) == 0
    p = B.rmx_params(*([0x1000] * 14))
    assert B.rmx_forward(cfg, 0x1000, p, 0x2000, 1 << 20, 0x3000) == B.RMX_ERR_INVALID_ARG


def test_bad_dtype_rejected(lib):
    cfg = B.rmx_config(2, 8, 64, 128, 7)
    assert B.rmx_saved_bytes(cfg) == 0


def test_null_and_misaligned_pointers(lib):
    cfg = B.make_config(2, 8, 64, 128, "f32")
    nbytes = B.rmx_saved_bytes(cfg)
    good = B.rmx_params(*([0x1000] * 14))
    nullp = B.rmx_params(*([0x1000] * 13 + [None]))
    mis = B.rmx_params(*([0x1000] * 13 + [0x1008]))
    assert B.rmx_forward(cfg, 0x1000, nullp, 0x2000, nbytes, 0x3000) == B.RMX_ERR_INVALID_ARG
    assert B.rmx_forward(cfg, 0x1000, mis, 0x2000, nbytes, 0x3000) == B.RMX_ERR_ALIGNMENT
    assert B.rmx_forward(cfg, 0x1004, good, 0x2000, nbytes, 0x3000) == B.RMX_ERR_ALIGNMENT
    assert B.rmx_forward(cfg, None, good, 0x2000, nbytes, 0x3000) == B.RMX_ERR_INVALID_ARG
    assert B.rmx_forward(cfg, 0x1000, good, 0x2000, nbytes, 0x1000) == B.RMX_ERR_INVALID_ARG  # x aliases y


def test_small_saved_buffer_rejected(lib):
    cfg = B.make_config(2, 8, 64, 128, "f32")
    nbytes = B.rmx_saved_bytes(cfg)
    p = B.rmx_params(*([0x1000] * 14))
    assert B.rmx_forward(cfg, 0x1000, p, 0x2000, nbytes - 1, 0x3000) == B.RMX_ERR_WORKSPACE
    g = B.rmx_grads(*([0x1000] * 14))
    ws = B.rmx_workspace_bytes(cfg)
    assert B.rmx_backward(cfg, 0x1000, 0x1100, 0x2000, nbytes, p, 0x3000, g, 0x4000, ws - 1) == B.RMX_ERR_WORKSPACE
    assert B.rmx_backward(cfg, 0x1000, 0x1100, 0x2000, nbytes, p, 0x3000, B.rmx_grads(*([None] * 14)),
                          0x4000, ws) == B.RMX_ERR_INVALID_ARG


def test_unsupported_row_width(lib):
    # The gate backward holds a whole FFN row per CTA: H above 3840 (k = 3 at
    # D = 1280, the widest the page's held-out domain reaches) is refused.
    cfg = B.make_config(2, 8, 64, 4096, "bf16")
    p = B.rmx_params(*([0x1000] * 14))
    assert B.rmx_forward(cfg, 0x1000, p, 0x2000, B.rmx_saved_bytes(cfg), 0x3000) == B.RMX_ERR_UNSUPPORTED


def test_padded_rows_reserve_their_copies(lib):
    # D = 36 is not a whole number of 16-byte bf16 vectors: the block runs on
    # copies padded to 40 columns (H = 72 -> 72), kept in `saved` (x, y and the
    # parameters) and in the scratch buffer (dy, dx and the gradients).
    e, Bn, T, D, H = 2, 3, 4, 36, 72
    cfg = B.make_config(Bn, T, D, H, "bf16")
    aligned = B.make_config(Bn, T, 40, H, "bf16")
    params_p = (T * 40 * 2 * H + T * 2 * H + T * H * 40 + T * 40 + 6 * 40 + 4 * H) * e
    acts_p = 2 * Bn * T * 40 * e
    assert B.rmx_saved_bytes(cfg) >= B.rmx_saved_bytes(aligned) + params_p + acts_p
    assert B.rmx_workspace_bytes(cfg) >= B.rmx_workspace_bytes(aligned) + params_p + acts_p


def test_empty_batch_forward_is_a_no_op(lib):
    cfg = B.make_config(0, 8, 64, 128, "bf16")
    p = B.rmx_params(*([0x1000] * 14))
    before = B.rmx_launch_count()
    assert B.rmx_forward(cfg, None, p, None, 0, None) == B.RMX_OK
    assert B.rmx_launch_count() == before


def test_host_step_rejects_missing_buffers(lib):
    cfg = B.make_config(2, 8, 64, 128, "f32")
    host = B.rmx_host_io(None, None, None, None)
    dev = B.rmx_device_io(0x1000, 0x1100, 0x1200, 0x1300)
    p = B.rmx_params(*([0x1000] * 14))
    g = B.rmx_grads(*([0x1000] * 14))
    assert B.rmx_step_host(cfg, host, dev, p, g, 0x2000, 1 << 20, 0x3000, 1 << 20) == B.RMX_ERR_INVALID_ARG


def test_test_hooks_validate_arguments(lib):
    assert B.rmx_test_bounded_wait(0) == B.RMX_ERR_INVALID_ARG
    assert B.rmx_test_gemm(3, "bf16", 8, 8, 8, 1, 0x1000, 0x1000, 0x1000) == B.RMX_ERR_INVALID_ARG
    assert B.rmx_test_gemm(0, "bf16", 8, 8, 8, 1, 0x1008, 0x1000, 0x1000) == B.RMX_ERR_ALIGNMENT


def test_graph_entry_points_validate_arguments(lib):
    import ctypes
    assert B.lib().rmx_graph_create(None, None, None, None, None, 0, None, None, None, None, 0, None) == \
        B.RMX_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    bad = B.make_config(2, 3, 64, 128, "bf16")      # D % T != 0
    p = B.rmx_params(*([0x1000] * 14))
    g = B.rmx_grads(*([0x1000] * 14))
    assert B.lib().rmx_graph_create(ctypes.byref(bad), 0x1000, 0x1000, ctypes.byref(p), 0x1000, 1 << 20, 0x1000,
                                    0x1000, ctypes.byref(g), 0x1000, 1 << 20, ctypes.byref(h)) == B.RMX_ERR_INVALID_ARG
    assert h.value is None
    assert B.rmx_graph_launch(None) == B.RMX_ERR_INVALID_ARG
    assert B.rmx_graph_destroy(None) == B.RMX_OK
