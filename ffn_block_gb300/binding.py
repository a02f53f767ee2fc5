"""ctypes binding of librmx.so: the C ABI of include/rmx.h, same names.

Argument marshalling only: every step of the block runs in the library's CUDA
kernels.  Pointer arguments accept a torch tensor (its data_ptr()), an int
address or None; stream arguments accept a torch.cuda.Stream, an int handle
or None (the legacy default stream).  There is no fallback: if the library
has not been built, every call raises.
"""

from __future__ import annotations

import ctypes
import os
import re

from .inputs import PARAM_NAMES

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "librmx.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "rmx.h")

RMX_OK = 0
RMX_ERR_INVALID_ARG = 1
RMX_ERR_UNSUPPORTED = 2
RMX_ERR_ALIGNMENT = 3
RMX_ERR_WORKSPACE = 4
RMX_ERR_CUDA = 5
RMX_ERR_TIMEOUT = 6

# "tf32": float32 storage, contractions on the tensor cores with TF32 operands.
DTYPE_CODES = {"f32": 0, "bf16": 1, "f16": 2, "tf32": 3}


class RmxError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_str(status)}" if what else status_str(status))


class rmx_config(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("D", ctypes.c_int),
                ("H", ctypes.c_int), ("dtype", ctypes.c_int)]


class rmx_params(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in PARAM_NAMES]


class rmx_grads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in PARAM_NAMES]


class rmx_host_io(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("dy", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("dx", ctypes.c_void_p)]


class rmx_device_io(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("dy", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("dx", ctypes.c_void_p)]


_VP, _SZ, _I, _P = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.POINTER
_SIGNATURES = {
    "rmx_saved_bytes": (_SZ, [_P(rmx_config)]),
    "rmx_workspace_bytes": (_SZ, [_P(rmx_config)]),
    "rmx_forward": (_I, [_P(rmx_config), _VP, _P(rmx_params), _VP, _SZ, _VP, _VP]),
    "rmx_backward": (_I, [_P(rmx_config), _VP, _VP, _VP, _SZ, _P(rmx_params), _VP, _P(rmx_grads),
                          _VP, _SZ, _VP]),
    "rmx_step_host": (_I, [_P(rmx_config), _P(rmx_host_io), _P(rmx_device_io), _P(rmx_params),
                           _P(rmx_grads), _VP, _SZ, _VP, _SZ, _VP]),
    "rmx_check": (_I, [_VP]),
    "rmx_status_str": (ctypes.c_char_p, [_I]),
    "rmx_version": (_I, []),
    "rmx_launch_count": (ctypes.c_longlong, []),
    "rmx_profile_enable": (_I, [_I]),
    "rmx_profile_select": (_I, [ctypes.c_char_p]),
    "rmx_profile_read": (_I, [_P(ctypes.c_char_p), _P(ctypes.c_longlong), _P(ctypes.c_double), _I]),
    "rmx_test_bounded_wait": (_I, [_I, _VP]),
    "rmx_test_gemm": (_I, [_I, _I, _I, _I, _I, _I, _VP, _VP, _VP, _VP]),
    "rmx_ln2_backward_noalloc": (_I, [_P(rmx_config), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "rmx_graph_create": (_I, [_P(rmx_config), _VP, _VP, _P(rmx_params), _VP, _SZ, _VP, _VP, _P(rmx_grads), _VP,
                              _SZ, _P(_VP)]),
    "rmx_graph_launch": (_I, [_VP, _VP]),
    "rmx_graph_destroy": (_I, [_VP]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """Load librmx.so once; raise if it is missing (no fallback path)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m ffn_block_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def header_functions(path: str = HEADER_PATH) -> list[str]:
    """Names of every function declared in include/rmx.h."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rmx_[a-z0-9_]+)\s*\(", text)))


def _ptr(v) -> int | None:
    if v is None:
        return None
    if isinstance(v, int):
        return v
    return v.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def make_config(B: int, T: int, D: int, H: int, dtype: str | int) -> rmx_config:
    code = DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype)
    return rmx_config(B, T, D, H, code)


def make_params(tensors: dict) -> rmx_params:
    return rmx_params(*[_ptr(tensors[n]) for n in PARAM_NAMES])


def make_grads(tensors: dict) -> rmx_grads:
    return rmx_grads(*[_ptr(tensors[n]) for n in PARAM_NAMES])


def status_str(status: int) -> str:
    return lib().rmx_status_str(status).decode()


def check(status: int, what: str = "") -> None:
    if status != RMX_OK:
        raise RmxError(status, what)


# ------------------------------------------------------------------ the ABI calls

def rmx_saved_bytes(cfg: rmx_config) -> int:
    return lib().rmx_saved_bytes(ctypes.byref(cfg))


def rmx_workspace_bytes(cfg: rmx_config) -> int:
    return lib().rmx_workspace_bytes(ctypes.byref(cfg))


def rmx_forward(cfg, x, params: rmx_params, saved, saved_bytes: int, y, stream=None) -> int:
    return lib().rmx_forward(ctypes.byref(cfg), _ptr(x), ctypes.byref(params), _ptr(saved),
                             saved_bytes, _ptr(y), _stream(stream))


def rmx_backward(cfg, x, dy, saved, saved_bytes: int, params: rmx_params, dx, grads: rmx_grads,
                 ws, ws_bytes: int, stream=None) -> int:
    return lib().rmx_backward(ctypes.byref(cfg), _ptr(x), _ptr(dy), _ptr(saved), saved_bytes,
                              ctypes.byref(params), _ptr(dx), ctypes.byref(grads), _ptr(ws), ws_bytes,
                              _stream(stream))


def rmx_step_host(cfg, host: rmx_host_io, dev: rmx_device_io, params: rmx_params, grads: rmx_grads,
                  saved, saved_bytes: int, ws, ws_bytes: int, stream=None) -> int:
    return lib().rmx_step_host(ctypes.byref(cfg), ctypes.byref(host), ctypes.byref(dev),
                               ctypes.byref(params), ctypes.byref(grads), _ptr(saved), saved_bytes,
                               _ptr(ws), ws_bytes, _stream(stream))


def rmx_check(stream=None) -> int:
    return lib().rmx_check(_stream(stream))


def rmx_version() -> int:
    return lib().rmx_version()


def rmx_launch_count() -> int:
    return lib().rmx_launch_count()


def rmx_profile_enable(on: bool) -> int:
    return lib().rmx_profile_enable(1 if on else 0)


def rmx_profile_select(name) -> int:
    return lib().rmx_profile_select(name.encode() if name else None)


def rmx_profile_read(cap: int = 64) -> dict:
    names = (ctypes.c_char_p * cap)()
    launches = (ctypes.c_longlong * cap)()
    total = (ctypes.c_double * cap)()
    n = lib().rmx_profile_read(names, launches, total, cap)
    return {names[i].decode(): (int(launches[i]), float(total[i])) for i in range(min(n, cap))}


def rmx_test_bounded_wait(limit_us: int, stream=None) -> int:
    return lib().rmx_test_bounded_wait(limit_us, _stream(stream))


def rmx_test_gemm(kind: int, dtype, M: int, N: int, K: int, G: int, A, Bm, C, stream=None) -> int:
    code = DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype)
    return lib().rmx_test_gemm(kind, code, M, N, K, G, _ptr(A), _ptr(Bm), _ptr(C), _stream(stream))


def rmx_ln2_backward_noalloc(cfg, dy, s2, mean2, rstd2, gamma2, ds2, dgamma2, dbeta2, dbout,
                             stream=None) -> int:
    """norm2 backward with the library's fixed scratch array (no allocation)."""
    return lib().rmx_ln2_backward_noalloc(ctypes.byref(cfg), _ptr(dy), _ptr(s2), _ptr(mean2), _ptr(rstd2),
                                          _ptr(gamma2), _ptr(ds2), _ptr(dgamma2), _ptr(dbeta2), _ptr(dbout),
                                          _stream(stream))


def rmx_graph_create(cfg, x, dy, params: rmx_params, saved, saved_bytes: int, y, dx, grads: rmx_grads, ws,
                     ws_bytes: int) -> int:
    """Returns an opaque graph handle (an int); raises on failure."""
    h = ctypes.c_void_p()
    check(lib().rmx_graph_create(ctypes.byref(cfg), _ptr(x), _ptr(dy), ctypes.byref(params), _ptr(saved),
                                 saved_bytes, _ptr(y), _ptr(dx), ctypes.byref(grads), _ptr(ws), ws_bytes,
                                 ctypes.byref(h)), "rmx_graph_create")
    return h.value


def rmx_graph_launch(g: int, stream=None) -> int:
    return lib().rmx_graph_launch(g, _stream(stream))


def rmx_graph_destroy(g: int) -> int:
    return lib().rmx_graph_destroy(g)
