"""ctypes binding of libds4moe.so (argument marshalling only; every step runs in the library).

The names mirror the C ABI in include/ds4moe.h. Pointers are plain integers (for example
``tensor.data_ptr()``) or numpy arrays, which are passed by address and must stay alive for
the duration of the call. Streams are raw cudaStream_t values (``torch.cuda.current_stream()
.cuda_stream``); 0 is the legacy default stream.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libds4moe.so")

DS4MOE_OK = 0
DS4MOE_ERR_INVALID_ARG = -1
DS4MOE_ERR_UNSUPPORTED_FORMAT = -2
DS4MOE_ERR_DEVICE_MISMATCH = -3
DS4MOE_ERR_CAPACITY = -4
DS4MOE_ERR_OOM = -5
DS4MOE_ERR_CUDA = -6

DS4MOE_FMT_Q8_0 = 0
DS4MOE_FMT_Q2_K = 1
FORMATS = {"q8_0": DS4MOE_FMT_Q8_0, "q2_k": DS4MOE_FMT_Q2_K}

EXPORTED = ("ds4moe_create", "ds4moe_create_subset", "ds4moe_forward", "ds4moe_forward_ex", "ds4moe_forward_host",
            "ds4moe_get_route", "ds4moe_get_stats", "ds4moe_device_bytes",
            "ds4moe_launches_per_forward", "ds4moe_set_profiling", "ds4moe_get_phase_times", "ds4moe_route_noalloc",
            "ds4moe_set_test_stall",
            "ds4moe_destroy", "ds4moe_last_error")
DS4MOE_NOALLOC_MAX_LOGITS = 262144


class ds4moe_shapes(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("f_routed", ctypes.c_int32), ("f_shared", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("fmt_gate_up", ctypes.c_int32), ("fmt_down", ctypes.c_int32), ("fmt_shared", ctypes.c_int32),
                ("has_bias", ctypes.c_int32), ("hash_vocab", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
                ("device", ctypes.c_int32), ("reserved", ctypes.c_int32), ("workspace_limit", ctypes.c_int64)]


class ds4moe_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("router_w", "router_b", "gate", "up", "down", "shared_gate",
                                               "shared_up", "shared_down", "hash_table")]


class ds4moe_stats(ctypes.Structure):
    _fields_ = [("n_tokens", ctypes.c_int32), ("distinct_experts", ctypes.c_int32),
                ("error_flags", ctypes.c_int32), ("reserved", ctypes.c_int32), ("counts", ctypes.c_int32 * 256)]


class Ds4MoeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"ds4moe error {code}: {msg}")
        self.code = code


_lib = None


def lib() -> ctypes.CDLL:
    """Loads the in-tree library; raises if it has not been built (there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with quantized_moe_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        L.ds4moe_create.argtypes = [ctypes.POINTER(ds4moe_weights), ctypes.POINTER(ds4moe_shapes), ctypes.POINTER(vp)]
        L.ds4moe_create.restype = ctypes.c_int
        L.ds4moe_create_subset.argtypes = [ctypes.POINTER(ds4moe_weights), ctypes.POINTER(ds4moe_shapes), vp, i32,
                                           i32, ctypes.POINTER(vp)]
        L.ds4moe_create_subset.restype = ctypes.c_int
        L.ds4moe_forward.argtypes = [vp, vp, i32, vp, vp]
        L.ds4moe_forward.restype = ctypes.c_int
        L.ds4moe_forward_ex.argtypes = [vp, vp, i32, vp, i32, vp, vp]
        L.ds4moe_forward_ex.restype = ctypes.c_int
        L.ds4moe_forward_host.argtypes = [vp, vp, i32, vp, i32, vp, vp]
        L.ds4moe_forward_host.restype = ctypes.c_int
        L.ds4moe_get_route.argtypes = [vp, vp, vp, i32]
        L.ds4moe_get_route.restype = ctypes.c_int
        L.ds4moe_get_stats.argtypes = [vp, ctypes.POINTER(ds4moe_stats)]
        L.ds4moe_get_stats.restype = ctypes.c_int
        L.ds4moe_device_bytes.argtypes = [vp]
        L.ds4moe_device_bytes.restype = i64
        L.ds4moe_launches_per_forward.argtypes = [vp, i32]
        L.ds4moe_launches_per_forward.restype = i32
        L.ds4moe_set_profiling.argtypes = [vp, i32]
        L.ds4moe_set_profiling.restype = ctypes.c_int
        L.ds4moe_get_phase_times.argtypes = [vp, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_char_p), i32,
                                             ctypes.POINTER(i32)]
        L.ds4moe_get_phase_times.restype = ctypes.c_int
        L.ds4moe_route_noalloc.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp]
        L.ds4moe_route_noalloc.restype = ctypes.c_int
        L.ds4moe_set_test_stall.argtypes = [vp, i32]
        L.ds4moe_set_test_stall.restype = ctypes.c_int
        L.ds4moe_destroy.argtypes = [vp]
        L.ds4moe_destroy.restype = None
        L.ds4moe_last_error.argtypes = []
        L.ds4moe_last_error.restype = ctypes.c_char_p
        _lib = L
    return _lib


def ds4moe_last_error() -> str:
    return lib().ds4moe_last_error().decode()


def _check(rc: int) -> None:
    if rc != DS4MOE_OK:
        raise Ds4MoeError(rc, ds4moe_last_error())


def _ptr(a) -> Optional[int]:
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if isinstance(a, np.ndarray):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("arrays must be C-contiguous")
        return a.ctypes.data
    if hasattr(a, "data_ptr"):
        return a.data_ptr()
    raise TypeError(f"cannot take the address of {type(a)}")


def make_shapes(d, f_routed, f_shared, n_experts, top_k, n_shared, fmt_gate_up, fmt_down, fmt_shared,
                has_bias, hash_vocab, max_tokens, device=0, workspace_limit=0) -> ds4moe_shapes:
    fm = lambda f: FORMATS[f] if isinstance(f, str) else int(f)
    return ds4moe_shapes(d, f_routed, f_shared, n_experts, top_k, n_shared, fm(fmt_gate_up), fm(fmt_down),
                         fm(fmt_shared), int(bool(has_bias)), hash_vocab, max_tokens, device, 0, workspace_limit)


def make_weights(router_w, router_b, gate, up, down, shared_gate=None, shared_up=None, shared_down=None,
                 hash_table=None) -> ds4moe_weights:
    return ds4moe_weights(*(_ptr(a) for a in (router_w, router_b, gate, up, down, shared_gate, shared_up,
                                               shared_down, hash_table)))


def ds4moe_create(weights: ds4moe_weights, shapes: ds4moe_shapes) -> int:
    h = ctypes.c_void_p()
    _check(lib().ds4moe_create(ctypes.byref(weights), ctypes.byref(shapes), ctypes.byref(h)))
    return h.value


def ds4moe_create_subset(weights: ds4moe_weights, shapes: ds4moe_shapes, owned, include_shared: bool) -> int:
    """A handle holding only the routed experts in `owned` (see the header); returns its address."""
    ids = np.ascontiguousarray(np.asarray(owned, dtype=np.int32).reshape(-1))
    buf = ids if ids.size else np.zeros(1, np.int32)  # a valid address even for an empty list
    h = ctypes.c_void_p()
    _check(lib().ds4moe_create_subset(ctypes.byref(weights), ctypes.byref(shapes), buf.ctypes.data, int(ids.size),
                                      int(bool(include_shared)), ctypes.byref(h)))
    return h.value


def ds4moe_forward(h: int, x, n_tokens: int, out, stream: int = 0) -> None:
    _check(lib().ds4moe_forward(h, _ptr(x), n_tokens, _ptr(out), stream))


def ds4moe_forward_ex(h: int, x, n_tokens: int, token_ids, n_hash: int, out, stream: int = 0) -> None:
    _check(lib().ds4moe_forward_ex(h, _ptr(x), n_tokens, _ptr(token_ids), n_hash, _ptr(out), stream))


def ds4moe_forward_host(h: int, x, n_tokens: int, token_ids, n_hash: int, out, stream: int = 0) -> None:
    _check(lib().ds4moe_forward_host(h, _ptr(x), n_tokens, _ptr(token_ids), n_hash, _ptr(out), stream))


def ds4moe_get_route(h: int, n_tokens: int, top_k: int):
    idx = np.zeros((n_tokens, top_k), np.int32)
    w = np.zeros((n_tokens, top_k), np.float32)
    _check(lib().ds4moe_get_route(h, idx.ctypes.data, w.ctypes.data, n_tokens))
    return idx, w


def ds4moe_get_stats(h: int) -> dict:
    st = ds4moe_stats()
    _check(lib().ds4moe_get_stats(h, ctypes.byref(st)))
    return dict(n_tokens=st.n_tokens, distinct_experts=st.distinct_experts, error_flags=st.error_flags,
                counts=np.array(st.counts[:], dtype=np.int32))


def ds4moe_device_bytes(h: int) -> int:
    return lib().ds4moe_device_bytes(h)


def ds4moe_launches_per_forward(h: int, n_tokens: int) -> int:
    return lib().ds4moe_launches_per_forward(h, n_tokens)


def ds4moe_set_profiling(h: int, enable: bool) -> None:
    _check(lib().ds4moe_set_profiling(h, int(bool(enable))))


def ds4moe_get_phase_times(h: int) -> list:
    """[(launch name, stream milliseconds)] of the last profiled forward."""
    cap = 16
    ms = (ctypes.c_float * cap)()
    names = (ctypes.c_char_p * cap)()
    n = ctypes.c_int32()
    _check(lib().ds4moe_get_phase_times(h, ms, names, cap, ctypes.byref(n)))
    return [(names[i].decode(), float(ms[i])) for i in range(min(n.value, cap))]


def ds4moe_route_noalloc(router_w, router_b, x, n_tokens: int, d: int, n_experts: int, top_k: int, idx, w,
                         stream: int = 0) -> None:
    """Routing without any device allocation (for callers that cannot allocate); see the header."""
    _check(lib().ds4moe_route_noalloc(_ptr(router_w), _ptr(router_b), _ptr(x), n_tokens, d, n_experts, top_k,
                                      _ptr(idx), _ptr(w), stream))


def ds4moe_set_test_stall(h: int, stage: int) -> None:
    """Test hook: the next batched forward's GEMM withholds one arrival and its waits give up (see the header)."""
    _check(lib().ds4moe_set_test_stall(h, stage))


def ds4moe_destroy(h: Optional[int]) -> None:
    lib().ds4moe_destroy(h)
