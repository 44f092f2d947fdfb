"""Python binding of libgdpa (the C ABI in include/gdpa.h).

Argument marshalling only: every step of the forward pass runs in the CUDA
library.  Functions keep the C names.  Device tensors may be torch tensors or
raw integer addresses; host arrays are numpy arrays.  A non-OK status raises
:class:`GdpaError`.  If ``libgdpa.so`` has not been built the import of the
library fails loudly -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdpa.so")

GDPA_ACT_SOFTMAX = 0
GDPA_ACT_GELU_TANH = 1

GDPA_ROUTE_SFU = 0
GDPA_ROUTE_ALU = 1

GDPA_OK = 0
GDPA_ERR_INVALID_ARG = 1
GDPA_ERR_UNSUPPORTED = 2
GDPA_ERR_CUDA = 3
GDPA_ERR_DEVICE_TIMEOUT = 4
GDPA_ERR_NO_MEMORY = 5

# Every symbol include/gdpa.h declares.
EXPORTS = ("gdpa_fwd", "gdpa_fwd_async", "gdpa_fwd_lse", "gdpa_fwd_sliding", "gdpa_fwd_mx", "gdpa_fwd_mxfp8", "gdpa_bwd", "gdpa_bwd_sliding", "gdpa_fwd_noalloc", "gdpa_plan_create", "gdpa_plan_create_sliding", "gdpa_fwd_planned", "gdpa_plan_destroy", "gdpa_plan_num_items",
           "gdpa_plan_num_ctas", "gdpa_fwd_host", "gdpa_plan_enumerate", "gdpa_act_eval", "gdpa_set_act_route",
           "gdpa_get_act_route", "gdpa_device_status", "gdpa_wait_selftest", "gdpa_status_string", "gdpa_version")


class GdpaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s failed: %s" % (where, gdpa_status_string(code)))


class WorkItem(ctypes.Structure):
    _fields_ = [("seq", ctypes.c_int32), ("head", ctypes.c_int32), ("q0", ctypes.c_int32), ("kv0", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libgdpa.so (raises if it was never built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError("libgdpa.so is not built (%s); run jagged_attention_recommender_gb300.build" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    P, I, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    L.gdpa_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, F, P, P]
    L.gdpa_fwd_async.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, F, P, P]
    L.gdpa_fwd_noalloc.argtypes = [P, P, P, P, P, I, I, I, I, I, F, P, P]
    L.gdpa_fwd_lse.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, F, P, P, P]
    L.gdpa_fwd_sliding.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, F, P, P, P]
    L.gdpa_fwd_mx.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, F, P, P, P]
    L.gdpa_fwd_mxfp8.argtypes = [P, P, P, P, P, P, P, P, P, P, I, I, I, I, F, P, P, P]
    L.gdpa_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, F, P, P, P, P]
    L.gdpa_bwd_sliding.argtypes = [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, F, P, P, P, P]
    L.gdpa_plan_create.argtypes = [P, P, I, I, I, I, I, ctypes.POINTER(P)]
    L.gdpa_plan_create_sliding.argtypes = [P, P, I, I, I, I, I, ctypes.POINTER(P)]
    L.gdpa_fwd_planned.argtypes = [P, P, P, P, P, P, F, P, P]
    L.gdpa_plan_destroy.argtypes = [P]
    L.gdpa_plan_destroy.restype = None
    L.gdpa_plan_num_items.argtypes = [P]
    L.gdpa_plan_num_items.restype = I64
    L.gdpa_plan_num_ctas.argtypes = [P]
    L.gdpa_fwd_host.argtypes = [P, P, P, P, P, I, I, I, I, I, F, P, P]
    L.gdpa_plan_enumerate.argtypes = [P, P, I, I, I, I, I, I, P, I64, P, P, ctypes.POINTER(I64),
                                      ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
    L.gdpa_act_eval.argtypes = [I, P, P, I64, P]
    L.gdpa_set_act_route.argtypes = [I]
    L.gdpa_get_act_route.argtypes = []
    L.gdpa_get_act_route.restype = I
    L.gdpa_device_status.argtypes = [P]
    L.gdpa_wait_selftest.argtypes = [I, P]
    L.gdpa_status_string.argtypes = [I]
    L.gdpa_status_string.restype = ctypes.c_char_p
    L.gdpa_version.argtypes = []
    L.gdpa_version.restype = ctypes.c_char_p
    for name in ("gdpa_fwd", "gdpa_fwd_async", "gdpa_fwd_lse", "gdpa_fwd_sliding", "gdpa_fwd_mxfp8", "gdpa_bwd", "gdpa_bwd_sliding", "gdpa_fwd_noalloc", "gdpa_plan_create", "gdpa_plan_create_sliding", "gdpa_fwd_planned", "gdpa_plan_num_ctas", "gdpa_fwd_host",
                 "gdpa_plan_enumerate", "gdpa_act_eval", "gdpa_set_act_route", "gdpa_device_status", "gdpa_wait_selftest"):
        getattr(L, name).restype = I
    _lib = L
    return L


def _addr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _check(code: int, where: str):
    if code != GDPA_OK:
        raise GdpaError(code, where)


def gdpa_status_string(code: int) -> str:
    return lib().gdpa_status_string(int(code)).decode()


def gdpa_version() -> str:
    return lib().gdpa_version().decode()


def gdpa_fwd(q, k, v, q_offsets, kv_offsets, B, H, D, act, window_blocks, scale, out, stream=None):
    _check(lib().gdpa_fwd(_addr(q), _addr(k), _addr(v), _addr(q_offsets), _addr(kv_offsets), int(B), int(H),
                          int(D), int(act), int(window_blocks), float(scale), _addr(out), _stream(stream)),
           "gdpa_fwd")


def gdpa_fwd_noalloc(q, k, v, q_offsets, kv_offsets, B, H, D, act, window_blocks, scale, out, stream=None):
    """gdpa_fwd without any allocation (fixed 4 MiB device work-list array; see include/gdpa.h)."""
    _check(lib().gdpa_fwd_noalloc(_addr(q), _addr(k), _addr(v), _addr(q_offsets), _addr(kv_offsets), int(B), int(H),
                                  int(D), int(act), int(window_blocks), float(scale), _addr(out), _stream(stream)),
           "gdpa_fwd_noalloc")


def gdpa_fwd_async(q, k, v, h_q_offsets, h_kv_offsets, q_offsets, kv_offsets, B, H, D, act, window_blocks, scale,
                   out, stream=None):
    """Host offsets (numpy int32) plan the work; device offsets feed the kernel.  No sync."""
    qo, ko = _i32(h_q_offsets), _i32(h_kv_offsets)
    _check(lib().gdpa_fwd_async(_addr(q), _addr(k), _addr(v), qo.ctypes.data, ko.ctypes.data, _addr(q_offsets),
                                _addr(kv_offsets), int(B), int(H), int(D), int(act), int(window_blocks),
                                float(scale), _addr(out), _stream(stream)), "gdpa_fwd_async")


def gdpa_fwd_lse(q, k, v, h_q_offsets, h_kv_offsets, q_offsets, kv_offsets, B, H, D, act, window_blocks, scale,
                 out, lse, stream=None):
    """gdpa_fwd_async that also writes the softmax row logsumexp ``lse`` (device fp32 [Tq, H])."""
    qo, ko = _i32(h_q_offsets), _i32(h_kv_offsets)
    _check(lib().gdpa_fwd_lse(_addr(q), _addr(k), _addr(v), qo.ctypes.data, ko.ctypes.data, _addr(q_offsets),
                              _addr(kv_offsets), int(B), int(H), int(D), int(act), int(window_blocks), float(scale),
                              _addr(out), _addr(lse), _stream(stream)), "gdpa_fwd_lse")


def gdpa_fwd_sliding(q, k, v, h_q_offsets, h_kv_offsets, q_offsets, kv_offsets, B, H, D, act, window_tokens, scale,
                     out, lse=None, stream=None):
    """The forward with a causal sliding window of ``window_tokens`` tokens (optional ``lse`` output)."""
    qo, ko = _i32(h_q_offsets), _i32(h_kv_offsets)
    _check(lib().gdpa_fwd_sliding(_addr(q), _addr(k), _addr(v), qo.ctypes.data, ko.ctypes.data, _addr(q_offsets),
                                  _addr(kv_offsets), int(B), int(H), int(D), int(act), int(window_tokens),
                                  float(scale), _addr(out), _addr(lse), _stream(stream)), "gdpa_fwd_sliding")


def gdpa_fwd_mx(q8, q_sf, k8, k_sf, v, h_q_offsets, h_kv_offsets, q_offsets, kv_offsets, B, H, D, act, scale, out,
                lse=None, stream=None):
    """The forward with MXFP8 ``q8``/``k8`` (e4m3 codes) and E8M0 block scales ``q_sf``/``k_sf``."""
    qo, ko = _i32(h_q_offsets), _i32(h_kv_offsets)
    _check(lib().gdpa_fwd_mx(_addr(q8), _addr(q_sf), _addr(k8), _addr(k_sf), _addr(v), qo.ctypes.data,
                             ko.ctypes.data, _addr(q_offsets), _addr(kv_offsets), int(B), int(H), int(D), int(act),
                             float(scale), _addr(out), _addr(lse), _stream(stream)), "gdpa_fwd_mx")


def gdpa_fwd_mxfp8(q8, q_sf, k8, k_sf, vt8, vt_sf, h_q_offsets, h_kv_offsets, q_offsets, kv_offsets, B, H, D, act,
                   scale, out, lse=None, stream=None):
    """The forward with ``q8``/``k8`` and the key-major ``vt8`` all MXFP8 (e4m3 codes with E8M0 scales)."""
    qo, ko = _i32(h_q_offsets), _i32(h_kv_offsets)
    _check(lib().gdpa_fwd_mxfp8(_addr(q8), _addr(q_sf), _addr(k8), _addr(k_sf), _addr(vt8), _addr(vt_sf),
                                qo.ctypes.data, ko.ctypes.data, _addr(q_offsets), _addr(kv_offsets), int(B), int(H),
                                int(D), int(act), float(scale), _addr(out), _addr(lse), _stream(stream)),
           "gdpa_fwd_mxfp8")


def gdpa_bwd(q, k, v, out, dout, lse, h_q_offsets, h_kv_offsets, q_offsets, kv_offsets, B, H, D, act, window_blocks,
             scale, dq, dk, dv, stream=None):
    """Gradients dq, dk, dv (device bf16) of the forward for the upstream gradient ``dout``."""
    qo, ko = _i32(h_q_offsets), _i32(h_kv_offsets)
    _check(lib().gdpa_bwd(_addr(q), _addr(k), _addr(v), _addr(out), _addr(dout), _addr(lse), qo.ctypes.data,
                          ko.ctypes.data, _addr(q_offsets), _addr(kv_offsets), int(B), int(H), int(D), int(act),
                          int(window_blocks), float(scale), _addr(dq), _addr(dk), _addr(dv), _stream(stream)),
           "gdpa_bwd")


def gdpa_bwd_sliding(q, k, v, out, dout, lse, h_q_offsets, h_kv_offsets, q_offsets, kv_offsets, B, H, D, act,
                     window_tokens, scale, dq, dk, dv, stream=None):
    """gdpa_bwd for the causal sliding window of ``window_tokens`` tokens."""
    qo, ko = _i32(h_q_offsets), _i32(h_kv_offsets)
    _check(lib().gdpa_bwd_sliding(_addr(q), _addr(k), _addr(v), _addr(out), _addr(dout), _addr(lse), qo.ctypes.data,
                                  ko.ctypes.data, _addr(q_offsets), _addr(kv_offsets), int(B), int(H), int(D),
                                  int(act), int(window_tokens), float(scale), _addr(dq), _addr(dk), _addr(dv),
                                  _stream(stream)), "gdpa_bwd_sliding")


class Plan:
    """Owns a gdpa_plan_t; freed by gdpa_plan_destroy (or when collected)."""

    def __init__(self, handle: int):
        self.handle = handle

    @property
    def num_items(self) -> int:
        return lib().gdpa_plan_num_items(self.handle)

    @property
    def num_ctas(self) -> int:
        return lib().gdpa_plan_num_ctas(self.handle)

    def __del__(self):
        if getattr(self, "handle", None):
            try:
                lib().gdpa_plan_destroy(self.handle)
            except Exception:
                pass
            self.handle = None


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def gdpa_plan_create(h_q_offsets, h_kv_offsets, B, H, D, act, window_blocks) -> Plan:
    qo, ko = _i32(h_q_offsets), _i32(h_kv_offsets)
    h = ctypes.c_void_p()
    _check(lib().gdpa_plan_create(qo.ctypes.data, ko.ctypes.data, int(B), int(H), int(D), int(act),
                                  int(window_blocks), ctypes.byref(h)), "gdpa_plan_create")
    return Plan(h.value)


def gdpa_plan_create_sliding(h_q_offsets, h_kv_offsets, B, H, D, act, window_tokens) -> Plan:
    """The plan of gdpa_fwd_sliding (causal window of ``window_tokens`` tokens), for gdpa_fwd_planned."""
    qo, ko = _i32(h_q_offsets), _i32(h_kv_offsets)
    h = ctypes.c_void_p()
    _check(lib().gdpa_plan_create_sliding(qo.ctypes.data, ko.ctypes.data, int(B), int(H), int(D), int(act),
                                          int(window_tokens), ctypes.byref(h)), "gdpa_plan_create_sliding")
    return Plan(h.value)


def gdpa_fwd_planned(plan: Plan, q, k, v, q_offsets, kv_offsets, scale, out, stream=None):
    _check(lib().gdpa_fwd_planned(plan.handle, _addr(q), _addr(k), _addr(v), _addr(q_offsets), _addr(kv_offsets),
                                  float(scale), _addr(out), _stream(stream)), "gdpa_fwd_planned")


def gdpa_plan_destroy(plan: Plan):
    if plan.handle:
        lib().gdpa_plan_destroy(plan.handle)
        plan.handle = None


def gdpa_fwd_host(h_q, h_k, h_v, h_q_offsets, h_kv_offsets, B, H, D, act, window_blocks, scale, h_out,
                  stream=None):
    qo, ko = _i32(h_q_offsets), _i32(h_kv_offsets)
    _check(lib().gdpa_fwd_host(_addr(h_q), _addr(h_k), _addr(h_v), qo.ctypes.data, ko.ctypes.data, int(B),
                               int(H), int(D), int(act), int(window_blocks), float(scale), _addr(h_out),
                               _stream(stream)), "gdpa_fwd_host")


def gdpa_plan_enumerate(h_q_offsets, h_kv_offsets, B, H, D, act, window_blocks, num_ctas, with_rows=False):
    """Host planner only: returns (items [n, 4] int32, cta_begin [num_ctas+1], cost [n])
    (and, when ``with_rows``, the query rows per item and the keys per K/V tile)."""
    qo, ko = _i32(h_q_offsets), _i32(h_kv_offsets)
    n = ctypes.c_int64(0)
    rows = ctypes.c_int32(0)
    kvt = ctypes.c_int32(0)
    cta = np.zeros(num_ctas + 1, dtype=np.int32)
    code = lib().gdpa_plan_enumerate(qo.ctypes.data, ko.ctypes.data, int(B), int(H), int(D), int(act),
                                     int(window_blocks), int(num_ctas), None, 0, cta.ctypes.data, None,
                                     ctypes.byref(n), ctypes.byref(rows), ctypes.byref(kvt))
    if code not in (GDPA_OK, GDPA_ERR_NO_MEMORY):
        raise GdpaError(code, "gdpa_plan_enumerate")
    items = np.zeros((max(n.value, 1), 4), dtype=np.int32)
    cost = np.zeros(max(n.value, 1), dtype=np.int64)
    _check(lib().gdpa_plan_enumerate(qo.ctypes.data, ko.ctypes.data, int(B), int(H), int(D), int(act),
                                     int(window_blocks), int(num_ctas), items.ctypes.data, n.value,
                                     cta.ctypes.data, cost.ctypes.data, ctypes.byref(n), ctypes.byref(rows),
                                     ctypes.byref(kvt)),
           "gdpa_plan_enumerate")
    if with_rows:
        return items[:n.value], cta, cost[:n.value], rows.value, kvt.value
    return items[:n.value], cta, cost[:n.value]


def gdpa_act_eval(act, x, y, *, stream=None):
    """y = act(x) elementwise on the device (``stream`` keyword-only: a stray
    positional argument must not be taken for a stream handle)."""
    _check(lib().gdpa_act_eval(int(act), _addr(x), _addr(y), int(x.numel()), _stream(stream)), "gdpa_act_eval")


def gdpa_set_act_route(route) -> None:
    """Selects the sigma route of the GELU / SiLU activations for later
    launches (GDPA_ROUTE_SFU or GDPA_ROUTE_ALU)."""
    _check(lib().gdpa_set_act_route(int(route)), "gdpa_set_act_route")


def gdpa_get_act_route() -> int:
    return int(lib().gdpa_get_act_route())


def gdpa_device_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device status code."""
    return lib().gdpa_device_status(_stream(stream))


def gdpa_wait_selftest(timeout_ms: int, stream=None):
    _check(lib().gdpa_wait_selftest(int(timeout_ms), _stream(stream)), "gdpa_wait_selftest")
