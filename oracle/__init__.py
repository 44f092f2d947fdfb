"""fp64 CPU oracle for the jagged GDPA forward and backward passes -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it and
shares no code with it.  The arithmetic lives in ``gdpa_oracle.c`` (plain C,
built with gcc by :func:`build`); this module only marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdpa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with gcc (plain C, -O2, pthreads)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp.%d" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared", "-pthread",
                           "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        lib.oracle_gdpa_fwd.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_double, P, ctypes.c_int]
        lib.oracle_gdpa_fwd.restype = ctypes.c_int
        lib.oracle_gdpa_bwd.argtypes = [P, P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_double, P, P, P, P, ctypes.c_int]
        lib.oracle_gdpa_bwd.restype = ctypes.c_int
        lib.oracle_gelu_tanh_grad.argtypes = [ctypes.c_double]
        lib.oracle_gelu_tanh_grad.restype = ctypes.c_double
        lib.oracle_silu.argtypes = [ctypes.c_double]
        lib.oracle_silu.restype = ctypes.c_double
        lib.oracle_silu_grad.argtypes = [ctypes.c_double]
        lib.oracle_silu_grad.restype = ctypes.c_double
        lib.oracle_gelu_tanh.argtypes = [ctypes.c_double]
        lib.oracle_gelu_tanh.restype = ctypes.c_double
        lib.oracle_num_cpus.restype = ctypes.c_int
        lib.oracle_gdpa_fwd_mx.argtypes = [P, P, P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_double, P, ctypes.c_int]
        lib.oracle_gdpa_fwd_mx.restype = ctypes.c_int
        lib.oracle_gdpa_fwd_mxfp8.argtypes = [P, P, P, P, P, P, ctypes.c_int64, P, P, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, P,
                                              ctypes.c_int]
        lib.oracle_gdpa_fwd_mxfp8.restype = ctypes.c_int
        lib.oracle_vt_columns.argtypes = [P, ctypes.c_int]
        lib.oracle_vt_columns.restype = ctypes.c_int64
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_double.restype = ctypes.c_double
        lib.oracle_e8m0_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e8m0_to_double.restype = ctypes.c_double
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def gdpa_fwd(q, k, v, q_offsets, kv_offsets, H: int, D: int, act: int, window_blocks: int,
             scale: float, nthreads: int = 0) -> np.ndarray:
    """Oracle output, fp64 ``[Tq, H, D]``.

    ``q``, ``k``, ``v`` are uint16 bf16 bit patterns ``[tokens, H, D]``;
    offsets are int32 prefix sums ``[B+1]``.
    """
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    qo = np.ascontiguousarray(q_offsets, dtype=np.int32)
    ko = np.ascontiguousarray(kv_offsets, dtype=np.int32)
    B = len(qo) - 1
    out = np.zeros((int(qo[-1]), H, D), dtype=np.float64)
    rc = lib.oracle_gdpa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(qo), _ptr(ko), B, H, D, act,
                             window_blocks, float(scale), _ptr(out), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gdpa_fwd returned %d" % rc)
    return out


def gdpa_fwd_batch(batch, nthreads: int = 0) -> np.ndarray:
    w = batch.workload
    return gdpa_fwd(batch.q, batch.k, batch.v, batch.q_offsets, batch.kv_offsets, w.H, w.D, w.act,
                    w.window_blocks, w.scale, nthreads)


def gdpa_fwd_mx(q8, q_sf, k8, k_sf, v, q_offsets, kv_offsets, H: int, D: int, act: int,
                window_blocks: int, scale: float, nthreads: int = 0) -> np.ndarray:
    """Oracle output, fp64 ``[Tq, H, D]``, for MXFP8 Q and K.

    ``q8``, ``k8``: uint8 e4m3 codes ``[tokens, H, D]``; ``q_sf``, ``k_sf``:
    uint8 E8M0 scales ``[tokens, H, D // 32]``; ``v``: uint16 bf16 bits.
    """
    lib = _load()
    arrs = [np.ascontiguousarray(a, dtype=np.uint8) for a in (q8, q_sf, k8, k_sf)]
    v = np.ascontiguousarray(v, dtype=np.uint16)
    qo = np.ascontiguousarray(q_offsets, dtype=np.int32)
    ko = np.ascontiguousarray(kv_offsets, dtype=np.int32)
    B = len(qo) - 1
    out = np.zeros((int(qo[-1]), H, D), dtype=np.float64)
    rc = lib.oracle_gdpa_fwd_mx(*[_ptr(a) for a in arrs], _ptr(v), _ptr(qo), _ptr(ko), B, H, D, act,
                                window_blocks, float(scale), _ptr(out), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gdpa_fwd_mx returned %d" % rc)
    return out


def gdpa_fwd_mx_batch(batch, nthreads: int = 0) -> np.ndarray:
    w = batch.workload
    return gdpa_fwd_mx(batch.q8, batch.q_sf, batch.k8, batch.k_sf, batch.v, batch.q_offsets, batch.kv_offsets,
                       w.H, w.D, w.act, w.window_blocks, w.scale, nthreads)


def gdpa_fwd_mxfp8(q8, q_sf, k8, k_sf, vt8, vt_sf, q_offsets, kv_offsets, H: int, D: int, act: int,
                   window_blocks: int, scale: float, nthreads: int = 0) -> np.ndarray:
    """Oracle output, fp64 ``[Tq, H, D]``, for Q, K and V all in MXFP8.

    ``q8``, ``k8``, ``q_sf``, ``k_sf`` as :func:`gdpa_fwd_mx`; ``vt8``: uint8
    e4m3 codes ``[H*D, VT]`` of V, key-major; ``vt_sf``: uint8 E8M0 scales
    ``[VT // 32, H*D]`` (layout in ``gdpa_oracle.c``).
    """
    lib = _load()
    arrs = [np.ascontiguousarray(a, dtype=np.uint8) for a in (q8, q_sf, k8, k_sf, vt8, vt_sf)]
    qo = np.ascontiguousarray(q_offsets, dtype=np.int32)
    ko = np.ascontiguousarray(kv_offsets, dtype=np.int32)
    B = len(qo) - 1
    VT = int(arrs[4].shape[1]) if arrs[4].ndim == 2 else -1
    out = np.zeros((int(qo[-1]), H, D), dtype=np.float64)
    rc = lib.oracle_gdpa_fwd_mxfp8(*[_ptr(a) for a in arrs], VT, _ptr(qo), _ptr(ko), B, H, D, act,
                                   window_blocks, float(scale), _ptr(out), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gdpa_fwd_mxfp8 returned %d" % rc)
    return out


def gdpa_fwd_mxfp8_batch(batch, nthreads: int = 0) -> np.ndarray:
    w = batch.workload
    return gdpa_fwd_mxfp8(batch.q8, batch.q_sf, batch.k8, batch.k_sf, batch.vt8, batch.vt_sf, batch.q_offsets,
                          batch.kv_offsets, w.H, w.D, w.act, w.window_blocks, w.scale, nthreads)


def vt_columns(kv_offsets) -> int:
    """VT, the row length of the key-major V layout, as the oracle counts it."""
    ko = np.ascontiguousarray(kv_offsets, dtype=np.int32)
    return int(_load().oracle_vt_columns(_ptr(ko), len(ko) - 1))


def e4m3_to_double(code: int) -> float:
    return _load().oracle_e4m3_to_double(int(code))


def e8m0_to_double(code: int) -> float:
    return _load().oracle_e8m0_to_double(int(code))


def gdpa_bwd(q, k, v, dout, q_offsets, kv_offsets, H: int, D: int, act: int, window_blocks: int,
             scale: float, nthreads: int = 0):
    """Oracle gradients ``(dq, dk, dv, lse)`` in fp64 for the upstream gradient ``dout``.

    ``dout`` is uint16 bf16 bits ``[Tq, H, D]`` like ``q``; ``lse`` is ``[Tq, H]``
    (natural log; -inf for an empty key set, 0 for GELU rows).
    """
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    do = np.ascontiguousarray(dout, dtype=np.uint16)
    qo = np.ascontiguousarray(q_offsets, dtype=np.int32)
    ko = np.ascontiguousarray(kv_offsets, dtype=np.int32)
    B = len(qo) - 1
    Tq, Tkv = int(qo[-1]), int(ko[-1])
    dq = np.zeros((Tq, H, D), dtype=np.float64)
    dk = np.zeros((Tkv, H, D), dtype=np.float64)
    dv = np.zeros((Tkv, H, D), dtype=np.float64)
    lse = np.zeros((Tq, H), dtype=np.float64)
    rc = lib.oracle_gdpa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(qo), _ptr(ko), B, H, D, act,
                             window_blocks, float(scale), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(lse), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gdpa_bwd returned %d" % rc)
    return dq, dk, dv, lse


def gdpa_bwd_batch(batch, dout, nthreads: int = 0):
    w = batch.workload
    return gdpa_bwd(batch.q, batch.k, batch.v, dout, batch.q_offsets, batch.kv_offsets, w.H, w.D, w.act,
                    w.window_blocks, w.scale, nthreads)


def gelu_tanh_grad(x: float) -> float:
    return _load().oracle_gelu_tanh_grad(float(x))


def silu(x: float) -> float:
    return _load().oracle_silu(float(x))


def silu_grad(x: float) -> float:
    return _load().oracle_silu_grad(float(x))


def gelu_tanh(x: float) -> float:
    return _load().oracle_gelu_tanh(float(x))


def num_cpus() -> int:
    return _load().oracle_num_cpus()
