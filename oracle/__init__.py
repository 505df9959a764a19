"""Oracle for the virtual-rank bf16 allreduce -- TEST INFRASTRUCTURE ONLY.

This package wraps ``oracle.c`` (plain single-threaded C) through ctypes.  It
may be imported only by the tests, by ``__graft_entry__.smoke()`` and by the
CPU-baseline leg of ``bench.py``; the GPU library never imports it and shares
no code with it.

The definition it computes (fp32 accumulation in rank order 0..R-1, one
round-to-nearest-even to bf16, identical output for every rank) and the
passages it follows are stated at the top of ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
CFLAGS = [
    "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
    "-fexcess-precision=standard", "-fPIC", "-shared",
]
LIBS = ["-lm"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile ``oracle.c`` into a shared library with gcc and return its path."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", *CFLAGS, src, "-o", tmp, *LIBS])
    os.replace(tmp, out)
    return out


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) and return the oracle library."""
    global _lib
    with _lock:
        if path is not None:
            return _declare(ctypes.CDLL(path))
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
        return _lib


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    u16p = ctypes.POINTER(ctypes.c_uint16)
    lib.oracle_f32_to_bf16_rne.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16_rne.restype = ctypes.c_uint16
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f32.restype = ctypes.c_float
    lib.oracle_f32_to_bf16_array.argtypes = [
        ctypes.POINTER(ctypes.c_float), u16p, ctypes.c_size_t]
    lib.oracle_f32_to_bf16_array.restype = None
    lib.oracle_allreduce_bf16.argtypes = [
        ctypes.c_int, ctypes.c_size_t, ctypes.POINTER(u16p), ctypes.POINTER(u16p)]
    lib.oracle_allreduce_bf16.restype = ctypes.c_int
    lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_f32.restype = ctypes.c_float
    lib.oracle_f32_to_f16_rne.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_f16_rne.restype = ctypes.c_uint16
    lib.oracle_f32_to_f16_array.argtypes = [
        ctypes.POINTER(ctypes.c_float), u16p, ctypes.c_size_t]
    lib.oracle_f32_to_f16_array.restype = None
    f32p = ctypes.POINTER(ctypes.c_float)
    lib.oracle_allreduce_f16.argtypes = [
        ctypes.c_int, ctypes.c_size_t, ctypes.POINTER(u16p), ctypes.POINTER(u16p)]
    lib.oracle_allreduce_f16.restype = ctypes.c_int
    lib.oracle_allreduce_f32.argtypes = [
        ctypes.c_int, ctypes.c_size_t, ctypes.POINTER(f32p), ctypes.POINTER(f32p)]
    lib.oracle_allreduce_f32.restype = ctypes.c_int
    for name in ("oracle_reduce_scatter_bf16", "oracle_all_gather_bf16"):
        fn = getattr(lib, name)
        fn.argtypes = [ctypes.c_int, ctypes.c_size_t, ctypes.POINTER(u16p), ctypes.POINTER(u16p)]
        fn.restype = ctypes.c_int
    return lib


def _u16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 buffers are passed as uint16 bit patterns")
    return a


def f32_to_bf16(x: np.ndarray, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Round an fp32 array to bf16 bit patterns (round to nearest, ties to even)."""
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16)
    lib.oracle_f32_to_bf16_array(
        x.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
        y.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)), x.size)
    return y


def allreduce_bf16(inputs, lib: ctypes.CDLL | None = None, outputs=None):
    """Allreduce R bf16 buffers (uint16 bit patterns, equal length).

    Returns the list of R outputs (all identical).  ``outputs`` may be given
    to write into caller buffers, including the inputs themselves (in place).
    """
    lib = lib or load()
    ins = [_u16(a) for a in inputs]
    R = len(ins)
    if R < 1:
        raise ValueError("need at least one rank")
    count = ins[0].size
    if any(a.size != count for a in ins):
        raise ValueError("all ranks must hold the same element count")
    outs = outputs if outputs is not None else [np.empty(count, np.uint16) for _ in range(R)]
    outs = [_u16(o) for o in outs]
    u16p = ctypes.POINTER(ctypes.c_uint16)
    in_tbl = (u16p * R)(*[a.ctypes.data_as(u16p) for a in ins])
    out_tbl = (u16p * R)(*[o.ctypes.data_as(u16p) for o in outs])
    rc = lib.oracle_allreduce_bf16(R, count, in_tbl, out_tbl)
    if rc != 0:
        raise ValueError("oracle rejected R=%d" % R)
    return outs


def _tables(bufs):
    u16p = ctypes.POINTER(ctypes.c_uint16)
    return (u16p * len(bufs))(*[b.ctypes.data_as(u16p) for b in bufs])


def reduce_scatter_bf16(inputs, lib: ctypes.CDLL | None = None):
    """Reduce-scatter of R inputs of R*recvcount elements; returns R outputs
    of recvcount elements (output r = rank-order sum of block r)."""
    lib = lib or load()
    ins = [_u16(a) for a in inputs]
    R = len(ins)
    total = ins[0].size
    if total % R or any(a.size != total for a in ins):
        raise ValueError("inputs must all hold R * recvcount elements")
    rc = total // R
    outs = [np.empty(rc, np.uint16) for _ in range(R)]
    if lib.oracle_reduce_scatter_bf16(R, rc, _tables(ins), _tables(outs)) != 0:
        raise ValueError("oracle rejected R=%d" % R)
    return outs


def all_gather_bf16(inputs, lib: ctypes.CDLL | None = None):
    """All-gather of R inputs of sendcount elements; returns R outputs of
    R*sendcount elements (the inputs concatenated in rank order)."""
    lib = lib or load()
    ins = [_u16(a) for a in inputs]
    R = len(ins)
    sc = ins[0].size
    if any(a.size != sc for a in ins):
        raise ValueError("inputs must hold the same element count")
    outs = [np.empty(R * sc, np.uint16) for _ in range(R)]
    if lib.oracle_all_gather_bf16(R, sc, _tables(ins), _tables(outs)) != 0:
        raise ValueError("oracle rejected R=%d" % R)
    return outs


def f32_to_f16(x: np.ndarray, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Round an fp32 array to fp16 bit patterns (round to nearest, ties to even)."""
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16)
    lib.oracle_f32_to_f16_array(
        x.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
        y.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)), x.size)
    return y


def allreduce_f16(inputs, lib: ctypes.CDLL | None = None):
    """Allreduce of R fp16 buffers (uint16 bit patterns); returns output 0."""
    lib = lib or load()
    ins = [_u16(a) for a in inputs]
    R, count = len(ins), ins[0].size
    outs = [np.empty(count, np.uint16) for _ in range(R)]
    if lib.oracle_allreduce_f16(R, count, _tables(ins), _tables(outs)) != 0:
        raise ValueError("oracle rejected R=%d" % R)
    return outs


def allreduce_f32(inputs, lib: ctypes.CDLL | None = None):
    """Allreduce of R fp32 buffers; returns the R outputs."""
    lib = lib or load()
    ins = [np.ascontiguousarray(a, dtype=np.float32) for a in inputs]
    R, count = len(ins), ins[0].size
    outs = [np.empty(count, np.float32) for _ in range(R)]
    f32p = ctypes.POINTER(ctypes.c_float)
    it = (f32p * R)(*[a.ctypes.data_as(f32p) for a in ins])
    ot = (f32p * R)(*[o.ctypes.data_as(f32p) for o in outs])
    if lib.oracle_allreduce_f32(R, count, it, ot) != 0:
        raise ValueError("oracle rejected R=%d" % R)
    return outs
