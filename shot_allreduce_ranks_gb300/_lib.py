"""ctypes declarations of the C ABI in include/ar.h.

Loading fails loudly when libar_gb300.so has not been built: there is no
fallback implementation of any kind.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libar_gb300.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "ar.h")

AR_OK, AR_ERR_INVALID_ARG, AR_ERR_UNSUPPORTED, AR_ERR_OOM, AR_ERR_CUDA, AR_ERR_TIMEOUT = range(6)
AR_BF16, AR_FP16, AR_FP32 = 0, 1, 2
AR_AUTO, AR_ONESHOT_PULL, AR_ONESHOT_FANOUT, AR_TWOPHASE, AR_FUSED_LL8 = range(5)
AR_ONESHOT_FANOUT_BULK, AR_FUSED_LL8_STAGED, AR_PACKET_3OP = 5, 6, 7
VARIANTS = {
    "auto": AR_AUTO,
    "oneshot_pull": AR_ONESHOT_PULL,
    "oneshot_fanout": AR_ONESHOT_FANOUT,
    "twophase": AR_TWOPHASE,
    "fused_ll8": AR_FUSED_LL8,
    "oneshot_fanout_bulk": AR_ONESHOT_FANOUT_BULK,
    "fused_ll8_staged": AR_FUSED_LL8_STAGED,
    "packet_3op": AR_PACKET_3OP,
}
AR_MAX_RANKS = 16
AR_MAX_PACKET_RANKS = 8


class ArInfo(ctypes.Structure):
    _fields_ = [
        ("R", ctypes.c_int),
        ("dtype", ctypes.c_int),
        ("max_count", ctypes.c_size_t),
        ("scratch_bytes", ctypes.c_size_t),
        ("num_sms", ctypes.c_int),
        ("fused_max_ctas", ctypes.c_int),
        ("fused_threads", ctypes.c_int),
        ("device", ctypes.c_int),
    ]


_H = ctypes.c_void_p
_VP = ctypes.c_void_p
_SZ = ctypes.c_size_t
_I = ctypes.c_int
_ST = ctypes.c_int

PROTOTYPES = {
    "ar_create": (_ST, [_I, _SZ, _I, ctypes.POINTER(_H)]),
    "ar_allreduce": (_ST, [_H, _VP, _VP, _SZ, _VP]),
    "ar_destroy": (_ST, [_H]),
    "ar_set_variant": (_ST, [_H, _I]),
    "ar_select": (_ST, [_H, _SZ, ctypes.POINTER(_I)]),
    "ar_set_launch": (_ST, [_H, _I, _I, _I]),
    "ar_set_spin_limit_ns": (_ST, [_H, ctypes.c_uint64]),
    "ar_get_device_status": (_ST, [_H, _VP]),
    "ar_last_timeout": (_ST, [_H, ctypes.POINTER(_I), ctypes.POINTER(_I),
                              ctypes.POINTER(ctypes.c_uint32)]),
    "ar_query": (_ST, [_H, ctypes.POINTER(ArInfo)]),
    "ar_status_string": (ctypes.c_char_p, [_I]),
    "ar_variant_name": (ctypes.c_char_p, [_I]),
    "ar_reserve_host_staging": (_ST, [_H]),
    "ar_allreduce_host": (_ST, [_H, _VP, _VP, _SZ, _VP]),
    "ar_debug_skip_producer": (_ST, [_H, _I]),
    "ar_debug_check_guards": (_ST, [_H, ctypes.POINTER(_I)]),
    "ar_debug_delay_producer": (_ST, [_H, _I, ctypes.c_uint64]),
    "ar_debug_set_epoch": (_ST, [_H, ctypes.c_uint32]),
    "ar_debug_get_epoch": (_ST, [_H, ctypes.POINTER(ctypes.c_uint32)]),
    "ar_allreduce_fused_noalloc": (_ST, [_I, _VP, _VP, _SZ, _VP]),
    "ar_reduce_scatter": (_ST, [_H, _VP, _VP, _SZ, _VP]),
    "ar_all_gather": (_ST, [_H, _VP, _VP, _SZ, _VP]),
}

AR_NOALLOC_SCRATCH_BYTES = 32 << 20


def noalloc_max_count(R: int) -> int:
    """Largest count ar_allreduce_fused_noalloc accepts for R ranks."""
    if R <= 1:
        return (1 << 64) - 1
    return (AR_NOALLOC_SCRATCH_BYTES // (32 * R * (R - 1))) * 8 * R


_lock = threading.Lock()
_lib = None


def header_functions(path: str = HEADER):
    """Names of the functions declared in include/ar.h."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ar_[a-z0-9_]+)\s*\(", text)))


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is not None and path == LIB_PATH:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                "libar_gb300.so is not built (%s); run "
                "`python -m shot_allreduce_ranks_gb300.build`" % path)
        lib = ctypes.CDLL(path)
        for name, (res, args) in PROTOTYPES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path == LIB_PATH:
            _lib = lib
        return lib


class ArError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = load().ar_status_string(status).decode()
        super().__init__("%s%s (status %d)" % (what + ": " if what else "", msg, status))


def check(status: int, what: str = "") -> None:
    if status != AR_OK:
        raise ArError(status, what)
