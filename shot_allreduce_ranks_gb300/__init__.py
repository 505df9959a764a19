"""GB300-native bf16 allreduce over R virtual ranks held as HBM buffers.

Thin Python binding of libar_gb300.so (C ABI in include/ar.h).  PyTorch only
provides device memory and streams here; every step of the reduction runs in
the library's CUDA kernels.  Importing this package does not load the
library; the first ``AllReduce`` does, and fails loudly if it is not built.
"""
from __future__ import annotations

import ctypes

from ._lib import (AR_AUTO, AR_BF16, AR_FP16, AR_FP32, AR_FUSED_LL8,  # noqa: F401
                   AR_MAX_PACKET_RANKS, AR_MAX_RANKS, AR_ONESHOT_FANOUT, AR_ONESHOT_PULL,
                   AR_TWOPHASE, VARIANTS, ArError, ArInfo, check, load)

__all__ = ["AllReduce", "ArError", "VARIANTS", "allreduce_fused_noalloc", "load"]


def _variant_id(v) -> int:
    if v is None:
        return AR_AUTO
    if isinstance(v, str):
        return VARIANTS[v]
    return int(v)


def _dtype_code(dtype) -> int:
    import torch
    codes = {torch.bfloat16: AR_BF16, torch.float16: AR_FP16, torch.float32: AR_FP32}
    if dtype not in codes:
        raise ValueError("dtype must be torch.bfloat16, torch.float16 or torch.float32")
    return codes[dtype]


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


class AllReduce:
    """A handle for R virtual ranks of up to ``max_count`` elements each.

    ``ar(inputs, outputs)`` leaves in every ``outputs[r]`` the rank-order fp32
    sum of all ``inputs``, rounded once to the element type (bf16, fp16; fp32
    is not rounded).  Buffers are contiguous CUDA tensors of ``dtype`` on the
    handle's device; ``outputs`` may be ``inputs`` (in place).  Calls are
    asynchronous on the current (or given) stream.
    """

    def __init__(self, R: int, max_count: int, device=None, dtype=None):
        import torch
        self._lib = load()
        self.R = int(R)
        self.max_count = int(max_count)
        self.dtype = torch.bfloat16 if dtype is None else dtype
        code = _dtype_code(self.dtype)
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None
                                   else torch.device(device).index or 0)
        h = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            check(self._lib.ar_create(self.R, self.max_count, code, ctypes.byref(h)), "ar_create")
        self._h = h
        self._tables = {}

    # -- lifetime ----------------------------------------------------------
    def close(self) -> None:
        if getattr(self, "_h", None):
            import torch
            with torch.cuda.device(self.device):
                check(self._lib.ar_destroy(self._h), "ar_destroy")
            self._h = None
            self._tables.clear()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # -- pointer tables ----------------------------------------------------
    def tables(self, inputs, outputs):
        """Device int64 tensors of the R input and R output pointers (cached)."""
        import torch
        key = tuple(t.data_ptr() for t in inputs) + tuple(t.data_ptr() for t in outputs)
        tbl = self._tables.get(key)
        if tbl is None:
            if len(self._tables) > 64:
                self._tables.clear()
            ptrs = torch.tensor(list(key), dtype=torch.int64)
            dev = ptrs.to(self.device)
            tbl = (dev[: self.R], dev[self.R:])
            self._tables[key] = tbl
        return tbl

    def _check_buffers(self, bufs, count):
        import torch
        if len(bufs) != self.R:
            raise ValueError("expected %d buffers, got %d" % (self.R, len(bufs)))
        for t in bufs:
            if t.dtype != self.dtype or not t.is_cuda or t.device != self.device:
                raise ValueError("buffers must be %s CUDA tensors on %s" % (self.dtype, self.device))
            if not t.is_contiguous() or t.numel() < count:
                raise ValueError("buffers must be contiguous with >= %d elements" % count)

    # -- calls -------------------------------------------------------------
    def allreduce_tables(self, in_tbl, out_tbl, count: int, stream=None) -> None:
        """Raw call: device pointer tables (int64 CUDA tensors or addresses)."""
        ip = in_tbl if isinstance(in_tbl, int) else in_tbl.data_ptr()
        op = out_tbl if isinstance(out_tbl, int) else out_tbl.data_ptr()
        check(self._lib.ar_allreduce(self._h, ip, op, int(count), _stream_handle(stream)),
              "ar_allreduce")

    def __call__(self, inputs, outputs=None, count=None, variant=None, stream=None):
        import torch
        if count is None:
            count = inputs[0].numel()
        if outputs is None:
            outputs = [torch.empty_like(t) for t in inputs]
        self._check_buffers(inputs, count)
        self._check_buffers(outputs, count)
        if variant is not None:
            self.set_variant(variant)
        in_tbl, out_tbl = self.tables(inputs, outputs)
        self.allreduce_tables(in_tbl, out_tbl, count, stream)
        return outputs

    def reduce_scatter(self, inputs, outputs=None, recvcount=None, stream=None):
        """outputs[r] <- block r of the rank-order sum; inputs hold R*recvcount."""
        import torch
        if recvcount is None:
            recvcount = inputs[0].numel() // self.R
        if outputs is None:
            outputs = [torch.empty(recvcount, dtype=self.dtype, device=self.device)
                       for _ in range(self.R)]
        self._check_buffers(inputs, self.R * recvcount)
        self._check_buffers(outputs, recvcount)
        in_tbl, out_tbl = self.tables(inputs, outputs)
        check(self._lib.ar_reduce_scatter(self._h, in_tbl.data_ptr(), out_tbl.data_ptr(),
                                          int(recvcount), _stream_handle(stream)),
              "ar_reduce_scatter")
        return outputs

    def all_gather(self, inputs, outputs=None, sendcount=None, stream=None):
        """outputs[r] <- concatenation of all inputs in rank order."""
        import torch
        if sendcount is None:
            sendcount = inputs[0].numel()
        if outputs is None:
            outputs = [torch.empty(self.R * sendcount, dtype=self.dtype, device=self.device)
                       for _ in range(self.R)]
        self._check_buffers(inputs, sendcount)
        self._check_buffers(outputs, self.R * sendcount)
        in_tbl, out_tbl = self.tables(inputs, outputs)
        check(self._lib.ar_all_gather(self._h, in_tbl.data_ptr(), out_tbl.data_ptr(),
                                      int(sendcount), _stream_handle(stream)), "ar_all_gather")
        return outputs

    def allreduce_host(self, host_inputs, host_outputs, count=None, stream=None) -> None:
        """End-to-end call on HOST tensors (pinned for asynchronous copies)."""
        if count is None:
            count = host_inputs[0].numel()
        n = self.R
        ins = (ctypes.c_void_p * n)(*[t.data_ptr() for t in host_inputs])
        outs = (ctypes.c_void_p * n)(*[t.data_ptr() for t in host_outputs])
        check(self._lib.ar_allreduce_host(self._h, ctypes.cast(ins, ctypes.c_void_p),
                                          ctypes.cast(outs, ctypes.c_void_p), int(count),
                                          _stream_handle(stream)), "ar_allreduce_host")

    def reserve_host_staging(self) -> None:
        check(self._lib.ar_reserve_host_staging(self._h), "ar_reserve_host_staging")

    # -- configuration -----------------------------------------------------
    def set_variant(self, variant) -> None:
        check(self._lib.ar_set_variant(self._h, _variant_id(variant)), "ar_set_variant")

    def select(self, count: int) -> str:
        v = ctypes.c_int()
        check(self._lib.ar_select(self._h, int(count), ctypes.byref(v)), "ar_select")
        return self._lib.ar_variant_name(v.value).decode()

    def set_launch(self, variant, ctas: int = 0, threads: int = 0) -> None:
        check(self._lib.ar_set_launch(self._h, _variant_id(variant), int(ctas), int(threads)),
              "ar_set_launch")

    def set_spin_limit_ns(self, ns: int) -> None:
        check(self._lib.ar_set_spin_limit_ns(self._h, int(ns)), "ar_set_spin_limit_ns")

    def query(self) -> ArInfo:
        info = ArInfo()
        check(self._lib.ar_query(self._h, ctypes.byref(info)), "ar_query")
        return info

    def device_status(self, stream=None) -> int:
        """AR_OK, or AR_ERR_TIMEOUT if a fused call gave up waiting (clears it)."""
        return self._lib.ar_get_device_status(self._h, _stream_handle(stream))

    def last_timeout(self):
        """(waiting rank, lowest missing rank, waits that gave up) of the last
        timeout device_status() reported; (-1, -1, 0) if none."""
        w, m, n = ctypes.c_int(), ctypes.c_int(), ctypes.c_uint32()
        check(self._lib.ar_last_timeout(self._h, ctypes.byref(w), ctypes.byref(m),
                                        ctypes.byref(n)), "ar_last_timeout")
        return w.value, m.value, n.value

    # -- test hooks ----------------------------------------------------------
    def debug_skip_producer(self, rank: int) -> None:
        check(self._lib.ar_debug_skip_producer(self._h, int(rank)), "ar_debug_skip_producer")

    def debug_guards_intact(self) -> bool:
        """True if nothing wrote outside the handle's packet regions."""
        ok = ctypes.c_int()
        check(self._lib.ar_debug_check_guards(self._h, ctypes.byref(ok)), "ar_debug_check_guards")
        return bool(ok.value)

    def debug_delay_producer(self, rank: int, ns: int) -> None:
        check(self._lib.ar_debug_delay_producer(self._h, int(rank), int(ns)),
              "ar_debug_delay_producer")

    def debug_set_epoch(self, epoch: int) -> None:
        check(self._lib.ar_debug_set_epoch(self._h, int(epoch)), "ar_debug_set_epoch")

    def debug_get_epoch(self) -> int:
        e = ctypes.c_uint32()
        check(self._lib.ar_debug_get_epoch(self._h, ctypes.byref(e)), "ar_debug_get_epoch")
        return e.value


def allreduce_fused_noalloc(R: int, in_tbl, out_tbl, count: int, stream=None) -> None:
    """Fused LL8 allreduce for callers that cannot allocate device memory.

    No handle: the packet scratch is a fixed array inside the library's
    device image, set up on the first call per device (make that call before
    any stream capture).  ``in_tbl`` / ``out_tbl`` are device int64 tensors
    (or addresses) of R buffer pointers; ``count`` must not exceed
    ``_lib.noalloc_max_count(R)``.  Calls that overlap on the GPU race.
    """
    lib = load()
    ip = in_tbl if isinstance(in_tbl, int) else in_tbl.data_ptr()
    op = out_tbl if isinstance(out_tbl, int) else out_tbl.data_ptr()
    check(lib.ar_allreduce_fused_noalloc(int(R), ip, op, int(count), _stream_handle(stream)),
          "ar_allreduce_fused_noalloc")
