"""Helpers shared by the GPU tests: run the CUDA path through the C ABI and
compare it with the oracle bit for bit."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from shot_allreduce_ranks_gb300 import AllReduce, build, inputs

DEV = "cuda"
PARITY_VARIANTS = ["oneshot_pull", "oneshot_fanout", "twophase", "fused_ll8",
                   "oneshot_fanout_bulk", "fused_ll8_staged", "packet_3op"]

_handles = {}


def ensure_built():
    build.build()


def handle(R: int, max_count: int) -> AllReduce:
    key = (R, max_count)
    h = _handles.get(key)
    if h is None:
        ensure_built()
        h = AllReduce(R, max_count)
        _handles[key] = h
    return h


def release_handles():
    for h in list(_handles.values()):
        h.close()
    _handles.clear()


def is_nan_bits(a: np.ndarray) -> np.ndarray:
    return ((a & 0x7F80) == 0x7F80) & ((a & 0x007F) != 0)


def mismatches(got: np.ndarray, want: np.ndarray) -> np.ndarray:
    """Indices where two bf16 bit arrays differ (any NaN equals any NaN)."""
    gn, wn = is_nan_bits(got), is_nan_bits(want)
    bad = (got != want) & ~(gn & wn)
    return np.nonzero(bad)[0]


def assert_bitexact(got: np.ndarray, want: np.ndarray, what: str = ""):
    bad = mismatches(got, want)
    if bad.size:
        i = int(bad[0])
        raise AssertionError(
            "%s: %d of %d elements differ; first at %d: got 0x%04x want 0x%04x"
            % (what, bad.size, want.size, i, int(got[i]), int(want[i])))


def oracle_expect(xs_cpu):
    """Oracle result (uint16 bits) for CPU bf16 inputs."""
    outs = oracle.allreduce_bf16([inputs.bits(x) for x in xs_cpu])
    return outs[0]


def to_device(xs_cpu):
    return [x.to(DEV) for x in xs_cpu]


def device_bits(t: torch.Tensor) -> np.ndarray:
    return inputs.bits(t.cpu())


def run_variant(ar: AllReduce, xs_dev, variant, outs=None, count=None):
    ar.set_variant(variant)
    outs = ar(xs_dev, outs, count=count)
    torch.cuda.synchronize()
    return outs


def check_all_outputs(outs, want, what, count=None):
    for r, o in enumerate(outs):
        got = device_bits(o)
        if count is not None:
            got = got[:count]
        assert_bitexact(got, want, "%s rank %d" % (what, r))
