"""Pins for the oracle: checks against facts fixed by IEEE 754 arithmetic and
by library routines, never against the oracle itself.

Each ``pin_*`` function takes a loaded oracle library (the real one, or a
deliberately broken copy compiled by the mutation tests) and returns a list
of failure descriptions; an empty list means the pin holds.

The pages print no numeric worked example of the reduction (their tables are
timings), so the closed-form cases below are derived by hand from the
definition of fp32 addition and of round-to-nearest-even; each derivation is
written next to its case.
"""
from __future__ import annotations

import struct

import numpy as np
import torch

import oracle
from shot_allreduce_ranks_gb300 import inputs


def bf16_bits_of(x: float) -> int:
    """Bits of a value that is exactly representable in bf16 (checked)."""
    u = struct.unpack("<I", struct.pack("<f", x))[0]
    if u & 0xFFFF:
        raise ValueError("%r is not exactly representable in bf16" % x)
    if struct.unpack("<f", struct.pack("<I", u))[0] != x and x == x:
        raise ValueError("%r is not exactly representable in fp32" % x)
    return u >> 16


def value_of_bits(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (b & 0xFFFF) << 16))[0]


def run(lib, rank_bits):
    """Allreduce a list of per-rank uint16 arrays; returns the R outputs."""
    return oracle.allreduce_bf16([np.asarray(a, np.uint16) for a in rank_bits], lib=lib)


def _all_equal(outs, expect):
    return all(np.array_equal(o, expect) for o in outs)


# --------------------------------------------------------------------------
# R = 1 is the identity on every non-NaN bit pattern, NaN stays NaN.

def pin_identity(lib):
    fails = []
    x = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    (y,) = run(lib, [x])
    is_nan = ((x & 0x7F80) == 0x7F80) & ((x & 0x007F) != 0)
    if not np.array_equal(y[~is_nan], x[~is_nan]):
        bad = np.nonzero(y[~is_nan] != x[~is_nan])[0][:4]
        fails.append("R=1 not identity at bit patterns %s" % [hex(int(v)) for v in x[~is_nan][bad]])
    ynan = y[is_nan]
    if not np.all(((ynan & 0x7F80) == 0x7F80) & ((ynan & 0x007F) != 0)):
        fails.append("R=1 NaN input did not stay NaN")
    return fails


# --------------------------------------------------------------------------
# Sums that are exact: their value does not depend on rounding or order.

def pin_all_ones(lib):
    fails = []
    for R in range(1, 9):
        outs = run(lib, [np.full(37, bf16_bits_of(1.0), np.uint16)] * R)
        if not _all_equal(outs, np.full(37, bf16_bits_of(float(R)), np.uint16)):
            fails.append("all-ones R=%d did not give exactly %d" % (R, R))
    return fails


def _exact_int_check(lib, R, count, seed, fill):
    xs = inputs.make_inputs(R, count, seed, fill)
    ints = [x.to(torch.int64).numpy() for x in xs]
    exact = np.sum(np.stack(ints), axis=0)          # integer arithmetic
    assert np.abs(exact).max() <= 256               # exact in bf16
    expect = np.array([bf16_bits_of(float(v)) for v in exact.tolist()], np.uint16)
    outs = run(lib, [inputs.bits(x) for x in xs])
    return _all_equal(outs, expect)


def pin_small_integers(lib):
    fails = []
    for R in range(1, 9):
        for seed in (0, 1, 2):
            if not _exact_int_check(lib, R, 1000 + 7 * R + seed, seed, "ints"):
                fails.append("ints in [-8,8] R=%d seed=%d not summed exactly" % (R, seed))
    return fails


def pin_position_fill(lib):
    fails = []
    for R in (2, 3, 8):
        if not _exact_int_check(lib, R, 4099, 0, "position"):
            fails.append("position-dependent fill R=%d not summed exactly" % R)
    return fails


# --------------------------------------------------------------------------
# Hand-derived closed forms (rank order, a single final rounding, ties to
# even, signed zeros, subnormals, overflow).

P24 = float(1 << 24)
CLOSED_FORMS = [
    # (ranks' values, exact expected result, derivation)
    ([P24, 1.0, 1.0, -P24], 0.0,
     "rank order: 2^24+1 is a tie between 2^24 and 2^24+2 in fp32, even -> 2^24;"
     " +1 -> 2^24 again; -2^24 -> 0.  Any other order gives 1 or 2."),
    ([1.0, 2.0 ** -9, 2.0 ** -9, 2.0 ** -9], 1.0 + 2.0 ** -7,
     "fp32 sum 1+3*2^-9 is exact; one bf16 rounding (spacing 2^-7 at 1): 3/4 of a"
     " spacing above 1 -> 1+2^-7.  Rounding after each add would stay at 1."),
    ([1.0, 2.0 ** -8], 1.0,
     "1+2^-8 is exactly halfway between 1 and 1+2^-7; tie to even -> 1."),
    ([1.0 + 2.0 ** -7, 2.0 ** -8], 1.0 + 2.0 ** -6,
     "1+2^-7+2^-8 is halfway between 1+2^-7 (odd last bit) and 1+2^-6 (even) -> 1+2^-6."),
    ([-0.0], -0.0, "R=1 keeps the sign of zero."),
    ([-0.0, -0.0], -0.0, "(-0)+(-0) = -0 under round to nearest."),
    ([-0.0, 0.0], 0.0, "(-0)+(+0) = +0 under round to nearest."),
    ([3.0, -3.0, 5.0], 5.0, "exact: 3-3 = +0, +5 = 5."),
    ([value_of_bits(0x7F7F), value_of_bits(0x7F7F)], float("inf"),
     "2 x largest finite bf16 (~3.39e38) exceeds the fp32 range -> +inf."),
    ([value_of_bits(0xFF7F), value_of_bits(0xFF7F)], float("-inf"), "negative overflow -> -inf."),
    ([value_of_bits(0x0001)] * 8, value_of_bits(0x0008),
     "8 x smallest subnormal bf16 (2^-133) = 2^-130, exact, no flush to zero."),
    ([value_of_bits(0x0080), -value_of_bits(0x0001)], value_of_bits(0x007F),
     "smallest normal minus smallest subnormal = largest subnormal, exact."),
    ([float("inf"), 1.0], float("inf"), "inf + finite = inf."),
]


def pin_closed_forms(lib):
    fails = []
    for vals, expect, why in CLOSED_FORMS:
        xs = [np.array([bf16_bits_of(v)], np.uint16) for v in vals]
        outs = run(lib, xs)
        want = bf16_bits_of(expect)
        got = [int(o[0]) for o in outs]
        if any(g != want for g in got):
            fails.append("closed form %s: got %s want %s (%s)"
                         % (vals, [hex(g) for g in got], hex(want), why))
    # inf + (-inf) is invalid: the result must be a NaN.
    (y,) = run(lib, [np.array([0x7F80], np.uint16), np.array([0xFF80], np.uint16)])[:1]
    if not (int(y[0]) & 0x7F80 == 0x7F80 and int(y[0]) & 0x7F):
        fails.append("inf + -inf did not give NaN")
    return fails


# --------------------------------------------------------------------------
# Rounding against a library routine (torch's fp32 -> bf16 conversion).

def _rounding_subset():
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = [0x0000, 0x0001, 0x3FFF, 0x7FFF, 0x8000, 0x8001, 0xBFFF, 0xFFFE, 0xFFFF]
    rng = np.random.default_rng(12345)
    lows += [int(v) for v in rng.integers(0, 1 << 16, 7)]
    parts = [hi | np.uint32(lo) for lo in lows]
    parts.append(rng.integers(0, 1 << 32, 1 << 22, dtype=np.uint64).astype(np.uint32))
    return np.concatenate(parts)


def compare_rounding(lib, u32: np.ndarray):
    """Returns the bit patterns where the oracle and torch disagree."""
    f = u32.view(np.float32)
    mine = oracle.f32_to_bf16(f, lib=lib)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan_in = np.isnan(f)
    mine_nan = ((mine & 0x7F80) == 0x7F80) & ((mine & 0x7F) != 0)
    bad = (~nan_in & (mine != ref)) | (nan_in & ~mine_nan)
    return u32[bad]


def pin_rounding(lib):
    bad = compare_rounding(lib, _rounding_subset())
    if bad.size:
        return ["fp32->bf16 differs from torch at %s" % [hex(int(v)) for v in bad[:4]]]
    return []


# --------------------------------------------------------------------------
# Whole path against library routines on tiny inputs: torch's fp32 additions
# in rank order followed by torch's bf16 conversion.

def library_rank_order_sum(xs):
    acc = xs[0].to(torch.float32)
    for x in xs[1:]:
        acc = acc + x.to(torch.float32)
    return inputs.bits(acc.to(torch.bfloat16))


def pin_tiny_brute_force(lib):
    fails = []
    for R in range(1, 9):
        for count in list(range(1, 68, 3)) + [67]:
            xs = inputs.make_inputs(R, count, seed=R * 100 + count, fill="normal")
            # widen the dynamic range so cancellation and rounding both occur
            scale = torch.tensor([2.0 ** ((k % 9) - 4) for k in range(count)], dtype=torch.float32)
            xs = [(x.float() * scale).to(torch.bfloat16) for x in xs]
            expect = library_rank_order_sum(xs)
            outs = run(lib, [inputs.bits(x) for x in xs])
            if not _all_equal(outs, expect):
                fails.append("brute force R=%d count=%d differs from torch rank-order sum" % (R, count))
                break
    return fails


def pin_outputs_identical_and_in_place(lib):
    fails = []
    xs = [inputs.bits(x).copy() for x in inputs.make_inputs(5, 257, 3, "normal")]
    outs = run(lib, xs)
    if not all(np.array_equal(outs[0], o) for o in outs):
        fails.append("ranks' outputs differ")
    expect = library_rank_order_sum([inputs.from_bits(x) for x in xs])
    bufs = [x.copy() for x in xs]
    oracle.allreduce_bf16(bufs, lib=lib, outputs=bufs)
    if not all(np.array_equal(b, expect) for b in bufs):
        fails.append("in-place call differs from the rank-order sum")
    return fails


# --------------------------------------------------------------------------
# Reduce-scatter and all-gather (the other two collectives the one-shot
# kernel of the torchcomms relay page serves).

def pin_reduce_scatter_exact(lib):
    fails = []
    for R, rc in ((1, 13), (2, 7), (4, 1003), (8, 129)):
        for fill in ("ints", "position"):
            xs = inputs.make_inputs(R, R * rc, seed=R + rc, fill=fill)
            ints = np.stack([x.to(torch.int64).numpy() for x in xs])
            outs = oracle.reduce_scatter_bf16([inputs.bits(x) for x in xs], lib=lib)
            for r in range(R):
                exact = ints[:, r * rc:(r + 1) * rc].sum(axis=0)
                want = np.array([bf16_bits_of(float(v)) for v in exact.tolist()], np.uint16)
                if not np.array_equal(outs[r], want):
                    fails.append("reduce-scatter %s R=%d rc=%d block %d not exact" % (fill, R, rc, r))
    return fails


def pin_reduce_scatter_order(lib):
    """The rank-order closed form placed in one block of a 4-rank call."""
    fails = []
    R, rc = 4, 5
    vals = [P24, 1.0, 1.0, -P24]
    for blk in range(R):
        xs = []
        for s in range(R):
            a = np.zeros(R * rc, np.uint16)
            a[blk * rc:(blk + 1) * rc] = bf16_bits_of(vals[s])
            xs.append(a)
        outs = oracle.reduce_scatter_bf16(xs, lib=lib)
        for r in range(R):
            want = 0 if r != blk else bf16_bits_of(0.0)
            if not (outs[r] == want).all():
                fails.append("reduce-scatter order case, block %d, rank %d" % (blk, r))
    return fails


def pin_all_gather_exact(lib):
    fails = []
    for R, sc in ((1, 9), (3, 17), (8, 257)):
        xs = inputs.make_inputs(R, sc, seed=0, fill="position")
        outs = oracle.all_gather_bf16([inputs.bits(x) for x in xs], lib=lib)
        for r in range(R):
            for s in range(R):
                # the position fill written out again from its formula
                want = [bf16_bits_of(float(((7 * j + 13 * s) % 17) - 8)) for j in range(sc)]
                if outs[r][s * sc:(s + 1) * sc].tolist() != want:
                    fails.append("all-gather R=%d rank %d block %d" % (R, r, s))
    return fails


# --------------------------------------------------------------------------
# fp16 and fp32 element types.

def f16_bits_of(x: float) -> int:
    """Bits of a value exactly representable in fp16 (checked with numpy)."""
    h = np.array([x], dtype=np.float16)
    if float(h[0]) != x and x == x:
        raise ValueError("%r is not exactly representable in fp16" % x)
    return int(h.view(np.uint16)[0])


def compare_rounding_f16(lib, u32: np.ndarray):
    f = u32.view(np.float32)
    mine = oracle.f32_to_f16(f, lib=lib)
    ref = torch.from_numpy(f.copy()).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    nan_in = np.isnan(f)
    mine_nan = ((mine & 0x7C00) == 0x7C00) & ((mine & 0x3FF) != 0)
    bad = (~nan_in & (mine != ref)) | (nan_in & ~mine_nan)
    return u32[bad]


def pin_f16_rounding(lib):
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = [0x0000, 0x0001, 0x0FFF, 0x1000, 0x1001, 0x1FFF, 0x2000, 0x2001, 0x7FFF, 0x8000,
            0xFFFF]
    rng = np.random.default_rng(99)
    parts = [hi | np.uint32(lo) for lo in lows]
    parts.append(rng.integers(0, 1 << 32, 1 << 22, dtype=np.uint64).astype(np.uint32))
    bad = compare_rounding_f16(lib, np.concatenate(parts))
    return ["fp32->fp16 differs from torch at %s" % [hex(int(v)) for v in bad[:4]]] if bad.size else []


def pin_f16_widening(lib):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    mine = np.array([lib.oracle_f16_to_f32(int(v)) for v in h], dtype=np.float32)
    ref = torch.from_numpy(h.view(np.int16)).view(torch.float16).float().numpy()
    nan = np.isnan(ref)
    bad = (~nan & (mine.view(np.uint32) != ref.view(np.uint32))) | (nan & ~np.isnan(mine))
    return ["fp16->fp32 differs from torch at %s" % [hex(int(v)) for v in h[bad][:4]]] if bad.any() else []


F16_CLOSED_FORMS = [
    ([1.0, 2.0 ** -11], 1.0, "1+2^-11 is halfway between 1 and 1+2^-10; tie to even -> 1."),
    ([1.0 + 2.0 ** -10, 2.0 ** -11], 1.0 + 2.0 ** -9,
     "halfway between 1+2^-10 (odd) and 1+2^-9 (even) -> 1+2^-9."),
    ([1.0, 2.0 ** -12, 2.0 ** -12, 2.0 ** -12], 1.0 + 2.0 ** -10,
     "1+3*2^-12 is exact in fp32; one rounding: 3/4 of an fp16 spacing -> 1+2^-10."),
    ([65504.0, 16.0], float("inf"),
     "65520 is halfway between 65504 (odd last bit) and 65536 (= overflow) -> inf."),
    ([65504.0, 15.0], 65504.0, "65519 is below the halfway point 65520 -> 65504."),
    ([2.0 ** -24] * 8, 2.0 ** -21, "8 x smallest subnormal = 2^-21, exact, no flush."),
    ([2.0 ** -14, -(2.0 ** -24)], 2.0 ** -14 - 2.0 ** -24, "largest subnormal, exact."),
    ([2.0 ** -25, 2.0 ** -26], 2.0 ** -24,
     "3*2^-26 is 3/4 of the subnormal spacing 2^-24 -> 2^-24."),
    ([2.0 ** -25], 0.0, "2^-25 is halfway between 0 (even) and 2^-24 -> +0."),
    ([-0.0, -0.0], -0.0, "(-0)+(-0) = -0."),
]


def pin_f16_closed_forms(lib):
    fails = []
    for vals, expect, why in F16_CLOSED_FORMS:
        # 2^-25 and 2^-26 are not fp16 values: feed them as fp32 sums of fp16 inputs where
        # needed; every input below is exact in fp16 except those two, which only appear
        # in the rounding cases and are applied through the fp32 -> fp16 routine directly.
        if any(v != 0 and abs(v) < 2.0 ** -24 for v in vals):
            acc = np.float32(vals[0])
            for v in vals[1:]:
                acc = np.float32(acc + np.float32(v))
            got = int(oracle.f32_to_f16(np.array([acc], np.float32), lib=lib)[0])
        else:
            xs = [np.array([f16_bits_of(v)], np.uint16) for v in vals]
            got = int(oracle.allreduce_f16(xs, lib=lib)[0][0])
        want = f16_bits_of(expect)
        if got != want:
            fails.append("fp16 closed form %s: got %s want %s (%s)" % (vals, hex(got), hex(want), why))
    return fails


def pin_f32_exact(lib):
    fails = []
    for R in (1, 3, 8):
        xs = [np.array([((7 * i + 13 * r) % 17) - 8 for i in range(301)], np.float32)
              for r in range(R)]
        exact = np.sum(np.stack(xs).astype(np.int64), axis=0).astype(np.float32)
        outs = oracle.allreduce_f32(xs, lib=lib)
        if not all(np.array_equal(o, exact) for o in outs):
            fails.append("fp32 integer sums R=%d" % R)
    outs = oracle.allreduce_f32([np.array([v], np.float32) for v in (P24, 1.0, 1.0, -P24)], lib=lib)
    if float(outs[0][0]) != 0.0:
        fails.append("fp32 rank order closed form gave %r" % float(outs[0][0]))
    return fails


ALL_PINS = [
    pin_identity, pin_all_ones, pin_small_integers, pin_position_fill,
    pin_closed_forms, pin_rounding, pin_tiny_brute_force,
    pin_outputs_identical_and_in_place, pin_reduce_scatter_exact, pin_reduce_scatter_order,
    pin_all_gather_exact, pin_f16_rounding, pin_f16_widening, pin_f16_closed_forms,
    pin_f32_exact,
]


def all_failures(lib):
    fails = []
    for pin in ALL_PINS:
        fails += pin(lib)
    return fails
