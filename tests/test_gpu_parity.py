"""CUDA path vs oracle, bit for bit (tolerance 0 ULP), through the C ABI.

Every variant must produce exactly the oracle's result: fp32 accumulation in
rank order 0..R-1 and one round-to-nearest-even to bf16, identical in every
rank's output.  Where floating point could decide nothing else, NaN payloads
are the only freedom (any NaN equals any NaN).
"""
import numpy as np
import pytest
import torch

from shot_allreduce_ranks_gb300 import ArError, inputs
from shot_allreduce_ranks_gb300._lib import AR_ERR_INVALID_ARG
from tests import gpu_helpers as G
from tests import oracle_pins as P

pytestmark = pytest.mark.gpu

RAGGED = [1, 7, 8, 9, 63, 4095, 4097, 3 * 65536 + 5]


@pytest.fixture(scope="module", autouse=True)
def _cleanup():
    yield
    G.release_handles()


@pytest.mark.parametrize("variant", G.PARITY_VARIANTS)
@pytest.mark.parametrize("R", [1, 2, 3, 4, 5, 6, 7, 8])
def test_ragged_counts(variant, R):
    ar = G.handle(R, max(RAGGED))
    for count in RAGGED:
        xs = inputs.make_inputs(R, count, seed=count % 7, fill="normal")
        want = G.oracle_expect(xs)
        outs = G.run_variant(ar, G.to_device(xs), variant)
        G.check_all_outputs(outs, want, "%s R=%d count=%d" % (variant, R, count))
    assert ar.debug_guards_intact(), "%s R=%d wrote outside a packet region" % (variant, R)


FULL = ["r8_4096", "r8_440x5120", "r8_512x5120", "r8_512x7168", "r8_512x8192",
        "r8_632x5120", "r8_680x5120"] + [
    n for n in inputs.WORKLOADS if n.startswith("r8_") and n.endswith(("_ints", "_normal"))
] + ["r4_64mib", "r8_64mib"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_configs(name):
    """Every benchmark workload at its full size, default launch shapes (the
    ones bench.py times), every variant plus the selector, all outputs."""
    w = inputs.WORKLOADS[name]
    ar = G.handle(w.R, w.count)
    seeds = (0, 1, 2)
    for seed in seeds:
        xs = inputs.make_inputs(w.R, w.count, seed, w.fill)
        want = G.oracle_expect(xs)
        xd = G.to_device(xs)
        outs = [torch.empty_like(x) for x in xd]
        for variant in G.PARITY_VARIANTS + ["auto"]:
            for o in outs:
                o.fill_(float("nan"))
            G.run_variant(ar, xd, variant, outs)
            G.check_all_outputs(outs, want, "%s %s seed=%d" % (name, variant, seed))
        del xd, outs
    assert ar.debug_guards_intact(), "%s: a write outside a packet region" % name
    torch.cuda.empty_cache()


@pytest.mark.parametrize("variant", G.PARITY_VARIANTS)
def test_exact_integer_sums_without_oracle(variant):
    """Integers in [-8, 8] sum exactly: pins the GPU independently of the oracle."""
    R, count = 8, 1 << 20
    ar = G.handle(R, count)
    for fill in ("ints", "position"):
        xs = inputs.make_inputs(R, count, seed=5, fill=fill)
        exact = torch.stack([x.to(torch.int64) for x in xs]).sum(0)
        want = inputs.bits(exact.to(torch.bfloat16))
        outs = G.run_variant(ar, G.to_device(xs), variant)
        G.check_all_outputs(outs, want, "%s %s" % (variant, fill))


@pytest.mark.parametrize("variant", G.PARITY_VARIANTS)
def test_closed_forms_on_gpu(variant):
    """The hand-derived closed forms of the oracle pins hold on the GPU too
    (rank order, single rounding, ties to even, signed zero, subnormals,
    overflow, infinities, NaN)."""
    cases = P.CLOSED_FORMS + [([float("inf"), float("-inf")], None, "NaN")]
    for vals, expect, why in cases:
        R = len(vals)
        ar = G.handle(R, 64)
        # the same case in every element of a 3-group buffer, ragged tail
        count = 21
        xs = [inputs.from_bits(np.full(count, P.bf16_bits_of(v), np.uint16)) for v in vals]
        outs = G.run_variant(ar, G.to_device(xs), variant)
        for o in outs:
            got = G.device_bits(o)
            if expect is None:
                assert G.is_nan_bits(got).all(), (variant, vals)
            else:
                want = np.full(count, P.bf16_bits_of(expect), np.uint16)
                G.assert_bitexact(got, want, "%s %s (%s)" % (variant, vals, why))


@pytest.mark.parametrize("variant", G.PARITY_VARIANTS)
def test_special_values_mixed(variant):
    """Random bit patterns (all classes: subnormal, huge, inf, NaN) vs oracle."""
    R, count = 8, 40_000
    rng = np.random.default_rng(7)
    xs = [inputs.from_bits(rng.integers(0, 1 << 16, count, dtype=np.uint64).astype(np.uint16))
          for _ in range(R)]
    want = G.oracle_expect(xs)
    outs = G.run_variant(G.handle(R, count), G.to_device(xs), variant)
    G.check_all_outputs(outs, want, variant)


@pytest.mark.parametrize("variant", G.PARITY_VARIANTS)
@pytest.mark.parametrize("which", ["inputs", "outputs", "both"])
def test_misaligned_pointers(variant, which):
    """Pointers offset by one element (2 bytes): the call takes the element
    path and still matches."""
    R, count = 8, 4099
    ar = G.handle(R, count + 8)
    xs = inputs.make_inputs(R, count, seed=11, fill="normal")
    want = G.oracle_expect(xs)
    base_in = [torch.empty(count + 8, dtype=torch.bfloat16, device=G.DEV) for _ in range(R)]
    base_out = [torch.empty(count + 8, dtype=torch.bfloat16, device=G.DEV) for _ in range(R)]
    off_in = 1 if which in ("inputs", "both") else 0
    off_out = 1 if which in ("outputs", "both") else 0
    xin = [b[off_in:off_in + count] for b in base_in]
    xout = [b[off_out:off_out + count] for b in base_out]
    for d, x in zip(xin, xs):
        d.copy_(x)
    G.run_variant(ar, xin, variant, xout)
    G.check_all_outputs(xout, want, "%s misaligned %s" % (variant, which))


@pytest.mark.parametrize("variant", G.PARITY_VARIANTS)
def test_in_place(variant):
    R, count = 8, (1 << 20) + 3
    ar = G.handle(R, count)
    xs = inputs.make_inputs(R, count, seed=3, fill="normal")
    want = G.oracle_expect(xs)
    bufs = G.to_device(xs)
    G.run_variant(ar, bufs, variant, bufs)
    G.check_all_outputs(bufs, want, "%s in place" % variant)


@pytest.mark.parametrize("variant", G.PARITY_VARIANTS)
def test_guard_canaries(variant):
    """Nothing is written outside [0, count) of any output, nor outside the
    handle's packet regions."""
    R, count, pad = 8, 1000 * 8 + 5, 64
    ar = G.handle(R, count)
    xs = inputs.make_inputs(R, count, seed=2, fill="normal")
    want = G.oracle_expect(xs)
    bases = [torch.full((count + 2 * pad,), 12345.0, dtype=torch.bfloat16, device=G.DEV)
             for _ in range(R)]
    outs = [b[pad:pad + count] for b in bases]
    G.run_variant(ar, G.to_device(xs), variant, outs)
    G.check_all_outputs(outs, want, variant)
    canary = inputs.bits(torch.tensor([12345.0], dtype=torch.bfloat16))[0]
    for b in bases:
        bits = G.device_bits(b)
        assert (bits[:pad] == canary).all() and (bits[pad + count:] == canary).all()
    assert ar.debug_guards_intact()


def test_back_to_back_calls_with_changing_inputs():
    """Twenty fused calls in a row on one stream, inputs changing every call,
    no synchronisation between them: a stale flag or stale packet would show
    up as wrong data in some call."""
    R, count = 8, 300_000 + 3
    ar = G.handle(R, count)
    ar.set_variant("fused_ll8")
    bufs = [torch.empty(count, dtype=torch.bfloat16, device=G.DEV) for _ in range(R)]
    outs = [torch.empty_like(b) for b in bufs]
    in_tbl, out_tbl = ar.tables(bufs, outs)
    snaps, wants = [], []
    for call in range(20):
        xs = inputs.make_inputs(R, count, seed=100 + call, fill="normal")
        wants.append(G.oracle_expect(xs))
        for b, x in zip(bufs, xs):
            b.copy_(x, non_blocking=False)
        ar.allreduce_tables(in_tbl, out_tbl, count)
        snaps.append([o.clone() for o in outs])
    torch.cuda.synchronize()
    for call, (snap, want) in enumerate(zip(snaps, wants)):
        G.check_all_outputs(snap, want, "call %d" % call)


@pytest.mark.parametrize("R", [8, 4, 3])
def test_fused_launch_shapes(R):
    """The fused kernel is correct for every CTA count it can be given,
    down to one CTA per rank, and for 128/256/512 threads (narrowed to 256
    for R <= 4, the bound that kernel is compiled for)."""
    count = 200_003
    ar = G.handle(R, count)
    if R <= 4:
        assert ar.query().fused_threads <= 256
    xs = inputs.make_inputs(R, count, seed=9, fill="normal")
    want = G.oracle_expect(xs)
    xd = G.to_device(xs)
    for threads in (128, 256, 512):
        for ctas in (R, 3 * R, 64, 152 * 2, 0):
            ar.set_launch("fused_ll8", ctas, threads)
            outs = G.run_variant(ar, xd, "fused_ll8")
            G.check_all_outputs(outs, want, "fused ctas=%d threads=%d" % (ctas, threads))
    ar.set_launch("fused_ll8", 0, 0)


@pytest.mark.parametrize("variant", ["oneshot_pull", "oneshot_fanout", "twophase"])
def test_grid_stride_shapes(variant):
    R, count = 8, 100_001
    ar = G.handle(R, count)
    xs = inputs.make_inputs(R, count, seed=4, fill="normal")
    want = G.oracle_expect(xs)
    xd = G.to_device(xs)
    shapes = ((1, 128), (R, 128), (40, 512), (0, 512), (0, 0))
    if variant != "oneshot_fanout":
        shapes += ((1, 64), (40, 512))
    for ctas, threads in shapes:
        ar.set_launch(variant, ctas, threads)
        outs = G.run_variant(ar, xd, variant)
        G.check_all_outputs(outs, want, "%s ctas=%d threads=%d" % (variant, ctas, threads))
    ar.set_launch(variant, 0, 0)


def test_count_zero_and_bounds():
    R = 4
    ar = G.handle(R, 1000)
    xs = G.to_device(inputs.make_inputs(R, 1000, 0))
    outs = [torch.full_like(x, 7.0) for x in xs]
    ar(xs, outs, count=0)
    torch.cuda.synchronize()
    assert all((o == 7.0).all() for o in outs)
    in_tbl, out_tbl = ar.tables(xs, outs)
    with pytest.raises(ArError) as e:
        ar.allreduce_tables(in_tbl, out_tbl, 1001)
    assert e.value.status == AR_ERR_INVALID_ARG


def test_selector_picks_a_real_variant_and_matches():
    R = 8
    ar = G.handle(R, 1 << 22)
    ar.set_variant("auto")
    for count in (4096, 65536, 1 << 20, 1 << 22):
        assert ar.select(count) in G.PARITY_VARIANTS
        xs = inputs.make_inputs(R, count, seed=1)
        outs = G.run_variant(ar, G.to_device(xs), "auto")
        G.check_all_outputs(outs, G.oracle_expect(xs), "auto count=%d" % count)


def test_host_buffer_path_pageable():
    """Pageable host buffers take the staging-copy path."""
    R, count = 8, 50_003
    ar = G.handle(R, count)
    ar.reserve_host_staging()
    xs = inputs.make_inputs(R, count, seed=16)
    want = G.oracle_expect(xs)
    hout = [torch.empty(count, dtype=torch.bfloat16) for _ in range(R)]
    for variant in ("auto", "fused_ll8", "oneshot_fanout"):
        ar.set_variant(variant)
        ar.allreduce_host(xs, hout)
        torch.cuda.synchronize()
        for r in range(R):
            G.assert_bitexact(inputs.bits(hout[r]), want, "pageable %s rank %d" % (variant, r))


def test_host_buffer_path():
    R, count = 8, 123_457
    ar = G.handle(R, count)
    ar.reserve_host_staging()
    xs = inputs.make_inputs(R, count, seed=6)
    want = G.oracle_expect(xs)
    hin = [x.pin_memory() for x in xs]
    hout = [torch.empty(count, dtype=torch.bfloat16).pin_memory() for _ in range(R)]
    for variant in G.PARITY_VARIANTS + ["auto"]:
        ar.set_variant(variant)
        ar.allreduce_host(hin, hout)
        torch.cuda.synchronize()
        for r in range(R):
            G.assert_bitexact(inputs.bits(hout[r]), want, "host path %s rank %d" % (variant, r))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32],
                         ids=["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("R", [2, 4, 8, 16])
def test_selector_boundaries_bracket_the_measured_crossover(R, dtype):
    """Pull up to about 1.75 MiB / R per rank (fp32: half the elements of
    bf16/fp16), then fan-out; at R = 16 the bulk-copy fan-out up to 720 KiB
    per rank first."""
    from shot_allreduce_ranks_gb300 import AllReduce
    eb = 4 if dtype == torch.float32 else 2
    edge = 917504 * 2 // eb // R // 64 * 64
    bulk_edge = 368640 * 2 // eb if R >= 16 else edge
    with AllReduce(R, max(edge, bulk_edge) + 4096, dtype=dtype) as ar:
        assert ar.select(1) == "oneshot_pull"
        assert ar.select(edge) == "oneshot_pull"
        if R >= 16:
            assert ar.select(edge + 1) == "oneshot_fanout_bulk"
            assert ar.select(bulk_edge) == "oneshot_fanout_bulk"
        assert ar.select(bulk_edge + 1) == "oneshot_fanout"
        assert ar.select(bulk_edge + 4096) == "oneshot_fanout"
        ar.set_variant("fused_ll8" if R <= 8 else "twophase")
        assert ar.select(5) == ("fused_ll8" if R <= 8 else "twophase")


def test_tuning_file_and_forced_variant_env(tmp_path, monkeypatch):
    from shot_allreduce_ranks_gb300 import AllReduce
    table = tmp_path / "table.txt"
    table.write_text("# R max_count variant ctas threads\n8 1000 twophase 0 128\n0 -1 fused_ll8\n")
    monkeypatch.setenv("AR_TUNING_FILE", str(table))
    with AllReduce(8, 5000) as ar:
        assert ar.select(1000) == "twophase"
        assert ar.select(1001) == "fused_ll8"
        xs = inputs.make_inputs(8, 3000, seed=8)
        outs = G.run_variant(ar, G.to_device(xs), "auto")
        G.check_all_outputs(outs, G.oracle_expect(xs), "tuning-file auto")
    monkeypatch.delenv("AR_TUNING_FILE")
    # a table written from sweep timings (bench.py --sweep --write-tuning)
    import bench
    rows = bench.tuning_rows(8, {4096: {"oneshot_pull": 2.0, "oneshot_fanout": 2.5},
                                 16384: {"oneshot_pull": 3.0, "oneshot_fanout": 2.6},
                                 65536: {"twophase": 1.0, "oneshot_fanout": 2.6}})
    written = tmp_path / "written.txt"
    bench.write_tuning(str(written), rows, "test")
    monkeypatch.setenv("AR_TUNING_FILE", str(written))
    with AllReduce(8, 100000) as ar:
        assert ar.select(4096) == "oneshot_pull"
        assert ar.select(8192) == "oneshot_pull"       # up to sqrt(4096 * 16384)
        assert ar.select(8193) == "oneshot_fanout"
        assert ar.select(16384) == "oneshot_fanout"
        assert ar.select(65536) == "twophase"
        assert ar.select(100000) == "twophase"
    monkeypatch.delenv("AR_TUNING_FILE")
    monkeypatch.setenv("AR_VARIANT", "twophase")
    with AllReduce(4, 100) as ar:
        assert ar.select(10) == "twophase"


@pytest.mark.parametrize("pdl", ["1", "0"], ids=["pdl", "no_pdl"])
@pytest.mark.parametrize("variant", ["oneshot_pull", "oneshot_fanout", "twophase",
                                     "oneshot_fanout_bulk"])
def test_chained_calls_see_the_previous_result(variant, pdl, monkeypatch):
    """Each call reads the previous call's outputs, with no host
    synchronisation in between, eagerly and replayed from a CUDA graph.
    With programmatic dependent launch a call is scheduled before the
    previous one has finished; it must still read that call's results."""
    import oracle
    from shot_allreduce_ranks_gb300 import AllReduce
    monkeypatch.setenv("AR_PDL", pdl)
    R, count, calls = 8, 30_001, 6
    xs = inputs.make_inputs(R, count, seed=5, fill="ints")
    cur = [inputs.bits(x) for x in xs]
    for _ in range(calls):
        cur = oracle.allreduce_bf16(cur)
    want = cur[0]
    with AllReduce(R, count) as ar:
        ar.set_variant(variant)
        a = G.to_device(xs)
        b = [torch.empty_like(t) for t in a]
        tabs = [ar.tables(a, b), ar.tables(b, a)]

        def chain():
            for k in range(calls):
                ar.allreduce_tables(*tabs[k % 2], count)

        chain()
        torch.cuda.synchronize()
        G.check_all_outputs(a if calls % 2 == 0 else b, want, "%s eager" % variant)
        for t, x in zip(a, xs):
            t.copy_(x)
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                chain()
        torch.cuda.synchronize()
        for t, x in zip(a, xs):
            t.copy_(x)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        G.check_all_outputs(a if calls % 2 == 0 else b, want, "%s graph" % variant)
        assert ar.device_status() == 0


@pytest.mark.parametrize("variant", ["oneshot_fanout", "oneshot_pull", "twophase"])
def test_two_handles_on_two_streams(variant):
    """One handle per concurrent stream (the threading rule of ar.h): two
    handles run calls on two streams at the same time, inputs changing every
    call, and every call of each stream is exact."""
    import oracle
    from shot_allreduce_ranks_gb300 import AllReduce
    R, count, calls = 8, 200_003, 4
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    with AllReduce(R, count) as h1, AllReduce(R, count) as h2:
        h1.set_variant(variant)
        h2.set_variant(variant)
        runs = []
        for k in range(calls):
            for h, s, seed in ((h1, s1, 300 + k), (h2, s2, 400 + k)):
                xs = inputs.make_inputs(R, count, seed=seed)
                with torch.cuda.stream(s):
                    xd = [x.to(G.DEV, non_blocking=False) for x in xs]
                    outs = h(xd, stream=s)
                runs.append((xs, outs))
        torch.cuda.synchronize()
        for k, (xs, outs) in enumerate(runs):
            want = oracle.allreduce_bf16([inputs.bits(x) for x in xs])[0]
            G.check_all_outputs(outs, want, "%s stream %d call %d" % (variant, k % 2, k // 2))


WIDE = 1 << 21  # bf16 elements in 2^18 groups: where the fan-out starts 32-byte requests


@pytest.mark.parametrize("count", [WIDE - 8, WIDE, WIDE + 8, WIDE + 8 + 3],
                         ids=["below", "at", "odd_groups", "odd_and_partial"])
def test_fanout_wide_requests_edges(count):
    """The fan-out's 32-byte path for large calls: at and around its size
    threshold, with an odd number of whole groups and with a partial last
    group; and pointers that are 16- but not 32-byte aligned, which must take
    the 16-byte path.  All bit-exact against the oracle."""
    R = 8
    ar = G.handle(R, WIDE + 64)
    xs = inputs.make_inputs(R, count, seed=count % 11)
    want = G.oracle_expect(xs)
    ar.set_variant("oneshot_fanout")
    outs = ar(G.to_device(xs))
    torch.cuda.synchronize()
    G.check_all_outputs(outs, want, "fanout count=%d" % count)
    # 16-byte aligned, not 32-byte aligned: views 8 elements into bigger buffers
    base_in = [torch.zeros(count + 8, dtype=torch.bfloat16, device=G.DEV) for _ in range(R)]
    base_out = [torch.zeros(count + 8, dtype=torch.bfloat16, device=G.DEV) for _ in range(R)]
    vin = [b[8:] for b in base_in]
    vout = [b[8:] for b in base_out]
    assert all(v.data_ptr() % 32 == 16 for v in vin + vout)
    for v, x in zip(vin, xs):
        v.copy_(x)
    ar(vin, vout)
    torch.cuda.synchronize()
    G.check_all_outputs(vout, want, "fanout 16B-aligned count=%d" % count)
    ar.set_variant("auto")


@pytest.mark.parametrize("R,count", [(8, (1 << 22) + 8 + 3), (8, 3 * (1 << 22) - 5),
                                     (16, (1 << 22) + 1), (3, (1 << 23) + 13)])
def test_fanout_large_call_grid(R, count):
    """Large calls run the fan-out on a grid of several waves (a thread takes
    at most two 32-byte pairs, or one pass of two groups above eight ranks)
    instead of the co-resident grid: ragged ends (odd whole groups, a partial
    group) at sizes above the switch, bit-exact against the oracle."""
    ar = G.handle(R, count)
    xs = inputs.make_inputs(R, count, seed=count % 13)
    want = G.oracle_expect(xs)
    ar.set_variant("oneshot_fanout")
    outs = ar(G.to_device(xs))
    torch.cuda.synchronize()
    G.check_all_outputs(outs, want, "fanout R=%d count=%d" % (R, count))
    assert ar.device_status() == 0
    ar.set_variant("auto")


@pytest.mark.parametrize("variant", ["oneshot_pull", "oneshot_fanout", "twophase", "fused_ll8",
                                     "fused_ll8_staged", "oneshot_fanout_bulk"])
def test_tables_rewritten_by_copies_between_back_to_back_calls(variant):
    """One pair of device pointer tables, rewritten by a host-to-device copy
    on the call's stream before each of six back-to-back calls (no
    synchronisation in between; small calls, so launched with programmatic
    dependent launch, whose kernels read the tables before waiting for the
    previous kernel): each call must use its own tables."""
    R, count, calls = 8, 4096 * 3 + 5, 6
    ar = G.handle(R, count)
    ar.set_variant(variant)
    xs = [inputs.make_inputs(R, count, seed=900 + c) for c in range(calls)]
    ins = [G.to_device(x) for x in xs]
    outs = [[torch.empty(count, dtype=torch.bfloat16, device=G.DEV) for _ in range(R)]
            for _ in range(calls)]
    tin = torch.empty(R, dtype=torch.int64, device=G.DEV)
    tout = torch.empty(R, dtype=torch.int64, device=G.DEV)
    hosts = [(torch.tensor([t.data_ptr() for t in ins[c]], dtype=torch.int64).pin_memory(),
              torch.tensor([t.data_ptr() for t in outs[c]], dtype=torch.int64).pin_memory())
             for c in range(calls)]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for c in range(calls):
            tin.copy_(hosts[c][0], non_blocking=True)
            tout.copy_(hosts[c][1], non_blocking=True)
            ar.allreduce_tables(tin, tout, count, s)
    s.synchronize()
    for c in range(calls):
        G.check_all_outputs(outs[c], G.oracle_expect(xs[c]), "%s call %d" % (variant, c))
    assert ar.device_status() == 0
    ar.set_variant("auto")
