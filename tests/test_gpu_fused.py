"""Fused LL8 kernel: flag rotation, stale-packet rejection, bounded waits
(made to run out from the host side, no GPU fault), epoch wrap and CUDA-graph
replay."""
import pytest
import torch

from shot_allreduce_ranks_gb300 import inputs
from shot_allreduce_ranks_gb300._lib import AR_ERR_TIMEOUT, AR_OK
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu

R, COUNT = 8, 65_536 * 8 + 11


@pytest.fixture(scope="module")
def ar():
    h = G.handle(R, COUNT)
    h.set_variant("fused_ll8")
    yield h
    h.set_spin_limit_ns(100_000_000)
    G.release_handles()


PACKET_VARIANTS = ["fused_ll8", "fused_ll8_staged", "packet_3op"]


def _bufs(xs):
    bufs = G.to_device(xs)
    return bufs, [torch.empty_like(b) for b in bufs]


def test_epoch_advances_once_per_call(ar):
    xs = inputs.make_inputs(R, COUNT, 1)
    bufs, outs = _bufs(xs)
    e0 = ar.debug_get_epoch()
    for _ in range(5):
        ar(bufs, outs)
    assert ar.debug_get_epoch() == e0 + 5
    G.check_all_outputs(outs, G.oracle_expect(xs), "after 5 calls")


def _flag_after(e, k):
    """The k-th epoch after e in the sequence 1 .. 2^32-1 that skips 0."""
    return (e - 1 + k) % 0xFFFFFFFF + 1


@pytest.mark.parametrize("variant", ["fused_ll8", "packet_3op"])
def test_epoch_wraps_to_one_skipping_zero(ar, variant):
    """A call moves the epoch by one flag value.  Started just below 2^32,
    three calls carry the flags across the wrap, skipping 0, and every one
    is correct."""
    ar.set_variant(variant)
    xs = inputs.make_inputs(R, COUNT, 2)
    want = G.oracle_expect(xs)
    bufs, outs = _bufs(xs)
    e0 = ar.debug_get_epoch()
    ar(bufs, outs)
    step = ar.debug_get_epoch() - e0
    assert step == 1
    e = 0xFFFFFFFF - step
    ar.debug_set_epoch(e)
    for call in range(3):
        for o in outs:
            o.zero_()
        ar(bufs, outs)
        e = _flag_after(e, step)
        assert ar.debug_get_epoch() == e
        G.check_all_outputs(outs, want, "%s call %d near the wrap" % (variant, call))
    assert ar.device_status() == AR_OK
    ar.set_variant("fused_ll8")


@pytest.mark.parametrize("variant", PACKET_VARIANTS)
def test_epoch_advances_once_per_call_every_packet_variant(ar, variant):
    """By one per call."""
    xs = inputs.make_inputs(R, COUNT, 11)
    bufs, outs = _bufs(xs)
    ar.set_variant(variant)
    e0 = ar.debug_get_epoch()
    ar(bufs, outs)
    step = ar.debug_get_epoch() - e0
    assert step == 1
    for _ in range(2):
        ar(bufs, outs)
    assert ar.debug_get_epoch() == e0 + 3 * step
    G.check_all_outputs(outs, G.oracle_expect(xs), variant)
    ar.set_variant("fused_ll8")


@pytest.mark.parametrize("variant", PACKET_VARIANTS)
@pytest.mark.parametrize("skip", [0, 3, R - 1])
def test_missing_producer_times_out_and_next_call_recovers(ar, variant, skip):
    """Rank `skip` stores no packets for one call: its owners' waits run out
    after the (short) spin limit, the device error word says so, and the
    next call, with a newer epoch, is correct."""
    ar.set_variant(variant)
    xs = inputs.make_inputs(R, COUNT, 3)
    want = G.oracle_expect(xs)
    bufs, outs = _bufs(xs)
    assert ar.device_status() == AR_OK
    ar.set_spin_limit_ns(2_000_000)
    ar.debug_skip_producer(skip)
    ar(bufs, outs)
    assert ar.device_status() == AR_ERR_TIMEOUT
    waiting, missing, waits = ar.last_timeout()
    assert missing == skip, (waiting, missing, waits)
    assert 0 <= waiting < R and waiting != skip and waits >= 1
    assert ar.device_status() == AR_OK  # reading clears it
    assert ar.last_timeout() == (waiting, missing, waits)  # the last one reported stays
    ar(bufs, outs)
    assert ar.device_status() == AR_OK
    G.check_all_outputs(outs, want, "call after a timeout")
    ar.set_spin_limit_ns(100_000_000)
    ar.set_variant("fused_ll8")


def test_stale_packets_are_rejected(ar):
    """Call A fills every packet slot with epoch e.  Call B (epoch e+1) gets
    no packets from rank 2: with a constant flag (Flag = 1) it would consume
    A's packets and return A's data silently; with rotation it must time out."""
    xa = inputs.make_inputs(R, COUNT, 4)
    bufs, outs = _bufs(xa)
    ar(bufs, outs)
    assert ar.device_status() == AR_OK
    xb = inputs.make_inputs(R, COUNT, 5)
    for b, x in zip(bufs, xb):
        b.copy_(x)
    ar.set_spin_limit_ns(2_000_000)
    ar.debug_skip_producer(2)
    ar(bufs, outs)
    assert ar.device_status() == AR_ERR_TIMEOUT
    ar.set_spin_limit_ns(100_000_000)
    ar(bufs, outs)
    assert ar.device_status() == AR_OK
    G.check_all_outputs(outs, G.oracle_expect(xb), "after stale-packet timeout")


def test_graph_replay_with_changing_inputs(ar):
    """Capture one fused call into a CUDA graph, then replay it with inputs
    that change between replays.  The epoch lives on the device, so every
    replay rotates it (a by-value epoch would be baked into the graph)."""
    bufs = [torch.empty(COUNT, dtype=torch.bfloat16, device=G.DEV) for _ in range(R)]
    outs = [torch.empty_like(b) for b in bufs]
    in_tbl, out_tbl = ar.tables(bufs, outs)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ar.allreduce_tables(in_tbl, out_tbl, COUNT)  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ar.allreduce_tables(in_tbl, out_tbl, COUNT)
    torch.cuda.synchronize()
    e0 = ar.debug_get_epoch()
    for rep in range(6):
        xs = inputs.make_inputs(R, COUNT, 50 + rep)
        for b, x in zip(bufs, xs):
            b.copy_(x)
        g.replay()
        torch.cuda.synchronize()
        G.check_all_outputs(outs, G.oracle_expect(xs), "replay %d" % rep)
    assert ar.debug_get_epoch() == e0 + 6
    assert ar.device_status() == AR_OK


def _replay_time_us(g):
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3


@pytest.mark.parametrize("rank", [0, 5])
def test_graph_replay_with_a_skewed_producer(ar, rank):
    """The capture-and-replay check of "Add HIP-graph capture coverage for
    the sharded-relay collectives" (torchcomms #3850, summary), with one
    producer late: the warps of virtual rank `rank` wait 40 us of the device
    timer before their first packet store on every replay (the delay is a
    launch argument, so the captured call keeps it), and the inputs change
    between replays.  Owners therefore poll for that rank's packets while
    its slots still hold the previous replay's packets; a flag that did not
    rotate per replay (a by-value or hardcoded epoch) would accept them and
    return the previous replay's sums.  Every replay must equal the oracle,
    the epoch must move by one per replay, and no wait may run out."""
    delay_ns = 40_000
    bufs = [torch.empty(COUNT, dtype=torch.bfloat16, device=G.DEV) for _ in range(R)]
    outs = [torch.empty_like(b) for b in bufs]
    in_tbl, out_tbl = ar.tables(bufs, outs)
    ar.set_variant("fused_ll8")
    ar.debug_delay_producer(rank, delay_ns)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ar.allreduce_tables(in_tbl, out_tbl, COUNT)  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ar.allreduce_tables(in_tbl, out_tbl, COUNT)
    ar.debug_delay_producer(-1, 0)  # later launches run undelayed; the graph keeps its copy
    torch.cuda.synchronize()
    e0 = ar.debug_get_epoch()
    reps = 8
    for rep in range(reps):
        xs = inputs.make_inputs(R, COUNT, 70 + rep)
        for b, x in zip(bufs, xs):
            b.copy_(x)
        torch.cuda.synchronize()
        assert _replay_time_us(g) >= delay_ns / 1e3  # the producer really was late
        G.check_all_outputs(outs, G.oracle_expect(xs), "skewed replay %d" % rep)
    assert ar.debug_get_epoch() == e0 + reps
    assert ar.device_status() == AR_OK
    # and an undelayed eager call afterwards is correct too
    xs = inputs.make_inputs(R, COUNT, 99)
    for b, x in zip(bufs, xs):
        b.copy_(x)
    ar.allreduce_tables(in_tbl, out_tbl, COUNT)
    torch.cuda.synchronize()
    G.check_all_outputs(outs, G.oracle_expect(xs), "eager after skewed replays")


def test_delay_hook_bounds():
    from shot_allreduce_ranks_gb300 import ArError
    h = G.handle(R, COUNT)
    with pytest.raises(ArError):
        h.debug_delay_producer(R, 1000)
    with pytest.raises(ArError):
        h.debug_delay_producer(0, 20_000_000)  # above the 10 ms bound
    h.debug_delay_producer(-1, 0)


RING_COUNT = 3 * 65_536 * 8 + 5


@pytest.fixture(params=[1, 2], ids=["lead1", "lead2"])
def ring_handle(request, monkeypatch):
    """A handle whose fused calls use the per-CTA packet rings (forced: the
    automatic choice takes them only for messages of several L2 sizes), on a
    grid of 3 CTAs, so that every ring slot is reused hundreds of times in a
    call and the flag moves on once per round."""
    from shot_allreduce_ranks_gb300 import AllReduce
    monkeypatch.setenv("AR_FUSED_RING", "1")
    monkeypatch.setenv("AR_FUSED_LEAD", str(request.param))
    G.ensure_built()
    h = AllReduce(R, RING_COUNT)
    h.set_variant("fused_ll8")
    h.set_launch("fused_ll8", 3, 0)
    yield h
    h.close()


def _rounds_per_call(h, count):
    tr = h.query().fused_threads // R
    groups = (count + 7) // 8
    tiles = ((groups + R - 1) // R + tr - 1) // tr
    return (tiles + 3 - 1) // 3  # 3 CTAs


def test_ring_mode_many_rounds_and_changing_inputs(ring_handle):
    h = ring_handle
    bufs = [torch.empty(RING_COUNT, dtype=torch.bfloat16, device=G.DEV) for _ in range(R)]
    outs = [torch.empty_like(b) for b in bufs]
    in_tbl, out_tbl = h.tables(bufs, outs)
    steps = _rounds_per_call(h, RING_COUNT)
    assert steps > 100
    e0 = h.debug_get_epoch()
    snaps, wants = [], []
    for call in range(4):
        xs = inputs.make_inputs(R, RING_COUNT, seed=300 + call)
        wants.append(G.oracle_expect(xs))
        for b, x in zip(bufs, xs):
            b.copy_(x)
        h.allreduce_tables(in_tbl, out_tbl, RING_COUNT)
        snaps.append([o.clone() for o in outs])
    torch.cuda.synchronize()
    assert h.device_status() == AR_OK
    assert h.debug_get_epoch() == _flag_after(e0, 4 * steps)  # one flag per round
    for call, (snap, want) in enumerate(zip(snaps, wants)):
        G.check_all_outputs(snap, want, "ring call %d" % call)


def test_ring_mode_flags_wrap_inside_a_call(ring_handle):
    """Started 100 flags below 2^32, a call's rounds carry the flag across
    the wrap (skipping 0) partway through; the next call starts after it."""
    h = ring_handle
    xs = inputs.make_inputs(R, RING_COUNT, seed=310)
    want = G.oracle_expect(xs)
    bufs, outs = _bufs(xs)
    steps = _rounds_per_call(h, RING_COUNT)
    e = 0xFFFFFFFF - 100
    h.debug_set_epoch(e)
    for call in range(2):
        for o in outs:
            o.zero_()
        h(bufs, outs)
        e = _flag_after(e, steps)
        assert h.debug_get_epoch() == e
        G.check_all_outputs(outs, want, "ring call %d across the wrap" % call)
    assert h.device_status() == AR_OK


@pytest.mark.parametrize("skip", [0, R - 1])
def test_ring_mode_missing_producer_times_out_and_recovers(ring_handle, skip):
    """A rank that stores nothing: its owners' waits run out, every warp of
    the CTA leaves the loop through the same barrier, the error word says
    so, and the next call is correct."""
    h = ring_handle
    xs = inputs.make_inputs(R, RING_COUNT, seed=320)
    want = G.oracle_expect(xs)
    bufs, outs = _bufs(xs)
    h.set_spin_limit_ns(2_000_000)
    h.debug_skip_producer(skip)
    h(bufs, outs)
    assert h.device_status() == AR_ERR_TIMEOUT
    waiting, missing, _ = h.last_timeout()
    assert missing == skip and waiting != skip, (waiting, missing)
    h(bufs, outs)
    assert h.device_status() == AR_OK
    G.check_all_outputs(outs, want, "ring call after a timeout")
    h.set_spin_limit_ns(100_000_000)


@pytest.mark.parametrize("mode,variant", [("drop", "fused_ll8"), ("ring", "fused_ll8"),
                                          ("drop", "fused_ll8_staged"),
                                          ("drop_lead1", "fused_ll8_staged")])
@pytest.mark.parametrize("ranks", [3, 4, 8])
def test_forced_packet_modes_on_ragged_counts(mode, variant, ranks, monkeypatch):
    """The line drops (their boundary: only lines holding a group below the
    shard's end are dropped; without write mode, also the result packets'
    lines) and the rings, forced on counts that end in a partial tile, a
    partial group and an odd shard, two calls in a row per count with
    different inputs: a line dropped from the wrong slot, or a stale packet
    taken for a new one, would show up as a wrong sum or a timeout."""
    from shot_allreduce_ranks_gb300 import AllReduce
    if mode.startswith("drop"):
        monkeypatch.setenv("AR_FUSED_DISCARD", "1")
        monkeypatch.setenv("AR_FUSED_RING", "0")
    else:
        monkeypatch.setenv("AR_FUSED_RING", "1")
    if mode == "drop_lead1":
        monkeypatch.setenv("AR_FUSED_LEAD", "1")
    counts = [9, 4097, 65_541, 300_003]
    G.ensure_built()
    with AllReduce(ranks, max(counts)) as h:
        h.set_variant(variant)
        for count in counts:
            for call in range(2):
                xs = inputs.make_inputs(ranks, count, seed=500 + call + count % 97)
                outs = h([x.to(G.DEV) for x in xs])
                torch.cuda.synchronize()
                G.check_all_outputs(outs, G.oracle_expect(xs), "%s %s R=%d count=%d call %d"
                                    % (variant, mode, ranks, count, call))
        assert h.debug_guards_intact(), "a packet store landed outside its region"
        assert h.device_status() == AR_OK


@pytest.mark.parametrize("variant,count,calls", [("fused_ll8", 4096 * 3 + 5, 200_000),
                                                 ("fused_ll8", 65_536 * 8 + 11, 20_000),
                                                 ("fused_ll8_staged", 4096 * 3 + 5, 50_000)])
def test_soak_many_graph_replayed_calls(variant, count, calls):
    """Many back-to-back calls replayed from one CUDA graph of 1000 calls (the
    epoch advancing on every one): no packet wait may run out, the epoch must
    have moved by the number of calls, and the last call's outputs are
    bit-exact."""
    R = 8
    ar = G.handle(R, count)
    ar.set_variant(variant)
    xs = inputs.make_inputs(R, count, seed=77)
    bufs = G.to_device(xs)
    outs = [torch.empty_like(b) for b in bufs]
    in_tbl, out_tbl = ar.tables(bufs, outs)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ar.allreduce_tables(in_tbl, out_tbl, count)
    torch.cuda.synchronize()
    per_graph = 1000
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(per_graph):
            ar.allreduce_tables(in_tbl, out_tbl, count)
    torch.cuda.synchronize()
    e0 = ar.debug_get_epoch()
    for o in outs:
        o.zero_()
    for _ in range(calls // per_graph):
        g.replay()
    torch.cuda.synchronize()
    assert ar.device_status() == AR_OK
    assert ar.debug_get_epoch() == _flag_after(e0, (calls // per_graph) * per_graph)
    G.check_all_outputs(outs, G.oracle_expect(xs), "%s after %d calls" % (variant, calls))
    ar.set_variant("fused_ll8")


# Packet handling the handle picks per call on a GB300 (its L2 size decides):
# (R, elements per rank) -> (lead, line drops, ring rounds).  The benchmark
# sizes, and the measured crossovers of the rules (scratch left alone while
# packets, inputs and outputs fit L2; drops above; rings above 2 L2 of
# packets).
AUTO_MODES = [
    (8, 2_252_800, (2, 0, 0)),    # 440x5120: 63 MB of packets, 135 MB in all
    (8, 4_194_304, (2, 1, 0)),    # 512x8192: 117 MB of packets
    (8, 10_485_760, (1, 0, 2)),   # 294 MB of packets, above 2 L2
    (8, 33_554_432, (1, 0, 2)),   # 64 MiB per rank
    (4, 4_194_304, (2, 0, 0)),    # 50 MB of packets, 117 MB in all
    (4, 33_554_432, (1, 0, 2)),   # 64 MiB per rank: 403 MB of packets
    (3, 8_388_608, (2, 1, 0)),    # 67 MB of packets, 168 MB in all
]


@pytest.mark.parametrize("R_, count, want", AUTO_MODES)
def test_automatic_packet_mode(R_, count, want, monkeypatch, capfd):
    """The call's packet handling, as AR_LOG reports it, is the one the
    measured rules give for this size; the call is still correct."""
    import re

    from shot_allreduce_ranks_gb300 import AllReduce
    for k in ("AR_FUSED_RING", "AR_FUSED_DISCARD", "AR_FUSED_LEAD"):
        monkeypatch.delenv(k, raising=False)
    monkeypatch.setenv("AR_LOG", "1")
    bufs = [torch.full((count,), float(r + 1), dtype=torch.bfloat16, device=G.DEV)
            for r in range(R_)]
    outs = [torch.empty_like(b) for b in bufs]
    with AllReduce(R_, count) as h:
        h.set_variant("fused_ll8")
        capfd.readouterr()
        h(bufs, outs)
        torch.cuda.synchronize()
        assert h.device_status() == AR_OK
    err = capfd.readouterr().err
    m = re.search(r"packets: lead=(\d+) discard=(\d+) ring_rounds=(\d+)", err)
    assert m, err
    assert tuple(int(x) for x in m.groups()) == want
    total = float(R_ * (R_ + 1) // 2)  # exact in bf16 for R <= 8
    for o in outs:
        assert bool((o == total).all())
    del bufs, outs
    torch.cuda.empty_cache()
