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


PACKET_VARIANTS = ["fused_ll8", "fused_ll8_staged", "packet_3op", "fused_ll8_ring"]


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


@pytest.mark.parametrize("variant", ["fused_ll8", "fused_ll8_ring", "packet_3op"])
def test_epoch_wraps_to_one_skipping_zero(ar, variant):
    """A call moves the epoch by its number of flag values (one for the
    full-scratch kernels, one per round for the ring).  Started just below
    2^32, three calls carry the flags across the wrap, skipping 0, and every
    one is correct."""
    ar.set_variant(variant)
    xs = inputs.make_inputs(R, COUNT, 2)
    want = G.oracle_expect(xs)
    bufs, outs = _bufs(xs)
    e0 = ar.debug_get_epoch()
    ar(bufs, outs)
    step = ar.debug_get_epoch() - e0
    assert 1 <= step <= 8
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
    """By one per call (the ring: by its rounds per call, the same every call)."""
    xs = inputs.make_inputs(R, COUNT, 11)
    bufs, outs = _bufs(xs)
    ar.set_variant(variant)
    e0 = ar.debug_get_epoch()
    ar(bufs, outs)
    step = ar.debug_get_epoch() - e0
    assert step == 1 or (variant == "fused_ll8_ring" and 1 <= step <= 8)
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
    assert ar.device_status() == AR_OK  # reading clears it
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


@pytest.mark.parametrize("depth_calls", [(0, 2), (3 * R, 5)])
def test_ring_many_rounds(depth_calls):
    """The ring kernel over many rounds (a small grid forces K >> D), so that
    every ring slot is reused and every credit wait is exercised; several
    calls in a row with changing inputs."""
    ctas, calls = depth_calls
    h = G.handle(R, 3 * 65536 * 8 + 5)
    h.set_variant("fused_ll8_ring")
    h.set_launch("fused_ll8_ring", ctas if ctas else R, 128)
    count = 3 * 65536 * 8 + 5
    bufs = [torch.empty(count, dtype=torch.bfloat16, device=G.DEV) for _ in range(R)]
    outs = [torch.empty_like(b) for b in bufs]
    in_tbl, out_tbl = h.tables(bufs, outs)
    snaps, wants = [], []
    for call in range(calls):
        xs = inputs.make_inputs(R, count, seed=200 + call)
        wants.append(G.oracle_expect(xs))
        for b, x in zip(bufs, xs):
            b.copy_(x)
        h.allreduce_tables(in_tbl, out_tbl, count)
        snaps.append([o.clone() for o in outs])
    torch.cuda.synchronize()
    assert h.device_status() == AR_OK
    for call, (snap, want) in enumerate(zip(snaps, wants)):
        G.check_all_outputs(snap, want, "ring call %d" % call)
    h.set_launch("fused_ll8_ring", 0, 0)
