"""The allocation-free entry point (ar_allreduce_fused_noalloc), for callers
that cannot allocate device memory themselves: its outputs must equal those
of the handle-based entry point bit for bit (the tolerance of every parity
test here: 0 ULP), on two calls in a row with different inputs.

Named to be collected last, so that a run stopping at the first failure has
already run every other test.  It needs nothing from earlier tests and
passes alone in a fresh process as well."""
import numpy as np
import pytest
import torch

from shot_allreduce_ranks_gb300 import AllReduce, _lib, build, inputs

pytestmark = pytest.mark.gpu


def _bits(t):
    return inputs.bits(t.cpu())


@pytest.mark.parametrize("R,count", [(8, 1_000_003), (3, 4097)])
def test_noalloc_matches_handle_entry_point_twice(R, count):
    build.build()
    lib = _lib.load()
    assert count <= _lib.noalloc_max_count(R)
    with AllReduce(R, count) as ar:
        ar.set_variant("fused_ll8")
        bufs = [torch.empty(count, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        ref = [torch.empty_like(b) for b in bufs]
        new = [torch.full_like(b, float("nan")) for b in bufs]
        ref_tbl = ar.tables(bufs, ref)
        new_tbl = ar.tables(bufs, new)
        for call in range(2):
            for b, x in zip(bufs, inputs.make_inputs(R, count, seed=40 + call)):
                b.copy_(x)
            ar.allreduce_tables(ref_tbl[0], ref_tbl[1], count)
            st = lib.ar_allreduce_fused_noalloc(
                R, new_tbl[0].data_ptr(), new_tbl[1].data_ptr(), count,
                torch.cuda.current_stream().cuda_stream)
            assert st == _lib.AR_OK, st
            torch.cuda.synchronize()
            want = _bits(ref[0])
            for r in range(R):
                assert np.array_equal(_bits(ref[r]), want)
                got = _bits(new[r])
                bad = np.nonzero(got != want)[0]
                assert bad.size == 0, "call %d rank %d: %d elements differ, first at %d" % (
                    call, r, bad.size, int(bad[0]))


def test_noalloc_rejects_counts_beyond_its_fixed_scratch():
    build.build()
    lib = _lib.load()
    R = 8
    limit = _lib.noalloc_max_count(R)
    bufs = [torch.zeros(16, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    tbl = torch.tensor([b.data_ptr() for b in bufs], dtype=torch.int64, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.ar_allreduce_fused_noalloc(R, tbl.data_ptr(), tbl.data_ptr(), limit + 1,
                                          stream) == _lib.AR_ERR_INVALID_ARG
    assert lib.ar_allreduce_fused_noalloc(R, tbl.data_ptr(), tbl.data_ptr(), 0,
                                          stream) == _lib.AR_OK
    assert lib.ar_allreduce_fused_noalloc(9, tbl.data_ptr(), tbl.data_ptr(), 8,
                                          stream) == _lib.AR_ERR_INVALID_ARG
    assert lib.ar_allreduce_fused_noalloc(R, None, tbl.data_ptr(), 8,
                                          stream) == _lib.AR_ERR_INVALID_ARG


def test_noalloc_switching_counts_and_ranks_against_the_oracle():
    """The fixed array is shared by every call on the device, and its packet
    layout moves with each call's count and R: only the rotating flag keeps
    a packet of an earlier call from being taken for a new one.  Alternate
    the largest count the array holds with a small ragged one, switch R from
    8 to 3 and back, and make an R = 1 call (the identity); every output of
    every call must equal the oracle bit for bit and the handle path's."""
    import oracle
    build.build()
    lib = _lib.load()
    stream = torch.cuda.current_stream().cuda_stream
    plan = [(8, _lib.noalloc_max_count(8)), (8, 4097), (8, _lib.noalloc_max_count(8)),
            (3, 100_003), (8, 65_541), (1, 12_345), (8, 4097)]
    for call, (R, count) in enumerate(plan):
        xs = inputs.make_inputs(R, count, seed=60 + call)
        want = oracle.allreduce_bf16([inputs.bits(x) for x in xs])[0]
        bufs = [x.to("cuda") for x in xs]
        outs = [torch.full_like(b, float("nan")) for b in bufs]
        in_tbl = torch.tensor([b.data_ptr() for b in bufs], dtype=torch.int64, device="cuda")
        out_tbl = torch.tensor([o.data_ptr() for o in outs], dtype=torch.int64, device="cuda")
        st = lib.ar_allreduce_fused_noalloc(R, in_tbl.data_ptr(), out_tbl.data_ptr(), count,
                                            stream)
        assert st == _lib.AR_OK, (call, st)
        torch.cuda.synchronize()
        for r in range(R):
            got = _bits(outs[r])
            bad = np.nonzero(got != want)[0]
            assert bad.size == 0, "call %d (R=%d, count=%d) rank %d: %d differ, first at %d" % (
                call, R, count, r, bad.size, int(bad[0]))
        if R == 1:
            assert np.array_equal(_bits(outs[0]), inputs.bits(xs[0]))
        with AllReduce(R, count) as ar:
            ar.set_variant("fused_ll8")
            ref = ar(bufs)
            torch.cuda.synchronize()
            assert np.array_equal(_bits(ref[0]), want)
        del bufs, outs
