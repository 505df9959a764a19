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
