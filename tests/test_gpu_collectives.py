"""Reduce-scatter and all-gather on the GPU vs the oracle, bit for bit."""
import numpy as np
import pytest
import torch

from shot_allreduce_ranks_gb300 import ArError, inputs
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu

import oracle  # noqa: E402

BLOCKS = [1, 7, 8, 9, 4097, 65536 + 8, 3 * 65536 + 5]


@pytest.fixture(scope="module", autouse=True)
def _cleanup():
    yield
    G.release_handles()


@pytest.mark.parametrize("R", [1, 2, 3, 8])
def test_reduce_scatter_matches_oracle(R):
    ar = G.handle(R, R * max(BLOCKS))
    for rc in BLOCKS:
        xs = inputs.make_inputs(R, R * rc, seed=rc % 5, fill="normal")
        want = oracle.reduce_scatter_bf16([inputs.bits(x) for x in xs])
        outs = ar.reduce_scatter(G.to_device(xs), recvcount=rc)
        torch.cuda.synchronize()
        for r in range(R):
            G.assert_bitexact(G.device_bits(outs[r]), want[r], "RS R=%d rc=%d rank %d" % (R, rc, r))


@pytest.mark.parametrize("R", [1, 2, 3, 8])
def test_all_gather_matches_oracle(R):
    ar = G.handle(R, R * max(BLOCKS))
    for sc in BLOCKS:
        xs = inputs.make_inputs(R, sc, seed=sc % 3, fill="normal")
        want = oracle.all_gather_bf16([inputs.bits(x) for x in xs])
        outs = ar.all_gather(G.to_device(xs), sendcount=sc)
        torch.cuda.synchronize()
        for r in range(R):
            G.assert_bitexact(G.device_bits(outs[r]), want[r], "AG R=%d sc=%d rank %d" % (R, sc, r))


def test_reduce_scatter_exact_integers_without_oracle():
    R, rc = 8, 1 << 17
    ar = G.handle(R, R * rc)
    xs = inputs.make_inputs(R, R * rc, seed=3, fill="ints")
    outs = ar.reduce_scatter(G.to_device(xs), recvcount=rc)
    exact = torch.stack([x.to(torch.int64) for x in xs]).sum(0)
    torch.cuda.synchronize()
    for r in range(R):
        want = inputs.bits(exact[r * rc:(r + 1) * rc].to(torch.bfloat16))
        G.assert_bitexact(G.device_bits(outs[r]), want, "RS ints rank %d" % r)


def test_reduce_scatter_is_a_slice_of_allreduce():
    """Same numerics: block r of the allreduce equals reduce-scatter output r."""
    R, rc = 8, 40_000
    ar = G.handle(R, R * rc)
    xs = G.to_device(inputs.make_inputs(R, R * rc, seed=9))
    rs = ar.reduce_scatter(xs, recvcount=rc)
    ar.set_variant("fused_ll8")
    full = ar(xs)
    torch.cuda.synchronize()
    for r in range(R):
        assert torch.equal(rs[r].view(torch.int16), full[0][r * rc:(r + 1) * rc].view(torch.int16))


def test_block_bounds():
    R = 4
    ar = G.handle(R, 100)
    big = G.to_device(inputs.make_inputs(R, 104, 0))
    with pytest.raises(ArError):          # R * 26 = 104 > max_count = 100
        ar.reduce_scatter(big, recvcount=26)
    xs = [x[:100] for x in big]
    with pytest.raises(ArError):
        ar.all_gather([x[:26] for x in xs], outputs=[torch.empty(104, dtype=torch.bfloat16,
                                                                 device="cuda") for _ in xs])
    outs = ar.reduce_scatter(xs, recvcount=25)
    torch.cuda.synchronize()
    assert all(o.numel() == 25 for o in outs)
    np.testing.assert_array_equal(G.device_bits(outs[0]),
                                  oracle.reduce_scatter_bf16([inputs.bits(x.cpu()) for x in xs])[0])


@pytest.mark.parametrize("R,block", [(8, 281_600), (8, 281_608), (16, 131_072)],
                         ids=["r8_even_groups", "r8_odd_groups", "r16"])
def test_large_blocks_and_32_byte_requests(R, block):
    """Large blocks (the benchmark message split R ways, even and odd group
    counts, R = 8 and 16) and pointers that are 16- but not 32-byte aligned;
    reduce-scatter (R <= 8) and all-gather."""
    ar = G.handle(R, R * block + 64)
    xs = inputs.make_inputs(R, R * block, seed=block % 7, fill="normal")
    ins = G.to_device(xs)
    checks = []
    if R <= 8:
        want_rs = oracle.reduce_scatter_bf16([inputs.bits(x) for x in xs])
        checks.append(("RS", ar.reduce_scatter(ins, recvcount=block), want_rs))
    small = [x[:block] for x in xs]
    want_ag = oracle.all_gather_bf16([inputs.bits(x) for x in small])
    checks.append(("AG", ar.all_gather([t[:block].contiguous() for t in ins], sendcount=block),
                   want_ag))
    torch.cuda.synchronize()
    for what, outs, want in checks:
        for r in range(R):
            G.assert_bitexact(G.device_bits(outs[r]), want[r], "%s R=%d block=%d rank %d" % (
                what, R, block, r))
    # 16-byte aligned, not 32-byte aligned: views 8 elements into larger buffers
    def offset_copy(ts):
        out = []
        for t in ts:
            b = torch.zeros(t.numel() + 8, dtype=t.dtype, device=G.DEV)
            v = b[8:]
            v.copy_(t)
            out.append(v)
        return out
    vins = offset_copy([t[:block] for t in ins])
    vouts = offset_copy([torch.zeros(R * block, dtype=torch.bfloat16, device=G.DEV)
                         for _ in range(R)])
    assert all(v.data_ptr() % 32 == 16 for v in vins + vouts)
    outs = ar.all_gather(vins, vouts, sendcount=block)
    torch.cuda.synchronize()
    for r in range(R):
        G.assert_bitexact(G.device_bits(outs[r]), want_ag[r], "AG 16B-aligned rank %d" % r)
