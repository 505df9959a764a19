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
