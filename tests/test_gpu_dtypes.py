"""fp16 and fp32 element types, and R up to 16 ranks, on the GPU vs the
oracle, bit for bit (NaN payloads aside)."""
import numpy as np
import pytest
import torch

import oracle
from shot_allreduce_ranks_gb300 import AllReduce, ArError, build, inputs
from shot_allreduce_ranks_gb300._lib import AR_ERR_UNSUPPORTED

pytestmark = pytest.mark.gpu

ONE_SHOT = ["oneshot_pull", "oneshot_fanout", "oneshot_fanout_bulk", "twophase"]
PACKET = ["fused_ll8", "fused_ll8_staged", "packet_3op"]
COUNTS = [1, 7, 9, 4097, 3 * 65536 + 5]

_handles = {}


def handle(R, count, dtype):
    key = (R, count, dtype)
    if key not in _handles:
        build.build()
        _handles[key] = AllReduce(R, count, dtype=dtype)
    return _handles[key]


@pytest.fixture(scope="module", autouse=True)
def _cleanup():
    yield
    for h in _handles.values():
        h.close()
    _handles.clear()


def nan_mask(bits, dtype):
    if dtype == torch.float16:
        return ((bits & 0x7C00) == 0x7C00) & ((bits & 0x3FF) != 0)
    if dtype == torch.float32:
        return ((bits & 0x7F800000) == 0x7F800000) & ((bits & 0x7FFFFF) != 0)
    return ((bits & 0x7F80) == 0x7F80) & ((bits & 0x7F) != 0)


def expect(xs, dtype):
    if dtype == torch.float16:
        return oracle.allreduce_f16([inputs.bits(x) for x in xs])[0]
    if dtype == torch.float32:
        return oracle.allreduce_f32([x.numpy() for x in xs])[0].view(np.uint32)
    return oracle.allreduce_bf16([inputs.bits(x) for x in xs])[0]


def check(outs, want, dtype, what):
    for r, o in enumerate(outs):
        got = inputs.bits(o.cpu())
        gn, wn = nan_mask(got, dtype), nan_mask(want, dtype)
        bad = np.nonzero((got != want) & ~(gn & wn))[0]
        assert bad.size == 0, "%s rank %d: %d differ, first at %d (0x%x vs 0x%x)" % (
            what, r, bad.size, bad[0], int(got[bad[0]]), int(want[bad[0]]))


@pytest.mark.parametrize("dtype", [torch.float16, torch.float32], ids=["fp16", "fp32"])
@pytest.mark.parametrize("variant", ONE_SHOT + PACKET + ["auto"])
def test_dtype_parity(dtype, variant):
    R = 8
    ar = handle(R, max(COUNTS), dtype)
    ar.set_variant(variant)
    for count in COUNTS:
        xs = inputs.make_inputs(R, count, seed=count % 5, dtype=dtype)
        outs = ar([x.cuda() for x in xs])
        torch.cuda.synchronize()
        check(outs, expect(xs, dtype), dtype, "%s %s count=%d" % (dtype, variant, count))
    assert ar.device_status() == 0


@pytest.mark.parametrize("dtype", [torch.float16, torch.float32], ids=["fp16", "fp32"])
def test_dtype_special_values(dtype):
    """Random bit patterns of every class (subnormal, huge, inf, NaN)."""
    R, count = 8, 20_003
    rng = np.random.default_rng(3)
    if dtype == torch.float16:
        xs = [torch.from_numpy(rng.integers(0, 1 << 16, count, dtype=np.uint64)
                               .astype(np.uint16).view(np.int16)).view(torch.float16)
              for _ in range(R)]
    else:
        xs = [torch.from_numpy(rng.integers(0, 1 << 32, count, dtype=np.uint64)
                               .astype(np.uint32).view(np.int32)).view(torch.float32)
              for _ in range(R)]
    want = expect(xs, dtype)
    ar = handle(R, count, dtype)
    for variant in ONE_SHOT + PACKET:
        ar.set_variant(variant)
        outs = ar([x.cuda() for x in xs])
        torch.cuda.synchronize()
        check(outs, want, dtype, "%s special %s" % (dtype, variant))


@pytest.mark.parametrize("dtype", [torch.float16, torch.float32], ids=["fp16", "fp32"])
def test_dtype_misaligned_and_in_place(dtype):
    R, count = 4, 4099
    ar = handle(R, count + 8, dtype)
    xs = inputs.make_inputs(R, count, seed=12, dtype=dtype)
    want = expect(xs, dtype)
    for variant in ONE_SHOT + PACKET:
        ar.set_variant(variant)
        base = [torch.empty(count + 8, dtype=dtype, device="cuda") for _ in range(R)]
        bufs = [b[1:1 + count] for b in base]          # one element off alignment
        for b, x in zip(bufs, xs):
            b.copy_(x)
        ar(bufs, bufs)                                  # in place
        torch.cuda.synchronize()
        check(bufs, want, dtype, "%s misaligned in place %s" % (dtype, variant))


def test_fp32_exact_integer_sums_without_oracle():
    R, count = 16, 1 << 18
    ar = handle(R, count, torch.float32)
    xs = inputs.make_inputs(R, count, seed=2, fill="ints", dtype=torch.float32)
    exact = torch.stack([x.to(torch.int64) for x in xs]).sum(0).to(torch.float32)
    for variant in ONE_SHOT + ["auto"]:
        ar.set_variant(variant)
        outs = ar([x.cuda() for x in xs])
        torch.cuda.synchronize()
        for o in outs:
            assert torch.equal(o.cpu(), exact), variant


@pytest.mark.parametrize("R", [9, 12, 16])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
def test_many_ranks(R, dtype):
    count = 100_003
    ar = handle(R, R * count, dtype)
    xs = inputs.make_inputs(R, count, seed=R, dtype=dtype)
    want = expect(xs, dtype)
    for variant in ONE_SHOT + ["auto"]:
        ar.set_variant(variant)
        outs = ar([x.cuda() for x in xs])
        torch.cuda.synchronize()
        check(outs, want, dtype, "R=%d %s" % (R, variant))
    # reduce-scatter / all-gather at the same R
    big = inputs.make_inputs(R, R * 1001, seed=1, dtype=dtype)
    rs = ar.reduce_scatter([x.cuda() for x in big], recvcount=1001)
    ag = ar.all_gather([x[:1001].cuda() for x in big], sendcount=1001)
    torch.cuda.synchronize()
    full = expect(big, dtype)
    for r in range(R):
        got = inputs.bits(rs[r].cpu())
        assert np.array_equal(got[~nan_mask(got, dtype)],
                              full[r * 1001:(r + 1) * 1001][~nan_mask(got, dtype)])
        cat = np.concatenate([inputs.bits(x[:1001]) for x in big])
        assert np.array_equal(inputs.bits(ag[r].cpu()), cat)


def test_packet_variants_need_at_most_8_ranks():
    ar = handle(12, 1000, torch.bfloat16)
    xs = [torch.zeros(1000, dtype=torch.bfloat16, device="cuda") for _ in range(12)]
    for variant in PACKET:
        ar.set_variant(variant)
        with pytest.raises(ArError) as e:
            ar(xs)
        assert e.value.status == AR_ERR_UNSUPPORTED
    ar.set_variant("auto")
    ar(xs)
    torch.cuda.synchronize()


@pytest.mark.parametrize("R", [4, 16])
@pytest.mark.parametrize("dtype", [torch.float16, torch.float32], ids=["fp16", "fp32"])
def test_host_buffer_paths(dtype, R):
    """ar_allreduce_host for the other element types and for R > 8: page-locked
    buffers (kernel on the host memory in place) and pageable ones (staging)."""
    count = 70_001
    ar = handle(R, count, dtype)
    ar.reserve_host_staging()
    xs = inputs.make_inputs(R, count, 17, "normal", dtype)
    want = expect(xs, dtype)
    pinned_in = [x.pin_memory() for x in xs]
    pinned_out = [torch.empty(count, dtype=dtype).pin_memory() for _ in range(R)]
    pageable_out = [torch.empty(count, dtype=dtype) for _ in range(R)]
    variants = ["auto", "oneshot_fanout", "twophase"] + (["fused_ll8"] if R <= 8 else [])
    for v in variants:
        ar.set_variant(v)
        ar.allreduce_host(pinned_in, pinned_out)
        ar.allreduce_host(xs, pageable_out)
        torch.cuda.synchronize()
        check(pinned_out, want, dtype, "host page-locked %s R=%d" % (v, R))
        check(pageable_out, want, dtype, "host pageable %s R=%d" % (v, R))
    ar.set_variant("auto")


def test_host_path_refuses_stream_capture():
    """ar_allreduce_host copies its device pointer table from memory that
    lives only for the call, so a captured graph would keep a dangling
    source: under capture the call must refuse (AR_ERR_UNSUPPORTED) and
    enqueue nothing, and work again once capture has ended."""
    from shot_allreduce_ranks_gb300 import _lib
    import ctypes
    R, count = 4, 4097
    ar = handle(R, count, torch.bfloat16)
    ar.reserve_host_staging()
    xs = inputs.make_inputs(R, count, seed=3, fill="normal")
    pinned_in = [x.pin_memory() for x in xs]
    pinned_out = [torch.empty(count, dtype=torch.bfloat16).pin_memory() for _ in range(R)]
    ins = (ctypes.c_void_p * R)(*[t.data_ptr() for t in pinned_in])
    outs = (ctypes.c_void_p * R)(*[t.data_ptr() for t in pinned_out])
    lib = _lib.load()
    side = torch.cuda.Stream()
    dummy = torch.zeros(16, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        dummy.add_(1.0)  # keep the captured graph non-empty
        st = lib.ar_allreduce_host(ar._h, ctypes.cast(ins, ctypes.c_void_p),
                                   ctypes.cast(outs, ctypes.c_void_p), count,
                                   side.cuda_stream)
    assert st == AR_ERR_UNSUPPORTED
    g.replay()
    torch.cuda.synchronize()
    ar.set_variant("auto")
    ar.allreduce_host(pinned_in, pinned_out)
    torch.cuda.synchronize()
    check(pinned_out, expect(xs, torch.bfloat16), torch.bfloat16, "host path after capture")


@pytest.mark.parametrize("block", [4096 + 24, 1001], ids=["vector", "element"])
@pytest.mark.parametrize("R", [4, 8])
@pytest.mark.parametrize("dtype", [torch.float16, torch.float32], ids=["fp16", "fp32"])
def test_reduce_scatter_and_all_gather_types(dtype, R, block):
    """fp16/fp32 reduce-scatter and all-gather on both access paths: a block
    that is a whole number of 16-byte groups (vector path) and one that is
    not (element path).  Reduce-scatter block r must equal block r of the
    oracle's allreduce; all-gather must be the plain concatenation."""
    ar = handle(R, R * block, dtype)
    big = inputs.make_inputs(R, R * block, seed=3, dtype=dtype)
    rs = ar.reduce_scatter([x.cuda() for x in big], recvcount=block)
    ag = ar.all_gather([x[:block].cuda() for x in big], sendcount=block)
    torch.cuda.synchronize()
    full = expect(big, dtype)
    cat = np.concatenate([inputs.bits(x[:block]) for x in big])
    for r in range(R):
        got = inputs.bits(rs[r].cpu())
        want = full[r * block:(r + 1) * block]
        keep = ~(nan_mask(got, dtype) & nan_mask(want, dtype))
        assert np.array_equal(got[keep], want[keep]), "reduce-scatter rank %d" % r
        assert np.array_equal(inputs.bits(ag[r].cpu()), cat), "all-gather rank %d" % r


@pytest.mark.parametrize("count", [(1 << 20) - 4, 1 << 20, (1 << 20) + 4 + 1],
                         ids=["below", "at", "odd_and_partial"])
def test_fp32_fanout_wide_requests(count):
    """fp32 fan-out around the 32-byte path's threshold (2^18 groups of 4)."""
    R = 8
    ar = handle(R, (1 << 20) + 64, torch.float32)
    xs = inputs.make_inputs(R, count, 23, "normal", torch.float32)
    want = expect(xs, torch.float32)
    ar.set_variant("oneshot_fanout")
    outs = ar([x.cuda() for x in xs])
    torch.cuda.synchronize()
    check(outs, want, torch.float32, "fp32 fanout count=%d" % count)
    ar.set_variant("auto")


@pytest.mark.parametrize("dtype", [torch.float16, torch.float32], ids=["fp16", "fp32"])
def test_fused_ring_mode_types(dtype, monkeypatch):
    """The fused kernel's per-CTA packet rings (forced, on a grid of 3 CTAs
    so that every slot is reused many times) for fp16 and fp32, ragged
    count, two calls with different inputs."""
    monkeypatch.setenv("AR_FUSED_RING", "1")
    R, count = 8, 3 * 65536 * 4 + 3
    build.build()
    with AllReduce(R, count, dtype=dtype) as ar:
        ar.set_variant("fused_ll8")
        ar.set_launch("fused_ll8", 3, 0)
        for call in range(2):
            xs = inputs.make_inputs(R, count, seed=400 + call, fill="normal", dtype=dtype)
            outs = ar([x.to("cuda") for x in xs])
            torch.cuda.synchronize()
            check(outs, expect(xs, dtype), dtype, "ring %s call %d" % (dtype, call))
        assert ar.device_status() == 0
