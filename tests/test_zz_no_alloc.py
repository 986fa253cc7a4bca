"""purlin_all_reduce_noalloc: AllReduce with no device allocation.

Some callers cannot call cudaMalloc when they reduce: code running under
CUDA graph capture, or an engine that has already given all free device
memory to its own pool.  This entry point keeps its scratch (flags and an
error word) in a fixed device array inside the library instead of memory the
context allocates.  Its output must equal, bit for bit, the CPU oracle's
AllReduce and the output of the context entry point purlin_all_reduce in
the composed mode, which runs the same kernel on the same fixed rank order.

This file is collected last so that a run stopping at its first failure has
already run every other test.  It builds what it needs and also passes when
run alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def P():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__

    __graft_entry__.build()
    import collective_datapath_atom_gb300 as mod

    torch.cuda.set_device(0)
    return mod


def _host_inputs(R, n, dtype, seed):
    return workloads.normals(seed, R, n, workloads.F32 if dtype == 0 else workloads.BF16)


def _inputs(R, n, dtype, seed):
    xs = _host_inputs(R, n, dtype, seed)
    if dtype == 0:
        return [torch.from_numpy(x).cuda() for x in xs]
    return [torch.from_numpy(x.view(np.int16)).cuda() for x in xs]


def _oracle_on_device(xs, dtype):
    """The oracle's AllReduce output (the same for every destination)."""
    want = oracle.all_reduce_one(xs, dtype)
    return torch.from_numpy(want if dtype == 0 else want.view(np.int16)).cuda()


def _call_noalloc(P, R, src, dst, n, dtype, stream):
    """Straight through the C ABI (ctypes), as a C caller would."""
    ps = (ctypes.c_void_p * R)(*[t.data_ptr() for t in src])
    pd = (ctypes.c_void_p * R)(*[t.data_ptr() for t in dst])
    return P.lib.purlin_all_reduce_noalloc(
        R, ctypes.cast(ps, ctypes.POINTER(ctypes.c_void_p)),
        ctypes.cast(pd, ctypes.POINTER(ctypes.c_void_p)), n, dtype, P.PURLIN_SUM,
        P.purlin_layout(P.PURLIN_SCATTERED, P.PURLIN_SCATTERED),
        ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("dtype", [0, 1], ids=["f32", "bf16"])
@pytest.mark.parametrize("R,n", [(8, 1 << 20), (8, 100003), (3, 4096 + 7), (2, 40), (31, 31 * 4099)])
def test_noalloc_matches_context_allreduce_twice(P, dtype, R, n):
    stream = torch.cuda.current_stream()
    ctx = P.purlin_init(R, stream)
    try:
        P.purlin_set_option(ctx, P.PURLIN_OPT_VARIANT, 2)
        P.purlin_set_option(ctx, P.PURLIN_OPT_AR_MODE, 2)
        tdt = src_dtype = torch.float32 if dtype == 0 else torch.int16
        for call in range(2):    # two calls in a row share (and reuse) the static scratch
            xs = _host_inputs(R, n, dtype, seed=100 + call)
            src = [torch.from_numpy(x if dtype == 0 else x.view(np.int16)).cuda() for x in xs]
            exact = _oracle_on_device(xs, dtype)
            want = [torch.empty(n, dtype=tdt, device="cuda") for _ in range(R)]
            got = [torch.full((n,), -1, dtype=src_dtype, device="cuda") for _ in range(R)]
            P.purlin_all_reduce(ctx, src, want, n, dtype)
            P.purlin_check(ctx)
            st = _call_noalloc(P, R, src, got, n, dtype, stream)
            assert st == P.PURLIN_OK, P.status_string(st)
            st = P.lib.purlin_noalloc_check(ctypes.c_void_p(stream.cuda_stream))
            assert st == P.PURLIN_OK, P.status_string(st)   # no device-side wait expired
            torch.cuda.synchronize()
            for d in range(R):
                assert torch.equal(got[d], exact), f"call {call} rank {d}: differs from the oracle"
                assert torch.equal(got[d], want[d]), f"call {call} rank {d}"
    finally:
        ctx.close()


def test_noalloc_allocates_no_device_memory(P):
    R, n = 8, 1 << 18
    stream = torch.cuda.current_stream()
    src = _inputs(R, n, 1, seed=7)
    dst = [torch.empty(n, dtype=torch.int16, device="cuda") for _ in range(R)]
    assert _call_noalloc(P, R, src, dst, n, 1, stream) == P.PURLIN_OK   # set-up call
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _call_noalloc(P, R, src, dst, n, 1, stream) == P.PURLIN_OK
        assert P.lib.purlin_noalloc_check(ctypes.c_void_p(stream.cuda_stream)) == P.PURLIN_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_noalloc_rejects_sizes_past_its_scratch(P):
    stream = torch.cuda.current_stream()
    R = 8
    # 8192 chunks of 12 KiB per source is the limit at R = 8: 96 MiB per rank
    limit_elems = 8192 * ((98304 // R) & ~15) // 2    # bf16 elements per rank
    # small integers: every bf16 sum is exact, and the call at the limit uses
    # the last flag of the array
    rng = np.random.default_rng(3)
    ints = [rng.integers(-8, 9, size=limit_elems + 4096).astype(np.float32) for _ in range(R)]
    xs = [(x.view(np.uint32) >> 16).astype(np.uint16) for x in ints]   # exact in bf16
    src = [torch.from_numpy(x.view(np.int16)).cuda() for x in xs]
    dst = [torch.full((limit_elems + 4096,), -1, dtype=torch.int16, device="cuda")
           for _ in range(R)]
    st = _call_noalloc(P, R, src, dst, limit_elems + 4096, 1, stream)
    assert st == P.PURLIN_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert all(bool((t == -1).all().item()) for t in dst), "a refused call wrote its outputs"
    st = _call_noalloc(P, R, src, dst, limit_elems, 1, stream)
    assert st == P.PURLIN_OK
    torch.cuda.synchronize()
    want = _oracle_on_device([x[:limit_elems] for x in xs], 1)
    for d in range(R):
        assert torch.equal(dst[d][:limit_elems], want), f"rank {d} at the size limit"
        assert bool((dst[d][limit_elems:] == -1).all().item()), "wrote past n"
    del src, dst, want
    big_r = 32
    srcs = [torch.empty(64, dtype=torch.int16, device="cuda") for _ in range(big_r)]
    dsts = [torch.empty(64, dtype=torch.int16, device="cuda") for _ in range(big_r)]
    assert _call_noalloc(P, big_r, srcs, dsts, 64, 1, stream) == P.PURLIN_ERR_INVALID_ARG
