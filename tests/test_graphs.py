"""Calls captured into a CUDA graph stay correct at every replay.

The modes whose CTAs notify one another (the composed AllReduce with chunk
flags, the latency path's packets, the no-allocation AllReduce, and a
device-side collective) take their epoch from device memory: a replayed
launch has its parameters frozen at capture, yet must not take the flags or
packets of an earlier replay for its own.  Each test captures a few calls,
then replays the graph several times with new inputs copied in between, and
checks every replay bit for bit against the CPU oracle.
"""
import numpy as np
import pytest

import oracle
from test_parity_gpu import gen_inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

R = 8


@pytest.fixture(scope="module")
def P():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__

    __graft_entry__.build()
    import collective_datapath_atom_gb300 as mod

    torch.cuda.set_device(0)
    return mod


def replay_and_check(P, stream, call, src, dst, n, replays=4, calls_per_graph=2):
    """Capture `calls_per_graph` calls of `call`, then replay with fresh inputs."""
    call()                                   # compile and cache the plan before capture
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(calls_per_graph):
            call()
    for k in range(replays):
        ins = gen_inputs([n] * R, 1, seed=7000 + k)
        with torch.cuda.stream(stream):
            for s, x in zip(src, ins):
                s.copy_(torch.from_numpy(x.view(np.int16)), non_blocking=False)
            for d in dst:
                d.zero_()
        stream.synchronize()
        g.replay()
        stream.synchronize()
        want = oracle.all_reduce(ins, 1)
        for d in range(R):
            got = dst[d].cpu().numpy().view(np.uint16)
            assert np.array_equal(got, want[d]), f"replay {k}: rank {d} differs"


def buffers(n):
    src = [torch.empty(n, dtype=torch.int16, device="cuda") for _ in range(R)]
    dst = [torch.zeros(n, dtype=torch.int16, device="cuda") for _ in range(R)]
    return src, dst


@pytest.mark.parametrize("mode", [2, 3], ids=["chunk-flags", "packets"])
def test_composed_allreduce_in_a_graph(P, mode):
    stream = torch.cuda.Stream()
    ctx = P.purlin_init(R, stream)
    try:
        P.purlin_set_option(ctx, P.PURLIN_OPT_AR_MODE, mode)
        P.purlin_set_option(ctx, P.PURLIN_OPT_VARIANT, 2 if mode == 2 else 0)
        n = (3 << 20) // 2 + 5 if mode == 2 else (1 << 20) // 2 - 3
        src, dst = buffers(n)
        replay_and_check(P, stream, lambda: P.purlin_all_reduce(ctx, src, dst, n, 1), src, dst, n)
        assert P.purlin_last_launch(ctx)["variant"] == (3 if mode == 2 else 5)
        assert P.purlin_check_status(ctx) == P.PURLIN_OK
    finally:
        ctx.close()


def test_noalloc_allreduce_in_a_graph(P):
    stream = torch.cuda.Stream()
    n = (5 << 20) // 2 + 1
    src, dst = buffers(n)
    replay_and_check(P, stream,
                     lambda: P.purlin_all_reduce_noalloc(R, src, dst, n, 1, stream=stream),
                     src, dst, n, calls_per_graph=3)
    P.purlin_noalloc_check(stream)   # raises if a replayed call's device wait expired


def test_device_collective_in_a_graph(P):
    from collective_datapath_atom_gb300 import examples as X

    stream = torch.cuda.Stream()
    ctx = P.purlin_init(R, stream)
    try:
        P.purlin_set_option(ctx, P.PURLIN_OPT_AR_MODE, 2)
        n = (2 << 20) // 2 + 7
        src, dst = buffers(n)
        blocks = torch.cuda.get_device_properties(0).multi_processor_count
        d = P.purlin_device_prepare(ctx, P.PURLIN_COLL_ALL_REDUCE, src, dst, n=n, dtype=1,
                                    blocks=blocks)
        assert d.composed == 1
        replay_and_check(P, stream, lambda: X.collective(d, stream=stream), src, dst, n)
        assert P.purlin_device_check(d, stream) == P.PURLIN_OK
        P.purlin_device_release(ctx, d)
    finally:
        ctx.close()


def test_alltoallv_graph_survives_plan_cache_pressure(P):
    """An AllToAllV plan (its segment table in device memory) used in a
    captured graph stays valid while more than the cache's 64 other shapes
    pass through it; replays after that are still correct."""
    import workloads

    stream = torch.cuda.Stream()
    ctx = P.purlin_init(R, stream)
    try:
        part = workloads.zipf_partition(300001)
        C = workloads.rotated_counts(part)
        counts = C.reshape(-1).tolist()
        T = int(C.sum(axis=1)[0])
        src = [torch.empty(T, dtype=torch.int16, device="cuda") for _ in range(R)]
        dst = [torch.zeros(int(C[:, d].sum()), dtype=torch.int16, device="cuda") for d in range(R)]
        call = lambda: P.purlin_all_to_all_v(ctx, src, dst, counts, 1)   # noqa: E731
        call()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            call()

        def check(k):
            ins = gen_inputs([T] * R, 1, seed=8000 + k)
            with torch.cuda.stream(stream):
                for s, x in zip(src, ins):
                    s.copy_(torch.from_numpy(x.view(np.int16)))
                for d in dst:
                    d.zero_()
            stream.synchronize()
            g.replay()
            stream.synchronize()
            want = oracle.all_to_all_v(ins, C, 1)
            for d in range(R):
                assert np.array_equal(dst[d].cpu().numpy().view(np.uint16), want[d]), \
                    f"replay {k}: rank {d}"

        check(0)
        # 70 other shapes through the 64-entry plan cache
        small = [torch.empty(4096, dtype=torch.int16, device="cuda") for _ in range(2 * R)]
        for k in range(70):
            cs = [1 + (k + i) % 7 for i in range(R * R)]
            need_in = max(sum(cs[s * R:(s + 1) * R]) for s in range(R))
            need_out = max(sum(cs[s * R + d] for s in range(R)) for d in range(R))
            assert need_in <= 4096 and need_out <= 4096
            P.purlin_all_to_all_v(ctx, small[:R], small[R:], cs, 1)
        P.purlin_check(ctx)
        check(1)
    finally:
        ctx.close()


def test_first_call_of_a_large_plan_during_capture_is_refused(P):
    """A plan whose table must be uploaded cannot be compiled while the
    stream is being captured: the call returns UNSUPPORTED instead of
    recording an upload the graph could not replay."""
    stream = torch.cuda.Stream()
    ctx = P.purlin_init(R, stream)
    try:
        counts = [3] * (R * R)
        src = [torch.empty(3 * R, dtype=torch.int16, device="cuda") for _ in range(R)]
        dst = [torch.empty(3 * R, dtype=torch.int16, device="cuda") for _ in range(R)]
        g = torch.cuda.CUDAGraph()
        with pytest.raises(P.PurlinError) as e:
            with torch.cuda.graph(g, stream=stream):
                P.purlin_all_to_all_v(ctx, src, dst, counts, 1)
        assert e.value.status == P.PURLIN_ERR_UNSUPPORTED
        torch.cuda.synchronize()
        # outside capture the same call works
        P.purlin_all_to_all_v(ctx, src, dst, counts, 1)
        P.purlin_check(ctx)
    finally:
        ctx.close()


def test_device_count_alltoallv_graph_with_new_counts_each_replay(P):
    """MoE dispatch in a graph: the counts live in device memory and change
    between replays (as a router on the GPU would write them); each replay
    dispatches by the counts it finds, with no host involvement."""
    import workloads

    H = 64
    tokens = 96
    stream = torch.cuda.Stream()
    ctx = P.purlin_init(R, stream)
    try:
        cap_out = R * tokens * H
        src = [torch.empty(tokens * H, dtype=torch.int16, device="cuda") for _ in range(R)]
        dst = [torch.zeros(cap_out, dtype=torch.int16, device="cuda") for _ in range(R)]
        d_counts = torch.zeros(R * R, dtype=torch.int64, device="cuda")
        call = lambda: P.purlin_all_to_all_v_device_counts(   # noqa: E731
            ctx, src, dst, d_counts, tokens * H, cap_out, 1)
        call()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            call()
        for k in range(4):
            C, _ = workloads.moe_dispatch(seed=20 + k, tokens=tokens, hidden=H, payload=False)
            counts = (C * H).reshape(-1)
            ins = gen_inputs([tokens * H] * R, 1, seed=9000 + k)
            with torch.cuda.stream(stream):
                d_counts.copy_(torch.from_numpy(counts))
                for s, x in zip(src, ins):
                    s.copy_(torch.from_numpy(x.view(np.int16)))
                for d in dst:
                    d.zero_()
            stream.synchronize()
            g.replay()
            stream.synchronize()
            want = oracle.all_to_all_v(ins, counts.reshape(R, R), 1)
            for d in range(R):
                got = dst[d][:want[d].size].cpu().numpy().view(np.uint16)
                assert np.array_equal(got, want[d]), f"replay {k}: rank {d}"
                assert int(dst[d][want[d].size:].abs().sum().item()) == 0
        assert P.purlin_check_status(ctx) == P.PURLIN_OK
    finally:
        ctx.close()
