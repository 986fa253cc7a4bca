"""GPU parity of the composed AllReduce on the latency path (PURLIN_OPT_AR_MODE
= 3): reducing CTAs publish each 8-byte unit as a 16-byte payload+flag packet
and gathering CTAs poll the packets ("Purlin: Separating Orchestration from
the Datapath of Collectives" §3.2 latency path; §4.1 two 2 MiB staging
buffers; §4.3 epoch parity).  Bit for bit against the CPU oracle.
"""
import numpy as np
import pytest

import oracle
from test_parity_gpu import ES, assert_same, gen_inputs, run

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


MAX_PAYLOAD = 1 << 20   # bytes per rank that fit one staging buffer


@pytest.mark.parametrize("dtype", [0, 1], ids=["f32", "bf16"])
@pytest.mark.parametrize("R", [2, 3, 8, 16])
def test_packet_allreduce_parity(P, dtype, R):
    ctx = P.purlin_init(R, torch.cuda.current_stream())
    try:
        P.purlin_set_option(ctx, P.PURLIN_OPT_AR_MODE, 3)
        es = ES[dtype]
        sizes = [1, 2, 3, 4, 5, 7, 8, 9, 4096 + 3, 70001, MAX_PAYLOAD // es]
        for k, n in enumerate(sizes):
            ins = gen_inputs([n] * R, dtype, seed=300 + k * 7 + R)
            got, _ = run(P, ctx, "all_reduce", ins, [n * es] * R, dtype, n)
            assert_same(got, oracle.all_reduce(ins, dtype), f"packets R={R} n={n}")
            assert P.purlin_last_launch(ctx)["variant"] == 5
        # one element past the staging buffer: the call runs as in mode 2
        # (the automatic variant choice, then the ring's composed mode)
        n = MAX_PAYLOAD // es + 1
        ins = gen_inputs([n] * R, dtype, seed=5)
        got, _ = run(P, ctx, "all_reduce", ins, [n * es] * R, dtype, n)
        assert_same(got, oracle.all_reduce(ins, dtype), "past the staging buffer")
        assert P.purlin_last_launch(ctx)["variant"] in (1, 3)
        P.purlin_set_option(ctx, P.PURLIN_OPT_VARIANT, 2)
        got, _ = run(P, ctx, "all_reduce", ins, [n * es] * R, dtype, n)
        assert_same(got, oracle.all_reduce(ins, dtype), "past the staging buffer, ring")
        assert P.purlin_last_launch(ctx)["variant"] == 3
    finally:
        ctx.close()


def test_packet_allreduce_repeated_and_in_place(P):
    """Calls in a row alternate staging buffers and flag values (the epoch);
    stale packets of earlier calls are never taken.  In place works too."""
    R, dtype, n = 8, 1, 100003
    stream = torch.cuda.current_stream()
    ctx = P.purlin_init(R, stream)
    try:
        P.purlin_set_option(ctx, P.PURLIN_OPT_AR_MODE, 3)
        epochs = []
        for k in range(6):
            # the same length every call: a stale packet would hold a valid-looking value
            ins = gen_inputs([n] * R, dtype, seed=k)
            got, _ = run(P, ctx, "all_reduce", ins, [n * 2] * R, dtype, n)
            assert_same(got, oracle.all_reduce(ins, dtype), f"call {k}")
            info = P.purlin_last_launch(ctx)
            epochs.append((info["epoch"], info["epoch_next"]))
        assert all(b - a == 1 for a, b in epochs)
        ins = gen_inputs([n] * R, dtype, seed=99)
        bufs = [torch.from_numpy(x.view(np.int16).copy()).cuda() for x in ins]
        P.purlin_all_reduce(ctx, bufs, bufs, n, dtype)
        P.purlin_check(ctx)
        want = oracle.all_reduce(ins, dtype)
        for d in range(R):
            assert np.array_equal(bufs[d].cpu().numpy().view(np.uint16), want[d])
    finally:
        ctx.close()


def test_packet_dropped_notification_times_out(P):
    """A packet that is never stored: the gathering thread gives up after the
    bounded wait and reports TIMEOUT; the next call is correct."""
    R, dtype, n = 8, 1, 50000
    ctx = P.purlin_init(R, torch.cuda.current_stream())
    try:
        P.purlin_set_option(ctx, P.PURLIN_OPT_AR_MODE, 3)
        P.purlin_set_option(ctx, P.PURLIN_OPT_SPIN_TIMEOUT_NS, 20_000_000)
        P.purlin_set_option(ctx, P.PURLIN_OPT_DROP_NOTIFY, 1234)
        ins = gen_inputs([n] * R, dtype, seed=1)
        src = [torch.from_numpy(x.view(np.int16).copy()).cuda() for x in ins]
        dst = [torch.zeros(n, dtype=torch.int16, device="cuda") for _ in range(R)]
        P.purlin_all_reduce(ctx, src, dst, n, dtype)
        assert P.purlin_check_status(ctx) == P.PURLIN_ERR_TIMEOUT
        P.purlin_set_option(ctx, P.PURLIN_OPT_DROP_NOTIFY, -1)
        got, _ = run(P, ctx, "all_reduce", ins, [n * 2] * R, dtype, n)
        assert_same(got, oracle.all_reduce(ins, dtype), "after a timeout")
    finally:
        ctx.close()
