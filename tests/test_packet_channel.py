"""GPU parity of the packet channel of the device-side API: producer CTAs of a
compute kernel stream 8-byte results to consumer CTAs as 16-byte
payload+flag packets ("Purlin: Separating Orchestration from the Datapath of
Collectives" §3.2, the latency path; §4.1 two staging buffers; §4.3 the
epoch's parity picks the buffer and the epoch is the flag).

The kernel is the library's example (examples/device_examples.cu,
purlin_example_packet_stream): producers compute relu of every rank input
per unit and sum the ranks in order (SCORE), consumers write each received
unit to all R outputs.  The outputs must equal, bit for bit, the oracle's
AllReduce of the relu'd inputs; the inputs must be left as they were.
Also: launches in a row and graph replays (no reset between them), a
packet dropped on the host's request (TIMEOUT, then a correct launch), and
the host-side refusals.
"""
import numpy as np
import pytest

import oracle
from test_device_api import relu_bits
from test_parity_gpu import ES, assert_same, gen_inputs, outputs, upload

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


@pytest.fixture(scope="module")
def X(P):
    from collective_datapath_atom_gb300 import examples

    return examples


def sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


CAP = 1 << 20   # payload bytes per launch


def stream_once(X, ch, src, dst, n, dtype, relu, stream):
    X.packet_stream(ch, [b.ptr for b in src], [b.ptr for b in dst], n, dtype, relu, stream=stream)


@pytest.mark.parametrize("dtype", [0, 1], ids=["f32", "bf16"])
@pytest.mark.parametrize("R", [2, 3, 8, 16])
def test_packet_stream_parity(P, X, R, dtype):
    stream = torch.cuda.current_stream()
    ctx = P.purlin_init(R, stream)
    try:
        ch = P.purlin_packet_channel_create(ctx, CAP, 2 * sms())
        assert ch.capacity == CAP // 8 and ch.ctas == 2 * sms()
        es = ES[dtype]
        for k, n in enumerate((1, 2, 3, 5, 7, 4096 + 3, 70001, CAP // es)):
            for relu in (True, False):
                ins = gen_inputs([n] * R, dtype, seed=8000 + 37 * k + R + (1 if relu else 0))
                want = oracle.all_reduce([relu_bits(x, dtype) for x in ins] if relu else ins, dtype)
                src = upload(ins)
                dst = outputs([n * es] * R)
                stream_once(X, ch, src, dst, n, dtype, relu, stream)
                assert P.purlin_packet_channel_check(ch, stream) == P.PURLIN_OK
                assert_same([b.body() for b in dst], want, f"R={R} n={n} relu={relu}")
                assert_same([b.body() for b in src], ins, "the inputs changed")
                assert all(b.guards_ok() for b in src + dst)
        P.purlin_packet_channel_release(ctx, ch)
        assert ch.staging is None and ch.owner is None
    finally:
        ctx.close()


def test_packet_stream_launches_in_a_row_and_graph_replays(P, X):
    """Each launch advances the channel's epoch on the device: the next one
    uses the other packet set and a new flag, so stale packets of earlier
    launches (same units, same buffers) are never taken, also when the
    launches are replayed from a CUDA graph with frozen parameters."""
    R, dtype, n = 8, 1, 100003
    stream = torch.cuda.Stream()
    ctx = P.purlin_init(R, stream)
    try:
        ch = P.purlin_packet_channel_create(ctx, CAP, 2 * sms())
        src = upload(gen_inputs([n] * R, dtype, seed=1))
        dst = outputs([n * 2] * R)
        for k in range(6):
            ins = gen_inputs([n] * R, dtype, seed=100 + k)
            for b, x in zip(src, ins):
                b.t[256:256 + x.nbytes].copy_(torch.from_numpy(x.view(np.uint8).copy()))
            torch.cuda.synchronize()
            stream_once(X, ch, src, dst, n, dtype, k % 2 == 0, stream)
            assert P.purlin_packet_channel_check(ch, stream) == P.PURLIN_OK
            want = oracle.all_reduce([relu_bits(x, dtype) for x in ins] if k % 2 == 0 else ins,
                                     dtype)
            assert_same([b.body() for b in dst], want, f"launch {k}")
        # two launches captured in one graph, replayed with new inputs
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            stream_once(X, ch, src, dst, n, dtype, True, stream)
            stream_once(X, ch, src, dst, n, dtype, True, stream)
        for rep in range(4):
            ins = gen_inputs([n] * R, dtype, seed=200 + rep)
            for b, x in zip(src, ins):
                b.t[256:256 + x.nbytes].copy_(torch.from_numpy(x.view(np.uint8).copy()))
            for b in dst:
                b.t[256:256 + b.nbytes].fill_(0x11)
            torch.cuda.synchronize()
            g.replay()
            assert P.purlin_packet_channel_check(ch, stream) == P.PURLIN_OK
            want = oracle.all_reduce([relu_bits(x, dtype) for x in ins], dtype)
            assert_same([b.body() for b in dst], want, f"replay {rep}")
        del g
    finally:
        ctx.close()


def test_dropped_packet_times_out_and_the_next_launch_is_correct(P, X):
    """Fault injection on the host: one unit's packet is never sent.  Its
    consumer's bounded wait expires (TIMEOUT in the channel's error word, the
    other consumers give up at once), the launch ends, and the next launch,
    with nothing dropped, is correct: the epoch moved on as usual."""
    R, dtype, n = 8, 0, 50000
    stream = torch.cuda.current_stream()
    ctx = P.purlin_init(R, stream)
    try:
        ch = P.purlin_packet_channel_create(ctx, CAP, 2 * sms())
        assert ch.drop_unit == -1
        ins = gen_inputs([n] * R, dtype, seed=9)
        src = upload(ins)
        dst = outputs([n * 4] * R)
        ch.timeout_ns = 20_000_000   # 20 ms
        ch.drop_unit = 12345
        stream_once(X, ch, src, dst, n, dtype, True, stream)
        assert P.purlin_packet_channel_check(ch, stream) == P.PURLIN_ERR_TIMEOUT
        assert P.purlin_packet_channel_check(ch, stream) == P.PURLIN_OK   # cleared
        ch.drop_unit = -1
        for b in dst:
            b.t[256:256 + b.nbytes].fill_(0x33)
        stream_once(X, ch, src, dst, n, dtype, True, stream)
        assert P.purlin_packet_channel_check(ch, stream) == P.PURLIN_OK
        want = oracle.all_reduce([relu_bits(x, dtype) for x in ins], dtype)
        assert_same([b.body() for b in dst], want, "after the timeout")
        # the option set on the context reaches channels created after it
        P.purlin_set_option(ctx, P.PURLIN_OPT_DROP_NOTIFY, 7)
        ch2 = P.purlin_packet_channel_create(ctx, 4096, 2)
        assert ch2.drop_unit == 7
    finally:
        ctx.close()


def test_channel_refusals(P, X):
    R = 4
    stream = torch.cuda.current_stream()
    ctx = P.purlin_init(R, stream)
    try:
        for cap, ctas in ((0, 2), (1 << 35, 2), (64, 0), (64, 70000)):
            with pytest.raises(P.PurlinError) as e:
                P.purlin_packet_channel_create(ctx, cap, ctas)
            assert e.value.status == P.PURLIN_ERR_INVALID_ARG
        ch = P.purlin_packet_channel_create(ctx, 64, 2)
        assert ch.capacity == 8
        ins = gen_inputs([33] * R, 1, seed=3)    # 66 bytes: 9 units, one past the capacity
        src, dst = upload(ins), outputs([66] * R)
        with pytest.raises(P.PurlinError) as e:
            stream_once(X, ch, src, dst, 33, 1, True, stream)
        assert e.value.status == P.PURLIN_ERR_INVALID_ARG
        odd = P.purlin_packet_channel_create(ctx, 64, 3)     # producers and consumers pair up
        with pytest.raises(P.PurlinError):
            stream_once(X, odd, src, dst, 32, 1, True, stream)
        assert all((b.body() == 0x5A).all() for b in dst), "a refused launch wrote"
        # a channel of another context, or one released already
        other = P.purlin_init(R, stream)
        try:
            with pytest.raises(P.PurlinError):
                P.purlin_packet_channel_release(other, ch)
        finally:
            other.close()
        P.purlin_packet_channel_release(ctx, ch)
        P.purlin_packet_channel_release(ctx, ch)   # cleared: a no-op
    finally:
        ctx.close()
