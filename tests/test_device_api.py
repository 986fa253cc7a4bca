"""GPU parity of the device-side API: collectives and Atoms called from inside
user kernels (include/purlin_device.cuh), compared bit for bit with the CPU
oracle.

The kernels are the examples in collective_datapath_atom_gb300/examples,
written the way an application would write them ("Purlin" project README,
"Device-side" and "Samples"): a kernel whose CTAs call a prepared
collective; one that computes its inputs, passes a grid barrier and then
runs the collective (fusion with computation); one where only some CTAs
enter the collective; and CTAs that copy or reduce their own slice with the
Atom.
"""
import numpy as np
import pytest

import oracle
from test_parity_gpu import (COLLS, ES, Guarded, assert_same, gen_inputs, in_lengths, oracle_of,
                             out_sizes, outputs, size_cases, upload)

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


def prepare(P, ctx, coll, src, dst, n, counts, dtype, blocks, **kw):
    return P.purlin_device_prepare(ctx, COLLS.index(coll), [b.ptr for b in src],
                                   [b.ptr for b in dst], n=n, counts=counts, dtype=dtype,
                                   blocks=blocks, **kw)


def bodies(bufs):
    return [b.body() for b in bufs]


def guards(bufs):
    return all(b.guards_ok() for b in bufs)


# --------------------------------------------------- prepared collectives --

@pytest.mark.parametrize("coll", COLLS)
@pytest.mark.parametrize("dtype", [0, 1], ids=["f32", "bf16"])
@pytest.mark.parametrize("R", [3, 8])
def test_device_collective_parity(P, X, coll, dtype, R):
    """Every collective, called from a user kernel by `blocks` CTAs, twice
    per descriptor (the per-CTA epochs advance between calls)."""
    stream = torch.cuda.current_stream()
    ctx = P.purlin_init(R, stream)
    try:
        for k, (n, counts) in enumerate(size_cases(coll, R)):
            ins = gen_inputs(in_lengths(coll, R, n, counts), dtype, seed=500 + 10 * k + R)
            want = oracle_of(coll, ins, dtype, counts)
            src = upload(ins)
            dst = outputs(out_sizes(coll, R, n, counts, ES[dtype]))
            for blocks in (1, 7, sms()):
                d = prepare(P, ctx, coll, src, dst, n, counts, dtype, blocks)
                assert d.blocks == blocks and d.R == R and d.composed == 0
                for call in range(2):
                    for b in dst:
                        b.t[256:256 + b.nbytes].fill_(0x11)
                    X.collective(d, stream=stream)
                    assert P.purlin_device_check(d, stream) == P.PURLIN_OK
                    assert_same(bodies(dst), want,
                                f"{coll} R={R} dtype={dtype} n={n} blocks={blocks} call={call}")
                    assert guards(src + dst)
                P.purlin_device_release(ctx, d)
                assert d.owner is None and d.segs is None
    finally:
        ctx.close()


@pytest.mark.parametrize("dtype", [0, 1], ids=["f32", "bf16"])
def test_device_composed_allreduce(P, X, dtype):
    """Composed AllReduce inside a user kernel: reducing CTAs publish
    per-chunk flags, gathering CTAs acquire them ("Purlin: Separating Orchestration from the Datapath of Collectives"
    §3.2).  With
    256-byte chunks the 16 MiB-per-rank case has more notifying chunks than
    flag slots, so chunk flags take two generations within a call."""
    R = 8
    stream = torch.cuda.current_stream()
    ctx = P.purlin_init(R, stream)
    try:
        P.purlin_set_option(ctx, P.PURLIN_OPT_AR_MODE, 2)
        big = (16 << 20) // ES[dtype]
        for n, chunk in ((4096 + 3, 0), (100003, 0), (1 << 21, 0), (big, 256)):
            P.purlin_set_option(ctx, P.PURLIN_OPT_CHUNK_BYTES, chunk)
            ins = gen_inputs([n] * R, dtype, seed=n % 97)
            want = oracle.all_reduce(ins, dtype)
            src = upload(ins)
            dst = outputs([n * ES[dtype]] * R)
            d = prepare(P, ctx, "all_reduce", src, dst, n, None, dtype, sms())
            assert d.composed == 1 and d.flags is not None
            if chunk:
                assert d.epoch_inc >= 3, "expected two flag generations per call"
            for call in range(3):
                for b in dst:
                    b.t[256:256 + b.nbytes].fill_(0x22)
                X.collective(d, stream=stream)
                assert P.purlin_device_check(d, stream) == P.PURLIN_OK
                assert_same(bodies(dst), want, f"composed n={n} chunk={chunk} call={call}")
                assert guards(src + dst)
            P.purlin_device_release(ctx, d)
    finally:
        ctx.close()


def relu_bits(x, dtype):
    """max(x, 0) on raw bits: negatives and -0 become +0, NaN is kept."""
    if dtype == 0:
        u = x.view(np.uint32).copy()
        neg = ((u & 0x80000000) != 0) & ((u & 0x7FFFFFFF) <= 0x7F800000)
        u[neg] = 0
        return u.view(np.float32)
    u = x.view(np.uint16).copy()
    neg = ((u & 0x8000) != 0) & ((u & 0x7FFF) <= 0x7F80)
    u[neg] = 0
    return u


@pytest.mark.parametrize("mode", [1, 2], ids=["fused", "composed"])
@pytest.mark.parametrize("dtype", [0, 1], ids=["f32", "bf16"])
def test_device_allreduce_fused_with_compute(P, X, mode, dtype):
    """A kernel that computes its inputs (ReLU in place), passes a grid
    barrier and runs the AllReduce on them, in one launch."""
    R = 8
    stream = torch.cuda.current_stream()
    ctx = P.purlin_init(R, stream)
    try:
        P.purlin_set_option(ctx, P.PURLIN_OPT_AR_MODE, mode)
        for n in (37, 70001, 1 << 20):
            ins = gen_inputs([n] * R, dtype, seed=n % 89 + mode)
            ins[0][: min(n, 3)] = ins[0][: min(n, 3)] * 0   # some zeros (+0 and -0)
            if dtype == 0 and n > 10:
                ins[1][5] = np.float32(-0.0)
            relu = [relu_bits(x, dtype) for x in ins]
            want = oracle.all_reduce(relu, dtype)
            src = upload(ins)
            dst = outputs([n * ES[dtype]] * R)
            d = prepare(P, ctx, "all_reduce", src, dst, n, None, dtype, sms())
            # (messages under 16 bytes per rank per rank stay fused)
            assert d.composed == (1 if mode == 2 and n * ES[dtype] >= 16 * R else 0)
            X.relu_collective(d, n, stream=stream)
            assert P.purlin_device_check(d, stream) == P.PURLIN_OK
            assert_same(bodies(src), [r.view(np.uint8) for r in relu], f"relu inputs n={n}")
            assert_same(bodies(dst), want, f"relu+allreduce mode={mode} n={n}")
            assert guards(src + dst)
            P.purlin_device_release(ctx, d)
    finally:
        ctx.close()


@pytest.mark.parametrize("coll", ["all_gather", "all_reduce"])
def test_device_collective_on_a_subset_of_the_grid(P, X, coll):
    """Only CTAs [0, blocks) enter the collective; the kernel's other CTAs do
    unrelated work at the same time."""
    R, dtype = 8, 1
    stream = torch.cuda.current_stream()
    ctx = P.purlin_init(R, stream)
    try:
        if coll == "all_reduce":
            P.purlin_set_option(ctx, P.PURLIN_OPT_AR_MODE, 2)
        n = 300007 if coll == "all_reduce" else 131075
        ins = gen_inputs([n] * R, dtype, seed=4242)
        want = oracle_of(coll, ins, dtype)
        src = upload(ins)
        dst = outputs(out_sizes(coll, R, n, None, ES[dtype]))
        extra = 8
        d = prepare(P, ctx, coll, src, dst, n, None, dtype, sms() - extra)
        words = 5_000_003
        fill = torch.zeros(words, dtype=torch.int64, device="cuda")   # 8-byte words: room to check
        fill32 = fill.view(torch.int32)
        X.subset(d, extra, fill32.data_ptr(), words, stream=stream)
        assert P.purlin_device_check(d, stream) == P.PURLIN_OK
        assert_same(bodies(dst), want, f"{coll} on a subset")
        got = fill32[:words].cpu().numpy().view(np.uint32)
        exp = (np.arange(words, dtype=np.uint64) * 2654435761 % (1 << 32)).astype(np.uint32)
        assert np.array_equal(got, exp)
        assert int(fill32[words:].abs().sum().item()) == 0
        P.purlin_device_release(ctx, d)
    finally:
        ctx.close()


def test_device_workspace_cap(P, X):
    """A descriptor prepared under a small shared-memory cap uses a smaller
    ring and gives the same result."""
    R, dtype, n = 8, 1, 3 * 65536 + 5
    stream = torch.cuda.current_stream()
    ctx = P.purlin_init(R, stream)
    try:
        ins = gen_inputs([n] * R, dtype, seed=9)
        want = oracle.all_reduce(ins, dtype)
        src = upload(ins)
        dst = outputs([n * 2] * R)
        d = prepare(P, ctx, "all_reduce", src, dst, n, None, dtype, 2 * sms(),
                    max_workspace_bytes=40 * 1024)
        assert d.workspace_bytes <= 40 * 1024
        X.collective(d, stream=stream)
        assert P.purlin_device_check(d, stream) == P.PURLIN_OK
        assert_same(bodies(dst), want, "capped workspace")
        P.purlin_device_release(ctx, d)
    finally:
        ctx.close()


def test_device_errors_are_reported(P, X):
    """A block too small for the ring's roles is refused inside the kernel
    (nothing written, INVALID_ARG in the error word); a dropped notification
    in the composed AllReduce makes the waiting CTAs give up after the
    bounded wait (TIMEOUT); a descriptor prepared afterwards works."""
    R, dtype, n = 8, 1, 1 << 18
    stream = torch.cuda.current_stream()
    ctx = P.purlin_init(R, stream)
    try:
        ins = gen_inputs([n] * R, dtype, seed=3)
        want = oracle.all_reduce(ins, dtype)
        src = upload(ins)
        dst = outputs([n * 2] * R)
        d = prepare(P, ctx, "all_reduce", src, dst, n, None, dtype, 16)
        X.collective(d, threads=64, stream=stream)
        assert P.purlin_device_check(d, stream) == P.PURLIN_ERR_INVALID_ARG
        assert all((b.body() == 0x5A).all() for b in dst), "a refused call wrote output"
        assert P.purlin_device_check(d, stream) == P.PURLIN_OK   # cleared
        X.collective(d, stream=stream)
        assert P.purlin_device_check(d, stream) == P.PURLIN_OK
        assert_same(bodies(dst), want, "after a refused call")
        P.purlin_device_release(ctx, d)

        P.purlin_set_option(ctx, P.PURLIN_OPT_AR_MODE, 2)
        P.purlin_set_option(ctx, P.PURLIN_OPT_SPIN_TIMEOUT_NS, 20_000_000)
        P.purlin_set_option(ctx, P.PURLIN_OPT_DROP_NOTIFY, 3)
        d = prepare(P, ctx, "all_reduce", src, dst, n, None, dtype, sms())
        assert d.drop_notify == 3
        X.collective(d, stream=stream)
        assert P.purlin_device_check(d, stream) == P.PURLIN_ERR_TIMEOUT
        P.purlin_device_release(ctx, d)
        P.purlin_set_option(ctx, P.PURLIN_OPT_DROP_NOTIFY, -1)
        d = prepare(P, ctx, "all_reduce", src, dst, n, None, dtype, sms())
        for b in dst:
            b.t[256:256 + b.nbytes].fill_(0)
        X.collective(d, stream=stream)
        assert P.purlin_device_check(d, stream) == P.PURLIN_OK
        assert_same(bodies(dst), want, "after a timeout")
        P.purlin_device_release(ctx, d)
        P.purlin_device_release(ctx, d)   # a cleared descriptor: no-op
    finally:
        ctx.close()


# ------------------------------------------------------------------ Atoms --

@pytest.mark.parametrize("src_phase,dst_phase", [(0, 0), (0, 6), (10, 0), (4, 14), (2, 2)])
def test_atom_copy(P, X, src_phase, dst_phase):
    """The README's sample: CTA b copies its slice with the Atom.  Slices
    start at every 16-byte phase (shifted staging), sizes are ragged."""
    stream = torch.cuda.current_stream()
    rng = np.random.default_rng(src_phase * 16 + dst_phase)
    for total, per_block in ((2, 2), (46, 16), (1000, 1000), (65538, 4098), (3 << 20, 1 << 18),
                             ((3 << 20) + 6, 98306)):
        data = rng.integers(0, 256, total + 64, dtype=np.uint8)
        src = Guarded(total + 64, fill=0xC3)
        src.t[256:256 + total + 64].copy_(torch.from_numpy(data))
        dst = Guarded(total + 64)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        X.atom_copy(dst.ptr + dst_phase, src.ptr + src_phase, total, per_block, status.data_ptr(),
                    stream=stream)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got = dst.body()
        assert np.array_equal(got[dst_phase:dst_phase + total], data[src_phase:src_phase + total])
        assert (got[:dst_phase] == 0x5A).all() and (got[dst_phase + total:] == 0x5A).all()
        assert dst.guards_ok() and src.guards_ok()


def test_atom_copy_refuses_odd_addresses(P, X):
    stream = torch.cuda.current_stream()
    src = Guarded(4096, fill=0xC3)
    dst = Guarded(4096)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    X.atom_copy(dst.ptr + 1, src.ptr, 1024, 1024, status.data_ptr(), stream=stream)
    torch.cuda.synchronize()
    assert int(status.item()) == P.PURLIN_ERR_ALIGNMENT
    assert (dst.body() == 0x5A).all()


@pytest.mark.parametrize("dtype", [0, 1], ids=["f32", "bf16"])
@pytest.mark.parametrize("nsrc", [1, 2, 5, 8, 13])
def test_atom_reduce(P, X, dtype, nsrc):
    """Each CTA reduces its slice of nsrc sources (SCORE): equal, bit for bit,
    to the oracle's AllReduce over those sources."""
    stream = torch.cuda.current_stream()
    for elems, per_block in ((1, 1), (37, 8), (4099, 1024), (300001, 65536)):
        ins = gen_inputs([elems] * nsrc, dtype, seed=nsrc * 1000 + elems % 1000)
        want = oracle.all_reduce(ins, dtype)[0]
        src = upload(ins)
        dst = Guarded(elems * ES[dtype])
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        X.atom_reduce(dst.ptr, [b.ptr for b in src], elems, per_block, dtype, status.data_ptr(),
                      stream=stream)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_same([dst.body()], [want], f"atom reduce nsrc={nsrc} elems={elems}")
        assert dst.guards_ok()
