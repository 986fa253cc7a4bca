"""GPU parity of the V collectives whose counts live in device memory (no
host round trip: the kernel takes the prefix sums), bit for bit against the
CPU oracle.

Covers every collective × dtype, R ∈ {1, 3, 8, 16} (16 gives AllToAllV a
256-segment table that stays in the kernel's shared-memory build area),
forced vector-unit and ring modes plus the device's own choice, zero and
ragged counts, counts produced by a kernel on the GPU (an MoE router's
bincount) at the MoE-dispatch workload's full size, and counts that exceed
the declared capacities (refused on the device, nothing written).
"""
import numpy as np
import pytest

import oracle
import workloads
from test_parity_gpu import (ES, Guarded, assert_same, gen_inputs, in_lengths, oracle_of,
                             out_sizes, size_cases)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GUARD = 256


@pytest.fixture(scope="module")
def P():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__

    __graft_entry__.build()
    import collective_datapath_atom_gb300 as mod

    torch.cuda.set_device(0)
    return mod


def capacity_buffers(lengths, cap_elems, es, fill, arrays=None):
    """R buffers of cap_elems elements each (plus guards); arrays, if given,
    are written at the start of each."""
    out = []
    for r, L in enumerate(lengths):
        b = Guarded(cap_elems * es, fill=fill)
        if arrays is not None and arrays[r].nbytes:
            b.t[GUARD:GUARD + arrays[r].nbytes].copy_(torch.from_numpy(arrays[r].view(np.uint8).copy()))
        out.append(b)
    return out


def call(P, ctx, coll, src, dst, d_counts, in_cap, out_cap, dtype):
    f = getattr(P, f"purlin_{coll}_device_counts")
    f(ctx, [b.ptr for b in src], [b.ptr for b in dst], d_counts, in_cap, out_cap, dtype)


VCOLLS = ["all_gather_v", "reduce_scatter_v", "all_to_all_v"]


@pytest.mark.parametrize("coll", VCOLLS)
@pytest.mark.parametrize("dtype", [0, 1], ids=["f32", "bf16"])
@pytest.mark.parametrize("variant", [0, 1, 2], ids=["device-choice", "units", "ring"])
@pytest.mark.parametrize("R", [1, 3, 8, 16])
def test_device_counts_parity(P, coll, dtype, variant, R):
    stream = torch.cuda.current_stream()
    ctx = P.purlin_init(R, stream)
    try:
        P.purlin_set_option(ctx, P.PURLIN_OPT_VARIANT, variant)
        cases = size_cases(coll, R)
        if R > 8:
            cases = cases[:2]
        for k, (n, counts) in enumerate(cases):
            lengths = in_lengths(coll, R, n, counts)
            ins = gen_inputs(lengths, dtype, seed=900 + 10 * k + R)
            want = oracle_of(coll, ins, dtype, counts)
            es = ES[dtype]
            osz = [s // es for s in out_sizes(coll, R, n, counts, es)]
            in_cap = max(lengths) + 5            # capacities above what the counts use
            out_cap = max(osz) + 3
            src = capacity_buffers(lengths, in_cap, es, 0xC3, ins)
            dst = capacity_buffers(osz, out_cap, es, 0x5A)
            d_counts = torch.tensor(counts, dtype=torch.int64, device="cuda")
            call(P, ctx, coll, src, dst, d_counts, in_cap, out_cap, dtype)
            P.purlin_check(ctx)
            assert P.purlin_last_launch(ctx)["variant"] == 4
            for r, b in enumerate(dst):
                body = b.body()
                used = osz[r] * es
                assert np.array_equal(body[:used], want[r].view(np.uint8)), \
                    f"{coll} R={R} dtype={dtype} variant={variant} case {k}: rank {r}"
                assert (body[used:] == 0x5A).all(), "wrote past the counts"
                assert b.guards_ok()
    finally:
        ctx.close()


def test_device_counts_refuses_counts_past_the_capacities(P):
    """Counts that need more room than declared: nothing is written, the
    error word says INVALID_ARG, and the context stays usable."""
    R, dtype = 8, 1
    stream = torch.cuda.current_stream()
    ctx = P.purlin_init(R, stream)
    try:
        C = np.full((R, R), 100, dtype=np.int64)
        C[2, 5] = 1000                  # row 2 sums to 1700, column 5 to 1700
        ins = gen_inputs([int(C[s].sum()) for s in range(R)], dtype, seed=5)
        for in_cap, out_cap in ((1699, 4000), (4000, 1699)):
            src = capacity_buffers([in_cap] * R, in_cap, 2, 0xC3,
                                   [x[:in_cap] for x in ins])
            dst = capacity_buffers([out_cap] * R, out_cap, 2, 0x5A)
            d_counts = torch.from_numpy(C.reshape(-1)).cuda()
            call(P, ctx, "all_to_all_v", src, dst, d_counts, in_cap, out_cap, dtype)
            assert P.purlin_check_status(ctx) == P.PURLIN_ERR_INVALID_ARG
            assert all((b.body() == 0x5A).all() for b in dst)
        # the same call with room for it
        src = capacity_buffers([1700] * R, 1700, 2, 0xC3, ins)
        dst = capacity_buffers([1700] * R, 1700, 2, 0x5A)
        call(P, ctx, "all_to_all_v", src, dst, torch.from_numpy(C.reshape(-1)).cuda(), 1700, 1700,
             dtype)
        P.purlin_check(ctx)
        want = oracle.all_to_all_v(ins, C, dtype)
        for d in range(R):
            used = int(C[:, d].sum()) * 2
            assert np.array_equal(dst[d].body()[:used], want[d].view(np.uint8))
        # counts of 2^40 or more are refused whatever the capacities
        big = np.zeros(R, dtype=np.int64)
        big[0] = 1 << 40
        src = capacity_buffers([16] * R, 16, 2, 0xC3)
        dst = capacity_buffers([16] * R, 16, 2, 0x5A)
        call(P, ctx, "all_gather_v", src, dst, torch.from_numpy(big).cuda(), 16, 16, dtype)
        assert P.purlin_check_status(ctx) == P.PURLIN_ERR_INVALID_ARG
    finally:
        ctx.close()


def test_device_counts_host_checks(P):
    """What the host can check without the counts: the counts pointer, the
    capacities' extents (overlaps) and R."""
    stream = torch.cuda.current_stream()
    ctx = P.purlin_init(4, stream)
    try:
        a = torch.empty(4096, dtype=torch.int16, device="cuda")
        src = [a[i * 512:(i + 1) * 512] for i in range(4)]
        dst = [torch.empty(1024, dtype=torch.int16, device="cuda") for _ in range(4)]
        cnt = torch.zeros(4, dtype=torch.int64, device="cuda")
        with pytest.raises(P.PurlinError) as e:   # null counts
            P.purlin_all_gather_v_device_counts(ctx, src, dst, 0, 512, 1024, 1)
        assert e.value.status == P.PURLIN_ERR_INVALID_ARG
        with pytest.raises(P.PurlinError) as e:   # an output overlapping an input extent
            P.purlin_all_gather_v_device_counts(ctx, src, [a] + dst[1:], cnt, 512, 1024, 1)
        assert e.value.status == P.PURLIN_ERR_ALIAS
        P.purlin_all_gather_v_device_counts(ctx, src, dst, cnt, 512, 1024, 1)   # zero counts
        P.purlin_check(ctx)
    finally:
        ctx.close()
    ctx = P.purlin_init(17, stream)
    try:
        bufs = [torch.empty(64, dtype=torch.int16, device="cuda") for _ in range(34)]
        cnt = torch.zeros(17, dtype=torch.int64, device="cuda")
        with pytest.raises(P.PurlinError) as e:
            P.purlin_all_gather_v_device_counts(ctx, bufs[:17], bufs[17:], cnt, 2, 34, 1)
        assert e.value.status == P.PURLIN_ERR_UNSUPPORTED
    finally:
        ctx.close()


def test_moe_dispatch_with_router_counts_on_the_gpu(P):
    """The MoE-dispatch workload (8 ranks x 16384 tokens x 7168, Zipf(1.2)
    destinations) with its count matrix produced ON THE GPU by a router
    (bincount of each rank's token-to-expert assignment) and never copied to
    the host before the AllToAllV.  Checked against the host-count call
    (bit for bit) and the oracle in full."""
    R = 8
    C, ins = workloads.moe_dispatch()
    # per-rank expert ids in destination order, so the input is packed by
    # destination exactly as the workload's count matrix says
    ids = [np.repeat(np.arange(R), C[s]) for s in range(R)]
    stream = torch.cuda.current_stream()
    ctx = P.purlin_init(R, stream)
    try:
        src = [torch.from_numpy(x.view(np.int16)).cuda() for x in ins]
        H = workloads.MOE_HIDDEN
        d_ids = [torch.from_numpy(i).cuda() for i in ids]
        d_counts = torch.stack([torch.bincount(i, minlength=R) for i in d_ids]) * H   # the router
        in_cap = workloads.MOE_TOKENS * H
        out_cap = int(C.sum(axis=0).max()) * H
        dst = [torch.zeros(out_cap, dtype=torch.int16, device="cuda") for _ in range(R)]
        P.purlin_all_to_all_v_device_counts(ctx, src, dst, d_counts.reshape(-1), in_cap, out_cap, 1)
        P.purlin_check(ctx)
        counts = (C * H).reshape(-1)
        ref = [torch.zeros(int(C[:, d].sum()) * H, dtype=torch.int16, device="cuda")
               for d in range(R)]
        P.purlin_all_to_all_v(ctx, src, ref, counts.tolist(), 1)
        P.purlin_check(ctx)
        for d in range(R):
            n = ref[d].numel()
            assert torch.equal(dst[d][:n], ref[d]), f"rank {d}"
            assert int(dst[d][n:].abs().sum().item()) == 0
        # the oracle, every output element
        for d, o in enumerate(oracle.all_to_all_v(ins, counts.reshape(R, R), 1)):
            n = o.size
            assert torch.equal(dst[d][:n], torch.from_numpy(o.view(np.int16)).cuda()), f"rank {d}"
    finally:
        ctx.close()
