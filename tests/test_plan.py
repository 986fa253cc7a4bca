"""Host logic of the library, no GPU: argument validation and the layout
compiler ("Purlin: Separating Orchestration from the Datapath of
Collectives" §3.1 layouts -> one kernel's schedule; §3.2 composed AllReduce
dependencies).

The compiled segment list is executed by a small interpreter here (bytes
copied, reductions summed in rank order in binary32 via numpy, bf16 rounded
by torch) and the result is compared bit for bit with the CPU oracle.  The
cut into TMA chunks and vector units is checked against its invariants.
"""
import numpy as np
import pytest

import oracle
import workloads

P = None


@pytest.fixture(scope="module", autouse=True)
def _lib():
    global P
    import __graft_entry__

    __graft_entry__.build()
    import collective_datapath_atom_gb300 as mod

    P = mod
    yield


ES = {0: 4, 1: 2}
NP = {0: np.float32, 1: np.uint16}
COLLS = {
    "all_reduce": 0, "reduce_scatter": 1, "all_gather": 2, "all_to_all": 3,
    "all_gather_v": 4, "reduce_scatter_v": 5, "all_to_all_v": 6,
}


def fake_ptrs(sizes, base=0x7f0000000000, gap=1 << 32):
    return [base + i * gap for i in range(len(sizes))]


def sizes_of(coll, R, n, counts, es):
    if coll in ("all_reduce", "all_to_all"):
        return [n * es] * R, [n * es] * R
    if coll == "reduce_scatter":
        return [n * es] * R, [n // R * es] * R
    if coll == "all_gather":
        return [n * es] * R, [R * n * es] * R
    if coll == "all_gather_v":
        return [c * es for c in counts], [sum(counts) * es] * R
    if coll == "reduce_scatter_v":
        return [sum(counts) * es] * R, [c * es for c in counts]
    C = np.asarray(counts).reshape(R, R)
    return [int(C[s].sum()) * es for s in range(R)], [int(C[:, d].sum()) * es for d in range(R)]


def inspect(coll, R, n, counts, dtype, variant, ar_mode=0, chunk=0, src=None, dst=None):
    op, layout = P.LAYOUTS[coll]
    es = ES.get(dtype, 2)
    ib, ob = sizes_of(coll, R, n, counts, es)
    src = fake_ptrs(ib) if src is None else src
    dst = fake_ptrs(ob, base=0x7e0000000000) if dst is None else dst
    return P.purlin_plan_inspect(COLLS[coll], R, src, dst, n, counts, dtype, op, layout,
                                 variant, ar_mode, chunk)


def _to_f32(raw, dtype):
    if dtype == 0:
        return raw.view(np.float32)
    return (raw.view(np.uint16).astype(np.uint32) << 16).view(np.float32)


def _round(x32, dtype):
    if dtype == 0:
        return x32.astype(np.float32).view(np.uint8)
    return workloads.to_bf16_bits(x32).view(np.uint8)


def interpret(segs, R, ins, outs, dtype):
    """Execute a segment list on byte buffers."""
    for sg in segs:
        b = sg["bytes"]
        dsts = [sg["dst_rank"]] if sg["dst_rank"] >= 0 else \
            [d for d in range(R) if d != sg["skip_rank"]]
        if sg["src_rank"] >= 0:
            srcbuf = outs[sg["src_rank"]] if sg["src_is_dst"] else ins[sg["src_rank"]]
            data = srcbuf[sg["src_off"]:sg["src_off"] + b].copy()
        else:
            acc = _to_f32(ins[0][sg["src_off"]:sg["src_off"] + b], dtype).copy()
            for s in range(1, R):
                acc = (acc + _to_f32(ins[s][sg["src_off"]:sg["src_off"] + b], dtype)).astype(
                    np.float32)
            data = _round(acc, dtype)
        for d in dsts:
            outs[d][sg["dst_off"]:sg["dst_off"] + b] = data


def oracle_run(coll, ins, n, counts, dtype):
    if coll == "all_reduce":
        return oracle.all_reduce(ins, dtype)
    if coll == "reduce_scatter":
        return oracle.reduce_scatter(ins, dtype)
    if coll == "all_gather":
        return oracle.all_gather(ins, dtype)
    if coll == "all_to_all":
        return oracle.all_to_all(ins, dtype)
    if coll == "all_gather_v":
        return oracle.all_gather_v(ins, counts, dtype)
    if coll == "reduce_scatter_v":
        return oracle.reduce_scatter_v(ins, counts, dtype)
    return oracle.all_to_all_v(ins, np.asarray(counts).reshape(len(ins), -1), dtype)


def make_case(coll, R, rng, dtype, small=True):
    n, counts = 0, None
    if coll in ("all_reduce", "all_gather"):
        n = int(rng.integers(0, 200 if small else 5000))
    elif coll in ("reduce_scatter", "all_to_all"):
        n = R * int(rng.integers(0, 40 if small else 2000))
    elif coll in ("all_gather_v", "reduce_scatter_v"):
        counts = [int(x) for x in rng.integers(0, 90 if small else 3000, size=R)]
        if R > 1:
            counts[int(rng.integers(0, R))] = 0
    else:
        counts = [int(x) for x in rng.integers(0, 30 if small else 900, size=R * R)]
    es = ES[dtype]
    ib, ob = sizes_of(coll, R, n, counts, es)
    ins = []
    for b in ib:
        x = rng.standard_normal(b // es).astype(np.float32)
        ins.append(x if dtype == 0 else workloads.to_bf16_bits(x))
    return n, counts, ins, ob


CASES = [(c, R, dt) for c in COLLS for R in (1, 2, 3, 8) for dt in (0, 1)]


@pytest.mark.parametrize("coll,R,dtype", CASES)
@pytest.mark.parametrize("variant,ar_mode", [(1, 0), (2, 1), (2, 2)])
def test_plan_executes_to_the_oracle(coll, R, dtype, variant, ar_mode):
    rng = np.random.default_rng(hash((coll, R, dtype, variant, ar_mode)) & 0xFFFF)
    for trial in range(3):
        n, counts, ins, ob = make_case(coll, R, rng, dtype, small=trial < 2)
        chunk = [0, 48, 4096][trial]
        st, segs, nch, nun = inspect(coll, R, n, counts, dtype, variant, ar_mode, chunk)
        assert st == 0, P.status_string(st)
        outs = [np.full(b, 0xAB, dtype=np.uint8) for b in ob]
        interpret(segs, R, [x.view(np.uint8) for x in ins], outs, dtype)
        want = oracle_run(coll, ins, n, counts, dtype)
        for o, w in zip(outs, want):
            assert np.array_equal(o, w.view(np.uint8)), (coll, R, dtype, n, counts)


@pytest.mark.parametrize("coll,R,dtype", CASES)
def test_cut_invariants(coll, R, dtype):
    rng = np.random.default_rng(1 + hash((coll, R, dtype)) & 0xFFFF)
    for trial in range(4):
        n, counts, ins, ob = make_case(coll, R, rng, dtype, small=trial % 2 == 0)
        chunk = int(rng.choice([16, 64, 1024, 32768]))
        for variant, ar_mode in ((1, 0), (2, 1), (2, 2)):
            st, segs, nch, nun = inspect(coll, R, n, counts, dtype, variant, ar_mode, chunk)
            assert st == 0
            es = ES[dtype]
            chunk_total = unit_total = 0
            for sg in segs:
                assert sg["bytes"] > 0 and sg["bytes"] % es == 0
                assert sg["src_off"] % es == 0 and sg["dst_off"] % es == 0
                g = sg["src_off"] if sg["src_rank"] < 0 else sg["dst_off"]
                assert sg["chunk_begin"] == chunk_total and sg["unit_begin"] == unit_total
                if sg["tma"]:
                    assert variant == 2
                    body = sg["bytes"] - sg["head_bytes"] - sg["tail_bytes"]
                    assert body > 0 and body % 16 == 0
                    assert sg["head_bytes"] < 16 and sg["tail_bytes"] < 16
                    # the body is aligned on the grid the segment's units follow:
                    # a reduce's sources, a copy's destination
                    assert (g + sg["head_bytes"]) % 16 == 0
                    if (sg["src_rank"] >= 0 and sg["dst_rank"] < 0 and sg["sync"] == 0
                            and sg["bytes"] >= 144):
                        # a copy to every rank that waits on nothing starts its
                        # body on a 128-byte line (the bytes before it are a
                        # segment of their own on the vector path)
                        assert (g + sg["head_bytes"]) % 128 == 0
                    assert (sg["src_off"] - sg["dst_off"]) % 16 == sg["shift"]
                    assert sg["chunk_bytes"] % 16 == 0
                    chunk_total += -(-body // sg["chunk_bytes"])
                    unit_total += (sg["head_bytes"] > 0) + (sg["tail_bytes"] > 0)
                else:
                    # one unit per 16-byte window: a reduce's windows follow
                    # the sources' grid, a copy's the destination's
                    a, b = g, g + sg["bytes"]
                    unit_total += -(-b // 16) - a // 16
                    if variant == 2:   # the bytes before a line, or no whole aligned window
                        assert sg["bytes"] < 128 + 16
            assert chunk_total == nch and unit_total == nun
            # every access stays inside its buffer
            ib, ob = sizes_of(coll, R, n, counts, es)
            for sg in segs:
                srcs = ([sg["src_rank"]] if sg["src_rank"] >= 0 else list(range(R)))
                src_len = ob if sg["src_is_dst"] else ib
                for s in srcs:
                    assert sg["src_off"] + sg["bytes"] <= src_len[s]
                dsts = [sg["dst_rank"]] if sg["dst_rank"] >= 0 else \
                    [d for d in range(R) if d != sg["skip_rank"]]
                for d in dsts:
                    assert sg["dst_off"] + sg["bytes"] <= ob[d]
                if sg["tma"]:
                    assert max(sg["chunk_bytes"] * (R if sg["src_rank"] < 0 else 1),
                               sg["chunk_bytes"]) <= 1 << 20
                    # the staged source range starts on the 16-byte boundary at
                    # or before the first body byte and ends on the one at or
                    # after the last (a shifted copy's hull): never past the
                    # granule holding the buffer's end
                    lead = sg["shift"] if sg["src_rank"] >= 0 else 0
                    h0 = sg["src_off"] + sg["head_bytes"] - lead
                    body = sg["bytes"] - sg["head_bytes"] - sg["tail_bytes"]
                    h1 = h0 + body + (16 if lead else 0)
                    assert h0 >= 0 and h0 % 16 == 0
                    for s_ in srcs:
                        assert h1 <= -(-src_len[s_] // 16) * 16
            notify = [s for s in segs if s["sync"] == 1]
            wait = [s for s in segs if s["sync"] == 2]
            assert len(notify) == len(wait)
            for a, b in zip(notify, wait):
                assert a["bytes"] == b["bytes"] and a["src_off"] == b["src_off"]
                assert a["dst_rank"] == b["src_rank"] == b["skip_rank"] and b["src_is_dst"] == 1
                assert b["chunk_bytes"] == a["chunk_bytes"] * R and a["tma"] and b["tma"]
            if notify:
                assert coll == "all_reduce" and variant == 2 and ar_mode == 2
                last_notify = max(s["chunk_begin"] for s in notify)
                assert all(s["chunk_begin"] > last_notify for s in wait)


def test_moe_dispatch_plan_is_aligned():
    """The MoE-dispatch AllToAllV (7168-wide bf16 tokens) is entirely TMA."""
    C, _ = workloads.moe_dispatch(payload=False)
    counts = (C * workloads.MOE_HIDDEN).reshape(-1).tolist()
    st, segs, nch, nun = inspect("all_to_all_v", 8, 0, counts, 1, 2)
    assert st == 0 and nun == 0 and all(s["tma"] for s in segs)
    assert sum(s["bytes"] for s in segs) == 8 * workloads.MOE_TOKENS * workloads.MOE_HIDDEN * 2


# ------------------------------------------------------------ validation ----

def _call(coll, R, n, counts, dtype=1, op=None, layout=None, src=None, dst=None, variant=1):
    dop, dlayout = P.LAYOUTS[coll]
    es = ES.get(dtype, 2)
    ib, ob = sizes_of(coll, R, n, counts, es)
    src = fake_ptrs(ib) if src is None else src
    dst = fake_ptrs(ob, base=0x7e0000000000) if dst is None else dst
    return P.purlin_plan_inspect(COLLS[coll], R, src, dst, n, counts, dtype,
                                 dop if op is None else op,
                                 dlayout if layout is None else layout, variant)[0]


def test_wrong_op_or_layout_is_unsupported():
    S, PK, T = P.PURLIN_SCATTERED, P.PURLIN_PACKED, P.PURLIN_TRANSPOSED
    assert _call("all_reduce", 4, 64, None, op=P.PURLIN_COPY) == P.PURLIN_ERR_UNSUPPORTED
    assert _call("all_gather", 4, 64, None, op=P.PURLIN_SUM) == P.PURLIN_ERR_UNSUPPORTED
    assert _call("reduce_scatter", 4, 64, None, layout=(S, S)) == P.PURLIN_ERR_UNSUPPORTED
    assert _call("all_to_all", 4, 64, None, layout=(S, PK)) == P.PURLIN_ERR_UNSUPPORTED
    assert _call("all_gather", 4, 64, None, layout=(PK, T)) == P.PURLIN_ERR_UNSUPPORTED
    assert _call("all_reduce", 4, 64, None, layout=(9, S)) == P.PURLIN_ERR_INVALID_ARG
    assert _call("all_reduce", 4, 64, None, op=7) == P.PURLIN_ERR_INVALID_ARG
    assert _call("all_reduce", 4, 64, None, dtype=5) == P.PURLIN_ERR_INVALID_ARG


def test_divisibility_and_rank_limits():
    assert _call("reduce_scatter", 4, 66, None) == P.PURLIN_ERR_INVALID_ARG
    assert _call("all_to_all", 3, 10, None) == P.PURLIN_ERR_INVALID_ARG
    assert _call("reduce_scatter", 4, 0, None) == P.PURLIN_OK
    assert _call("all_reduce", 64, 16, None) == P.PURLIN_OK
    st = P.purlin_plan_inspect(0, 65, [0x10] * 65, [0x10] * 65, 4, None, 1, 1, (1, 1), 1)[0]
    assert st == P.PURLIN_ERR_INVALID_ARG
    st = P.purlin_plan_inspect(6, 2, fake_ptrs([16] * 2), fake_ptrs([16] * 2, base=1 << 44), 0,
                               None, 1, 0, (1, 2), 1)[0]
    assert st == P.PURLIN_ERR_INVALID_ARG


def test_null_and_alignment():
    base = fake_ptrs([128] * 4)
    outs = fake_ptrs([128] * 4, base=0x7e0000000000)
    bad = list(base)
    bad[2] = 0
    assert _call("all_reduce", 4, 32, None, src=bad, dst=outs) == P.PURLIN_ERR_INVALID_ARG
    bad[2] = base[2] + 8
    assert _call("all_reduce", 4, 32, None, src=bad, dst=outs) == P.PURLIN_ERR_ALIGNMENT
    odd = list(outs)
    odd[3] += 4
    assert _call("all_reduce", 4, 32, None, src=base, dst=odd) == P.PURLIN_ERR_ALIGNMENT
    # a rank with nothing to send may pass a null pointer
    st = _call("all_gather_v", 3, 0, [4, 0, 4], src=[base[0], 0, base[2]],
               dst=outs[:3])
    assert st == P.PURLIN_OK
    # V variants need their counts
    st = P.purlin_plan_inspect(4, 3, base[:3], outs[:3], 0, None, 1, 0, (0, 1), 1)[0]
    assert st == P.PURLIN_ERR_INVALID_ARG


def test_aliasing_rules():
    n, es = 64, 2
    outs = fake_ptrs([n * es] * 4, base=0x7e0000000000)
    # in-place AllReduce is allowed
    assert _call("all_reduce", 4, n, None, src=outs, dst=outs) == P.PURLIN_OK
    # ... but an input on another rank's output is not
    mixed = [outs[1]] + outs[1:]
    assert _call("all_reduce", 4, n, None, src=mixed, dst=outs) == P.PURLIN_ERR_ALIAS
    # overlapping outputs
    ov = list(outs)
    ov[1] = ov[0] + 32
    assert _call("all_reduce", 4, n, None, src=fake_ptrs([n * es] * 4), dst=ov) == \
        P.PURLIN_ERR_ALIAS
    # in-place AllGather: input r sits at slot r of output r
    R = 4
    ag_out = fake_ptrs([R * n * es] * R, base=0x7e0000000000)
    ag_in = [ag_out[r] + r * n * es for r in range(R)]
    assert _call("all_gather", R, n, None, src=ag_in, dst=ag_out) == P.PURLIN_OK
    wrong = list(ag_in)
    wrong[2] = ag_out[2]          # slot 0 of rank 2's output: not the in-place form
    assert _call("all_gather", R, n, None, src=wrong, dst=ag_out) == P.PURLIN_ERR_ALIAS
    # in-place ReduceScatter is not an allowed form
    rs_in = fake_ptrs([R * n * es] * R)
    rs_out = [rs_in[r] for r in range(R)]
    assert _call("reduce_scatter", R, R * n, None, src=rs_in, dst=rs_out) == P.PURLIN_ERR_ALIAS
    # inputs may overlap one another
    same = [outs[0]] * 4
    assert _call("all_reduce", 4, n, None, src=same,
                 dst=fake_ptrs([n * es] * 4, base=0x7d0000000000)) == P.PURLIN_OK


@pytest.mark.parametrize("R", [2, 3, 8])
@pytest.mark.parametrize("dtype", [0, 1])
def test_alltoall_units_follow_the_transposition(R, dtype):
    """The vector kernel's build for a uniform AllToAll of whole windows reads
    no segment table: it sends unit u, window k = u % W of block u // W =
    s*R + d, from offset (d*W + k)*16 of source s to offset (s*W + k)*16 of
    destination d ("Purlin: Separating Orchestration from the Datapath of
    Collectives" §3.1: AllToAll is the scattered -> transposed layout).  The
    compiled plan numbers its units exactly that way, so both agree on every
    unit; a block that is not a whole number of windows has no such plan."""
    es = ES[dtype]
    for M in (16 // es, 64 // es * 3, 512):   # elements per block: whole windows
        n = R * M
        st, segs, _, nunits = inspect("all_to_all", R, n, None, dtype, 1)
        assert st == P.PURLIN_OK
        W = M * es // 16
        assert nunits == R * R * W and len(segs) == R * R
        for u in range(nunits):
            blk, k = divmod(u, W)
            s, d = divmod(blk, R)
            g = segs[blk]
            assert (g["src_rank"], g["dst_rank"]) == (s, d)
            assert g["unit_begin"] + k == u
            assert g["src_off"] + 16 * k == (d * W + k) * 16
            assert g["dst_off"] + 16 * k == (s * W + k) * 16
    # a ragged block (not a multiple of 16 bytes) is cut differently
    M = 16 // es + 1
    st, segs, _, nunits = inspect("all_to_all", R, R * M, None, dtype, 1)
    assert st == P.PURLIN_OK and nunits != R * R * (M * es // 16)
