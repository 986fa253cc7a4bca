"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Every comparison is bit for bit: copies are bitwise and reductions follow
the same fixed rank order in binary32 with one rounding ("Purlin: Separating
Orchestration from the Datapath of Collectives" §3.3 SCORE; "Purlin" README,
"Deterministic Reduction").  Outputs sit between guard zones that must stay
untouched.
"""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GUARD = 256
ES = {0: 4, 1: 2}


@pytest.fixture(scope="module")
def P():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__

    __graft_entry__.build()
    import collective_datapath_atom_gb300 as mod

    torch.cuda.set_device(0)
    return mod


@pytest.fixture
def ctx8(P):
    c = P.purlin_init(8, torch.cuda.current_stream())
    yield c
    c.close()


def make_ctx(P, R):
    return P.purlin_init(R, torch.cuda.current_stream())


# ------------------------------------------------------------- buffers ----

class Guarded:
    """A device byte buffer with guard zones on both sides."""

    def __init__(self, nbytes, fill=0x5A):
        self.nbytes = nbytes
        self.t = torch.full((nbytes + 2 * GUARD,), fill, dtype=torch.uint8, device="cuda")
        self.fill = fill

    @property
    def ptr(self):
        return self.t.data_ptr() + GUARD

    def body(self):
        return self.t[GUARD:GUARD + self.nbytes].cpu().numpy()

    def guards_ok(self):
        g = torch.cat([self.t[:GUARD], self.t[GUARD + self.nbytes:]])
        return bool((g == self.fill).all().item())


def upload(arrays):
    out = []
    for a in arrays:
        b = Guarded(a.nbytes, fill=0xC3)
        if a.nbytes:
            b.t[GUARD:GUARD + a.nbytes].copy_(torch.from_numpy(a.view(np.uint8).copy()))
        out.append(b)
    return out


def outputs(sizes):
    return [Guarded(s) for s in sizes]


def run(P, ctx, coll, ins, out_sizes, dtype, n=0, counts=None):
    src = upload(ins)
    dst = outputs(out_sizes)
    f = getattr(P, "purlin_" + coll)
    arg = counts if coll.endswith("_v") else n
    f(ctx, [b.ptr for b in src], [b.ptr for b in dst], arg, dtype)
    P.purlin_check(ctx)
    for b in src + dst:
        assert b.guards_ok(), "guard zone overwritten"
    return [b.body() for b in dst], src


def oracle_of(coll, ins, dtype, counts=None, R=None):
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


def out_sizes(coll, R, n, counts, es):
    if coll in ("all_reduce", "all_to_all"):
        return [n * es] * R
    if coll == "reduce_scatter":
        return [n // R * es] * R
    if coll == "all_gather":
        return [R * n * es] * R
    if coll == "all_gather_v":
        return [sum(counts) * es] * R
    if coll == "reduce_scatter_v":
        return [c * es for c in counts]
    C = np.asarray(counts).reshape(R, R)
    return [int(C[:, d].sum()) * es for d in range(R)]


def in_lengths(coll, R, n, counts):
    if coll in ("all_reduce", "all_to_all", "reduce_scatter", "all_gather"):
        return [n] * R
    if coll == "all_gather_v":
        return list(counts)
    if coll == "reduce_scatter_v":
        return [sum(counts)] * R
    C = np.asarray(counts).reshape(R, R)
    return [int(C[s].sum()) for s in range(R)]


def gen_inputs(lengths, dtype, seed):
    rng = np.random.default_rng(seed)
    out = []
    for L in lengths:
        x = rng.standard_normal(L).astype(np.float32)
        out.append(x if dtype == 0 else workloads.to_bf16_bits(x))
    return out


def assert_same(got, want, what):
    for d, (g, w) in enumerate(zip(got, want)):
        w8 = w.view(np.uint8)
        if not np.array_equal(g, w8):
            bad = np.nonzero(g != w8)[0]
            raise AssertionError(f"{what}: rank {d} differs at byte {bad[0]} "
                                 f"({bad.size} bytes differ of {w8.size})")


# -------------------------------------------------------------- cases ----

def size_cases(coll, R):
    """(n, counts) pairs: tiny, ragged, several chunks, unaligned phases."""
    rng = np.random.default_rng(R * 31 + len(coll))
    if coll in ("all_reduce", "all_gather"):
        return [(n, None) for n in (1, 7, 8, 33, 4096, 70001, 3 * 65536 + 5)]
    if coll in ("reduce_scatter", "all_to_all"):
        return [(R * m, None) for m in (1, 3, 8, 517, 16384, 40000 + 3)]
    if coll in ("all_gather_v", "reduce_scatter_v"):
        cs = [[int(x) for x in rng.integers(0, 50, size=R)],
              [int(x) for x in rng.integers(1000, 90000, size=R)],
              [8192 * (k + 1) for k in range(R)]]
        cs[0][0] = 0
        return [(0, c) for c in cs]
    cs = [[int(x) for x in rng.integers(0, 20, size=R * R)],
          [int(x) for x in rng.integers(0, 9000, size=R * R)],
          [1024 * int(x) for x in rng.integers(0, 40, size=R * R)]]
    return [(0, c) for c in cs]


COLLS = ["all_reduce", "reduce_scatter", "all_gather", "all_to_all", "all_gather_v",
         "reduce_scatter_v", "all_to_all_v"]


@pytest.mark.parametrize("coll", COLLS)
@pytest.mark.parametrize("dtype", [0, 1], ids=["f32", "bf16"])
@pytest.mark.parametrize("variant", [1, 2], ids=["latency", "throughput"])
@pytest.mark.parametrize("R", [1, 3, 8])
def test_parity(P, coll, dtype, variant, R):
    ctx = make_ctx(P, R)
    try:
        P.purlin_set_option(ctx, P.PURLIN_OPT_VARIANT, variant)
        for k, (n, counts) in enumerate(size_cases(coll, R)):
            ins = gen_inputs(in_lengths(coll, R, n, counts), dtype, seed=1000 * k + R)
            got, _ = run(P, ctx, coll, ins, out_sizes(coll, R, n, counts, ES[dtype]), dtype, n,
                         counts)
            want = oracle_of(coll, ins, dtype, counts)
            assert_same(got, want, f"{coll} R={R} dtype={dtype} variant={variant} n={n}")
            info = P.purlin_last_launch(ctx)
            assert info["variant"] in (0, variant)
    finally:
        ctx.close()


@pytest.mark.parametrize("dtype", [0, 1], ids=["f32", "bf16"])
@pytest.mark.parametrize("R", [2, 3, 8])
def test_allreduce_composed_mode(P, dtype, R):
    """SNAC across CTAs: reducing CTAs notify per-chunk flags, gathering CTAs
    acquire them ("Purlin: Separating Orchestration from the Datapath of Collectives"
    §3.2, composed AllReduce)."""
    ctx = make_ctx(P, R)
    try:
        P.purlin_set_option(ctx, P.PURLIN_OPT_VARIANT, 2)
        P.purlin_set_option(ctx, P.PURLIN_OPT_AR_MODE, 2)
        for k, n in enumerate((64, 4096 + 3, 100003, 1 << 20)):
            for chunk in (0, 512):
                P.purlin_set_option(ctx, P.PURLIN_OPT_CHUNK_BYTES, chunk)
                ins = gen_inputs([n] * R, dtype, seed=77 + k)
                got, _ = run(P, ctx, "all_reduce", ins, [n * ES[dtype]] * R, dtype, n)
                assert_same(got, oracle.all_reduce(ins, dtype), f"composed n={n}")
                assert P.purlin_last_launch(ctx)["variant"] == 3
    finally:
        ctx.close()


@pytest.mark.parametrize("coll,n,spread", [
    ("all_reduce", 1024, True),     # 2 KiB per rank: 128 units of 16 vectors
    ("all_reduce", 1 << 17, True),  # 256 KiB per rank: 16384 units, the largest spread plan
    ("all_reduce", 1 << 18, False),  # 32768 units: more than a spread plan holds
    ("all_reduce", 512, False),     # 64 units: too light to spread
    ("all_gather", 512, True),      # 1 KiB per rank: 512 units of 9 vectors
    ("all_gather", 128, False),     # 256 B per rank: too light
    ("reduce_scatter", 1024, False),  # one store per unit: never spread
])
def test_small_all_rank_plans_spread(P, ctx8, coll, n, spread):
    """A small vector-kernel plan whose every unit stores to all R ranks runs
    about 16 CTAs of 32-128 threads; other plans keep blocks of up to 256.
    The results match the oracle either way."""
    dtype = 1
    ins = gen_inputs([n] * 8, dtype, seed=411)
    got, _ = run(P, ctx8, coll, ins, out_sizes(coll, 8, n, None, 2), dtype, n)
    assert_same(got, oracle_of(coll, ins, dtype), f"{coll} n={n}")
    info = P.purlin_last_launch(ctx8)
    assert info["variant"] == 1
    units = {"all_reduce": n // 8, "all_gather": n, "reduce_scatter": n // 8}[coll]
    assert info["units"] == units
    if spread:
        assert 32 <= info["block"] <= 128 and info["grid"] == -(-units // info["block"])
        assert info["grid"] >= min(16, units // 32)
    else:
        assert info["block"] == min(256, -(-units // 32) * 32)


@pytest.mark.parametrize("coll", ["all_gather", "reduce_scatter", "all_reduce", "all_to_all"])
def test_ring_grid_option_above_policy(P, ctx8, coll):
    """PURLIN_OPT_CTAS may ask for more throughput CTAs than the policy's CTAs
    per SM, up to what fits on the GPU at once: a small ring shape runs two
    CTAs per SM, an oversized request is capped, and the results stay exact."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    dtype = 1
    n = (1 << 20) + 40            # several chunks per CTA and a ragged tail
    n -= n % 8 if coll in ("reduce_scatter", "all_to_all") else 0
    P.purlin_set_option(ctx8, P.PURLIN_OPT_VARIANT, 2)
    P.purlin_set_option(ctx8, P.PURLIN_OPT_CONSUMER_WARPS, 4)
    P.purlin_set_option(ctx8, P.PURLIN_OPT_STAGES, 2)
    P.purlin_set_option(ctx8, P.PURLIN_OPT_CHUNK_BYTES, 2048)   # 32 KiB stages at most
    try:
        for k, want in enumerate((2 * sms, 1 << 20)):
            P.purlin_set_option(ctx8, P.PURLIN_OPT_CTAS, want)
            ins = gen_inputs([n] * 8, dtype, seed=301 + k)
            got, _ = run(P, ctx8, coll, ins, out_sizes(coll, 8, n, None, 2), dtype, n)
            assert_same(got, oracle_of(coll, ins, dtype), f"{coll} CTAs={want}")
            info = P.purlin_last_launch(ctx8)
            assert info["variant"] in (2, 3)
            if want == 2 * sms:
                assert info["grid"] == 2 * sms
            else:
                assert 2 * sms <= info["grid"] <= 32 * sms   # the occupancy limit
    finally:
        for opt in (P.PURLIN_OPT_CTAS, P.PURLIN_OPT_CONSUMER_WARPS, P.PURLIN_OPT_STAGES,
                    P.PURLIN_OPT_CHUNK_BYTES, P.PURLIN_OPT_VARIANT):
            P.purlin_set_option(ctx8, opt, 0)


def test_allreduce_composed_flag_generations(P, ctx8):
    """Composed AllReduce with more reducing chunks than flag slots per
    parity (256 MiB per rank, 65536 chunks of 4 KiB): chunk c publishes
    epoch + floor(pos / F) into slot pos mod F, pos its walk position.  The
    fused mode is compared with the oracle in full, and the composed mode
    with the fused mode bit for bit, twice in a row."""
    n = 128 << 20
    ins = workloads.ar_sweep_inputs(n // workloads.HIDDEN)
    src = [torch.from_numpy(x.view(np.int16)).cuda() for x in ins]
    fused = [torch.empty(n, dtype=torch.int16, device="cuda") for _ in range(8)]
    P.purlin_set_option(ctx8, P.PURLIN_OPT_VARIANT, 2)
    P.purlin_set_option(ctx8, P.PURLIN_OPT_AR_MODE, 1)
    P.purlin_all_reduce(ctx8, src, fused, n, 1)
    P.purlin_check(ctx8)
    want = torch.from_numpy(oracle.all_reduce_one(ins, 1).view(np.int16)).cuda()
    for d in range(8):
        assert torch.equal(fused[d], want), f"fused rank {d}"
    del want
    P.purlin_set_option(ctx8, P.PURLIN_OPT_AR_MODE, 2)
    P.purlin_set_option(ctx8, P.PURLIN_OPT_CHUNK_BYTES, 4096)   # 65536 reducing chunks
    try:
        for call in range(2):
            dst = [torch.zeros(n, dtype=torch.int16, device="cuda") for _ in range(8)]
            P.purlin_all_reduce(ctx8, src, dst, n, 1)
            P.purlin_check(ctx8)
            info = P.purlin_last_launch(ctx8)
            assert info["variant"] == 3 and info["epoch_next"] - info["epoch"] >= 3   # two generations
            for d in range(8):
                assert torch.equal(dst[d], fused[d]), f"call {call} rank {d}"
            del dst
        # the default composed ring (fewer, larger chunks) gives the same bits
        P.purlin_set_option(ctx8, P.PURLIN_OPT_CHUNK_BYTES, 0)
        dst = [torch.zeros(n, dtype=torch.int16, device="cuda") for _ in range(8)]
        P.purlin_all_reduce(ctx8, src, dst, n, 1)
        P.purlin_check(ctx8)
        assert P.purlin_last_launch(ctx8)["variant"] == 3
        for d in range(8):
            assert torch.equal(dst[d], fused[d]), f"default ring, rank {d}"
    finally:
        P.purlin_set_option(ctx8, P.PURLIN_OPT_CHUNK_BYTES, 0)


def test_repeated_calls_need_no_reset(P, ctx8):
    """Epoch parity and monotonic flags ("Purlin: Separating Orchestration from the Datapath of Collectives"
    §4.3): many calls in a
    row, no flag reset, each correct; the epoch advances by an odd amount."""
    P.purlin_set_option(ctx8, P.PURLIN_OPT_VARIANT, 2)
    P.purlin_set_option(ctx8, P.PURLIN_OPT_AR_MODE, 2)
    P.purlin_set_option(ctx8, P.PURLIN_OPT_CHUNK_BYTES, 256)
    n = 300000
    last = None
    for k in range(6):
        ins = gen_inputs([n] * 8, 1, seed=k)
        got, _ = run(P, ctx8, "all_reduce", ins, [2 * n] * 8, 1, n)
        assert_same(got, oracle.all_reduce(ins, 1), f"call {k}")
        info = P.purlin_last_launch(ctx8)
        assert (info["epoch_next"] - info["epoch"]) % 2 == 1
        if last is not None:
            assert info["epoch"] == last
        last = info["epoch_next"]


def test_in_place_allreduce(P, ctx8):
    for variant, mode in ((1, 0), (2, 1), (2, 2)):
        P.purlin_set_option(ctx8, P.PURLIN_OPT_VARIANT, variant)
        P.purlin_set_option(ctx8, P.PURLIN_OPT_AR_MODE, mode)
        n = 50001
        ins = gen_inputs([n] * 8, 1, seed=5)
        bufs = upload(ins)
        P.purlin_all_reduce(ctx8, [b.ptr for b in bufs], [b.ptr for b in bufs], n, 1)
        P.purlin_check(ctx8)
        want = oracle.all_reduce(ins, 1)
        assert_same([b.body() for b in bufs], want, f"in-place AR variant {variant}")
        assert all(b.guards_ok() for b in bufs)


def test_in_place_allgather(P, ctx8):
    for variant in (1, 2):
        P.purlin_set_option(ctx8, P.PURLIN_OPT_VARIANT, variant)
        for n in (4096, 336, 100008):
            ins = gen_inputs([n] * 8, 1, seed=n)
            outs = outputs([8 * n * 2] * 8)
            for r in range(8):
                outs[r].t[GUARD + r * n * 2:GUARD + (r + 1) * n * 2].copy_(
                    torch.from_numpy(ins[r].view(np.uint8).copy()))
            srcs = [outs[r].ptr + r * n * 2 for r in range(8)]
            P.purlin_all_gather(ctx8, srcs, [o.ptr for o in outs], n, 1)
            P.purlin_check(ctx8)
            assert_same([o.body() for o in outs], oracle.all_gather(ins, 1), "in-place AG")
    # r*n elements off a 16-byte boundary: the in-place input is misaligned
    n = 333
    outs = outputs([8 * n * 2] * 8)
    with pytest.raises(P.PurlinError) as e:
        P.purlin_all_gather(ctx8, [outs[r].ptr + r * n * 2 for r in range(8)],
                            [o.ptr for o in outs], n, 1)
    assert e.value.status == P.PURLIN_ERR_ALIGNMENT


def test_empty_calls_are_noops(P, ctx8):
    P.purlin_all_reduce(ctx8, [0] * 8, [0] * 8, 0, 1)
    assert P.purlin_last_launch(ctx8)["variant"] == 0
    P.purlin_all_gather_v(ctx8, [0] * 8, [0] * 8, [0] * 8, 1)
    P.purlin_all_to_all_v(ctx8, [0] * 8, [0] * 8, [0] * 64, 0)
    P.purlin_check(ctx8)


def test_argument_errors_enqueue_nothing(P, ctx8):
    n = 64
    ins = gen_inputs([n] * 8, 1, seed=1)
    src = upload(ins)
    dst = outputs([n * 2] * 8)
    with pytest.raises(P.PurlinError) as e:
        P.purlin_all_reduce(ctx8, [b.ptr for b in src], [b.ptr for b in dst], n, 1,
                            op=P.PURLIN_COPY)
    assert e.value.status == P.PURLIN_ERR_UNSUPPORTED
    with pytest.raises(P.PurlinError) as e:
        P.purlin_all_reduce(ctx8, [b.ptr + 2 for b in src], [b.ptr for b in dst], n - 1, 1)
    assert e.value.status == P.PURLIN_ERR_ALIGNMENT
    P.purlin_check(ctx8)
    assert all((torch.from_numpy(b.body()) == 0x5A).all() for b in dst)


def test_dropped_notify_times_out_and_recovers(P, ctx8):
    """Fault injection from the host: the notify of one chunk is skipped, so
    the gathering CTA's bounded acquire expires.  The kernel records
    PURLIN_ERR_TIMEOUT and ends; the context stays usable."""
    P.purlin_set_option(ctx8, P.PURLIN_OPT_VARIANT, 2)
    P.purlin_set_option(ctx8, P.PURLIN_OPT_AR_MODE, 2)
    P.purlin_set_option(ctx8, P.PURLIN_OPT_SPIN_TIMEOUT_NS, 2_000_000)   # 2 ms
    P.purlin_set_option(ctx8, P.PURLIN_OPT_DROP_NOTIFY, 3)
    n = 1 << 16
    ins = gen_inputs([n] * 8, 1, seed=9)
    src = upload(ins)
    dst = outputs([2 * n] * 8)
    P.purlin_all_reduce(ctx8, [b.ptr for b in src], [b.ptr for b in dst], n, 1)
    assert P.purlin_check_status(ctx8) == P.PURLIN_ERR_TIMEOUT
    assert P.purlin_check_status(ctx8) == P.PURLIN_OK   # the word was cleared
    P.purlin_set_option(ctx8, P.PURLIN_OPT_DROP_NOTIFY, -1)
    got, _ = run(P, ctx8, "all_reduce", ins, [2 * n] * 8, 1, n)
    assert_same(got, oracle.all_reduce(ins, 1), "after recovery")


def test_golden_fixtures_on_gpu(P):
    """The hand-derived fixtures, straight through the CUDA path."""
    import json
    import os

    gdir = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    g = json.load(open(os.path.join(gdir, "score_order_f32.json")))
    ins = [np.array([int(h, 16) for h in row], dtype=np.uint32).view(np.float32)
           for row in g["inputs_f32_hex"]]
    want = np.array([int(h, 16) for h in g["output_f32_hex"]], dtype=np.uint32)
    for variant in (1, 2):
        ctx = make_ctx(P, 3)
        P.purlin_set_option(ctx, P.PURLIN_OPT_VARIANT, variant)
        got, _ = run(P, ctx, "all_reduce", ins, [len(want) * 4] * 3, 0, len(want))
        ctx.close()
        for o in got:
            assert np.array_equal(o.view(np.uint32), want)
    g = json.load(open(os.path.join(gdir, "score_round_once_bf16.json")))
    for case in g["cases"]:
        ins = [np.array([int(h, 16) for h in row], dtype=np.uint16)
               for row in case["inputs_bf16_hex"]]
        want = np.array([int(h, 16) for h in case["output_bf16_hex"]], dtype=np.uint16)
        ctx = make_ctx(P, len(ins))
        got, _ = run(P, ctx, "all_reduce", ins, [2] * len(ins), 1, 1)
        ctx.close()
        for o in got:
            assert np.array_equal(o.view(np.uint16), want)


def test_nan_and_signed_zero_copies_are_bitwise(P, ctx8):
    n = 1000
    ins = [np.full(n, 0, dtype=np.uint32) for _ in range(8)]
    for s in range(8):
        ins[s][::3] = 0x7FC00000 | (s * 977 + 1)     # quiet NaNs with payloads
        ins[s][1::3] = 0x80000000                    # -0.0
        ins[s][2::3] = 0xFF800001 + s                # signalling NaN patterns
    ins = [x.view(np.float32) for x in ins]
    for variant in (1, 2):
        P.purlin_set_option(ctx8, P.PURLIN_OPT_VARIANT, variant)
        got, _ = run(P, ctx8, "all_gather", ins, [8 * n * 4] * 8, 0, n)
        assert_same(got, oracle.all_gather(ins, 0), "NaN AllGather")
        C = np.full((8, 8), n // 8)
        got, _ = run(P, ctx8, "all_to_all", ins, [n * 4] * 8, 0, n)
        assert_same(got, oracle.all_to_all(ins, 0), "NaN AllToAll")


# ----------------------------------------- the pages' V-collective workload --

@pytest.mark.parametrize("total_bytes", [1024, 2048, 8192, 1 << 20, 16 << 20])
def test_v_collectives_zipf_partition(P, ctx8, total_bytes):
    """AllGatherV / ReduceScatterV / AllToAllV on the Zipf(s = 0.125) split of
    a total T over 8 ranks (uniform at 1 and 2 KiB; AllToAllV rotates the
    split so every rank sends and receives T), "Purlin: Separating Orchestration from the Datapath of Collectives"
    §C.4."""
    T = total_bytes // 2
    part = workloads.zipf_partition(T)
    assert sum(part) == T
    for variant in (0, 1, 2):
        P.purlin_set_option(ctx8, P.PURLIN_OPT_VARIANT, variant)
        ins = gen_inputs(part, 1, seed=T + 1)
        got, _ = run(P, ctx8, "all_gather_v", ins, [T * 2] * 8, 1, counts=part)
        assert_same(got, oracle.all_gather_v(ins, part, 1), f"AGV T={T} v={variant}")
        ins = gen_inputs([T] * 8, 1, seed=T + 2)
        got, _ = run(P, ctx8, "reduce_scatter_v", ins, [c * 2 for c in part], 1, counts=part)
        assert_same(got, oracle.reduce_scatter_v(ins, part, 1), f"RSV T={T} v={variant}")
        C = workloads.rotated_counts(part)
        got, _ = run(P, ctx8, "all_to_all_v", ins, [T * 2] * 8, 1, counts=C.reshape(-1).tolist())
        assert_same(got, oracle.all_to_all_v(ins, C, 1), f"A2AV T={T} v={variant}")


# ------------------------------------------------------- full-size configs --

def _device(arrays):
    return [torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()
            for a in arrays]


def test_cfg_allreduce_f32_exact(P, ctx8):
    w = workloads.AR_F32_R8_4096
    ins = workloads.inputs_for(w)
    src = _device(ins)
    dst = [torch.empty(w.n, dtype=torch.float32, device="cuda") for _ in range(8)]
    P.purlin_all_reduce(ctx8, src, dst, w.n, 0)
    P.purlin_check(ctx8)
    exact = np.sum(np.stack(ins).astype(np.int64), axis=0).astype(np.float32)
    for d in range(8):
        got = dst[d].cpu().numpy()
        assert np.array_equal(got, exact)
        assert np.array_equal(got.view(np.uint32), oracle.all_reduce(ins, 0)[d].view(np.uint32))


def test_cfg_allgather_bf16_full(P, ctx8):
    """The default variant (the vector kernel) and the ring, each in full."""
    w = workloads.AG_BF16_R8_8MI
    ins = workloads.inputs_for(w)
    src = _device(ins)
    want = torch.from_numpy(np.concatenate(ins).view(np.int16)).cuda()   # concatenation invariant
    oracle_out = [torch.from_numpy(o.view(np.int16)).cuda() for o in oracle.all_gather(ins, 1)]
    try:
        for variant, ran in ((0, 1), (2, 2)):
            P.purlin_set_option(ctx8, P.PURLIN_OPT_VARIANT, variant)
            dst = [torch.full((8 * w.n,), -1, dtype=torch.int16, device="cuda") for _ in range(8)]
            P.purlin_all_gather(ctx8, src, dst, w.n, 1)
            P.purlin_check(ctx8)
            assert P.purlin_last_launch(ctx8)["variant"] == ran
            for d in range(8):
                assert torch.equal(dst[d], want)
                assert torch.equal(dst[d], oracle_out[d]), f"variant {ran} rank {d}"   # the oracle, in full
            del dst
    finally:
        P.purlin_set_option(ctx8, P.PURLIN_OPT_VARIANT, 0)


def test_cfg_reducescatter_bf16_full(P, ctx8):
    """The default variant (the vector kernel) and the ring, each in full."""
    w = workloads.RS_BF16_R8_128MI
    ins = workloads.inputs_for(w)
    src = _device(ins)
    M = w.n // 8
    want = oracle.reduce_scatter(ins, 1)
    try:
        for variant, ran in ((0, 1), (2, 2)):
            P.purlin_set_option(ctx8, P.PURLIN_OPT_VARIANT, variant)
            dst = [torch.full((M,), -1, dtype=torch.int16, device="cuda") for _ in range(8)]
            P.purlin_reduce_scatter(ctx8, src, dst, w.n, 1)
            P.purlin_check(ctx8)
            assert P.purlin_last_launch(ctx8)["variant"] == ran
            for r in range(8):
                assert np.array_equal(dst[r].cpu().numpy().view(np.uint16), want[r]), \
                    f"variant {ran} rank {r}"
    finally:
        P.purlin_set_option(ctx8, P.PURLIN_OPT_VARIANT, 0)


def test_cfg_alltoallv_moe_full(P, ctx8):
    C, ins = workloads.moe_dispatch()
    counts = (C * workloads.MOE_HIDDEN).reshape(-1)
    src = _device(ins)
    dst = [torch.empty(int(counts.reshape(8, 8)[:, d].sum()), dtype=torch.int16, device="cuda")
           for d in range(8)]
    P.purlin_all_to_all_v(ctx8, src, dst, counts.tolist(), 1)
    P.purlin_check(ctx8)
    want = oracle.all_to_all_v(ins, counts.reshape(8, 8), 1)
    for d in range(8):
        assert np.array_equal(dst[d].cpu().numpy().view(np.uint16), want[d])


@pytest.mark.parametrize("batch", workloads.AR_BF16_SWEEP_BATCHES)
def test_cfg_allreduce_sweep(P, ctx8, batch):
    """Every size with the default variant (the vector kernel); from 4 MiB
    per rank also with the fused ring."""
    w = workloads.ar_sweep_workload(batch)
    ins = workloads.inputs_for(w)
    src = _device(ins)
    # every output against the oracle's, element by element
    want = torch.from_numpy(oracle.all_reduce_one(ins, 1).view(np.int16)).cuda()
    try:
        for variant in ((0, 2) if batch >= 512 else (0,)):
            P.purlin_set_option(ctx8, P.PURLIN_OPT_VARIANT, variant)
            dst = [torch.full((w.n,), -1, dtype=torch.int16, device="cuda") for _ in range(8)]
            P.purlin_all_reduce(ctx8, src, dst, w.n, 1)
            P.purlin_check(ctx8)
            assert P.purlin_last_launch(ctx8)["variant"] == (1 if variant == 0 else 2)
            for d in range(8):
                if not torch.equal(dst[d], want):
                    bad = torch.nonzero(dst[d] != want)[0].item()
                    raise AssertionError(f"batch {batch} variant {variant}: rank {d} differs "
                                         f"first at element {bad}")
            del dst
    finally:
        P.purlin_set_option(ctx8, P.PURLIN_OPT_VARIANT, 0)


# --------------------------------------------------------------- wide R ----

@pytest.mark.parametrize("coll", COLLS)
@pytest.mark.parametrize("variant", [1, 2], ids=["latency", "throughput"])
@pytest.mark.parametrize("R", [16, 64])
def test_parity_wide_R(P, coll, variant, R):
    """More than 8 ranks: the rank pointers need the large parameter block and
    the segment tables live in device memory (AllToAll(V) at R = 64 has 4096
    segments, read from global memory rather than staged)."""
    ctx = make_ctx(P, R)
    try:
        P.purlin_set_option(ctx, P.PURLIN_OPT_VARIANT, variant)
        rng = np.random.default_rng(R + variant)
        if coll in ("all_reduce", "all_gather"):
            cases = [(37, None), (4099, None)]
        elif coll in ("reduce_scatter", "all_to_all"):
            cases = [(R * 3, None), (R * 517, None)]
        elif coll in ("all_gather_v", "reduce_scatter_v"):
            cases = [(0, [int(x) for x in rng.integers(0, 300, size=R)])]
        else:
            cases = [(0, [int(x) for x in rng.integers(0, 40, size=R * R)])]
        for k, (n, counts) in enumerate(cases):
            ins = gen_inputs(in_lengths(coll, R, n, counts), 1, seed=4000 + 10 * k + R)
            got, _ = run(P, ctx, coll, ins, out_sizes(coll, R, n, counts, 2), 1, n, counts)
            assert_same(got, oracle_of(coll, ins, 1, counts), f"{coll} R={R} v={variant} n={n}")
    finally:
        ctx.close()


@pytest.mark.parametrize("R", [16, 31, 64])
def test_composed_allreduce_wide_R(P, R):
    """Composed AllReduce (2R + 1 segments, notifying and waiting chunks)
    with more than 8 ranks, against the oracle."""
    ctx = make_ctx(P, R)
    try:
        P.purlin_set_option(ctx, P.PURLIN_OPT_VARIANT, 2)
        P.purlin_set_option(ctx, P.PURLIN_OPT_AR_MODE, 2)
        # the last case, with 256-byte chunks, has enough reducing chunks for
        # the ring to interleave its gathering chunks (more than lag + 1
        # groups of R: lag = 8 * 152 // (R + 1) groups on 152 CTAs, with the
        # ring's flag batches of 4)
        for k, (n, chunk) in enumerate(((R * 16 * 3 + 5, 0), (70001, 0), (300007, 256))):
            P.purlin_set_option(ctx, P.PURLIN_OPT_CHUNK_BYTES, chunk)
            ins = gen_inputs([n] * R, 1, seed=5000 + k + R)
            got, _ = run(P, ctx, "all_reduce", ins, [n * 2] * R, 1, n)
            assert_same(got, oracle.all_reduce(ins, 1), f"composed R={R} n={n} chunk={chunk}")
            assert P.purlin_last_launch(ctx)["variant"] == 3
    finally:
        ctx.close()
