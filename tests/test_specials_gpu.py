"""GPU parity of reductions over NaN, infinities, overflow and subnormals.

"Purlin: Separating Orchestration from the Datapath of Collectives" §3.3
(SCORE: each output is the sum of its sources in a fixed order, rounded
once) and the "Purlin" README, "Deterministic Reduction".  IEEE 754 fixes
every bit of such a sum except the payload and sign of a NaN that an
addition produces, so the rule here is: an output is NaN exactly where the
CPU oracle's is, and every other output equals the oracle's bit for bit
(infinities from overflow, the round-to-nearest-even tie at the top of the
bf16 range, subnormal sums that a flush to zero would lose).

Covered: AllReduce, ReduceScatter and ReduceScatterV, f32 and bf16, on the
vector (latency) kernel, the fused ring, the composed ring (chunk flags),
the packet path, the device-count kernel, a collective called from a user
kernel, and the allocation-free AllReduce.
"""
import ctypes

import numpy as np
import pytest

import oracle
from test_parity_gpu import ES, Guarded, run

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


# ------------------------------------------------------------- inputs ----

F32_SPECIALS = np.array([0x7FC00000, 0xFFC00000, 0x7FC12345, 0x7F800000, 0xFF800000,
                         0x7F7FFFFF, 0xFF7FFFFF, 0x00000001, 0x80000001, 0x007FFFFF,
                         0x80000000], dtype=np.uint32)
BF16_SPECIALS = np.array([0x7FC0, 0xFFC0, 0x7FC1, 0x7F80, 0xFF80, 0x7F7F, 0xFF7F, 0x0001,
                          0x8001, 0x007F, 0x8000], dtype=np.uint16)


def special_inputs(R, L, dtype, seed):
    """R rank buffers of L elements: N(0,1) values with specials planted.

    About 3% of positions get one special value in one random rank (NaN of
    either sign and payloads, infinities, the largest finite values,
    subnormals, -0).  Further positions get patterns over all ranks: every
    rank at the largest value (binary32 overflow, or for bf16 an overflow of
    the sum), +Inf in one rank and -Inf in another (invalid), rank 0 at the
    bf16 maximum plus 2^119 or 2^118 in rank 1 (the round-to-nearest-even tie
    that rounds up to +Inf, and the value just below it), and subnormals in
    every rank."""
    rng = np.random.default_rng(seed)
    if dtype == 0:
        xs = [rng.standard_normal(L).astype(np.float32).view(np.uint32) for _ in range(R)]
        sp = F32_SPECIALS
        big, tie, below, sub = 0x7F7FFFFF, None, None, 0x00000003
    else:
        xs = []
        for _ in range(R):
            u = rng.standard_normal(L).astype(np.float32).view(np.uint32)
            xs.append(((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16))   # finite normals
        sp = BF16_SPECIALS
        big, tie, below, sub = 0x7F7F, 0x7B00, 0x7A80, 0x0003
    for pos in rng.choice(L, size=max(1, L // 32), replace=False):
        xs[int(rng.integers(R))][pos] = sp[int(rng.integers(sp.size))]
    pattern_pos = rng.choice(L, size=max(4, L // 64), replace=False)
    for k, pos in enumerate(pattern_pos):
        kind = k % 5
        if kind == 0:
            for r in range(R):
                xs[r][pos] = big
        elif kind == 1 and R > 1:
            a, b = rng.choice(R, size=2, replace=False)
            xs[a][pos] = sp[3]
            xs[b][pos] = sp[4]
        elif kind == 2 and tie is not None and R > 1:
            for r in range(R):
                xs[r][pos] = 0
            xs[0][pos] = big
            xs[1][pos] = tie if k % 2 else below
        elif kind == 3:
            for r in range(R):
                xs[r][pos] = sub
        elif kind == 4 and R > 1:
            xs[0][pos] = big
            xs[1][pos] = big
            xs[R - 1][pos] = sp[6]
    if dtype == 0:
        return [x.view(np.float32) for x in xs]
    return xs


def assert_specials_match(got_bytes, want, dtype, what):
    """NaN exactly where the oracle has NaN; every other element bit for bit."""
    total = nans = 0
    for d, (g8, w) in enumerate(zip(got_bytes, want)):
        if dtype == 0:
            g = np.frombuffer(g8.tobytes(), dtype=np.uint32)
            wb = w.view(np.uint32)
            exp, man = 0x7F800000, 0x007FFFFF
        else:
            g = np.frombuffer(g8.tobytes(), dtype=np.uint16).astype(np.uint32)
            wb = w.astype(np.uint32)
            exp, man = 0x7F80, 0x007F
        assert g.size == wb.size, what
        g_nan = ((g & exp) == exp) & ((g & man) != 0)
        w_nan = ((wb & exp) == exp) & ((wb & man) != 0)
        total += wb.size
        nans += int(w_nan.sum())
        bad = np.nonzero((g_nan != w_nan) | (~w_nan & (g != wb)))[0]
        if bad.size:
            i = int(bad[0])
            raise AssertionError(f"{what}: rank {d} differs at element {i} "
                                 f"(got {g[i]:#x}, oracle {wb[i]:#x}; {bad.size} of {g.size})")
    assert nans > 0 or total < 2000, f"{what}: no NaN in the oracle's output"


def _counts(T, R, rng):
    cuts = np.sort(rng.integers(0, T + 1, size=R - 1))
    return np.diff(np.concatenate([[0], cuts, [T]])).astype(int).tolist()


# --------------------------------------------------------- host calls ----

PATHS = {
    # name: (PURLIN_OPT_VARIANT, PURLIN_OPT_AR_MODE)
    "latency": (1, 1),
    "ring": (2, 1),
    "composed": (2, 2),
    "packets": (0, 3),
}


@pytest.mark.parametrize("dtype", [0, 1], ids=["f32", "bf16"])
@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("R", [3, 8])
def test_allreduce_specials(P, R, path, dtype):
    variant, mode = PATHS[path]
    ctx = P.purlin_init(R, torch.cuda.current_stream())
    try:
        P.purlin_set_option(ctx, P.PURLIN_OPT_VARIANT, variant)
        P.purlin_set_option(ctx, P.PURLIN_OPT_AR_MODE, mode)
        es = ES[dtype]
        for k, n in enumerate((37, 4096 + 5, 100003, (3 << 18) + 11)):
            if path == "packets" and n * es > (1 << 20):
                continue   # past the packet staging buffer the call runs another path
            ins = special_inputs(R, n, dtype, seed=7000 + 31 * k + R)
            got, _ = run(P, ctx, "all_reduce", ins, [n * es] * R, dtype, n)
            assert_specials_match(got, oracle.all_reduce(ins, dtype), dtype,
                                  f"AllReduce {path} R={R} n={n}")
            v = P.purlin_last_launch(ctx)["variant"]
            want = {"latency": 1, "ring": 2, "composed": 3, "packets": 5}[path]
            if path == "composed" and n * es < 16 * R:
                want = 2   # under 16 bytes per owner slice: a plain ring plan
            assert v == want, (n, v)
    finally:
        ctx.close()


@pytest.mark.parametrize("dtype", [0, 1], ids=["f32", "bf16"])
@pytest.mark.parametrize("variant", [1, 2], ids=["latency", "ring"])
@pytest.mark.parametrize("R", [3, 8])
def test_reduce_scatter_specials(P, R, variant, dtype):
    ctx = P.purlin_init(R, torch.cuda.current_stream())
    rng = np.random.default_rng(R + 10 * variant + dtype)
    try:
        P.purlin_set_option(ctx, P.PURLIN_OPT_VARIANT, variant)
        es = ES[dtype]
        for k, M in enumerate((5, 4096 + 3, 50001)):
            n = M * R
            ins = special_inputs(R, n, dtype, seed=7100 + 31 * k + R)
            got, _ = run(P, ctx, "reduce_scatter", ins, [M * es] * R, dtype, n)
            assert_specials_match(got, oracle.reduce_scatter(ins, dtype), dtype,
                                  f"ReduceScatter variant={variant} R={R} M={M}")
            T = n + 7
            counts = _counts(T, R, rng)
            ins = special_inputs(R, T, dtype, seed=7200 + 31 * k + R)
            got, _ = run(P, ctx, "reduce_scatter_v", ins, [c * es for c in counts], dtype,
                         counts=counts)
            assert_specials_match(got, oracle.reduce_scatter_v(ins, counts, dtype), dtype,
                                  f"ReduceScatterV variant={variant} R={R} counts={counts}")
    finally:
        ctx.close()


# ---------------------------------------------- device counts, device API --

def _capacity(arrays, cap, es, fill):
    out = []
    for a in arrays:
        b = Guarded(cap * es, fill=fill)
        if a is not None and a.nbytes:
            b.t[GUARD:GUARD + a.nbytes].copy_(torch.from_numpy(a.view(np.uint8).copy()))
        out.append(b)
    return out


@pytest.mark.parametrize("dtype", [0, 1], ids=["f32", "bf16"])
@pytest.mark.parametrize("variant", [1, 2], ids=["units", "ring"])
def test_reduce_scatter_v_device_counts_specials(P, variant, dtype):
    R, es = 8, ES[dtype]
    ctx = P.purlin_init(R, torch.cuda.current_stream())
    rng = np.random.default_rng(77 + variant)
    try:
        P.purlin_set_option(ctx, P.PURLIN_OPT_VARIANT, variant)
        for T in (1000, 300007):
            counts = _counts(T, R, rng)
            ins = special_inputs(R, T, dtype, seed=7300 + T)
            want = oracle.reduce_scatter_v(ins, counts, dtype)
            src = _capacity(ins, T, es, 0xC3)
            dst = _capacity([None] * R, max(counts), es, 0x5A)
            d_counts = torch.tensor(counts, dtype=torch.int64, device="cuda")
            P.purlin_reduce_scatter_v_device_counts(ctx, [b.ptr for b in src],
                                                    [b.ptr for b in dst], d_counts, T,
                                                    max(counts), dtype)
            P.purlin_check(ctx)
            got = [b.body()[:c * es] for b, c in zip(dst, counts)]
            assert_specials_match(got, want, dtype, f"RSV device counts T={T}")
    finally:
        ctx.close()


@pytest.mark.parametrize("dtype", [0, 1], ids=["f32", "bf16"])
@pytest.mark.parametrize("mode", [0, 2], ids=["fused", "composed"])
def test_device_api_allreduce_specials(P, mode, dtype):
    from collective_datapath_atom_gb300 import examples
    from test_parity_gpu import COLLS, outputs, upload

    R, n = 8, 200003
    stream = torch.cuda.current_stream()
    ctx = P.purlin_init(R, stream)
    try:
        P.purlin_set_option(ctx, P.PURLIN_OPT_AR_MODE, mode)
        ins = special_inputs(R, n, dtype, seed=7400 + mode)
        src = upload(ins)
        dst = outputs([n * ES[dtype]] * R)
        blocks = torch.cuda.get_device_properties(0).multi_processor_count
        d = P.purlin_device_prepare(ctx, COLLS.index("all_reduce"), [b.ptr for b in src], [b.ptr for b in dst], n=n,
                                    counts=None, dtype=dtype, blocks=blocks)
        examples.collective(d, stream=stream)
        assert P.purlin_device_check(d, stream) == P.PURLIN_OK
        assert_specials_match([b.body() for b in dst], oracle.all_reduce(ins, dtype), dtype,
                              f"device API AllReduce mode={mode}")
        P.purlin_device_release(ctx, d)
    finally:
        ctx.close()


def test_noalloc_allreduce_specials(P):
    R, n = 8, 100003
    stream = torch.cuda.current_stream()
    for dtype in (0, 1):
        ins = special_inputs(R, n, dtype, seed=7500 + dtype)
        src = [torch.from_numpy(x.view(np.uint8).copy()).cuda() for x in ins]
        dst = [torch.empty(n * ES[dtype], dtype=torch.uint8, device="cuda") for _ in range(R)]
        ps = (ctypes.c_void_p * R)(*[t.data_ptr() for t in src])
        pd = (ctypes.c_void_p * R)(*[t.data_ptr() for t in dst])
        st = P.lib.purlin_all_reduce_noalloc(
            R, ctypes.cast(ps, ctypes.POINTER(ctypes.c_void_p)),
            ctypes.cast(pd, ctypes.POINTER(ctypes.c_void_p)), n, dtype, P.PURLIN_SUM,
            P.purlin_layout(P.PURLIN_SCATTERED, P.PURLIN_SCATTERED),
            ctypes.c_void_p(stream.cuda_stream))
        assert st == P.PURLIN_OK
        torch.cuda.synchronize()
        assert_specials_match([t.cpu().numpy() for t in dst], oracle.all_reduce(ins, dtype),
                              dtype, f"no-alloc AllReduce dtype={dtype}")
