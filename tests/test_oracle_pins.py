"""Pins for the CPU oracle: checks against what the pages and mathematics fix.

Nothing here compares the oracle with itself.  The pins are:
  * hand-derived worked examples in tests/golden/ (IEEE rounding worked by
    hand; each collective's contract written out element by element);
  * an independent definition of bf16 round-to-nearest-even (exact distance
    comparison in binary64) and torch's CPU conversion as a library routine;
  * exact integer sums (brute force in int64) on tiny inputs;
  * the recursive-summation error bound against exact rational sums;
  * the contract invariants: AllGather output = concatenation of inputs,
    AllGather(ReduceScatter(x)) == AllReduce(x) bitwise, AllToAllV with the
    transposed count matrix recovers the inputs, uniform-count V variants
    equal the plain ones, R = 1 is a copy.
The last part plants plausible mistakes in a copy of the oracle source and
checks that at least one pin fails for each.

Passages: "Purlin: Separating Orchestration from the Datapath of Collectives"
§2.1 (contracts, V variants), §3.1 (layouts; AllReduce = ReduceScatter then
AllGather), §3.3 (SCORE ordered accumulation), §C.4 (V-variant semantics).
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import BF16, F32

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
DTYPES = {"f32": F32, "bf16": BF16}


def _load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _f32_from_hex(hs):
    return np.array([int(h, 16) for h in hs], dtype=np.uint32).view(np.float32)


def _bf16_from_hex(hs):
    return np.array([int(h, 16) for h in hs], dtype=np.uint16)


def _as_dtype(values, dtype):
    x = np.asarray(values, dtype=np.float32)
    if dtype == F32:
        return x
    return (x.view(np.uint32) >> 16).astype(np.uint16)   # exact: the tests' values fit bf16


def _f32_of(arr, dtype):
    if dtype == F32:
        return arr.astype(np.float64)
    return (arr.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bits(arr):
    return arr.view(np.uint32) if arr.dtype == np.float32 else arr


# ----------------------------------------------------- independent codec ---

def ref_bf16_rne(bits_u32: np.ndarray) -> np.ndarray:
    """bf16 nearest-even from the definition: pick the closer of the two
    neighbouring bf16 values by exact binary64 distance, ties to the one with
    an even last mantissa bit; overflow past the largest finite value goes to
    infinity (which ties-to-even also reaches); NaN -> 0x7FC0."""
    u = np.asarray(bits_u32, dtype=np.uint32)
    sign = (u >> 31).astype(np.uint32)
    mag = u & np.uint32(0x7FFFFFFF)
    is_nan = mag > np.uint32(0x7F800000)
    x = mag.view(np.float32).astype(np.float64)
    lo_bits = mag & np.uint32(0xFFFF0000)
    lo = lo_bits.view(np.float32).astype(np.float64)
    exp = (lo_bits >> 23).astype(np.int64)
    # spacing of bf16 values with this exponent (subnormals share exponent 1's spacing)
    ulp = np.ldexp(1.0, np.maximum(exp, 1) - 127 - 7)
    hi = lo + ulp                           # for the top binade this is 2^128 (-> inf)
    dlo, dhi = x - lo, hi - x
    lo_even = ((lo_bits >> 16) & 1) == 0
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ~lo_even)
    out_mag = np.where(pick_hi, (lo_bits >> 16) + 1, lo_bits >> 16).astype(np.uint32)
    out_mag = np.where(mag >= np.uint32(0x7F800000), mag >> 16, out_mag)   # inf stays inf
    out = (sign << 15) | out_mag
    out = np.where(is_nan, np.uint32(0x7FC0), out)
    return out.astype(np.uint16)


def _codec_sample():
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x3FFF, 0x7FFF, 0x8000, 0x8001, 0xBFFF, 0xFFFF],
                    dtype=np.uint32)
    structured = (hi[:, None] | lows[None, :]).reshape(-1)
    rnd = np.random.default_rng(123).integers(0, 1 << 32, size=1 << 20, dtype=np.uint64)
    return np.concatenate([structured, rnd.astype(np.uint32)])


def _oracle_codec(bits):
    return oracle.f32_bits_to_bf16_array(bits)


def check_codec_definition():
    sub = _codec_sample()
    got = _oracle_codec(sub)
    want = ref_bf16_rne(sub)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"bf16 codec differs at {hex(int(sub[bad[0]]))}: " \
                          f"{hex(int(got[bad[0]]))} vs {hex(int(want[bad[0]]))}"


def check_codec_specials():
    cases = {
        0x3F800000: 0x3F80,   # 1.0
        0x3F808000: 0x3F80,   # 1 + 2^-8: tie, even stays
        0x3F818000: 0x3F82,   # (1 + 2^-7) + 2^-8: tie, odd rounds up
        0x3F808001: 0x3F81,   # just above the tie
        0x7F7FFFFF: 0x7F80,   # largest finite float rounds to +inf
        0xFF7FFFFF: 0xFF80,   # and its negative to -inf
        0x7F800000: 0x7F80,   # +inf
        0x80000000: 0x8000,   # -0
        0x00000001: 0x0000,   # smallest subnormal rounds to +0
        0x00008000: 0x0000,   # subnormal tie, even
        0x00018000: 0x0002,   # subnormal tie, odd -> up
        0x7FC00001: 0x7FC0,   # NaN -> quiet NaN
        0xFF800001: 0x7FC0,
    }
    for bits, want in cases.items():
        got = oracle.f32_bits_to_bf16(bits)
        assert got == want, f"{hex(bits)} -> {hex(got)}, want {hex(want)}"
    for b in (0x0000, 0x3F80, 0x8001, 0x7F80, 0xFFFF):
        assert oracle.bf16_to_f32_bits(b) == b << 16


def check_codec_vs_torch():
    torch = pytest.importorskip("torch")
    sample = _codec_sample()[::8]
    finite = sample[(sample & 0x7F800000) != 0x7F800000]
    t = torch.from_numpy(finite.view(np.float32).copy()).to(torch.bfloat16)
    want = t.view(torch.int16).numpy().view(np.uint16)
    got = ref_bf16_rne(finite)
    assert np.array_equal(got, want)
    assert np.array_equal(_oracle_codec(finite), want)


# ------------------------------------------------------------ golden -------

def check_golden_score_order():
    g = _load_golden("score_order_f32.json")
    ins = [_f32_from_hex(row) for row in g["inputs_f32_hex"]]
    want = np.array([int(h, 16) for h in g["output_f32_hex"]], dtype=np.uint32)
    outs = oracle.all_reduce(ins, F32)
    for o in outs:
        assert np.array_equal(o.view(np.uint32), want), (o.view(np.uint32), want)
    assert np.array_equal(oracle.all_reduce_one(ins, F32).view(np.uint32), want)


def check_golden_round_once():
    g = _load_golden("score_round_once_bf16.json")
    for case in g["cases"]:
        ins = [_bf16_from_hex(row) for row in case["inputs_bf16_hex"]]
        want = _bf16_from_hex(case["output_bf16_hex"])
        for o in oracle.all_reduce(ins, BF16):
            assert np.array_equal(o, want), (o, want)
        assert np.array_equal(oracle.all_reduce_one(ins, BF16), want)


def _specials_match(got_bits, want_hex, dtype):
    """The fixture's rule: "nan" matches any NaN, every other value bit for bit."""
    got_bits = np.asarray(got_bits).astype(np.uint32)
    exp_mask, man_mask = (0x7F800000, 0x007FFFFF) if dtype == F32 else (0x7F80, 0x007F)
    for i, w in enumerate(want_hex):
        g = int(got_bits[i])
        if w == "nan":
            assert (g & exp_mask) == exp_mask and (g & man_mask) != 0, (i, hex(g))
        else:
            assert g == int(w, 16), (i, hex(g), w)


def check_golden_specials():
    """NaN, infinities, overflow and subnormals in the ordered sum, worked by
    hand (tests/golden/score_specials.json): AllReduce, ReduceScatterV over
    a split of the same elements, and single points."""
    g = _load_golden("score_specials.json")
    for name, dtype in (("f32", F32), ("bf16", BF16)):
        case = g[name]
        ins = [_f32_from_hex(r) if dtype == F32 else _bf16_from_hex(r) for r in case["inputs_hex"]]
        want = case["output_hex"]
        for o in oracle.all_reduce(ins, dtype):
            _specials_match(_bits(o), want, dtype)
        _specials_match(_bits(oracle.all_reduce_one(ins, dtype)), want, dtype)
        n = len(want)
        counts = [n // 3 + (1 if r < n % 3 else 0) for r in range(3)]
        outs = oracle.reduce_scatter_v(ins, counts, dtype)
        at = 0
        for r, c in enumerate(counts):
            _specials_match(_bits(outs[r]), want[at:at + c], dtype)
            at += c
        for i in range(n):
            _specials_match(_bits(np.array([oracle.reduce_at(ins, dtype, i)])), [want[i]], dtype)


def _run_collective(case, dtype):
    ins = [_as_dtype(x, dtype) for x in case["inputs"]]
    c = case["collective"]
    if c == "all_gather":
        return oracle.all_gather(ins, dtype)
    if c == "all_gather_v":
        return oracle.all_gather_v(ins, case["counts"], dtype)
    if c == "reduce_scatter":
        return oracle.reduce_scatter(ins, dtype)
    if c == "reduce_scatter_v":
        return oracle.reduce_scatter_v(ins, case["counts"], dtype)
    if c == "all_reduce":
        return oracle.all_reduce(ins, dtype)
    if c == "all_to_all":
        return oracle.all_to_all(ins, dtype)
    if c == "all_to_all_v":
        return oracle.all_to_all_v(ins, np.array(case["C"]), dtype)
    raise KeyError(c)


def check_golden_contracts():
    g = _load_golden("small_contracts.json")
    for case in g["cases"]:
        for dtype in (F32, BF16):
            outs = _run_collective(case, dtype)
            assert len(outs) == case["R"]
            for o, w in zip(outs, case["outputs"]):
                assert np.array_equal(_bits(o), _bits(_as_dtype(w, dtype))), \
                    (case["collective"], dtype, o, w)


# --------------------------------------------------------- exact sums ------

def check_exact_integer_sums():
    rng = np.random.default_rng(7)
    for R in (1, 2, 3, 8):
        for n in (0, 1, 7, 16, 33):
            ints = [rng.integers(-8, 9, size=n * R) for _ in range(R)]
            exact = np.sum(np.stack(ints).astype(np.int64), axis=0) if n else np.zeros(0)
            for dtype in (F32, BF16):
                ins = [_as_dtype(x.astype(np.float32), dtype) for x in ints]
                for o in oracle.all_reduce(ins, dtype):
                    assert np.array_equal(_f32_of(o, dtype), exact.astype(np.float64))
                assert np.array_equal(_f32_of(oracle.all_reduce_one(ins, dtype), dtype),
                                      exact.astype(np.float64))
                rs = oracle.reduce_scatter(ins, dtype)
                for r in range(R):
                    assert np.array_equal(_f32_of(rs[r], dtype),
                                          exact[r * n:(r + 1) * n].astype(np.float64))
                counts = list(rng.multinomial(n * R, np.ones(R) / R))
                rsv = oracle.reduce_scatter_v(ins, counts, dtype)
                off = 0
                for r in range(R):
                    assert np.array_equal(_f32_of(rsv[r], dtype),
                                          exact[off:off + counts[r]].astype(np.float64))
                    off += counts[r]


def check_error_bound():
    """|oracle - exact| <= gamma_{R-1} sum|x| (binary32 recursive summation),
    plus half a bf16 spacing of the result for bf16 outputs."""
    rng = np.random.default_rng(11)
    for R in (2, 3, 8):
        for dtype in (F32, BF16):
            n = 48
            xs = [rng.standard_normal(n).astype(np.float32) * np.float32(2.0 ** rng.integers(-6, 6))
                  for _ in range(R)]
            ins = [_as_dtype(x, dtype) if dtype == F32 else
                   ref_bf16_rne(x.view(np.uint32)) for x in xs]
            vals = [_f32_of(a, dtype) for a in ins]
            out = _f32_of(oracle.all_reduce(ins, dtype)[0], dtype)
            u = 2.0 ** -24
            gamma = (R - 1) * u / (1 - (R - 1) * u)
            for i in range(n):
                exact = sum(Fraction(float(v[i])) for v in vals)
                absum = sum(abs(float(v[i])) for v in vals)
                bound = gamma * absum
                if dtype == BF16:
                    bound += 2.0 ** -8 * (abs(float(exact)) + bound)
                assert abs(Fraction(float(out[i])) - exact) <= Fraction(bound) * (1 + 1e-12), \
                    (R, dtype, i)


# --------------------------------------------------------- invariants ------

def _encoded(R, n):
    """Rank/index encoded fp32 bit patterns (some are NaN or -0 on purpose)."""
    return [((np.uint32(s) << np.uint32(24)) | np.arange(n, dtype=np.uint32)).view(np.float32)
            for s in range(R)]


def check_all_gather_concat():
    for R, n in ((1, 5), (3, 7), (8, 33)):
        ins = _encoded(R, n)
        ins[-1][:1] = np.array([0x7FC12345], dtype=np.uint32).view(np.float32)  # NaN payload
        want = np.concatenate(ins).view(np.uint32)
        for o in oracle.all_gather(ins, F32):
            assert np.array_equal(o.view(np.uint32), want)
        bins = [(x.view(np.uint32) & 0xFFFF).astype(np.uint16) ^ np.uint16(s << 12)
                for s, x in enumerate(ins)]
        for o in oracle.all_gather(bins, BF16):
            assert np.array_equal(o, np.concatenate(bins))


def check_rs_then_ag_is_ar():
    rng = np.random.default_rng(5)
    for R in (1, 2, 3, 8):
        for dtype in (F32, BF16):
            M = 37
            xs = [rng.standard_normal(R * M).astype(np.float32) for _ in range(R)]
            ins = xs if dtype == F32 else [ref_bf16_rne(x.view(np.uint32)) for x in xs]
            ar = oracle.all_reduce(ins, dtype)
            ag = oracle.all_gather(oracle.reduce_scatter(ins, dtype), dtype)
            for a, b in zip(ar, ag):
                assert np.array_equal(_bits(a), _bits(b))
            for a in ar[1:]:
                assert np.array_equal(_bits(a), _bits(ar[0]))


def check_a2a_inverse():
    rng = np.random.default_rng(9)
    for R in (1, 2, 3, 8):
        M = 5
        ins = [np.arange(R * M, dtype=np.float32) + 1000 * s for s in range(R)]
        twice = oracle.all_to_all(oracle.all_to_all(ins, F32), F32)
        for a, b in zip(ins, twice):
            assert np.array_equal(a, b)
        # AllToAll is AllToAllV with every count equal to M
        C = np.full((R, R), M)
        for a, b in zip(oracle.all_to_all(ins, F32), oracle.all_to_all_v(ins, C, F32)):
            assert np.array_equal(a, b)
        # ragged counts, including zero rows and columns: C^T undoes C
        for dtype in (F32, BF16):
            C = rng.integers(0, 6, size=(R, R))
            if R > 1:
                C[0, :] = 0
                C[:, -1] = 0
            xs = [(np.arange(C[s].sum(), dtype=np.uint32) | np.uint32(s << 20)) for s in range(R)]
            ins = [x.view(np.float32) if dtype == F32 else (x & 0xFFFF).astype(np.uint16)
                   for x in xs]
            out = oracle.all_to_all_v(ins, C, dtype)
            back = oracle.all_to_all_v(out, C.T.copy(), dtype)
            for a, b in zip(ins, back):
                assert np.array_equal(_bits(a), _bits(b))


def check_uniform_v_equals_plain():
    rng = np.random.default_rng(13)
    for R in (1, 3, 8):
        n = 9
        for dtype in (F32, BF16):
            xs = [rng.standard_normal(R * n).astype(np.float32) for _ in range(R)]
            ins = xs if dtype == F32 else [ref_bf16_rne(x.view(np.uint32)) for x in xs]
            short = [x[:n].copy() for x in ins]
            for a, b in zip(oracle.all_gather(short, dtype),
                            oracle.all_gather_v(short, [n] * R, dtype)):
                assert np.array_equal(_bits(a), _bits(b))
            for a, b in zip(oracle.reduce_scatter(ins, dtype),
                            oracle.reduce_scatter_v(ins, [n] * R, dtype)):
                assert np.array_equal(_bits(a), _bits(b))


def check_single_rank_is_copy():
    x = _encoded(1, 11)
    x[0][3] = np.float32(-0.0)
    for f in (oracle.all_gather, oracle.all_to_all):
        assert np.array_equal(f(x, F32)[0].view(np.uint32), x[0].view(np.uint32))
    y = [np.random.default_rng(2).standard_normal(11).astype(np.float32)]
    y[0][3] = np.float32(-0.0)
    for f in (oracle.all_reduce, oracle.reduce_scatter):
        assert np.array_equal(f(y, F32)[0].view(np.uint32), y[0].view(np.uint32))
    yb = [ref_bf16_rne(y[0].view(np.uint32))]
    assert np.array_equal(oracle.all_reduce(yb, BF16)[0], yb[0])


def check_points_match_full():
    rng = np.random.default_rng(17)
    R, n = 8, 64
    for dtype in (F32, BF16):
        xs = [rng.standard_normal(n).astype(np.float32) for _ in range(R)]
        ins = xs if dtype == F32 else [ref_bf16_rne(x.view(np.uint32)) for x in xs]
        full = oracle.all_reduce(ins, dtype)[0]
        assert np.array_equal(_bits(oracle.all_reduce_one(ins, dtype)), _bits(full))
        for i in (0, 1, 31, 63):
            assert _bits(np.array([oracle.reduce_at(ins, dtype, i)]))[0] == _bits(full)[i]
    C = rng.integers(0, 4, size=(4, 4))
    ins = [(np.arange(C[s].sum(), dtype=np.uint32) | np.uint32(s << 16)).view(np.float32)
           for s in range(4)]
    out = oracle.all_to_all_v(ins, C, F32)
    for d in range(4):
        for j in range(out[d].size):
            s, i = oracle.all_to_all_v_source(C, d, j)
            assert out[d].view(np.uint32)[j] == ins[s].view(np.uint32)[i]


PINS = [check_codec_definition, check_codec_specials, check_codec_vs_torch,
        check_golden_score_order, check_golden_round_once, check_golden_contracts,
        check_golden_specials,
        check_exact_integer_sums, check_error_bound, check_all_gather_concat,
        check_rs_then_ag_is_ar, check_a2a_inverse, check_uniform_v_equals_plain,
        check_single_rank_is_copy, check_points_match_full]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin()


def test_zipf_partition_preserves_total_and_shape():
    import workloads

    for T in (8, 1024, 1025, 4096, 1 << 20, (1 << 29) + 7):
        part = workloads.zipf_partition(T)
        assert sum(part) == T and len(part) == 8 and min(part) >= 0
        if T > 1024:
            assert part == sorted(part, reverse=True)       # weights fall with the rank
            assert 1.15 < part[0] / (T / 8) < 1.2            # 8 / sum k^-0.125 = 1.176
        C = workloads.rotated_counts(part)
        assert (C.sum(axis=0) == T).all() and (C.sum(axis=1) == T).all()


def test_independent_codec_matches_torch_exhaustive_top_halves():
    """Spot the independent reference itself against torch on every bf16
    neighbourhood (all 2^16 upper halves, tie and near-tie lower halves)."""
    torch = pytest.importorskip("torch")
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0x7FFF, 0x8000, 0x8001], dtype=np.uint32)
    s = (hi[:, None] | lows[None, :]).reshape(-1)
    s = s[(s & 0x7F800000) != 0x7F800000]
    want = torch.from_numpy(s.view(np.float32).copy()).to(torch.bfloat16)
    assert np.array_equal(ref_bf16_rne(s), want.view(torch.int16).numpy().view(np.uint16))


# ------------------------------------------------- planted mistakes -----------

MUTANTS = {
    # accumulate in reverse rank order
    "reverse_order": (
        "    float acc = load_as_f32(dtype, in[0], idx);\n"
        "    for (int s = 1; s < R; ++s) {\n"
        "        acc = acc + load_as_f32(dtype, in[s], idx);\n",
        "    float acc = load_as_f32(dtype, in[R - 1], idx);\n"
        "    for (int s = R - 2; s >= 0; --s) {\n"
        "        acc = acc + load_as_f32(dtype, in[s], idx);\n"),
    # drop the last rank's term
    "dropped_term": ("for (int s = 1; s < R; ++s) {", "for (int s = 1; s < R - 1; ++s) {"),
    # start the accumulator at +0.0 instead of rank 0's value
    "zero_start": (
        "    float acc = load_as_f32(dtype, in[0], idx);\n"
        "    for (int s = 1; s < R; ++s) {",
        "    float acc = 0.0f;\n"
        "    for (int s = 0; s < R; ++s) {"),
    # subtract instead of add for one operand
    "wrong_sign": ("acc = acc + load_as_f32", "acc = acc - load_as_f32"),
    # truncate instead of rounding to nearest even
    "truncating_bf16": ("u += 0x7FFFu + kept_lsb;", "u += 0u * kept_lsb;"),
    # ties away from zero
    "ties_away": ("u += 0x7FFFu + kept_lsb;", "u += 0x8000u + 0u * kept_lsb;"),
    # AllGather writes every contribution into the destination's own slot
    "ag_wrong_slot": ("copy_elem(out[d], (size_t)s * n + i, in[s], i, es);",
                      "copy_elem(out[d], (size_t)d * n + i, in[s], i, es);"),
    # ReduceScatter takes a strided instead of a contiguous slice
    "rs_strided_slice": ("ordered_sum(R, dtype, in, (size_t)r * M + i)",
                         "ordered_sum(R, dtype, in, i * (size_t)R + (size_t)r)"),
    # AllToAll transposed operands (source slot and destination slice swapped)
    "a2a_transposed": ("copy_elem(out[d], (size_t)s * M + i, in[s], (size_t)d * M + i, es);",
                       "copy_elem(out[d], (size_t)d * M + i, in[s], (size_t)s * M + i, es);"),
    # AllToAllV receive displacement from the row instead of the column
    "a2av_row_for_column": ("exclusive_scan(R, C + d, (size_t)R, Q); /* column d",
                            "exclusive_scan(R, C + (size_t)d * R, 1, Q); /* column d"),
    # AllGatherV displacement inclusive instead of exclusive
    "agv_inclusive_scan": ("        out[j] = run;\n        run += x[(size_t)j * stride];",
                           "        run += x[(size_t)j * stride];\n        out[j] = run;"),
}


# pins that need torch (a library cross-check); the planted-mistake children
# skip them so each child starts in well under a second
_TORCH_PINS = {"check_codec_vs_torch"}


def _run_pins_against(path: str, skip_torch: bool = True) -> list[str]:
    """Run the pins against another build of the oracle; return the names of
    the pins that failed."""
    failures = []
    with oracle.use_library(path):
        for pin in PINS:
            if skip_torch and pin.__name__ in _TORCH_PINS:
                continue
            try:
                pin()
            except (AssertionError, ValueError, IndexError):
                failures.append(pin.__name__)
    return failures


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    """Some mutants write out of bounds, so each runs in a child process; a
    pin failure or a crash of the child both count as caught."""
    import subprocess
    import sys

    old, new = MUTANTS[name]
    src = oracle.source_text()
    assert old in src, f"mutation anchor for {name} not found"
    path = oracle.compile_variant(src.replace(old, new), str(tmp_path / f"lib_{name}.so"))
    here = os.path.dirname(os.path.abspath(__file__))
    code = ("import sys; sys.path[:0] = [%r, %r]; import test_oracle_pins as t; "
            "f = t._run_pins_against(%r); print('FAILED:' + ','.join(f))"
            % (os.path.dirname(here), here, path))
    proc = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                          timeout=300)
    caught = proc.returncode != 0 or any(
        line.startswith("FAILED:") and line != "FAILED:" for line in proc.stdout.splitlines())
    assert caught, f"no pin caught the planted mistake {name}: {proc.stdout[-500:]}"


def test_openmp_build_gives_the_same_bits():
    """The CPU baseline's OpenMP build splits the element loops over threads;
    each element keeps its one thread and its order, so every collective
    returns the single-threaded build's bits."""
    rng = np.random.default_rng(23)
    R, n = 8, 8 * 4099
    xs32 = [rng.standard_normal(n).astype(np.float32) for _ in range(R)]
    xs16 = [ref_bf16_rne(x.view(np.uint32)) for x in xs32]
    counts = list(rng.multinomial(n, np.ones(R) / R))
    C = rng.integers(0, 600, size=(R, R))
    a2av = [ref_bf16_rne(rng.standard_normal(int(C[s].sum())).astype(np.float32).view(np.uint32))
            for s in range(R)]

    def run_all():
        out = []
        for dtype, xs in ((F32, xs32), (BF16, xs16)):
            out += oracle.all_reduce(xs, dtype) + [oracle.all_reduce_one(xs, dtype)]
            out += oracle.reduce_scatter(xs, dtype) + oracle.reduce_scatter_v(xs, counts, dtype)
            out += oracle.all_gather(xs, dtype) + oracle.all_gather_v(
                [x[:c] for x, c in zip(xs, counts)], counts, dtype)
            out += oracle.all_to_all(xs, dtype)
        return out + oracle.all_to_all_v(a2av, C, BF16)

    serial = run_all()
    with oracle.openmp(4) as omp:
        assert omp.threads == 4
        parallel = run_all()
    assert len(serial) == len(parallel)
    for a, b in zip(serial, parallel):
        assert np.array_equal(_bits(a), _bits(b))
