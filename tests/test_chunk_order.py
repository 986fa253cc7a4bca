"""The order in which a ring CTA takes its chunks (ChunkOrder and chunk_at in
csrc/plan.h), compiled here on the host from the library's own header.

"Purlin: Separating Orchestration from the Datapath of Collectives" §3.2:
a composed AllReduce's gathering chunks consume the reducing chunks of other
CTAs.  The walk interleaves them; these tests check, on the composed plans
the library compiles, that the walk takes every chunk exactly once, that
each gathering chunk comes after every reducing chunk it waits on (so the
earliest unfinished chunk can always proceed), and that plans without
flags keep their own order.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

DRIVER = r"""
#include <cstdio>
#include "plan.h"
int main() {
    unsigned long long nr, ng, ctas, batch;
    int R;
    while (std::scanf("%llu %llu %d %llu %llu", &nr, &ng, &R, &ctas, &batch) == 5) {
        const purlin::ChunkOrder o = purlin::make_chunk_order(nr, ng, R, (uint32_t)ctas, (int)batch);
        for (unsigned long long p = 0; p < nr + ng; ++p)
            std::printf("%llu ", (unsigned long long)purlin::chunk_at(o, p));
        std::printf("\n");
    }
    return 0;
}
"""


@pytest.fixture(scope="module")
def walk(tmp_path_factory):
    """walk(cases) -> one list of chunks per (nr, ng, R, ctas, batch) case."""
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no host C++ compiler")
    d = tmp_path_factory.mktemp("chunk_order")
    src = d / "driver.cpp"
    src.write_text(DRIVER)
    exe = d / "driver"
    subprocess.run([gxx, "-std=c++17", "-O1",
                    "-I", os.path.join(ROOT, "collective_datapath_atom_gb300", "csrc"),
                    str(src), "-o", str(exe)], check=True)

    def run(cases):
        text = "".join(f"{nr} {ng} {R} {c} {b}\n" for nr, ng, R, c, b in cases)
        out = subprocess.run([str(exe)], input=text, capture_output=True, text=True, check=True)
        return [[int(x) for x in line.split()] for line in out.stdout.splitlines()]

    return run


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__.build()
    import collective_datapath_atom_gb300 as mod

    return mod


def composed_plan(lib, R, n):
    """(nr, ng, deps): deps[G] = the last reducing chunk gathering chunk G
    waits on, from the plan's segments (gathering segment k waits on
    reducing segment k, and each gathering chunk covers R reducing chunks)."""
    src = [(i + 1) << 36 for i in range(R)]
    dst = [(i + 100) << 36 for i in range(R)]
    st, segs, nch, _ = lib.purlin_plan_inspect(0, R, src, dst, n, None, 1, 1, (1, 1), 2,
                                               ar_mode=2)
    assert st == 0
    notify = [s for s in segs if s["sync"] == 1]
    wait = [s for s in segs if s["sync"] == 2]
    assert wait and len(notify) == len(wait)
    nr = wait[0]["chunk_begin"]
    for s in segs:
        if s["sync"] == 0:
            assert not s["tma"], "chunks outside the notify/wait segments"
    deps = {}
    for a, b in zip(notify, wait):
        assert a["bytes"] == b["bytes"] and a["src_off"] == b["src_off"]
        if not b["tma"]:
            continue
        body = b["bytes"] - b["head_bytes"] - b["tail_bytes"]
        nred = -(-body // a["chunk_bytes"])
        for ci in range(-(-body // b["chunk_bytes"])):
            deps[b["chunk_begin"] - nr + ci] = a["chunk_begin"] + min(ci * R + R, nred) - 1
    return nr, nch - nr, deps


@pytest.mark.parametrize("R", [2, 3, 8, 16, 31])
def test_composed_walk_takes_each_chunk_once_after_its_dependencies(lib, walk, R):
    sizes = [16 * R, 1000 * R + 3, 123457, 1 << 20, 5 * R * 8192 + 77, (1 << 24) + 5]
    plans = [composed_plan(lib, R, n) for n in sizes]
    for ctas in (1, 7, 152):
        cases = [(nr, ng, R, ctas, 8) for nr, ng, _ in plans]
        for (nr, ng, deps), seq in zip(plans, walk(cases)):
            assert sorted(seq) == list(range(nr + ng)), "not a permutation of the chunks"
            pos = {c: p for p, c in enumerate(seq)}
            for G, last in deps.items():
                assert last < (G + 1) * R          # what the walk relies on
                assert pos[nr + G] > pos[last], (R, nr, ng, ctas, G)
            # the reducing chunks keep their own order, and so do the gathering ones
            red = [c for c in seq if c < nr]
            gat = [c for c in seq if c >= nr]
            assert red == sorted(red) and gat == sorted(gat)


def test_interleaving_starts_after_the_lag_and_plans_without_flags_keep_their_order(walk):
    # 4000 reducing chunks, 500 gathering chunks, R = 8, 152 CTAs, batches of 8:
    # lag = 12 * 152 // 9 = 202 groups, so gathering chunk 0 sits at position 203 * 8
    nr, ng, R = 4000, 500, 8
    seq, ident = walk([(nr, ng, R, 152, 8), (nr + ng, 0, R, 152, 8)])
    assert seq[:203 * 8] == list(range(203 * 8))
    assert seq[203 * 8] == nr
    assert seq[203 * 8 + 1:203 * 8 + 1 + R] == list(range(203 * 8, 203 * 8 + R))
    assert seq[203 * 8 + 1 + R] == nr + 1
    assert seq[-1] == nr + ng - 1
    assert ident == list(range(nr + ng))
    # too few groups for the lag: the plan's own order
    short, = walk([(100, 13, R, 152, 8)])
    assert short == list(range(113))
    # fewer gathering chunks than groups of R (no composed plan has this, the
    # walk still takes every chunk once): all of them interleaved, then the
    # remaining reducing chunks
    few, = walk([(4000, 100, R, 152, 8)])
    assert sorted(few) == list(range(4100))
    assert [c for c in few if c >= 4000] == list(range(4000, 4100))
    assert few[-1] == 3999 and few[203 * 8 + 99 * 9] == 4099


FLAG_DRIVER = r"""
#include <cstdio>
#include "plan.h"
int main() {
    unsigned long long nr, ng, ctas, batch, F;
    int R;
    while (std::scanf("%llu %llu %d %llu %llu %llu", &nr, &ng, &R, &ctas, &batch, &F) == 6) {
        const purlin::ChunkOrder o = purlin::make_chunk_order(nr, ng, R, (uint32_t)ctas, (int)batch);
        for (unsigned long long d = 0; d < nr; ++d) {
            const purlin::FlagAt f = purlin::flag_at(o, F, d);
            std::printf("%llu %llu %llu ", (unsigned long long)purlin::walk_pos(o, d),
                        (unsigned long long)f.slot, (unsigned long long)f.gen);
        }
        std::printf("\n");
    }
    return 0;
}
"""


@pytest.fixture(scope="module")
def flags(tmp_path_factory):
    """flags(cases) -> per (nr, ng, R, ctas, batch, F) case, a list of
    (walk position, slot, generation) for every notifying chunk d < nr."""
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no host C++ compiler")
    d = tmp_path_factory.mktemp("flag_at")
    src = d / "driver.cpp"
    src.write_text(FLAG_DRIVER)
    exe = d / "driver"
    subprocess.run([gxx, "-std=c++17", "-O1",
                    "-I", os.path.join(ROOT, "collective_datapath_atom_gb300", "csrc"),
                    str(src), "-o", str(exe)], check=True)

    def run(cases):
        text = "".join(" ".join(str(v) for v in c) + "\n" for c in cases)
        out = subprocess.run([str(exe)], input=text, capture_output=True, text=True, check=True)
        res = []
        for line in out.stdout.splitlines():
            v = [int(x) for x in line.split()]
            res.append(list(zip(v[0::3], v[1::3], v[2::3])))
        return res

    return run


def _slots_per_parity(ctas):
    return (65536 // ctas) * ctas   # the context's flag_geometry: a multiple of the grid


@pytest.mark.parametrize("R", [2, 3, 8, 31])
def test_reused_flag_slots_stay_on_one_cta_in_walk_order(walk, flags, R):
    """A consumer of notifying chunk d waits for its slot to reach this
    call's generation for d.  That is sound only if the slot's earlier
    generations are published before d and its later ones after: the slot's
    chunks must sit on one CTA, in walk order.  Checked with the walk itself
    (chunk_at), for plans with more notifying chunks than slots (the slots
    are then numbered by walk position) and plans with fewer (one slot per
    chunk, generation 0)."""
    for ctas in (7, 152, 304):
        F = _slots_per_parity(ctas)
        cases = []
        for nr in (F - 1, F, F + 1, 2 * F + 12345, 3 * F + 7):
            ng = -(-nr // R)
            cases.append((nr, ng, R, ctas, 4, F))
        seqs = walk([c[:5] for c in cases])
        for (nr, ng, _, _, _, _), seq, fl in zip(cases, seqs, flags(cases)):
            assert len(fl) == nr
            by_slot = {}
            for d, (pos, slot, gen) in enumerate(fl):
                assert seq[pos] == d, "walk_pos is not the inverse of chunk_at"
                assert slot < F
                if nr <= F:
                    assert (slot, gen) == (d, 0)
                else:
                    assert (slot, gen) == (pos % F, pos // F)
                    assert gen < -(-(nr + ng) // F)   # the epoch increment covers it
                by_slot.setdefault(slot, []).append((gen, pos))
            for slot, uses in by_slot.items():
                uses.sort()
                owners = {pos % ctas for _, pos in uses}
                assert len(owners) == 1, (nr, slot, uses[:4])
                positions = [pos for _, pos in uses]
                assert positions == sorted(positions)
                gens = [g for g, _ in uses]
                assert all(a < b for a, b in zip(gens, gens[1:])), (slot, gens)


def test_chunk_numbered_slots_would_cross_ctas(walk):
    """The reason for walk-position numbering: under the interleaved walk,
    notifying chunks d and d + F (numbered by chunk) usually land on
    different CTAs, so a consumer of d could pass on d + F's flag."""
    ctas, R = 152, 8
    F = _slots_per_parity(ctas)
    nr = F + 5000
    ng = -(-nr // R)
    seq, = walk([(nr, ng, R, ctas, 4)])
    pos = {c: p for p, c in enumerate(seq)}
    crossing = sum(pos[d] % ctas != pos[d + F] % ctas for d in range(nr - F))
    assert crossing > 0
