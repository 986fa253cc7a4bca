// plan.cpp -- argument validation and the layout compiler (host only).
//
// "Purlin: Separating Orchestration from the Datapath of Collectives":
//   §2.1  the contracts of AllGather, ReduceScatter, AllReduce, AllToAll and
//         their variable-length variants;
//   §3.1  each collective = (input layout, output layout, copy | reduce);
//         AllReduce = ReduceScatter then AllGather, scattered -> scattered;
//   §3.2  SNAC derives rank dependencies from the layouts; composed
//         AllReduce has reducing and gathering CTAs working on chunks;
//   §C.4  the variable-length variants.
// "Purlin" project README, "Note": addresses and byte counts are kept
// aligned for the Atom; here 16 bytes is required of every base pointer and
// the aligned body of each transfer goes through the TMA ring, the ragged
// head and tail through the vector path.
#include "plan.h"

#include <algorithm>

namespace purlin {

namespace {

constexpr uint64_t kMaxBufferBytes = 1ull << 48;

bool layout_is(const purlin_layout &l, int in, int out) { return l.in == in && l.out == out; }

uint64_t sum_counts(const size_t *c, int k, size_t stride) {
    uint64_t s = 0;
    for (int j = 0; j < k; ++j) s += c[(size_t)j * stride];
    return s;
}

bool ranges_overlap(uintptr_t a, uint64_t la, uintptr_t b, uint64_t lb) {
    if (la == 0 || lb == 0) return false;
    return a < b + lb && b < a + la;
}

struct RawSeg {
    uint64_t src_off, dst_off, bytes;
    int src_rank, dst_rank, skip_rank;
    bool src_is_dst;
    uint8_t sync;
};

}  // namespace

int elem_bytes(int dtype) {
    if (dtype == PURLIN_F32) return 4;
    if (dtype == PURLIN_BF16) return 2;
    return 0;
}

void buffer_bytes(const CallDesc &c, std::vector<uint64_t> &in_b, std::vector<uint64_t> &out_b) {
    const uint64_t es = (uint64_t)elem_bytes(c.dtype);
    const int R = c.R;
    in_b.assign(R, 0);
    out_b.assign(R, 0);
    switch (c.coll) {
        case PURLIN_COLL_ALL_REDUCE:
        case PURLIN_COLL_ALL_TO_ALL:
            for (int r = 0; r < R; ++r) in_b[r] = out_b[r] = c.n * es;
            break;
        case PURLIN_COLL_REDUCE_SCATTER:
            for (int r = 0; r < R; ++r) {
                in_b[r] = c.n * es;
                out_b[r] = (c.n / (uint64_t)R) * es;
            }
            break;
        case PURLIN_COLL_ALL_GATHER:
            for (int r = 0; r < R; ++r) {
                in_b[r] = c.n * es;
                out_b[r] = (uint64_t)R * c.n * es;
            }
            break;
        case PURLIN_COLL_ALL_GATHER_V: {
            uint64_t T = sum_counts(c.counts, R, 1);
            for (int r = 0; r < R; ++r) {
                in_b[r] = c.counts[r] * es;
                out_b[r] = T * es;
            }
            break;
        }
        case PURLIN_COLL_REDUCE_SCATTER_V: {
            uint64_t T = sum_counts(c.counts, R, 1);
            for (int r = 0; r < R; ++r) {
                in_b[r] = T * es;
                out_b[r] = c.counts[r] * es;
            }
            break;
        }
        case PURLIN_COLL_ALL_TO_ALL_V:
            for (int r = 0; r < R; ++r) {
                in_b[r] = sum_counts(c.counts + (size_t)r * R, R, 1) * es;
                out_b[r] = sum_counts(c.counts + r, R, (size_t)R) * es;
            }
            break;
    }
}

uint64_t algorithmic_bytes(const CallDesc &c) {
    std::vector<uint64_t> in_b, out_b;
    buffer_bytes(c, in_b, out_b);
    uint64_t t = 0;
    for (int r = 0; r < c.R; ++r) t += in_b[r] + out_b[r];
    return t;
}

purlin_status validate_shape(const CallDesc &c, const void *const src[], void *const dst[]) {
    if (c.R < 1 || c.R > PURLIN_MAX_RANKS) return PURLIN_ERR_INVALID_ARG;
    const int es = elem_bytes(c.dtype);
    if (es == 0) return PURLIN_ERR_INVALID_ARG;
    if (c.op != PURLIN_COPY && c.op != PURLIN_SUM) return PURLIN_ERR_INVALID_ARG;
    for (int k : {c.layout.in, c.layout.out})
        if (k < PURLIN_PACKED || k > PURLIN_TRANSPOSED) return PURLIN_ERR_INVALID_ARG;
    if (src == nullptr || dst == nullptr) return PURLIN_ERR_INVALID_ARG;

    // The one legal (op, layout) pair per collective, §3.1.
    int want_op = PURLIN_COPY, want_in = PURLIN_PACKED, want_out = PURLIN_SCATTERED;
    switch (c.coll) {
        case PURLIN_COLL_ALL_REDUCE:
            want_op = PURLIN_SUM; want_in = PURLIN_SCATTERED; want_out = PURLIN_SCATTERED; break;
        case PURLIN_COLL_REDUCE_SCATTER:
        case PURLIN_COLL_REDUCE_SCATTER_V:
            want_op = PURLIN_SUM; want_in = PURLIN_SCATTERED; want_out = PURLIN_PACKED; break;
        case PURLIN_COLL_ALL_GATHER:
        case PURLIN_COLL_ALL_GATHER_V:
            want_op = PURLIN_COPY; want_in = PURLIN_PACKED; want_out = PURLIN_SCATTERED; break;
        case PURLIN_COLL_ALL_TO_ALL:
        case PURLIN_COLL_ALL_TO_ALL_V:
            want_op = PURLIN_COPY; want_in = PURLIN_SCATTERED; want_out = PURLIN_TRANSPOSED; break;
        default:
            return PURLIN_ERR_INVALID_ARG;
    }
    if (c.op != want_op || !layout_is(c.layout, want_in, want_out)) return PURLIN_ERR_UNSUPPORTED;
    return PURLIN_OK;
}

purlin_status validate_extents(const CallDesc &c, const void *const src[], void *const dst[],
                               const std::vector<uint64_t> &in_b,
                               const std::vector<uint64_t> &out_b) {
    const uint64_t es64 = (uint64_t)elem_bytes(c.dtype);
    for (int r = 0; r < c.R; ++r) {
        if (in_b[r] && src[r] == nullptr) return PURLIN_ERR_INVALID_ARG;
        if (out_b[r] && dst[r] == nullptr) return PURLIN_ERR_INVALID_ARG;
        if (in_b[r] && ((uintptr_t)src[r] & 15u)) return PURLIN_ERR_ALIGNMENT;
        if (out_b[r] && ((uintptr_t)dst[r] & 15u)) return PURLIN_ERR_ALIGNMENT;
    }

    // Outputs never overlap one another.
    for (int a = 0; a < c.R; ++a)
        for (int b = a + 1; b < c.R; ++b)
            if (ranges_overlap((uintptr_t)dst[a], out_b[a], (uintptr_t)dst[b], out_b[b]))
                return PURLIN_ERR_ALIAS;
    // An input overlaps no output, except the in-place forms.
    for (int s = 0; s < c.R; ++s) {
        for (int d = 0; d < c.R; ++d) {
            if (!ranges_overlap((uintptr_t)src[s], in_b[s], (uintptr_t)dst[d], out_b[d])) continue;
            if (s == d && c.coll == PURLIN_COLL_ALL_REDUCE && src[s] == dst[d]) continue;
            if (s == d && c.coll == PURLIN_COLL_ALL_GATHER &&
                (uintptr_t)src[s] == (uintptr_t)dst[d] + (uint64_t)s * c.n * es64)
                continue;
            return PURLIN_ERR_ALIAS;
        }
    }
    return PURLIN_OK;
}

purlin_status validate_call(const CallDesc &c, const void *const src[], void *const dst[]) {
    purlin_status st = validate_shape(c, src, dst);
    if (st != PURLIN_OK) return st;
    const int es = elem_bytes(c.dtype);

    const bool is_v = c.coll == PURLIN_COLL_ALL_GATHER_V || c.coll == PURLIN_COLL_REDUCE_SCATTER_V ||
                      c.coll == PURLIN_COLL_ALL_TO_ALL_V;
    if (is_v) {
        if (c.counts == nullptr) return PURLIN_ERR_INVALID_ARG;
        const int k = c.coll == PURLIN_COLL_ALL_TO_ALL_V ? c.R * c.R : c.R;
        uint64_t total = 0;
        for (int j = 0; j < k; ++j) {
            if (c.counts[j] > kMaxBufferBytes / 4) return PURLIN_ERR_INVALID_ARG;
            total += c.counts[j];
        }
        if (total * (uint64_t)es > kMaxBufferBytes) return PURLIN_ERR_INVALID_ARG;
    } else {
        if (c.n > kMaxBufferBytes / 4 / (uint64_t)c.R) return PURLIN_ERR_INVALID_ARG;
        if ((c.coll == PURLIN_COLL_REDUCE_SCATTER || c.coll == PURLIN_COLL_ALL_TO_ALL) &&
            c.n % (size_t)c.R != 0)
            return PURLIN_ERR_INVALID_ARG;
    }

    std::vector<uint64_t> in_b, out_b;
    buffer_bytes(c, in_b, out_b);
    return validate_extents(c, src, dst, in_b, out_b);
}

namespace {

void raw_segments(const CallDesc &c, bool composed, uint32_t red_chunk, std::vector<RawSeg> &out) {
    const uint64_t es = (uint64_t)elem_bytes(c.dtype);
    const int R = c.R;
    out.clear();
    auto push = [&](uint64_t so, uint64_t dof, uint64_t b, int sr, int dr, int skip, bool sid,
                    uint8_t sync) {
        if (b == 0) return;
        out.push_back(RawSeg{so, dof, b, sr, dr, skip, sid, sync});
    };
    switch (c.coll) {
        case PURLIN_COLL_ALL_REDUCE: {
            const uint64_t total = c.n * es;
            if (!composed) {
                push(0, 0, total, kRankAll, kRankAll, -1, false, kSyncNone);
                break;
            }
            // Owner slices of the ReduceScatter half: R slices whose
            // boundaries fall on whole chunks, so each gather chunk depends
            // on exactly one reduce chunk.
            const uint64_t body = total & ~uint64_t(15);
            const uint64_t per = (body + R - 1) / R;
            const uint64_t L = std::max<uint64_t>(
                red_chunk, (per + red_chunk - 1) / red_chunk * red_chunk);
            for (int r = 0; r < R; ++r) {
                uint64_t a = std::min<uint64_t>((uint64_t)r * L, body);
                uint64_t b = std::min<uint64_t>((uint64_t)(r + 1) * L, body);
                push(a, a, b - a, kRankAll, r, -1, false, kSyncNotify);
            }
            for (int r = 0; r < R; ++r) {
                uint64_t a = std::min<uint64_t>((uint64_t)r * L, body);
                uint64_t b = std::min<uint64_t>((uint64_t)(r + 1) * L, body);
                push(a, a, b - a, r, kRankAll, r, true, kSyncWait);
            }
            // A ragged end (under 16 bytes) is reduced straight into every output.
            push(body, body, total - body, kRankAll, kRankAll, -1, false, kSyncNone);
            break;
        }
        case PURLIN_COLL_REDUCE_SCATTER: {
            const uint64_t M = c.n / (uint64_t)R;
            for (int r = 0; r < R; ++r)
                push((uint64_t)r * M * es, 0, M * es, kRankAll, r, -1, false, kSyncNone);
            break;
        }
        case PURLIN_COLL_ALL_GATHER:
            for (int s = 0; s < R; ++s)
                push(0, (uint64_t)s * c.n * es, c.n * es, s, kRankAll, -1, false, kSyncNone);
            break;
        case PURLIN_COLL_ALL_TO_ALL: {
            const uint64_t M = c.n / (uint64_t)R;
            for (int s = 0; s < R; ++s)
                for (int d = 0; d < R; ++d)
                    push((uint64_t)d * M * es, (uint64_t)s * M * es, M * es, s, d, -1, false,
                         kSyncNone);
            break;
        }
        case PURLIN_COLL_ALL_GATHER_V: {
            uint64_t D = 0;
            for (int s = 0; s < R; ++s) {
                push(0, D * es, c.counts[s] * es, s, kRankAll, -1, false, kSyncNone);
                D += c.counts[s];
            }
            break;
        }
        case PURLIN_COLL_REDUCE_SCATTER_V: {
            uint64_t D = 0;
            for (int r = 0; r < R; ++r) {
                push(D * es, 0, c.counts[r] * es, kRankAll, r, -1, false, kSyncNone);
                D += c.counts[r];
            }
            break;
        }
        case PURLIN_COLL_ALL_TO_ALL_V: {
            // Input of s packed by destination (row prefix); output of d
            // packed by source (column prefix).
            std::vector<uint64_t> S((size_t)R * R), Q((size_t)R * R);
            for (int s = 0; s < R; ++s) {
                uint64_t run = 0;
                for (int d = 0; d < R; ++d) {
                    S[(size_t)s * R + d] = run;
                    run += c.counts[(size_t)s * R + d];
                }
            }
            for (int d = 0; d < R; ++d) {
                uint64_t run = 0;
                for (int s = 0; s < R; ++s) {
                    Q[(size_t)s * R + d] = run;
                    run += c.counts[(size_t)s * R + d];
                }
            }
            for (int s = 0; s < R; ++s)
                for (int d = 0; d < R; ++d)
                    push(S[(size_t)s * R + d] * es, Q[(size_t)s * R + d] * es,
                         c.counts[(size_t)s * R + d] * es, s, d, -1, false, kSyncNone);
            break;
        }
    }
}

}  // namespace

constexpr uint64_t kLineBytes = 128;   // an L2 line
constexpr int kTransposeMaxR = 8;       // the vector kernel's build for whole_op 3

purlin_status compile_plan(const CallDesc &c, int variant, int ar_mode, uint32_t red_slot_bytes,
                           uint32_t copy_chunk, Plan *out) {
    Plan &p = *out;
    p = Plan{};
    p.variant = variant;
    const int R = c.R;
    uint32_t red_chunk = std::max<uint32_t>(16u, (red_slot_bytes / (uint32_t)R) & ~15u);
    copy_chunk = std::max<uint32_t>(16u, copy_chunk & ~15u);
    p.red_chunk = red_chunk;
    p.copy_chunk = copy_chunk;

    const uint64_t es = (uint64_t)elem_bytes(c.dtype);
    bool composed = c.coll == PURLIN_COLL_ALL_REDUCE && ar_mode == 2 &&
                    variant == kVariantThroughput && R > 1 && c.n * es >= 16ull * (uint64_t)R;
    p.composed = composed;

    std::vector<RawSeg> raw;
    raw_segments(c, composed, red_chunk, raw);

    uint64_t chunk = 0, unit = 0;
    std::vector<uint32_t> notify_begin;   // chunk_begin of the k-th notify segment
    p.segs.reserve(raw.size());
    // One piece [off, off + bytes) of a transfer; `ring` false keeps it on
    // the vector path.
    auto emit = [&](const RawSeg &r, uint64_t off, uint64_t bytes, bool ring) {
        Seg s{};
        s.src_off = r.src_off + off;
        s.dst_off = r.dst_off + off;
        s.bytes = bytes;
        s.src_rank = (int8_t)r.src_rank;
        s.dst_rank = (int8_t)r.dst_rank;
        s.skip_rank = (int8_t)r.skip_rank;
        s.src_is_dst = r.src_is_dst ? 1 : 0;
        s.sync = r.sync;
        const bool reduce = r.src_rank == kRankAll;
        // A gathering chunk of the composed AllReduce spans R reducing
        // chunks, so it fills a stage (R tiles) and waits on R flags.
        s.chunk_bytes = reduce ? red_chunk : r.sync == kSyncWait ? red_chunk * (uint32_t)R : copy_chunk;
        if (r.sync == kSyncWait) s.dep_ratio = (uint8_t)R;
        s.chunk_begin = (uint32_t)chunk;
        s.unit_begin = unit;
        uint64_t body = 0;
        if (ring) {
            // A copy's body is cut on the destination side (16-byte aligned
            // stores); a source at another 16-byte phase is staged as its
            // aligned hull, 16 bytes longer, and shifted into place by the
            // consumer warps.  A reduce's body is cut on the sources' side
            // (aligned stages, no shift), and its sums are stored at the
            // destination's phase.
            const Cut cut = cut_transfer(s.src_off, s.dst_off, bytes, reduce);
            body = cut.body;
            if (body > 0) {
                s.tma = 1;
                s.head = (uint8_t)cut.head;
                s.tail = (uint8_t)cut.tail;
                s.shift = (uint8_t)cut.shift;
            }
        }
        p.total_bytes += bytes;
        p.loose_bytes += bytes - body;
        if (s.tma) {
            uint64_t nch = (body + s.chunk_bytes - 1) / s.chunk_bytes;
            chunk += nch;
            unit += (s.head ? 1 : 0) + (s.tail ? 1 : 0);
            if (reduce) p.has_reduce = true;
            else p.has_copy_chunks = true;
            if (!reduce && s.shift) p.has_shifted_copies = true;
            if (reduce && s.shift) p.has_phase_reduce = true;
            if (r.sync == kSyncNotify) {
                notify_begin.push_back(s.chunk_begin);
                p.notify_chunks += nch;
            }
        } else {
            unit += units_in(unit_grid(s.src_off, s.dst_off, reduce), 0, bytes);
            s.whole = ((s.src_off | s.dst_off | bytes) & 15u) == 0 ? 1 : 0;
        }
        p.segs.push_back(s);
    };
    for (const RawSeg &r : raw) {
        const bool ring = variant == kVariantThroughput;
        // In the ring, a copy to every rank that waits on nothing (AllGather,
        // AllGatherV) starts its body on a 128-byte line of the destination,
        // so every chunk, and every warp's 512 contiguous bytes of stores in
        // it, covers whole L2 lines: the bytes before the line become a
        // segment of their own on the vector path.  (A warp whose run starts
        // mid-line touches five lines instead of four: 19% more L2 write
        // requests and partial-line writes, measured at 0.78 against 0.90 of
        // the copy peak on an AllGatherV of unequal shares.)  Point-to-point
        // copies (AllToAll(V): R*R segments, mostly stored in bulk) keep one
        // segment each: splitting them measured up to 34% slower, the
        // segment table outgrowing the ring's staged copy.  A gathering
        // segment of the composed AllReduce keeps the cut of the reducing
        // segment it waits on, so its chunks cover whole reducing chunks;
        // reduces are cut on their sources.
        const uint64_t lead = (kLineBytes - r.dst_off % kLineBytes) % kLineBytes;
        if (ring && r.src_rank != kRankAll && r.dst_rank == kRankAll && r.sync == kSyncNone &&
            lead >= 16 && r.bytes >= lead + 16) {
            emit(r, 0, lead, false);
            emit(r, lead, r.bytes - lead, true);
        } else {
            emit(r, 0, r.bytes, ring);
        }
    }
    // Each gather segment waits on the reduce segment of the same slice; the
    // two have equal length, and gather chunk i covers reduce chunks
    // [i*R, (i+1)*R) of it.
    size_t k = 0;
    for (Seg &s : p.segs)
        if (s.sync == kSyncWait) s.dep_chunk = k < notify_begin.size() ? notify_begin[k++] : 0;
    // A vector-path plan of whole-window copies only, or reductions only,
    // runs the vector kernel's build for that case (whole_unit).
    bool whole = variant == kVariantLatency && !p.segs.empty(), copies = true, reduces = true;
    for (const Seg &s : p.segs) {
        whole = whole && !s.tma && s.whole;
        copies = copies && s.src_rank >= 0;
        reduces = reduces && s.src_rank < 0;
    }
    p.whole_op = !whole ? 0 : copies ? 1 : reduces ? 2 : 0;
    // A uniform AllToAll of whole windows: block (s, d) is segment s*R + d,
    // W windows from offset d*W*16 of source s to offset s*W*16 of
    // destination d.  The vector kernel then computes each unit's addresses
    // from its index, with no table to fetch or search.
    const size_t R2 = (size_t)c.R * (size_t)c.R;
    if (p.whole_op == 1 && c.coll == PURLIN_COLL_ALL_TO_ALL && c.R <= kTransposeMaxR &&
        p.segs.size() == R2 && unit < (1ull << 32)) {
        const uint64_t B = p.segs[0].bytes, W = B / 16;
        bool uniform = B > 0 && B % 16 == 0 && unit == (uint64_t)R2 * W;
        for (size_t i = 0; uniform && i < R2; ++i) {
            const Seg &g = p.segs[i];
            const int sr = (int)(i / (size_t)c.R), dr = (int)(i % (size_t)c.R);
            uniform = g.src_rank == sr && g.dst_rank == dr && g.bytes == B &&
                      g.src_off == (uint64_t)dr * B && g.dst_off == (uint64_t)sr * B &&
                      g.unit_begin == (uint64_t)i * W;
        }
        if (uniform) p.whole_op = 3;
    }
    if (chunk > 0xFFFFFFF0ull) return PURLIN_ERR_INVALID_ARG;
    p.nchunks = chunk;
    p.nunits = unit;
    // A stage holds one tile per source; a shifted copy's tile (its aligned
    // hull) is 16 bytes longer.
    uint32_t slot = 0;
    for (const Seg &s : p.segs) {
        if (!s.tma) continue;
        const uint32_t tile = s.chunk_bytes + (s.src_rank != kRankAll && s.shift ? 16u : 0u);
        const uint32_t nsrc = s.src_rank == kRankAll ? (uint32_t)R : 1u;
        slot = std::max<uint32_t>(slot, tile * nsrc);
    }
    p.slot_bytes = slot;
    return PURLIN_OK;
}

}  // namespace purlin
