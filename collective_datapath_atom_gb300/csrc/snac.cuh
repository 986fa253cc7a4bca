// snac.cuh -- the device side of SNAC (stage, notify, consume) over the
// Atom primitives, as device functions.  The library's own kernels call them
// with their launch's CTA index and count; kernels written against the
// device API (include/purlin_device.cuh) call the same functions with the
// CTAs they hand to a collective.
//
// "Purlin: Separating Orchestration from the Datapath of Collectives":
//   §3.2  SNAC: chunks are staged, their readiness is notified, consumers
//         then copy or reduce them; composed AllReduce overlaps staging,
//         reduction and gathering on chunks.
//   §3.3  the Atom pipeline stages data in CTA-local shared memory so
//         fetches overlap with processing; SCORE reductions.
//   §4.3  a monotonic 64-bit epoch is the notification value and its
//         parity selects the buffer set.
// "Purlin" project README, "Device-side": Atoms and collectives are callable
// from inside a user kernel; exactly `blocks` CTAs enter a collective.
//
// Vector units (do_unit): one 16-byte destination window each; 128-bit
// loads of every source, ordered binary32 accumulation, 128-bit stores.
//
// The ring (run_ring): persistent CTAs with three warp roles over a ring of
// shared-memory stages.
//   warp 0     Stage: lane s issues cp.async.bulk global -> shared for
//              source s of the chunk (R tiles for a reduce, one for a
//              copy); completion on the stage's mbarrier.  A chunk that
//              depends on another CTA's chunk first acquires that chunk's
//              flag (bounded spin, whole warp).
//   warp 1     Consume (copy): lane d issues cp.async.bulk shared -> global
//              to destination d.  Notify: for a chunk other CTAs wait on,
//              once the consumer warps report it stored, release-store
//              epoch + generation into its flag (batched behind one
//              GPU-scope fence).
//   warps 2..  Consume (reduce, and copies that are shifted or stored with
//              vector stores): SCORE over the R tiles, each thread storing
//              its 16-byte results straight to one or all destinations;
//              also the ragged head/tail units.
// Every wait is bounded; an expired wait records PURLIN_ERR_TIMEOUT in the
// error word and the CTA winds down (its own bulk copies are waited for).
//
// Parameter objects (class P) expose: src[] and dst[] (rank buffer bases),
// segs / segs_dev (segment table), err, nchunks, nunits, timeout_ns,
// drop_notify, flag_slots, stages, slot_stride, nseg, R and vector_copies.
// The flag set and epoch of a launch are passed to run_ring separately.
#pragma once

#include <cuda_runtime.h>

#include "atom.cuh"
#include "plan.h"

namespace purlin {
namespace snac {

constexpr int kNotifyBatch = 4;                   // flags published behind one fence
constexpr uint64_t kRingWaitNs = 2000000000ull;   // 2 s bound on a ring wait
constexpr int kSmemSegs = 64;                     // segment table entries staged in the ring's workspace

// Error word layout: bits 0..7 status, 8..15 site, 16..63 chunk, unit or CTA.
enum ErrSite : uint64_t {
    kSiteFlagWait = 1,
    kSiteRingFull = 2,
    kSiteRingEmpty = 3,
    kSiteChunkDone = 4,
    kSiteDeviceArgs = 5,   // a device-API call with arguments that do not match its descriptor
    kSiteDeviceCounts = 6, // device-resident counts that exceed the declared capacities
    kSitePacketWait = 7,   // a latency-path packet that never arrived
    kSiteChannelArgs = 8,  // a packet-channel unit past the channel's capacity
};

struct Ctl {
    int abort;
    int pad;
    unsigned long long epoch;   // this CTA's epoch for the launch (device epoch, device API)
};

// Bytes of the ring's workspace: S stages of slot_stride bytes, 4*S
// mbarriers (full, empty, a 2*S completion ring) and the staged segment
// table.  Callers that keep a Ctl in the workspace add it after this.
__host__ __device__ constexpr uint32_t ring_workspace_bytes(uint32_t stages, uint32_t slot_stride) {
    return stages * slot_stride + 4 * stages * 8 + kSmemSegs * (uint32_t)sizeof(Seg);
}

template <class P>
__device__ __forceinline__ const Seg *seg_table(const P &p) {
    return p.segs_dev != nullptr ? p.segs_dev : p.segs;
}

// Copy the segment table (from the parameter block or device memory) into
// shared memory with every thread of the CTA: one round of parallel loads
// instead of a chain of dependent reads in each lookup.  Tables of more than
// `cap` segments stay where they are.  The caller synchronises the CTA
// before the table is read.
template <class P>
__device__ __forceinline__ const Seg *stage_segs(const P &p, Seg *sm, int cap) {
    if (p.nseg > cap || seg_table(p) == sm) return seg_table(p);   // too large, or already there
    const uint64_t *from = reinterpret_cast<const uint64_t *>(seg_table(p));
    uint64_t *to = reinterpret_cast<uint64_t *>(sm);
    const int words = p.nseg * (int)(sizeof(Seg) / sizeof(uint64_t));
    for (int i = threadIdx.x; i < words; i += blockDim.x) to[i] = from[i];
    return sm;
}

// Last segment whose first chunk (unit) index is <= x: the one holding x.
__device__ __forceinline__ int seg_of_chunk(const Seg *segs, int nseg, uint64_t x) {
    int lo = 0, hi = nseg;   // answer in [lo, hi)
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if ((uint64_t)segs[mid].chunk_begin <= x) lo = mid;
        else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ int seg_of_unit(const Seg *segs, int nseg, uint64_t x) {
    int lo = 0, hi = nseg;
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (segs[mid].unit_begin <= x) lo = mid;
        else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ void record_error(unsigned long long *err, uint64_t code, uint64_t site,
                                             uint64_t where) {
    unsigned long long v = (unsigned long long)((code & 0xFF) | ((site & 0xFF) << 8) |
                                                ((where & 0xFFFFFFFFFFFFull) << 16));
    atomicCAS(err, 0ull, v);
}

__device__ __forceinline__ bool error_set(const unsigned long long *err) {
    return *reinterpret_cast<const volatile unsigned long long *>(err) != 0ull;
}

// ------------------------------------------------------------ vector unit --

// Store bytes [b0, b0 + nb) of v at d (b0 + nb <= 16; d aligned to the
// element size) as 32-bit words, with a 16-bit piece at either end where d
// or the length is only 2-byte aligned.
template <int ES>
__device__ __forceinline__ void put_span_words(char *d, uint4 v, uint32_t b0, uint32_t nb) {
    if (b0 != 0) v = atom::shift_pair(v, v, b0);   // the span's first byte to byte 0
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    auto pick = [&](uint32_t i) { return i == 0 ? w[0] : i == 1 ? w[1] : i == 2 ? w[2] : w[3]; };
    if (ES == 4 || ((uintptr_t)d & 2u) == 0) {
#pragma unroll
        for (uint32_t i = 0; i < 4; ++i)
            if (4 * i + 4 <= nb) *reinterpret_cast<uint32_t *>(d + 4 * i) = w[i];
        if (ES == 2 && (nb & 2u))
            *reinterpret_cast<uint16_t *>(d + (nb & ~3u)) = (uint16_t)pick(nb >> 2);
    } else {   // d is 2 mod 4: a half word, whole words across x's words, a half word
        *reinterpret_cast<uint16_t *>(d) = (uint16_t)w[0];
#pragma unroll
        for (uint32_t i = 0; i < 3; ++i)
            if (4 * i + 6 <= nb)
                *reinterpret_cast<uint32_t *>(d + 2 + 4 * i) = __funnelshift_r(w[i], w[i + 1], 16);
        const uint32_t words = (nb - 2) >> 2;
        if ((nb - 2) & 2u)
            *reinterpret_cast<uint16_t *>(d + 2 + 4 * words) = (uint16_t)(pick(words) >> 16);
    }
}

// Store bytes [b0, b0 + nb) of v at d: one 128-bit store for a whole aligned
// window, else put_span_words.
template <int ES>
__device__ __forceinline__ void put_span(char *d, uint4 v, uint32_t b0, uint32_t nb) {
    if (b0 == 0 && nb == 16u && ((uintptr_t)d & 15u) == 0) atom::st_v4(d, v);
    else put_span_words<ES>(d, v, b0, nb);
}

// One 16-byte window of a segment: copy or reduce it to every destination.
//
// A reduce reads every source at the same offset, so its windows follow the
// sources' 16-byte grid (unit_grid): each source takes one aligned 128-bit
// load, all R in flight together, and the sum's window is stored at the
// destination's phase (put_span).  A copy's windows follow the destination's
// grid: its one source is fetched with at most two aligned 128-bit loads,
// each holding at least one of the window's bytes (no load leaves the
// source buffer's 16-byte granules), and shifted into place, so that the
// stores to the R destinations are aligned.  A ring segment's vector units
// are the bytes outside its aligned body (head and tail, on the same grid)
// (RING: the caller is the ring, whose segments may have a body; the
// one-shot kernels' never do).
// A unit of a segment made of whole aligned windows (Seg::whole, up to 8
// ranks): no window bounds, no shift, plain 128-bit stores.  Same loads, same
// rank-order sum and rounding as do_unit.  OP 1: a copy; OP 2: a reduction.
// The vector kernel has a build for plans made only of such copies or only of
// such reductions (kernels.cu): per call in a graph, AllReduce 2 KiB per rank
// 1.88 -> 1.63 us and 256 B 1.85 -> 1.45 us, AllGather 256 B 1.99 -> 1.72 us.
// One build with both operations made the reductions slower, and inlining
// the short path into do_unit made the 8-rank builds spill.
template <int DT, int MAXR, int OP, class P>
__device__ __forceinline__ void whole_unit(const P &p, const Seg &sg, uint64_t k) {
    using V = atom::Vec<DT>;
    const int R = p.R;
    const uint64_t so = sg.src_off + 16 * k, doff = sg.dst_off + 16 * k;
    uint4 out;
    const char *self = nullptr;
    if (OP == 2) {   // reduce (SCORE): rank order, binary32, one rounding
        uint4 v[MAXR];
#pragma unroll
        for (int j = 0; j < MAXR; ++j)
            if (j < R) v[j] = atom::ld_v4(static_cast<const char *>(p.src[j]) + so);
        float acc[V::VE];
        V::init(acc, v[0]);
#pragma unroll
        for (int j = 1; j < MAXR; ++j)
            if (j < R) V::add(acc, v[j]);
        out = V::pack(acc);
    } else {                 // copy, bitwise
        const char *sbase = static_cast<const char *>(sg.src_is_dst ? p.dst[sg.src_rank]
                                                                    : p.src[sg.src_rank]);
        self = sbase + so;   // in-place AllGather: the block is already there
        out = atom::ld_v4(self);
    }
    if (sg.dst_rank >= 0) {
        char *d = static_cast<char *>(p.dst[sg.dst_rank]) + doff;
        if (OP == 2 || d != self) atom::st_v4(d, out);
        return;
    }
#pragma unroll
    for (int r = 0; r < MAXR; ++r) {
        if (r >= R || r == sg.skip_rank) continue;
        char *d = static_cast<char *>(p.dst[r]) + doff;
        if (OP == 2 || d != self) atom::st_v4(d, out);
    }
}

// Unit u of a uniform AllToAll of whole windows (Plan::whole_op 3): window
// k = u % W of block (s, d) = (u / W / R, u / W % R), copied from offset
// (d*W + k)*16 of source s to offset (s*W + k)*16 of destination d.  The
// rank pointers are picked with static indices (parameter reads at fixed
// offsets), as in the reduce path's stores.
template <int MAXR, class P>
__device__ __forceinline__ void transposed_unit(const P &p, uint32_t u, uint32_t W) {
    const uint32_t R = (uint32_t)p.R;
    const uint32_t blk = u / W, k = u - blk * W;
    const uint32_t s = blk / R, d = blk - s * R;
    const char *sb = nullptr;
    char *db = nullptr;
#pragma unroll
    for (int j = 0; j < MAXR; ++j) {
        if ((uint32_t)j == s) sb = static_cast<const char *>(p.src[j]);
        if ((uint32_t)j == d) db = static_cast<char *>(p.dst[j]);
    }
    atom::st_v4(db + ((uint64_t)s * W + k) * 16u, atom::ld_v4(sb + ((uint64_t)d * W + k) * 16u));
}

template <int DT, int MAXR, bool RING, class P>
__device__ void do_unit(const P &p, const Seg &sg, uint64_t k) {
    using V = atom::Vec<DT>;
    constexpr int ES = DT == PURLIN_F32 ? 4 : 2;
    const bool reduce = sg.src_rank < 0;
    uint64_t lo, hi;
    if (RING && sg.tma) {
        if (k == 0 && sg.head) {
            lo = 0;
            hi = sg.head;
        } else {
            lo = sg.bytes - sg.tail;
            hi = sg.bytes;
        }
    } else {
        const uint64_t g = unit_grid(sg.src_off, sg.dst_off, reduce);
        const uint64_t a = (g / 16 + k) * 16;
        lo = (a > g ? a : g) - g;
        const uint64_t b = a + 16, e = g + sg.bytes;
        hi = (b < e ? b : e) - g;
    }
    const int R = p.R;
    const uint32_t nb = (uint32_t)(hi - lo);   // 1..16 bytes of this window
    const uint64_t sx = sg.src_off + lo;
    const uint32_t sh = (uint32_t)(sx & 15u);
    const bool two = sh + nb > 16u;            // the bytes straddle two aligned vectors
    const uint64_t doff = sg.dst_off + lo;

    // The window's source bytes in the buffer that starts at `base` (the rank
    // buffer itself: sx is the window's offset in it), in the low bytes of a
    // vector.
    auto fetch = [&](const char *base) -> uint4 {
        const char *a = base + (sx - sh);
        if (sh == 0) return atom::ld_v4(a);
        const uint4 v0 = atom::ld_v4_l1(a);
        return atom::shift_pair(v0, two ? atom::ld_v4_l1(a + 16) : v0, sh);
    };

    // A copy's store: its window lies on the destination's grid, so a whole
    // window is one aligned 128-bit store and a partial one element stores.
    auto put = [&](char *d, const uint4 &v) {
        if (nb == 16u) {
            atom::st_v4(d, v);
            return;
        }
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 16 / ES; ++j) {
            if ((uint32_t)(j * ES) >= nb) break;
            const uint32_t word = w[(j * ES) >> 2];
            if (ES == 4) *reinterpret_cast<uint32_t *>(d + j * ES) = word;
            else *reinterpret_cast<uint16_t *>(d + j * ES) = (uint16_t)(word >> (8 * ((j * ES) & 3)));
        }
    };

    if (!reduce) {   // copy, bitwise
        const char *sbase = static_cast<const char *>(sg.src_is_dst ? p.dst[sg.src_rank]
                                                                    : p.src[sg.src_rank]);
        const uint4 v = fetch(sbase);
        const char *self = sbase + sx;   // in-place AllGather: the block is already there
        if (sg.dst_rank >= 0) {
            char *d = static_cast<char *>(p.dst[sg.dst_rank]) + doff;
            if (d != self) put(d, v);
        } else {
            for (int r = 0; r < R; ++r) {
                if (r == sg.skip_rank) continue;
                char *d = static_cast<char *>(p.dst[r]) + doff;
                if (d != self) put(d, v);
            }
        }
        return;
    }

    // reduce (SCORE): rank order 0..R-1, binary32, one rounding at the end.
    // The window lies in one aligned vector of every source (its bytes are
    // [sh, sh + nb) of it); bytes outside the window are summed too and never
    // stored.  A group's loads all issue before any of its values is used.
    auto load = [&](int s) -> uint4 {
        return atom::ld_v4(static_cast<const char *>(p.src[s]) + (sx - sh));
    };
    float acc[V::VE];
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (j < R) v[j] = load(j);
    V::init(acc, v[0]);
#pragma unroll
    for (int j = 1; j < 8; ++j)
        if (j < R) V::add(acc, v[j]);
    if (MAXR > 8) {
        for (int s0 = 8; s0 < R; s0 += 8) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (s0 + j < R) v[j] = load(s0 + j);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (s0 + j < R) V::add(acc, v[j]);
        }
    }
    const uint4 out = V::pack(acc);
    if (sg.dst_rank >= 0) {
        put_span<ES>(static_cast<char *>(p.dst[sg.dst_rank]) + doff, out, sh, nb);
    } else if (MAXR <= 8) {
        // static indices: each destination pointer is read from the
        // parameters directly, not one indexed load per store
        if (sh == 0 && nb == 16u && (doff & 15u) == 0) {   // whole window (bases 16-B aligned)
#pragma unroll
            for (int r = 0; r < MAXR; ++r)
                if (r < R && r != sg.skip_rank) atom::st_v4(static_cast<char *>(p.dst[r]) + doff, out);
        } else {
#pragma unroll
            for (int r = 0; r < MAXR; ++r)
                if (r < R && r != sg.skip_rank)
                    put_span_words<ES>(static_cast<char *>(p.dst[r]) + doff, out, sh, nb);
        }
    } else {
        for (int r = 0; r < R; ++r)
            if (r != sg.skip_rank) put_span<ES>(static_cast<char *>(p.dst[r]) + doff, out, sh, nb);
    }
}

// Units u0, u0 + stride, ... of the plan: the first one's segment is found by
// binary search, later ones by walking forward (units only increase), so
// the search cost fades for threads that own many units.
// WHOLE: every segment is made of whole aligned windows (whole_unit).
template <int DT, int MAXR, bool RING, int WHOLE = 0, class P>
__device__ __forceinline__ void units_loop(const P &p, const Seg *segs, uint64_t u0,
                                           uint64_t stride) {
    if (u0 >= p.nunits) return;
    int si = seg_of_unit(segs, p.nseg, u0);
    for (uint64_t u = u0; u < p.nunits; u += stride) {
        while (si + 1 < p.nseg && segs[si + 1].unit_begin <= u) ++si;
        if constexpr (WHOLE != 0) whole_unit<DT, MAXR, WHOLE>(p, segs[si], u - segs[si].unit_begin);
        else do_unit<DT, MAXR, RING>(p, segs[si], u - segs[si].unit_begin);
    }
}

// ------------------------------------------------------------------ ring --

struct ChunkGeo {
    const Seg *sg;
    uint64_t ci;      // chunk index within the segment
    uint64_t off;     // byte offset of the chunk within the segment
    uint32_t bytes;   // bytes per source
};

__device__ __forceinline__ ChunkGeo chunk_geo(const Seg *segs, int nseg, uint64_t c) {
    ChunkGeo g;
    g.sg = &segs[seg_of_chunk(segs, nseg, c)];
    const Seg &sg = *g.sg;
    g.ci = c - sg.chunk_begin;
    const uint64_t body = sg.bytes - sg.head - sg.tail;
    const uint64_t done = g.ci * sg.chunk_bytes;
    g.off = sg.head + done;
    const uint64_t rem = body - done;
    g.bytes = (uint32_t)(rem < sg.chunk_bytes ? rem : sg.chunk_bytes);
    return g;
}

// Bounded wait on an mbarrier phase.  `abortable`: give up as soon as
// another role of the CTA has given up.
__device__ __forceinline__ bool ring_wait(uint64_t *bar, uint32_t parity, volatile Ctl *ctl,
                                          unsigned long long *err, uint64_t site, bool abortable) {
    if (atom::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = atom::globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (atom::mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 0) {
            if (abortable && ctl->abort) return false;
            if (atom::globaltimer_ns() - t0 > kRingWaitNs) {
                record_error(err, PURLIN_ERR_TIMEOUT, site, blockIdx.x);
                ctl->abort = 1;
                return false;
            }
        }
    }
}

// SNAC consume-side acquire, warp-wide: lane l waits until notifying chunks
// d0 + l, d0 + l + 32, ... hold at least this call's value for them, so the
// flags are polled in parallel rather than one dependent round trip after
// another.  Each wait is bounded; on expiry the error word is set and later
// waits of the launch are skipped.  __syncwarp then orders every lane's
// acquire before the bulk load lane 0 issues next.
template <class P>
__device__ void acquire_range(const P &p, const unsigned long long *flags, uint64_t epoch,
                              const ChunkOrder &order, uint64_t d0, uint64_t d1, int lane) {
    for (uint64_t d = d0 + (uint64_t)lane; d < d1; d += 32) {
        if (error_set(p.err)) break;
        const FlagAt fa = flag_at(order, p.flag_slots, d);
        const unsigned long long *f = flags + fa.slot;
        const unsigned long long want = epoch + fa.gen;
        if (atom::flag_acquire(f) >= want) continue;
        const uint64_t t0 = atom::globaltimer_ns();
        uint32_t ns = 32;
        while (atom::flag_acquire(f) < want) {
            if ((int64_t)(atom::globaltimer_ns() - t0) > p.timeout_ns) {
                record_error(p.err, PURLIN_ERR_TIMEOUT, kSiteFlagWait, d);
                break;
            }
            __nanosleep(ns);
            if (ns < 1024) ns <<= 1;
        }
    }
    __syncwarp();
    atom::fence_async_global();   // the staged reads that follow are async-proxy reads
}

// SNAC notify: publish a completed chunk (its stores are complete and
// ordered before this store by the caller).
template <class P>
__device__ __forceinline__ void notify_chunk(const P &p, unsigned long long *flags, uint64_t epoch,
                                             const ChunkOrder &order, uint64_t c) {
    if ((int64_t)c == p.drop_notify) return;   // host-side fault injection
    const FlagAt fa = flag_at(order, p.flag_slots, c);
    atom::flag_release(flags + fa.slot, epoch + fa.gen);
}

// ------------------------------------------------------------ packets --

// Bounded wait for the packet at pk to carry `flag`: true with its payload,
// or false once `timeout_ns` has passed (TIMEOUT recorded at the packet
// site with `where`) or when an earlier wait of the launch already gave up
// (the error word is set), so a lost packet costs one timeout, not one per
// unit.  The poll backs off in steps of 32 ns up to 256 ns.
__device__ __forceinline__ bool packet_wait(const unsigned char *pk, uint32_t flag,
                                            int64_t timeout_ns, unsigned long long *err,
                                            uint64_t where, uint64_t *payload) {
    if (atom::packet_load(pk, flag, payload)) return true;
    if (error_set(err)) return false;
    const uint64_t t0 = atom::globaltimer_ns();
    uint32_t ns = 0;
    while (!atom::packet_load(pk, flag, payload)) {
        if ((int64_t)(atom::globaltimer_ns() - t0) > timeout_ns) {
            record_error(err, PURLIN_ERR_TIMEOUT, kSitePacketWait, where);
            return false;
        }
        if (ns) __nanosleep(ns);
        ns = ns < 256 ? ns + 32 : 256;
    }
    return true;
}

// ------------------------------------------------------ device epoch --
//
// The epoch of a launch whose CTAs notify one another lives in device
// memory, so that a launch replayed from a CUDA graph (its parameters frozen
// at capture) still gets a new epoch: every CTA reads it on entry, and the
// last CTA to finish advances it by the launch's odd increment.  Every CTA
// increments `done` only after it has read the epoch, and the epoch moves
// only once `done` reaches the grid size, so all CTAs of a launch read the
// same value; the next launch on the stream reads the advanced one.
struct DevEpoch {
    unsigned long long epoch;
    unsigned long long done;
};

// Thread 0 reads the epoch into ctl->epoch; the caller synchronises the CTA.
__device__ __forceinline__ void epoch_enter(const DevEpoch *e, Ctl *ctl) {
    if (threadIdx.x == 0) ctl->epoch = *reinterpret_cast<const volatile unsigned long long *>(&e->epoch);
}

// Thread 0, after the whole CTA is done with the launch's work.
__device__ __forceinline__ void epoch_leave(DevEpoch *e, uint64_t inc, uint32_t ctas) {
    if (threadIdx.x != 0) return;
    if (atomicAdd(&e->done, 1ull) == (unsigned long long)ctas - 1ull) {
        e->done = 0;
        atomicAdd(&e->epoch, (unsigned long long)inc);
    }
}

// The consumer warps' share of a reduce chunk whose sources are staged on
// their own 16-byte grid (tile bytes apart, from sp) while the destination
// is at another phase: each thread sums its vectors over the sources in rank
// order and stores the sum at the destination's phase.
template <int DT, int MAXR, class P>
__device__ __forceinline__ void reduce_chunk_to_phase(const P &p, const Seg &sg,
                                                   const unsigned char *sp, uint32_t tile,
                                                   int nvec, uint64_t doff, int ctid, int nct) {
    using V = atom::Vec<DT>;
    constexpr int ES = DT == PURLIN_F32 ? 4 : 2;
    const int R = p.R;
    for (int v = ctid; v < nvec; v += nct) {
        const unsigned char *t = sp + 16 * (size_t)v;
        float acc[V::VE];
        V::init(acc, atom::lds_v4(t));
        if (MAXR <= 8) {
#pragma unroll
            for (int s = 1; s < MAXR; ++s)
                if (s < R) V::add(acc, atom::lds_v4(t + (size_t)s * tile));
        } else {
#pragma unroll 8
            for (int s = 1; s < R; ++s) V::add(acc, atom::lds_v4(t + (size_t)s * tile));
        }
        const uint4 out = V::pack(acc);
        const uint64_t o = doff + 16 * (uint64_t)v;
        if (sg.dst_rank >= 0) {
            put_span<ES>(static_cast<char *>(p.dst[sg.dst_rank]) + o, out, 0, 16);
        } else {
            for (int d = 0; d < R; ++d)
                if (d != sg.skip_rank) put_span<ES>(static_cast<char *>(p.dst[d]) + o, out, 0, 16);
        }
    }
}

// ------------------------------------------------------- chunk order --

// For plans whose chunks notify and wait (flags given): the first waiting
// segment's first chunk ends the reducing chunks (ChunkOrder in plan.h).
// Every thread calls it (measured: as fast as one thread's result shared
// through the control block, and the other collectives keep their speed).
__device__ __forceinline__ ChunkOrder chunk_order(const Seg *segs, int nseg, uint64_t nchunks,
                                                  int R, uint32_t nblk, bool composed) {
    if (!composed) return ChunkOrder{};
    for (int i = 0; i < nseg; ++i)
        if (segs[i].sync == kSyncWait && segs[i].tma)
            return make_chunk_order(segs[i].chunk_begin, nchunks - segs[i].chunk_begin, R, nblk,
                                    kNotifyBatch);
    return ChunkOrder{};
}

// The 16 bytes that start at byte 4K + r/8 of the 32-byte pair (a, b) (r: 0,
// 8, 16 or 24 bits): with the word offset K fixed at compile time the window
// is four funnel shifts, with no selects.
template <int K>
__device__ __forceinline__ uint4 window_at(const uint4 &a, const uint4 &b, uint32_t r) {
    static_assert(K >= 0 && K <= 3, "word offset");
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    return make_uint4(__funnelshift_r(w[K], w[K + 1], r), __funnelshift_r(w[K + 1], w[K + 2], r),
                      __funnelshift_r(w[K + 2], w[K + 3], r), __funnelshift_r(w[K + 3], w[K + 4], r));
}

// The consumer warps' share of a copy chunk staged as its 16-byte aligned
// hull (sp) whose source sits 4K + r/8 bytes past the destination's phase:
// each vector is read as the two aligned 128-bit shared vectors holding it
// (two conflict-free accesses per warp, against five 32-bit loads at a
// 16-byte lane stride, each a 4-way bank conflict) and shifted into place.
template <int K, class P>
__device__ __forceinline__ void copy_chunk_shifted(const P &p, const Seg &sg,
                                                   const unsigned char *sp, uint32_t r, int nvec,
                                                   uint64_t doff, const char *self, int ctid,
                                                   int nct) {
    const int R = p.R;
    for (int v = ctid; v < nvec; v += nct) {
        const unsigned char *t = sp + 16 * (size_t)v;
        const uint4 out = window_at<K>(atom::lds_v4(t), atom::lds_v4(t + 16), r);
        const uint64_t o = doff + 16 * (uint64_t)v;
        if (sg.dst_rank >= 0) {
            if (static_cast<const char *>(p.dst[sg.dst_rank]) + doff != self)
                atom::st_v4(static_cast<char *>(p.dst[sg.dst_rank]) + o, out);
        } else {
            for (int d = 0; d < R; ++d)
                if (d != sg.skip_rank && static_cast<const char *>(p.dst[d]) + doff != self)
                    atom::st_v4(static_cast<char *>(p.dst[d]) + o, out);
        }
    }
}

// flags/epoch: this launch's flag set (the parity the epoch selects) and its
// epoch, for plans whose chunks notify or wait (else unused).  RAGGED: the
// plan may hold chunks at another 16-byte phase than their destination:
// reduce chunks whose sums are stored at the destination's phase
// (reduce_chunk_to_phase, required for them) and shifted copies
// (copy_chunk_shifted).  A ring built without it takes no reduce chunk at
// another phase, shifts copies through its generic path, and keeps the
// consumer loop's code as it was.
template <int DT, int MAXR, bool RAGGED, class P>
__device__ void run_ring(const P &p, unsigned char *smem, Ctl *ctl_p, uint32_t bidx,
                         uint32_t nblk, unsigned long long *flags, uint64_t epoch) {
    using V = atom::Vec<DT>;
    Ctl &ctl = *ctl_p;
    // Generic-proxy writes made before this call (by this CTA, or by others
    // and ordered by the caller's grid barrier) precede the bulk loads below.
    atom::fence_async_global();

    const uint32_t S = p.stages;
    const int R = p.R;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ncw = (int)(blockDim.x >> 5) - 2;   // consumer warps

    unsigned char *ring = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)S * p.slot_stride);
    uint64_t *full = bars;           // S: producer arrive + transaction bytes
    uint64_t *empty = bars + S;      // S: ncw + 1 arrivals: every consumer warp and the writer
    uint64_t *cdone = bars + 2 * S;  // 2S: ncw arrivals: chunk k (entry k mod 2S) to publish
                                     //     has been stored
    // Every role waits on full[] for EVERY chunk, in order, and arrives once
    // per chunk on empty[]: a parity wait is only sound if the slot's
    // previous phase is known complete, and a slot is refilled only after
    // every role has passed it.  cdone[] has 2S entries: the writer's arrival
    // on empty[] for chunk k + S comes after its wait on cdone for chunk k,
    // so the consumer warps are never 2S chunks ahead of that wait.
    const uint32_t C = 2 * S;
    const Seg *segs = stage_segs(p, reinterpret_cast<Seg *>(bars + 4 * S), kSmemSegs);

    if (threadIdx.x == 0) {
        for (uint32_t i = 0; i < S; ++i) {
            atom::mbar_init(&full[i], 1);
            atom::mbar_init(&empty[i], (uint32_t)ncw + 1u);
        }
        for (uint32_t i = 0; i < C; ++i) atom::mbar_init(&cdone[i], (uint32_t)ncw);
        ctl.abort = 0;
        atom::mbar_init_fence();
    }
    __syncthreads();
    // (the staged table is complete)
    const ChunkOrder order = chunk_order(segs, p.nseg, p.nchunks, R, nblk, flags != nullptr);

    if (warp == 0) {
        // ---------------------------------------------------------- Stage --
        // The whole warp walks the chunk list; lane s issues the bulk load
        // of source s, so the R loads of a chunk go out in parallel.
        const uint64_t pol = atom::policy_evict_first();
        uint32_t k = 0;
        for (uint64_t pos = bidx; pos < p.nchunks; pos += nblk, ++k) {
            const uint64_t c = chunk_at(order, pos);
            const uint32_t slot = k % S;
            bool ok = true;
            if (k >= S)
                ok = ring_wait(&empty[slot], ((k / S) & 1u) ^ 1u, &ctl, p.err, kSiteRingEmpty, true);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            const ChunkGeo g = chunk_geo(segs, p.nseg, c);
            const Seg &sg = *g.sg;
            if (sg.sync == kSyncWait) {
                // the notifying chunks this one covers, polled by the whole warp
                const uint32_t ratio = sg.dep_ratio ? sg.dep_ratio : 1u;
                const uint32_t rc = sg.chunk_bytes / ratio;
                const uint64_t nred = (sg.bytes - sg.head - sg.tail + rc - 1) / rc;
                const uint64_t d0 = g.ci * ratio;
                const uint64_t d1 = d0 + ratio < nred ? d0 + ratio : nred;
                acquire_range(p, flags, epoch, order, sg.dep_chunk + d0, sg.dep_chunk + d1, lane);
            }
            unsigned char *sp = ring + (size_t)slot * p.slot_stride;
            const int nsrc = sg.src_rank < 0 ? R : 1;
            // A shifted copy's source is staged as its 16-byte aligned hull; a
            // reduce's sources are aligned on their own grid.
            const uint32_t lead = sg.src_rank >= 0 ? sg.shift : 0u;
            const uint32_t extra = lead ? 16u : 0u;
            const uint32_t tile = sg.chunk_bytes + extra;
            const uint32_t ld_bytes = g.bytes + extra;
            if (lane == 0) atom::mbar_arrive_expect_tx(&full[slot], ld_bytes * (uint32_t)nsrc);
            __syncwarp();
            for (int s = lane; s < nsrc; s += 32) {
                const char *base =
                    sg.src_rank < 0 ? static_cast<const char *>(p.src[s])
                                    : static_cast<const char *>(sg.src_is_dst ? p.dst[sg.src_rank]
                                                                              : p.src[sg.src_rank]);
                atom::bulk_load(sp + (size_t)s * tile, base + sg.src_off + g.off - lead, ld_bytes,
                                &full[slot], pol);
            }
        }
        // Every load this warp issued must land before the CTA exits.
        const uint32_t issued = k;
        if (lane == 0)
            for (uint32_t j = issued > S ? issued - S : 0; j < issued; ++j)
                ring_wait(&full[j % S], (j / S) & 1u, &ctl, p.err, kSiteRingFull, false);
    } else if (warp == 1) {
        // ------------------------- Consume (copy): write-back; Notify --
        // Lane d issues the bulk store to destination d; each lane tracks its
        // own bulk groups, and lane 0 hands a stage back once every lane's
        // stores have read it.
        // In a ragged plan the consumer warps store most chunks and this warp
        // mostly waits: it takes the segments' ragged head and tail windows
        // while the first stages load, and the consumer warps start on the
        // chunks at once.
        if (RAGGED) units_loop<DT, MAXR, true>(p, segs, (uint64_t)bidx * 32 + lane, (uint64_t)nblk * 32);
        const uint64_t pol = atom::policy_evict_first();
        uint32_t k = 0;
        int owed = -1;             // slot whose release waits on the newest bulk group
        uint64_t cd_phase = 0;     // per-slot phase bit of cdone (lane 0)
        // Chunks seen stored (cdone) whose flags are not yet published: one
        // GPU-scope fence covers a whole batch, off the stage-release path.
        uint64_t pend[kNotifyBatch];
        int npend = 0;
        auto publish = [&]() {
            if (lane == 0 && npend > 0) {
                atom::fence_acq_rel_gpu();   // the consumer warps' stores, at GPU scope
                for (int i = 0; i < npend; ++i) notify_chunk(p, flags, epoch, order, pend[i]);
            }
            npend = 0;
        };
        for (uint64_t pos = bidx; pos < p.nchunks; pos += nblk, ++k) {
            const uint64_t c = chunk_at(order, pos);
            const ChunkGeo g = chunk_geo(segs, p.nseg, c);
            const Seg &sg = *g.sg;
            const uint32_t slot = k % S;
            // Never wait on a chunk that depends on flags with flags of our own
            // still unpublished.
            if (sg.sync == kSyncWait) publish();
            if (sg.src_rank < 0 || sg.shift || p.vector_copies) {
                // A chunk the consumer warps store.  Settle the owed release
                // first (never hold a stage while waiting on another), pass
                // the chunk's full phase, then release it -- for a chunk others
                // wait on, once the consumer warps report it stored.
                atom::bulk_wait_read<0>();
                __syncwarp();
                bool ok = true;
                if (lane == 0) {
                    if (owed >= 0) atom::mbar_arrive(&empty[owed]);
                    ok = ring_wait(&full[slot], (k / S) & 1u, &ctl, p.err, kSiteRingFull, true);
                    if (ok) atom::mbar_arrive(&empty[slot]);
                    if (ok && sg.sync == kSyncNotify) {
                        const uint32_t e = k % C;
                        ok = ring_wait(&cdone[e], (uint32_t)(cd_phase >> e) & 1u, &ctl, p.err,
                                       kSiteChunkDone, true);
                        if (ok) {
                            cd_phase ^= 1ull << e;
                            pend[npend] = c;
                        }
                    }
                }
                owed = -1;
                if (!__shfl_sync(0xFFFFFFFFu, (int)ok, 0)) break;   // lane 0 decided
                if (sg.sync == kSyncNotify && ++npend == kNotifyBatch) publish();
                continue;
            }
            const bool ok = ring_wait(&full[slot], (k / S) & 1u, &ctl, p.err, kSiteRingFull, true);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            const unsigned char *from = ring + (size_t)slot * p.slot_stride;
            const char *self = static_cast<const char *>(sg.src_is_dst ? p.dst[sg.src_rank]
                                                                       : p.src[sg.src_rank]) +
                               sg.src_off + g.off;
            const uint64_t doff = sg.dst_off + g.off;
            if (sg.dst_rank >= 0) {
                char *d = static_cast<char *>(p.dst[sg.dst_rank]) + doff;
                if (lane == 0 && d != self) atom::bulk_store(d, from, g.bytes, pol);
            } else {
                for (int d = lane; d < R; d += 32) {
                    char *dp = static_cast<char *>(p.dst[d]) + doff;
                    if (d != sg.skip_rank && dp != self) atom::bulk_store(dp, from, g.bytes, pol);
                }
            }
            atom::bulk_commit();
            // The previous group has finished reading its stage: hand it back.
            atom::bulk_wait_read<1>();
            __syncwarp();
            if (lane == 0 && owed >= 0) atom::mbar_arrive(&empty[owed]);
            owed = (int)slot;
        }
        atom::bulk_wait_all<0>();
        atom::fence_async_global();   // the bulk stores, before generic accesses that follow
        __syncwarp();
        if (lane == 0 && owed >= 0) atom::mbar_arrive(&empty[owed]);
        publish();
    } else {
        // --------------------------------------------- Consume (reduce) --
        const int ctid = (int)threadIdx.x - 64;
        const int nct = (int)blockDim.x - 64;
        if (!RAGGED)
            units_loop<DT, MAXR, true>(p, segs, (uint64_t)bidx * nct + ctid, (uint64_t)nblk * nct);
        uint32_t k = 0;
        for (uint64_t pos = bidx; pos < p.nchunks; pos += nblk, ++k) {
            const uint64_t c = chunk_at(order, pos);
            const ChunkGeo g = chunk_geo(segs, p.nseg, c);
            const Seg &sg = *g.sg;
            const bool reduce = sg.src_rank < 0;
            const uint32_t slot = k % S;
            // Every lane waits (bounded) and the warp leaves together.
            const bool ok = ring_wait(&full[slot], (k / S) & 1u, &ctl, p.err, kSiteRingFull, true);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            if (!reduce && !sg.shift && !p.vector_copies) {   // the writer lane stores it
                __syncwarp();
                if (lane == 0) atom::mbar_arrive(&empty[slot]);
                continue;
            }
            const unsigned char *sp = ring + (size_t)slot * p.slot_stride;
            const uint32_t sh = reduce ? 0u : sg.shift;   // a copy's hull is shifted as it is read
            const uint32_t tile = sg.chunk_bytes + (sh ? 16u : 0u);
            const int nvec = (int)(g.bytes >> 4);
            const uint64_t doff = sg.dst_off + g.off;
            // in-place AllGather: the destination block that is the source itself
            const char *self =
                reduce ? nullptr
                       : static_cast<const char *>(sg.src_is_dst ? p.dst[sg.src_rank]
                                                                 : p.src[sg.src_rank]) +
                             sg.src_off + g.off;
            // 16 destination bytes of source tile s at vector v
            auto tile_v4 = [&](int s, int v) -> uint4 {
                const unsigned char *t = sp + (size_t)s * tile + 16 * (size_t)v;
                if (!sh) return atom::lds_v4(t);
                return atom::lds_v4_shifted(t, sh);
            };
            if (RAGGED && reduce && sg.shift) {
                // A reduce's body is aligned on the sources: its sums go to the
                // destination's phase.
                reduce_chunk_to_phase<DT, MAXR>(p, sg, sp, tile, nvec, doff, ctid, nct);
            } else if (RAGGED && sh) {
                // a copy's hull, shifted with the word offset fixed per loop
                const uint32_t r = (sh & 3u) * 8u;
                switch (sh >> 2) {
                    case 0: copy_chunk_shifted<0>(p, sg, sp, r, nvec, doff, self, ctid, nct); break;
                    case 1: copy_chunk_shifted<1>(p, sg, sp, r, nvec, doff, self, ctid, nct); break;
                    case 2: copy_chunk_shifted<2>(p, sg, sp, r, nvec, doff, self, ctid, nct); break;
                    default: copy_chunk_shifted<3>(p, sg, sp, r, nvec, doff, self, ctid, nct); break;
                }
            } else {
                for (int v = ctid; v < nvec; v += nct) {
                    uint4 out;
                    if (reduce) {
                        float acc[V::VE];
                        V::init(acc, tile_v4(0, v));
                        if (MAXR <= 8) {
#pragma unroll
                            for (int s = 1; s < MAXR; ++s)
                                if (s < R) V::add(acc, tile_v4(s, v));
                        } else {
#pragma unroll 8
                            for (int s = 1; s < R; ++s) V::add(acc, tile_v4(s, v));
                        }
                        out = V::pack(acc);
                    } else {
                        out = tile_v4(0, v);
                    }
                    const uint64_t o = doff + 16 * (uint64_t)v;
                    if (sg.dst_rank >= 0) {
                        if (static_cast<const char *>(p.dst[sg.dst_rank]) + doff != self)
                            atom::st_v4(static_cast<char *>(p.dst[sg.dst_rank]) + o, out);
                    } else {
                        for (int d = 0; d < R; ++d)
                            if (d != sg.skip_rank && static_cast<const char *>(p.dst[d]) + doff != self)
                                atom::st_v4(static_cast<char *>(p.dst[d]) + o, out);
                    }
                }
            }
            if (sg.sync == kSyncNotify) {
                // Others will read this chunk.  The stores are ordered before
                // the writer lane's publication by this mbarrier (release at
                // CTA scope), its wait (acquire), its GPU-scope fence and its
                // release-store: the pattern of a grid-wide barrier.
                __syncwarp();
                if (lane == 0) {
                    atom::mbar_arrive(&cdone[k % C]);
                    atom::mbar_arrive(&empty[slot]);
                }
            } else {
                __syncwarp();
                if (lane == 0) atom::mbar_arrive(&empty[slot]);
            }
        }
    }
    // Every role is done with the ring: retire its barriers so the caller
    // may reuse the workspace (another call, or its own data).
    __syncthreads();
    if (threadIdx.x == 0) {
        for (uint32_t i = 0; i < 2 * S; ++i) atom::mbar_inval(&bars[i]);
        for (uint32_t i = 0; i < C; ++i) atom::mbar_inval(&cdone[i]);
    }
    __syncthreads();
}

}  // namespace snac
}  // namespace purlin
