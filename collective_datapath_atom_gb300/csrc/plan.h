// plan.h -- the layout compiler's output: a list of contiguous transfers
// ("segments"), each cut into TMA chunks and 16-byte vector units.
//
// "Purlin: Separating Orchestration from the Datapath of Collectives",
// §3.1: a collective is named by its input layout, output layout and a copy
// or reduce operation; compatible transforms are composed into one kernel
// (AllReduce = ReduceScatter then AllGather, scattered -> scattered).
// §3.2: SNAC derives the dependencies between ranks from those layouts.
// Here a dependency exists only in the composed AllReduce, where the chunk a
// gathering CTA copies is the one a reducing CTA wrote and notified.
//
// This header is plain C++ (no CUDA types) and is shared by the host-side
// compiler and the kernels, which read the same struct from kernel
// parameters or device memory.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include "../../include/purlin.h"

#if defined(__CUDACC__)
#define PURLIN_HD __host__ __device__
#else
#define PURLIN_HD
#endif

namespace purlin {

constexpr int kRankAll = -1;

enum SyncKind : uint8_t {
    kSyncNone = 0,
    kSyncNotify = 1,   // release-store the chunk's flag once its stores completed
    kSyncWait = 2,     // acquire the producing chunk's flag before staging
};

enum Variant : int {
    kVariantNone = 0,
    kVariantLatency = 1,     // one-shot 128-bit vector loads/stores, a CTA per 256 windows
    kVariantThroughput = 2,  // persistent CTAs, cp.async.bulk shared-memory ring
};

// One contiguous transfer.  Offsets are bytes from the start of a rank
// buffer; every rank buffer is 16-byte aligned, so the 16-byte phase of an
// address is the phase of its offset.
struct Seg {
    uint64_t src_off;      // offset in src[src_rank] (or in every src, for a reduce)
    uint64_t dst_off;      // offset in dst[dst_rank] (or in every dst, for dst_rank -1)
    uint64_t bytes;        // bytes per source
    uint64_t unit_begin;   // global index of the segment's first vector unit
    uint32_t chunk_begin;  // global index of the segment's first TMA chunk
    uint32_t chunk_bytes;  // bytes per source per TMA chunk
    uint32_t dep_chunk;    // kSyncWait: global index of the notifying chunk for chunk 0
    uint8_t head;          // tma: bytes before the 16-byte aligned body
    uint8_t tail;          // tma: bytes after the body
    int8_t src_rank;       // >= 0 copy from that rank; -1 reduce over all ranks in order
    int8_t dst_rank;       // >= 0 that rank; -1 every rank (except skip_rank)
    int8_t skip_rank;      // with dst_rank -1: rank left out, or -1
    uint8_t src_is_dst;    // the source buffers are the destination buffers
    uint8_t sync;          // SyncKind
    uint8_t tma;           // the body goes through the TMA ring
    uint8_t shift;         // tma: 16-byte phase of the source relative to the destination
    uint8_t dep_ratio;     // kSyncWait: notifying chunks covered by one chunk of this segment
    uint8_t whole;         // vector path only: source and destination offsets and length are
                           // multiples of 16 (every unit a whole aligned window)
    uint8_t pad[1];
};
static_assert(sizeof(Seg) == 56, "Seg layout is part of the kernel parameter block");

// The offset whose 16-byte grid a segment's vector units follow.  A reduce
// reads every source at the same offset: on the sources' grid each source
// is one aligned 128-bit load and only the single sum is stored at another
// phase.  A copy reads one source: on the destination's grid that source is
// fetched (and shifted) once and every destination store is aligned.
PURLIN_HD inline uint64_t unit_grid(uint64_t src_off, uint64_t dst_off, bool reduce) {
    return reduce ? src_off : dst_off;
}

// The ring's cut of one transfer, on the 16-byte grid its vector units follow
// (unit_grid): the bytes before the grid's first boundary (head) and after
// its last (tail) go through the vector path; the aligned body goes through
// the ring in chunks.  shift is the source's 16-byte phase relative to the
// destination.  A copy's body is aligned on the destination: a shifted source
// is staged as its 16-byte aligned hull and shifted into place as it is read.
// A reduce's body is aligned on the sources: they are staged as they are,
// and the sum is stored at the destination's phase.  Used by the host plan
// compiler, the device-count kernel and the device-side Atom, so all cut a
// transfer the same way.
struct Cut {
    uint64_t body;
    uint32_t head, tail, shift;
};

PURLIN_HD inline Cut cut_transfer(uint64_t src_off, uint64_t dst_off, uint64_t bytes, bool reduce) {
    Cut c;
    const uint64_t grid = unit_grid(src_off, dst_off, reduce);
    const uint64_t lead = (16u - (grid & 15u)) & 15u;
    const uint64_t head = lead < bytes ? lead : bytes;
    const uint64_t rest = bytes - head;
    c.head = (uint32_t)head;
    c.tail = (uint32_t)(rest & 15u);
    c.body = rest - c.tail;
    c.shift = (uint32_t)((src_off - dst_off) & 15u);
    return c;
}

// The order in which a ring CTA takes its chunks (position pos of its walk
// -> chunk_at(order, pos)).  A composed AllReduce's plan numbers its reducing
// chunks [0, nr) (each notifies) before its gathering chunks [nr, nr + ng)
// (gathering chunk G waits on reducing chunks numbered below (G + 1) R).
// Taken in that order, every CTA runs a read-heavy phase and then a
// write-heavy one that starts on flags.  The walk instead puts gathering
// chunk G right after reducing chunk min(nr, (G + lag + 1) R) - 1: lag
// groups of R behind the chunks it depends on, enough for their flags to
// have gone out (a CTA publishes its flags in batches of up to `batch`
// chunks), and those chunks stay earlier in every CTA's walk (the launch is
// cooperative, so the earliest unfinished chunk can always proceed).  Other
// plans (ng == 0) keep their own order.  Chunk counts stay below 2^32.
struct ChunkOrder {
    uint32_t nr = 0;     // reducing chunks, numbered first
    uint32_t ng = 0;     // gathering chunks after them; 0: the plan's own order
    uint32_t g1 = 0;     // gathering chunks interleaved; the rest follow the last reducing chunk
    uint32_t base = 0;   // (lag + 1) R: the walk position of gathering chunk 0, when interleaved
    uint32_t R = 1;
};

PURLIN_HD inline ChunkOrder make_chunk_order(uint64_t nr, uint64_t ng, int R, uint32_t ctas,
                                             int batch) {
    ChunkOrder o;
    o.nr = (uint32_t)nr;
    o.ng = (uint32_t)ng;
    o.R = (uint32_t)R;
    uint32_t lag = (uint32_t)((uint64_t)(batch + 4) * ctas / ((uint64_t)R + 1u));
    lag = lag > 0 ? lag : 1u;
    // gathering chunk G is interleaved while (G + lag + 1) R < nr
    const uint32_t groups = (o.nr + o.R - 1) / o.R;
    const uint32_t g1 = groups > lag + 1 ? groups - lag - 1 : 0u;
    o.g1 = g1 < o.ng ? g1 : o.ng;
    o.base = (lag + 1) * o.R;
    return o;
}

// The chunk at position pos of the walk: gathering chunk G < g1 sits at
// position (R + 1) G + base, the others at nr + G, and the reducing chunks
// fill the other positions in their own order.
PURLIN_HD inline uint64_t chunk_at(const ChunkOrder &o, uint64_t pos64) {
    if (o.ng == 0) return pos64;
    const uint32_t pos = (uint32_t)pos64;
    if (pos >= o.nr + o.g1) return pos;   // gathering chunk pos - nr, numbered pos
    if (pos < o.base) return pos;         // before the first interleaved gathering chunk
    const uint32_t x = pos - o.base;
    const uint32_t q = x / (o.R + 1u);
    if (x == q * (o.R + 1u) && q < o.g1) return (uint64_t)o.nr + q;
    const uint32_t before = (x + o.R) / (o.R + 1u);   // gathering chunks placed earlier
    return pos - (before < o.g1 ? before : o.g1);      // (all g1, once ng < nr / R runs out)
}

// The walk position of reducing chunk d < nr: the inverse of chunk_at on the
// reducing chunks.  Before base they keep their own positions; after it each
// group of R follows one interleaved gathering chunk, until all g1 of them
// are placed.
PURLIN_HD inline uint64_t walk_pos(const ChunkOrder &o, uint64_t d) {
    if (o.ng == 0 || d < o.base) return d;
    const uint64_t q1 = (d - o.base) / o.R + 1u;   // gathering chunks placed before d
    return d + (q1 < o.g1 ? q1 : o.g1);
}

// The flag a notifying chunk d publishes (slot, generation), with F slots per
// parity.  When every notifying chunk has a slot of its own, slot = d.  When
// slots are reused (more than F notifying chunks), chunks are numbered by
// their walk position: F is a multiple of the grid, so position pos and
// pos + F belong to the same CTA, which publishes them in that order, and a
// slot's value only grows during a call.  Numbered by chunk instead, chunks d
// and d + F can sit on different CTAs under the interleaved walk, and a
// consumer of d could pass on d + F's flag before d is stored.  Every
// position of a call is below its chunk count, so ceil(nchunks / F)
// generations cover it.
struct FlagAt {
    uint64_t slot, gen;
};

PURLIN_HD inline FlagAt flag_at(const ChunkOrder &o, uint64_t F, uint64_t d) {
    const uint64_t i = o.nr <= F ? d : walk_pos(o, d);
    FlagAt f;
    f.slot = i % F;
    f.gen = i / F;
    return f;
}

// Vector units covering the bytes [grid + a, grid + b) of a segment whose
// units follow the 16-byte grid of offset `grid`: one unit per window.
PURLIN_HD inline uint64_t units_in(uint64_t grid, uint64_t a, uint64_t b) {
    if (b <= a) return 0;
    const uint64_t first = (grid + a) / 16;
    const uint64_t last = (grid + b + 15) / 16;
    return last - first;
}

struct Plan {
    std::vector<Seg> segs;
    uint64_t nchunks = 0;        // TMA chunks over all segments
    uint64_t nunits = 0;         // vector units over all segments
    uint64_t notify_chunks = 0;  // chunks that publish a flag (composed AllReduce)
    uint64_t total_bytes = 0;    // bytes per source over all segments
    uint64_t loose_bytes = 0;    // of those, bytes outside the TMA ring
    uint32_t slot_bytes = 0;     // largest shared-memory stage one chunk needs
    uint32_t red_chunk = 0;      // bytes per source per reduce chunk
    uint32_t copy_chunk = 0;     // bytes per copy chunk
    bool has_reduce = false;
    bool has_copy_chunks = false;
    bool has_shifted_copies = false;  // copies the consumer warps shift into place
    bool has_phase_reduce = false;    // reduce chunks stored at another 16-byte phase
    bool composed = false;
    int whole_op = 0;   // vector path, every segment of whole aligned 16-byte windows and
                        // all copies (1) or all reductions (2); 3: an AllToAll of R*R
                        // equal blocks of W windows in (source, destination) order and
                        // fewer than 2^32 units, whose unit u is window u % W of block
                        // u / W (no segment table needed); else 0
    int variant = kVariantNone;
};

// A plan with ring chunks at another 16-byte phase than their destination
// (reduce chunks stored at the destination's phase, or copies shifted into
// place): the ring kernel's RAGGED build runs it.
inline bool ragged_ring(const Plan &p) { return p.has_phase_reduce || p.has_shifted_copies; }

// Arguments of one call, as the C ABI received them.
struct CallDesc {
    purlin_collective coll;
    int R;
    int dtype;            // purlin_dtype
    size_t n;             // uniform collectives
    const size_t *counts; // R (AGV, RSV) or R*R (A2AV) entries, else null
    int op;               // purlin_op
    purlin_layout layout;
};

int elem_bytes(int dtype);

// Checks everything that can be checked without touching device memory:
// R, dtype, op, layout pair, divisibility, pointer nulls and alignment, and
// overlaps between the byte ranges of the buffers.
purlin_status validate_call(const CallDesc &c, const void *const src[], void *const dst[]);

// The two halves of validate_call.  validate_shape: R, dtype, op, layout
// pair and the array pointers.  validate_extents: pointer nulls and
// alignment, and overlaps, for the given byte extent of each buffer.
purlin_status validate_shape(const CallDesc &c, const void *const src[], void *const dst[]);
purlin_status validate_extents(const CallDesc &c, const void *const src[], void *const dst[],
                               const std::vector<uint64_t> &in_bytes,
                               const std::vector<uint64_t> &out_bytes);

// Byte lengths of each input and output buffer of a call (after validation
// of R and counts).
void buffer_bytes(const CallDesc &c, std::vector<uint64_t> &in_bytes,
                  std::vector<uint64_t> &out_bytes);

// Compile the layout of a (validated) call into segments and cut them for
// the given variant.  ar_mode: 0 auto, 1 fused, 2 composed.
// red_slot_bytes: shared memory for the R tiles of one reduce chunk;
// copy_chunk: bytes per copy chunk.
purlin_status compile_plan(const CallDesc &c, int variant, int ar_mode,
                           uint32_t red_slot_bytes, uint32_t copy_chunk, Plan *out);

// Total bytes every rank buffer must read plus write (the effective-bandwidth
// numerator of the benchmark).
uint64_t algorithmic_bytes(const CallDesc &c);

}  // namespace purlin
