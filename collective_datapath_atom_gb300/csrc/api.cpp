// api.cpp -- the C ABI declared in include/purlin.h.
//
// Host side of one call: validate (no partial work on error), compile the
// layout into a plan (cached by its key), pick the variant by message size
// (codesign policy, "Purlin: Separating Orchestration from the Datapath of Collectives"
// §4.2; push/latency vs pull/throughput,
// §3.2), size the launch (CTAs, ring depth: in-flight capacity near the
// bandwidth-delay product with few CTAs, §3.3), advance the epoch (§4.3)
// and enqueue one kernel.  Nothing here synchronises with the device
// except purlin_check, purlin_finalize and purlin_set_stream.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <list>
#include <new>
#include <string>
#include <unordered_map>

#include "launch.h"
#include "plan.h"

using namespace purlin;

namespace {

constexpr int kNumOptions = 12;
constexpr size_t kPlanCacheCap = 64;

// Built-in policy.
constexpr int64_t kInspectChunkBytes = 32 * 1024;        // plan_inspect default chunk
constexpr int64_t kDefaultTimeoutNs = 100 * 1000 * 1000; // 100 ms
constexpr int kLatBlock = 256;
constexpr int kCopyConsumerWarps = 4;
constexpr int kReduceConsumerWarps = 8;
constexpr int kShiftedCopyConsumerWarps = 6;

// Policy per collective (codesign policy, "Purlin: Separating Orchestration from the Datapath of Collectives"
// §4.2), measured on
// GB300 over 256 B..64 MiB per rank and at the workloads' sizes.
// Crossover: per-rank message bytes up to which the one-shot vector kernel
// beats the staged ring (it keeps ~150k threads' loads in flight, so for
// reductions it stays competitive up to several MiB).
// Ring shape:
//   ReduceScatter(V)  one destination per reduced chunk: large per-source
//                     chunks (96 KiB per stage), 2 stages;
//   AllReduce         R stores per reduced vector: 32 KiB per stage, 3 stages;
//   AllGather(V)      one staged tile written to R destinations: 16 KiB
//                     chunks, 4 stages, and the 8 consumer warps store the
//                     tile with 128-bit stores (0.956 of the copy peak versus
//                     0.92 with bulk stores from one warp);
//   AllToAll(V)       one load, one store per chunk: 16 KiB chunks, 3 stages,
//                     bulk stores (0.98).
struct Policy {
    uint32_t chunk;         // bytes per source per chunk
    uint32_t stages;
    uint64_t crossover;     // latency kernel at or below this many bytes per rank
    bool vector_copies;     // aligned copies stored by the consumer warps
    int consumer_warps;     // 0: by plan (8 with reductions or shifted copies, else 4)
};

Policy policy_for(purlin_collective coll, int R) {
    auto clamp16 = [](uint64_t v, uint64_t lo, uint64_t hi) {
        return (uint32_t)(std::min(hi, std::max(lo, v)) & ~uint64_t(15));
    };
    switch (coll) {
        case PURLIN_COLL_REDUCE_SCATTER:
        case PURLIN_COLL_REDUCE_SCATTER_V:
            return {clamp16(98304 / (uint64_t)R, 1024, 16384), 2, 8ull << 20, false, 0};
        case PURLIN_COLL_ALL_REDUCE:
            // (composed mode: the gather chunks are stored by the consumer warps)
            return {clamp16(32768 / (uint64_t)R, 512, 8192), 3, 8ull << 20, true, 0};
        case PURLIN_COLL_ALL_GATHER:
            return {16384, 4, 128ull << 10, true, 8};
        case PURLIN_COLL_ALL_GATHER_V:
            return {16384, 4, 1ull << 20, true, 8};
        default:
            return {16384, 3, 128ull << 10, false, 0};
    }
}

// Composed AllReduce (reducing CTAs notify, gathering CTAs wait): each
// gather chunk covers R reduce chunks and acquires R flags, so large chunks
// pay off: 96 KiB stages (12 KiB per source at R = 8), 2 stages, 12 consumer
// warps, one CTA per SM.  At 256 MiB per rank this measured 5.53 TB/s
// against 4.07 TB/s with the fused AllReduce's 4 KiB x 3-stage ring.
Policy composed_all_reduce_policy(int R) {
    const uint32_t chunk = (uint32_t)std::max<uint64_t>(512, (98304 / (uint64_t)R) & ~uint64_t(15));
    return {chunk, 2, 8ull << 20, true, 12};
}

// Device memory behind one purlin_device_coll.
struct DeviceCollMem {
    Seg *segs = nullptr;
    unsigned long long *flags = nullptr;
    unsigned long long *epochs = nullptr;
    unsigned long long *err = nullptr;
};

void free_device_coll(DeviceCollMem &m) {
    if (m.segs) cudaFree(m.segs);
    if (m.flags) cudaFree(m.flags);
    if (m.epochs) cudaFree(m.epochs);
    if (m.err) cudaFree(m.err);
    m = DeviceCollMem{};
}

struct CacheEntry {
    std::string key;
    Plan plan;
    Seg *segs_dev = nullptr;
    bool pinned = false;   // used while a CUDA graph was captured: kept until finalize
};

bool capturing(cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    return cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs != cudaStreamCaptureStatusNone;
}

int64_t env_or(const char *name, int64_t dflt) {
    const char *v = std::getenv(name);
    if (!v || !*v) return dflt;
    return std::strtoll(v, nullptr, 0);
}

}  // namespace

struct purlin_ctx {
    int R = 0;
    cudaStream_t stream = nullptr;
    int device = 0;
    int sms = 0;
    int max_smem = 0;
    unsigned long long *flags = nullptr;   // 2 x kFlagSlots
    unsigned char *packets = nullptr;      // 2 x kPacketStagingBytes (latency-path staging)
    unsigned long long *err = nullptr;     // 4 words: error word, pad, device epoch {epoch, done}
    unsigned long long *dev_epoch = nullptr;   // err + 2
    uint64_t epoch = 1;   // host count of the increments calls applied (reported in
                          // purlin_launch_info); the device epoch is the one kernels use
    int64_t opt[kNumOptions] = {};
    purlin_launch_info last = {};
    std::list<CacheEntry> lru;
    std::unordered_map<std::string, std::list<CacheEntry>::iterator> index;
    std::list<DeviceCollMem> device_colls;   // memory of purlin_device_prepare descriptors
};

namespace {

void append(std::string &k, const void *p, size_t n) { k.append(static_cast<const char *>(p), n); }

std::string plan_key(const CallDesc &c, int variant, int ar_mode, uint32_t red_slot,
                     uint32_t copy_chunk) {
    std::string k;
    int32_t hdr[5] = {(int32_t)c.coll, c.R, c.dtype, variant, ar_mode};
    append(k, hdr, sizeof hdr);
    uint32_t ch[2] = {red_slot, copy_chunk};
    append(k, ch, sizeof ch);
    uint64_t n = c.n;
    append(k, &n, sizeof n);
    if (c.counts) {
        size_t m = c.coll == PURLIN_COLL_ALL_TO_ALL_V ? (size_t)c.R * c.R : (size_t)c.R;
        append(k, c.counts, m * sizeof(size_t));
    }
    return k;
}

void drop_entry(CacheEntry &e) {
    if (e.segs_dev) cudaFree(e.segs_dev);   // synchronises the device: never on a hot path
    e.segs_dev = nullptr;
}

purlin_status get_plan(purlin_ctx *ctx, const CallDesc &c, int variant, int ar_mode,
                       uint32_t red_slot, uint32_t copy_chunk, CacheEntry **out) {
    std::string key = plan_key(c, variant, ar_mode, red_slot, copy_chunk);
    auto it = ctx->index.find(key);
    if (it != ctx->index.end()) {
        ctx->lru.splice(ctx->lru.begin(), ctx->lru, it->second);
        *out = &*ctx->lru.begin();
        return PURLIN_OK;
    }
    CacheEntry e;
    e.key = key;
    purlin_status st = compile_plan(c, variant, ar_mode, red_slot, copy_chunk, &e.plan);
    if (st != PURLIN_OK) return st;
    if (param_class(c.R, e.plan.segs.size()) != kClassSmall) {
        // An upload cannot be captured into a graph: the first call of such a
        // shape must come before capture.
        if (capturing(ctx->stream)) return PURLIN_ERR_UNSUPPORTED;
        // More segments than the small parameter block holds: the table
        // lives in device memory (uploaded once per cached plan) and the
        // kernels stage it into shared memory with coalesced loads.  A large
        // inline table would be read with divergent constant-cache accesses
        // and would lengthen every launch.  Uploaded from pageable memory,
        // which the runtime copies before returning.
        size_t bytes = e.plan.segs.size() * sizeof(Seg);
        if (cudaMalloc(&e.segs_dev, bytes) != cudaSuccess) return PURLIN_ERR_OOM;
        if (cudaMemcpyAsync(e.segs_dev, e.plan.segs.data(), bytes, cudaMemcpyHostToDevice,
                            ctx->stream) != cudaSuccess) {
            cudaFree(e.segs_dev);
            return PURLIN_ERR_CUDA;
        }
    }
    ctx->lru.push_front(std::move(e));
    ctx->index[key] = ctx->lru.begin();
    // Evict the least recently used plans past the cap, but never one that a
    // captured graph may still launch (its device table address is frozen in
    // the graph).
    auto it2 = ctx->lru.end();
    size_t unpinned_over = ctx->lru.size() > kPlanCacheCap ? ctx->lru.size() - kPlanCacheCap : 0;
    while (unpinned_over > 0 && it2 != ctx->lru.begin()) {
        --it2;
        if (it2->pinned) continue;
        drop_entry(*it2);
        ctx->index.erase(it2->key);
        it2 = ctx->lru.erase(it2);
        --unpinned_over;
    }
    *out = &*ctx->lru.begin();
    return PURLIN_OK;
}

uint64_t message_bytes(const CallDesc &c) {
    std::vector<uint64_t> in_b, out_b;
    buffer_bytes(c, in_b, out_b);
    uint64_t m = 0;
    for (int r = 0; r < c.R; ++r) m = std::max(m, in_b[r]);
    return m;
}

// Ring shape of a throughput launch: stages (reduced until the shared
// memory fits `limit`), stage stride, consumer warps and copy stores.
struct RingShape {
    uint32_t stages = 0;
    uint32_t slot_stride = 0;
    uint32_t smem = 0;
    int consumer_warps = 0;
    bool vector_copies = false;
};

purlin_status ring_shape(const purlin_ctx *ctx, const CallDesc &c, const Policy &shape,
                         const Plan &pl, uint32_t limit, RingShape *out) {
    RingShape r;
    r.slot_stride = (pl.slot_bytes + 127u) & ~127u;
    // Point-to-point copies at other 16-byte phases (ragged AllToAllV) go
    // through the consumer warps: 6 warps and a deeper ring keep two CTAs
    // per SM (measured +35% over 8 warps).
    const bool shifted_p2p = pl.has_shifted_copies && !shape.vector_copies &&
                             (c.coll == PURLIN_COLL_ALL_TO_ALL ||
                              c.coll == PURLIN_COLL_ALL_TO_ALL_V);
    uint32_t stages = (uint32_t)(ctx->opt[PURLIN_OPT_STAGES] > 0 ? ctx->opt[PURLIN_OPT_STAGES]
                                 : shifted_p2p ? 4u : shape.stages);
    stages = std::min<uint32_t>(32, std::max<uint32_t>(2, stages));
    while (stages > 2 && throughput_smem(stages, r.slot_stride) > limit) --stages;
    r.stages = stages;
    r.smem = throughput_smem(stages, r.slot_stride);
    if (r.smem > limit) return PURLIN_ERR_UNSUPPORTED;
    r.vector_copies = ctx->opt[PURLIN_OPT_COPY_STORES] == 0 ? shape.vector_copies
                                                            : ctx->opt[PURLIN_OPT_COPY_STORES] == 2;
    r.consumer_warps = ctx->opt[PURLIN_OPT_CONSUMER_WARPS] > 0
                           ? (int)ctx->opt[PURLIN_OPT_CONSUMER_WARPS]
                       : shape.consumer_warps > 0 ? shape.consumer_warps
                       : shifted_p2p ? kShiftedCopyConsumerWarps
                       : pl.has_reduce || pl.has_shifted_copies ? kReduceConsumerWarps
                                                                : kCopyConsumerWarps;
    *out = r;
    return PURLIN_OK;
}

// Per-parity flag slots for a grid of `grid` CTAs (a multiple of the grid,
// so a slot is always reused by the CTA that owns its chunks) and the odd
// epoch increment that keeps every generation of a call distinct.
void flag_geometry(uint64_t notify_chunks, int64_t grid, uint32_t *slots, uint64_t *epoch_inc) {
    *slots = (kFlagSlots / (uint32_t)grid) * (uint32_t)grid;
    uint64_t gens = (notify_chunks + *slots - 1) / *slots;
    if (gens == 0) gens = 1;
    *epoch_inc = gens | 1ull;   // odd: the parity flips every call
}

// AllReduce mode for the ring: the packet mode (3) runs the ring's composed
// mode where packets do not apply.
int ring_ar_mode(const purlin_ctx *ctx) {
    const int m = (int)ctx->opt[PURLIN_OPT_AR_MODE];
    return m == 3 ? 2 : m;
}

Policy call_policy(const purlin_ctx *ctx, const CallDesc &c) {
    return c.coll == PURLIN_COLL_ALL_REDUCE && ring_ar_mode(ctx) == 2
               ? composed_all_reduce_policy(c.R)
               : policy_for(c.coll, c.R);
}

purlin_status run_packets(purlin_ctx *ctx, const CallDesc &c, const void *const src[],
                          void *const dst[], uint64_t nbytes) {
    PktLaunch a;
    a.src = src;
    a.dst = dst;
    a.staging = ctx->packets;
    a.dev_epoch = ctx->dev_epoch;
    a.err = ctx->err;
    a.nbytes = nbytes;
    a.timeout_ns = ctx->opt[PURLIN_OPT_SPIN_TIMEOUT_NS] > 0 ? ctx->opt[PURLIN_OPT_SPIN_TIMEOUT_NS]
                                                            : kDefaultTimeoutNs;
    a.drop_unit = ctx->opt[PURLIN_OPT_DROP_NOTIFY];
    a.R = c.R;
    a.dtype = c.dtype;
    a.stream = ctx->stream;
    const uint64_t units = (nbytes + 7) / 8;
    const uint64_t per = (uint64_t)packet_threads();
    a.G = (int)std::max<uint64_t>(1, std::min<uint64_t>((units + per - 1) / per, (uint64_t)ctx->sms));
    if (launch_packet_all_reduce(a) != cudaSuccess) return PURLIN_ERR_CUDA;
    purlin_launch_info info = {};
    info.variant = 5;
    info.grid = 2 * a.G;
    info.block = (int32_t)per;
    info.units = (int64_t)units;
    info.epoch = ctx->epoch;
    ctx->epoch += 1;   // odd: the parity (staging buffer) flips every call
    info.epoch_next = ctx->epoch;
    ctx->last = info;
    return PURLIN_OK;
}

purlin_status run(purlin_ctx *ctx, const CallDesc &c, const void *const src[], void *const dst[]) {
    if (ctx == nullptr) return PURLIN_ERR_INVALID_ARG;
    if (c.R != ctx->R) return PURLIN_ERR_INVALID_ARG;
    purlin_status st = validate_call(c, src, dst);
    if (st != PURLIN_OK) return st;

    // ---- composed AllReduce on the latency path: packets (§3.2, §4.1)
    int ar_mode = (int)ctx->opt[PURLIN_OPT_AR_MODE];
    if (c.coll == PURLIN_COLL_ALL_REDUCE && ar_mode == 3) {
        const uint64_t nbytes = (uint64_t)c.n * (uint64_t)elem_bytes(c.dtype);
        if (nbytes > 0 && c.R > 1 && nbytes <= kPacketPayloadBytes)
            return run_packets(ctx, c, src, dst, nbytes);
        ar_mode = 2;   // past the staging buffer: the ring's composed mode
    }

    // ---- policy (§4.2)
    const Policy shape = ar_mode == 2 && c.coll == PURLIN_COLL_ALL_REDUCE
                             ? composed_all_reduce_policy(c.R)
                             : policy_for(c.coll, c.R);
    int variant = (int)ctx->opt[PURLIN_OPT_VARIANT];
    if (variant == 0) {
        const uint64_t xo = ctx->opt[PURLIN_OPT_CROSSOVER_BYTES] > 0
                                ? (uint64_t)ctx->opt[PURLIN_OPT_CROSSOVER_BYTES]
                                : shape.crossover;
        variant = message_bytes(c) <= xo ? kVariantLatency : kVariantThroughput;
    }
    const int64_t chunk_opt = ctx->opt[PURLIN_OPT_CHUNK_BYTES];
    // CHUNK_BYTES is bytes per source per chunk: a reduce stage holds R of them.
    const uint32_t chunk = (uint32_t)(chunk_opt > 0 ? chunk_opt : shape.chunk);
    const uint32_t copy_chunk = chunk;
    const uint32_t red_slot = chunk * (uint32_t)c.R;

    CacheEntry *e = nullptr;
    st = get_plan(ctx, c, variant, ar_mode, red_slot, copy_chunk, &e);
    if (st != PURLIN_OK) return st;
    if (ctx->opt[PURLIN_OPT_VARIANT] == 0 && variant == kVariantThroughput &&
        2 * e->plan.loose_bytes > e->plan.total_bytes) {
        // Most bytes sit at 16-byte phases the ring cannot move (ragged V
        // counts): the vector kernel, with every thread shifting, is faster.
        variant = kVariantLatency;
        st = get_plan(ctx, c, variant, ar_mode, red_slot, copy_chunk, &e);
        if (st != PURLIN_OK) return st;
    }
    const Plan &pl = e->plan;
    if (e->segs_dev != nullptr && !e->pinned && capturing(ctx->stream)) e->pinned = true;

    purlin_launch_info info = {};
    info.segments = (int64_t)pl.segs.size();
    info.chunks = (int64_t)pl.nchunks;
    info.units = (int64_t)pl.nunits;
    info.epoch = ctx->epoch;
    if (pl.nchunks == 0 && pl.nunits == 0) {   // nothing to move
        info.variant = kVariantNone;
        info.epoch_next = ctx->epoch;
        ctx->last = info;
        return PURLIN_OK;
    }

    LaunchArgs a;
    a.plan = &pl;
    a.segs_dev = e->segs_dev;
    a.src = src;
    a.dst = dst;
    a.R = c.R;
    a.dtype = c.dtype;
    a.err = ctx->err;
    a.timeout_ns = ctx->opt[PURLIN_OPT_SPIN_TIMEOUT_NS] > 0 ? ctx->opt[PURLIN_OPT_SPIN_TIMEOUT_NS]
                                                            : kDefaultTimeoutNs;
    a.drop_notify = ctx->opt[PURLIN_OPT_DROP_NOTIFY];
    a.stream = ctx->stream;
    a.flags = ctx->flags;   // both parities; the device epoch selects one

    uint64_t epoch_inc = 1;
    cudaError_t ce;
    if (variant == kVariantLatency) {
        const int64_t cap = ctx->opt[PURLIN_OPT_LAT_CTAS] > 0 ? ctx->opt[PURLIN_OPT_LAT_CTAS]
                                                              : 4 * (int64_t)ctx->sms;
        const int max_block = ctx->opt[PURLIN_OPT_LAT_BLOCK] > 0
                                  ? (int)ctx->opt[PURLIN_OPT_LAT_BLOCK] : kLatBlock;
        int block = (int)std::min<uint64_t>(max_block, (pl.nunits + 31) / 32 * 32);
        uint64_t want = (pl.nunits + block - 1) / block;
        a.block = block;
        a.grid = (int)std::max<uint64_t>(1, std::min<uint64_t>(want, (uint64_t)cap));
        info.variant = kVariantLatency;
        ce = launch_latency(a);
    } else {
        RingShape rs;
        st = ring_shape(ctx, c, shape, pl, (uint32_t)ctx->max_smem - 1024, &rs);
        if (st != PURLIN_OK) return st;
        const uint32_t stages = rs.stages, slot_stride = rs.slot_stride, smem = rs.smem;
        const bool vector_copies = rs.vector_copies;
        const int block = 32 * (2 + rs.consumer_warps);
        const int pclass = launch_class(c.R, pl.segs.size(), e->segs_dev != nullptr);
        int per_sm = 0;
        if (throughput_occupancy(c.dtype, pclass, block, smem, &per_sm) != cudaSuccess ||
            per_sm < 1)
            return PURLIN_ERR_UNSUPPORTED;
        int64_t grid = (int64_t)ctx->sms * per_sm;
        if (ctx->opt[PURLIN_OPT_CTAS] > 0) grid = std::min<int64_t>(grid, ctx->opt[PURLIN_OPT_CTAS]);
        int64_t work = (int64_t)std::max<uint64_t>(pl.nchunks, (pl.nunits + 255) / 256);
        grid = std::max<int64_t>(1, std::min<int64_t>(grid, work));
        a.grid = (int)grid;
        a.block = block;
        a.smem = smem;
        a.stages = stages;
        a.slot_stride = slot_stride;
        a.cooperative = pl.composed;
        a.vector_copies = vector_copies;
        if (pl.composed) {
            // flag slot reuse stays on one CTA (slots a multiple of the grid),
            // so a later generation of a slot implies the earlier one landed.
            flag_geometry(pl.notify_chunks, grid, &a.flag_slots, &epoch_inc);
            a.dev_epoch = ctx->dev_epoch;
            a.epoch_inc = epoch_inc;
        }
        info.variant = pl.composed ? 3 : kVariantThroughput;
        info.stages = (int32_t)stages;
        info.smem_bytes = smem;
        info.chunk_bytes = pl.has_reduce ? pl.red_chunk : pl.copy_chunk;
        ce = launch_throughput(a);
    }
    if (ce != cudaSuccess) return PURLIN_ERR_CUDA;
    info.grid = a.grid;
    info.block = a.block;
    ctx->epoch += epoch_inc;
    info.epoch_next = ctx->epoch;
    ctx->last = info;
    return PURLIN_OK;
}

// A V collective whose counts are in device memory (vcounts.cu): the host
// checks what it can (shape, pointers, the declared capacities' overlaps)
// and sizes the ring for the worst case of any counts; the kernel derives
// the displacements and checks the counts against the capacities.
purlin_status run_vcounts(purlin_ctx *ctx, purlin_collective coll, const void *const src[],
                          void *const dst[], const size_t *d_counts, size_t in_cap,
                          size_t out_cap, int dtype, int op, purlin_layout layout) {
    if (ctx == nullptr) return PURLIN_ERR_INVALID_ARG;
    CallDesc c;
    c.coll = coll;
    c.R = ctx->R;
    c.dtype = dtype;
    c.n = 0;
    c.counts = nullptr;
    c.op = op;
    c.layout = layout;
    purlin_status st = validate_shape(c, src, dst);
    if (st != PURLIN_OK) return st;
    if (c.R > kVcMaxRanks) return PURLIN_ERR_UNSUPPORTED;
    if (d_counts == nullptr || ((uintptr_t)d_counts & 7u) != 0) return PURLIN_ERR_INVALID_ARG;
    const uint64_t es = (uint64_t)elem_bytes(dtype);
    if (in_cap > (1ull << 44) || out_cap > (1ull << 44)) return PURLIN_ERR_INVALID_ARG;
    std::vector<uint64_t> in_b((size_t)c.R, in_cap * es), out_b((size_t)c.R, out_cap * es);
    st = validate_extents(c, src, dst, in_b, out_b);
    if (st != PURLIN_OK) return st;

    const Policy shape = policy_for(coll, c.R);
    const int64_t chunk_opt = ctx->opt[PURLIN_OPT_CHUNK_BYTES];
    const uint32_t chunk = (uint32_t)(chunk_opt > 0 ? chunk_opt : shape.chunk) & ~15u;
    const bool reduce = coll == PURLIN_COLL_REDUCE_SCATTER_V;
    // Any count may put a source at another 16-byte phase: room for the hull.
    const uint32_t slot = reduce ? (chunk + 16u) * (uint32_t)c.R : chunk + 16u;
    const uint32_t slot_stride = (slot + 127u) & ~127u;
    // AllToAllV: 3 stages and 6 consumer warps (two CTAs per SM) measured
    // best for both 16-byte aligned counts (the MoE dispatch: equal to the
    // host-count call) and ragged ones (Zipf V split: 4% faster than it).
    uint32_t stages = (uint32_t)(ctx->opt[PURLIN_OPT_STAGES] > 0 ? ctx->opt[PURLIN_OPT_STAGES]
                                                                 : shape.stages);
    stages = std::min<uint32_t>(32, std::max<uint32_t>(2, stages));
    const uint32_t limit = (uint32_t)ctx->max_smem - 1024;
    while (stages > 2 && vcounts_smem(coll, c.R, stages, slot_stride) > limit) --stages;
    const uint32_t smem = vcounts_smem(coll, c.R, stages, slot_stride);
    if (smem > limit) return PURLIN_ERR_UNSUPPORTED;
    const int cw = ctx->opt[PURLIN_OPT_CONSUMER_WARPS] > 0 ? (int)ctx->opt[PURLIN_OPT_CONSUMER_WARPS]
                   : shape.consumer_warps > 0 ? shape.consumer_warps
                   : coll == PURLIN_COLL_ALL_TO_ALL_V ? kShiftedCopyConsumerWarps
                                                      : kReduceConsumerWarps;
    const int block = 32 * (2 + cw);
    int per_sm = 0;
    if (vcounts_occupancy(dtype, c.R, block, smem, &per_sm) != cudaSuccess || per_sm < 1)
        return PURLIN_ERR_UNSUPPORTED;

    VcLaunch a;
    a.src = src;
    a.dst = dst;
    a.counts = reinterpret_cast<const unsigned long long *>(d_counts);
    a.err = ctx->err;
    a.in_cap = in_cap;
    a.out_cap = out_cap;
    const int64_t variant = ctx->opt[PURLIN_OPT_VARIANT];
    a.crossover = variant == kVariantLatency      ? ~0ull
                  : variant == kVariantThroughput ? 0ull
                  : ctx->opt[PURLIN_OPT_CROSSOVER_BYTES] > 0
                      ? (uint64_t)ctx->opt[PURLIN_OPT_CROSSOVER_BYTES]
                      : shape.crossover;
    a.timeout_ns = ctx->opt[PURLIN_OPT_SPIN_TIMEOUT_NS] > 0 ? ctx->opt[PURLIN_OPT_SPIN_TIMEOUT_NS]
                                                            : kDefaultTimeoutNs;
    a.red_chunk = chunk;
    a.copy_chunk = chunk;
    a.stages = stages;
    a.slot_stride = slot_stride;
    a.R = c.R;
    a.coll = coll;
    a.dtype = dtype;
    a.vector_copies = ctx->opt[PURLIN_OPT_COPY_STORES] == 0 ? shape.vector_copies
                                                            : ctx->opt[PURLIN_OPT_COPY_STORES] == 2;
    int64_t grid = (int64_t)ctx->sms * per_sm;
    if (ctx->opt[PURLIN_OPT_CTAS] > 0) grid = std::min<int64_t>(grid, ctx->opt[PURLIN_OPT_CTAS]);
    a.grid = (int)grid;
    a.block = block;
    a.smem = smem;
    a.stream = ctx->stream;
    if (launch_vcounts(a) != cudaSuccess) return PURLIN_ERR_CUDA;
    purlin_launch_info info = {};
    info.variant = 4;   // decided on the device from the counts
    info.grid = a.grid;
    info.block = a.block;
    info.stages = (int32_t)stages;
    info.chunk_bytes = chunk;
    info.segments = coll == PURLIN_COLL_ALL_TO_ALL_V ? (int64_t)c.R * c.R : c.R;
    info.smem_bytes = smem;
    info.epoch = info.epoch_next = ctx->epoch;
    ctx->last = info;
    return PURLIN_OK;
}

CallDesc make_desc(purlin_collective coll, int R, size_t n, const size_t *counts, int dtype,
                   int op, purlin_layout layout) {
    CallDesc c;
    c.coll = coll;
    c.R = R;
    c.dtype = dtype;
    c.n = n;
    c.counts = counts;
    c.op = op;
    c.layout = layout;
    return c;
}

}  // namespace

extern "C" {

purlin_status purlin_init(int R, purlin_stream stream, purlin_ctx **out) {
    if (out == nullptr) return PURLIN_ERR_INVALID_ARG;
    *out = nullptr;
    if (R < 1 || R > PURLIN_MAX_RANKS) return PURLIN_ERR_INVALID_ARG;
    purlin_ctx *ctx = new (std::nothrow) purlin_ctx();
    if (!ctx) return PURLIN_ERR_OOM;
    ctx->R = R;
    ctx->stream = static_cast<cudaStream_t>(stream);
    for (int i = 0; i < kNumOptions; ++i) ctx->opt[i] = 0;
    ctx->opt[PURLIN_OPT_DROP_NOTIFY] = -1;
    ctx->opt[PURLIN_OPT_VARIANT] = env_or("PURLIN_VARIANT", 0);
    ctx->opt[PURLIN_OPT_CROSSOVER_BYTES] = env_or("PURLIN_CROSSOVER_BYTES", 0);
    ctx->opt[PURLIN_OPT_STAGES] = env_or("PURLIN_STAGES", 0);
    ctx->opt[PURLIN_OPT_CHUNK_BYTES] = env_or("PURLIN_CHUNK_BYTES", 0);
    ctx->opt[PURLIN_OPT_CTAS] = env_or("PURLIN_CTAS", 0);
    ctx->opt[PURLIN_OPT_AR_MODE] = env_or("PURLIN_AR_MODE", 0);
    auto fail = [&](purlin_status s) {
        if (ctx->flags) cudaFree(ctx->flags);
        if (ctx->packets) cudaFree(ctx->packets);
        if (ctx->err) cudaFree(ctx->err);
        delete ctx;
        return s;
    };
    if (cudaGetDevice(&ctx->device) != cudaSuccess) return fail(PURLIN_ERR_CUDA);
    if (cudaDeviceGetAttribute(&ctx->sms, cudaDevAttrMultiProcessorCount, ctx->device) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&ctx->max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                               ctx->device) != cudaSuccess)
        return fail(PURLIN_ERR_CUDA);
    if (configure_kernels(ctx->max_smem - 1024) != cudaSuccess ||
        configure_vcounts(ctx->max_smem - 1024) != cudaSuccess)
        return fail(PURLIN_ERR_CUDA);
    if (cudaMalloc(&ctx->flags, 2 * (size_t)kFlagSlots * sizeof(unsigned long long)) !=
            cudaSuccess ||
        cudaMalloc(&ctx->packets, 2 * kPacketStagingBytes) != cudaSuccess ||
        cudaMalloc(&ctx->err, 4 * sizeof(unsigned long long)) != cudaSuccess)
        return fail(PURLIN_ERR_OOM);
    ctx->dev_epoch = ctx->err + 2;
    if (cudaMemsetAsync(ctx->packets, 0, 2 * kPacketStagingBytes, ctx->stream) != cudaSuccess)
        return fail(PURLIN_ERR_CUDA);
    if (cudaMemsetAsync(ctx->flags, 0, 2 * (size_t)kFlagSlots * sizeof(unsigned long long),
                        ctx->stream) != cudaSuccess ||
        cudaMemsetAsync(ctx->err, 0, 4 * sizeof(unsigned long long), ctx->stream) != cudaSuccess)
        return fail(PURLIN_ERR_CUDA);
    // the device epoch starts at 1 (flags start at 0, below any epoch)
    static const unsigned long long kFirstEpoch = 1;
    if (cudaMemcpyAsync(ctx->dev_epoch, &kFirstEpoch, sizeof kFirstEpoch, cudaMemcpyHostToDevice,
                        ctx->stream) != cudaSuccess ||
        cudaStreamSynchronize(ctx->stream) != cudaSuccess)
        return fail(PURLIN_ERR_CUDA);
    ctx->epoch = 1;
    *out = ctx;
    return PURLIN_OK;
}

purlin_status purlin_finalize(purlin_ctx *ctx) {
    if (ctx == nullptr) return PURLIN_OK;
    purlin_status st = PURLIN_OK;
    if (cudaStreamSynchronize(ctx->stream) != cudaSuccess) st = PURLIN_ERR_CUDA;
    for (CacheEntry &e : ctx->lru) drop_entry(e);
    for (DeviceCollMem &m : ctx->device_colls) free_device_coll(m);
    if (ctx->flags) cudaFree(ctx->flags);
    if (ctx->packets) cudaFree(ctx->packets);
    if (ctx->err) cudaFree(ctx->err);
    delete ctx;
    return st;
}

purlin_status purlin_set_stream(purlin_ctx *ctx, purlin_stream stream) {
    if (ctx == nullptr) return PURLIN_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(ctx->stream) != cudaSuccess) return PURLIN_ERR_CUDA;
    ctx->stream = static_cast<cudaStream_t>(stream);
    return PURLIN_OK;
}

purlin_status purlin_all_reduce(purlin_ctx *ctx, const void *const src[], void *const dst[],
                                size_t n, purlin_dtype dtype, purlin_op op, purlin_layout layout) {
    return run(ctx, make_desc(PURLIN_COLL_ALL_REDUCE, ctx ? ctx->R : 0, n, nullptr, dtype, op,
                              layout),
               src, dst);
}

purlin_status purlin_reduce_scatter(purlin_ctx *ctx, const void *const src[], void *const dst[],
                                    size_t n, purlin_dtype dtype, purlin_op op,
                                    purlin_layout layout) {
    return run(ctx, make_desc(PURLIN_COLL_REDUCE_SCATTER, ctx ? ctx->R : 0, n, nullptr, dtype, op,
                              layout),
               src, dst);
}

purlin_status purlin_all_gather(purlin_ctx *ctx, const void *const src[], void *const dst[],
                                size_t n, purlin_dtype dtype, purlin_op op, purlin_layout layout) {
    return run(ctx, make_desc(PURLIN_COLL_ALL_GATHER, ctx ? ctx->R : 0, n, nullptr, dtype, op,
                              layout),
               src, dst);
}

purlin_status purlin_all_to_all(purlin_ctx *ctx, const void *const src[], void *const dst[],
                                size_t n, purlin_dtype dtype, purlin_op op, purlin_layout layout) {
    return run(ctx, make_desc(PURLIN_COLL_ALL_TO_ALL, ctx ? ctx->R : 0, n, nullptr, dtype, op,
                              layout),
               src, dst);
}

purlin_status purlin_all_gather_v(purlin_ctx *ctx, const void *const src[], void *const dst[],
                                  const size_t counts[], purlin_dtype dtype, purlin_op op,
                                  purlin_layout layout) {
    return run(ctx, make_desc(PURLIN_COLL_ALL_GATHER_V, ctx ? ctx->R : 0, 0, counts, dtype, op,
                              layout),
               src, dst);
}

purlin_status purlin_reduce_scatter_v(purlin_ctx *ctx, const void *const src[],
                                      void *const dst[], const size_t counts[],
                                      purlin_dtype dtype, purlin_op op, purlin_layout layout) {
    return run(ctx, make_desc(PURLIN_COLL_REDUCE_SCATTER_V, ctx ? ctx->R : 0, 0, counts, dtype,
                              op, layout),
               src, dst);
}

purlin_status purlin_all_to_all_v(purlin_ctx *ctx, const void *const src[], void *const dst[],
                                  const size_t counts[], purlin_dtype dtype, purlin_op op,
                                  purlin_layout layout) {
    return run(ctx, make_desc(PURLIN_COLL_ALL_TO_ALL_V, ctx ? ctx->R : 0, 0, counts, dtype, op,
                              layout),
               src, dst);
}

purlin_status purlin_all_gather_v_device_counts(purlin_ctx *ctx, const void *const src[],
                                                void *const dst[], const size_t counts[],
                                                size_t in_capacity, size_t out_capacity,
                                                purlin_dtype dtype, purlin_op op,
                                                purlin_layout layout) {
    return run_vcounts(ctx, PURLIN_COLL_ALL_GATHER_V, src, dst, counts, in_capacity,
                       out_capacity, dtype, op, layout);
}

purlin_status purlin_reduce_scatter_v_device_counts(purlin_ctx *ctx, const void *const src[],
                                                    void *const dst[], const size_t counts[],
                                                    size_t in_capacity, size_t out_capacity,
                                                    purlin_dtype dtype, purlin_op op,
                                                    purlin_layout layout) {
    return run_vcounts(ctx, PURLIN_COLL_REDUCE_SCATTER_V, src, dst, counts, in_capacity,
                       out_capacity, dtype, op, layout);
}

purlin_status purlin_all_to_all_v_device_counts(purlin_ctx *ctx, const void *const src[],
                                                void *const dst[], const size_t counts[],
                                                size_t in_capacity, size_t out_capacity,
                                                purlin_dtype dtype, purlin_op op,
                                                purlin_layout layout) {
    return run_vcounts(ctx, PURLIN_COLL_ALL_TO_ALL_V, src, dst, counts, in_capacity,
                       out_capacity, dtype, op, layout);
}

purlin_status purlin_empty_launch(purlin_stream stream) {
    return launch_empty(static_cast<cudaStream_t>(stream)) == cudaSuccess ? PURLIN_OK
                                                                          : PURLIN_ERR_CUDA;
}

purlin_status purlin_check(purlin_ctx *ctx) {
    if (ctx == nullptr) return PURLIN_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(ctx->stream) != cudaSuccess) return PURLIN_ERR_CUDA;
    unsigned long long word = 0;
    if (cudaMemcpy(&word, ctx->err, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return PURLIN_ERR_CUDA;
    if (word == 0) return PURLIN_OK;
    if (cudaMemset(ctx->err, 0, sizeof word) != cudaSuccess) return PURLIN_ERR_CUDA;
    return static_cast<purlin_status>(word & 0xFF);
}

const char *purlin_status_string(purlin_status s) {
    switch (s) {
        case PURLIN_OK: return "ok";
        case PURLIN_ERR_INVALID_ARG: return "invalid argument";
        case PURLIN_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
        case PURLIN_ERR_UNSUPPORTED: return "unsupported op, layout or configuration";
        case PURLIN_ERR_ALIAS: return "forbidden overlap between buffers";
        case PURLIN_ERR_OOM: return "out of memory";
        case PURLIN_ERR_CUDA: return "CUDA runtime error";
        case PURLIN_ERR_TIMEOUT: return "bounded device wait expired";
    }
    return "unknown status";
}

purlin_status purlin_set_option(purlin_ctx *ctx, purlin_option opt, int64_t value) {
    if (ctx == nullptr || (int)opt < 0 || (int)opt >= kNumOptions) return PURLIN_ERR_INVALID_ARG;
    switch (opt) {
        case PURLIN_OPT_VARIANT:
            if (value < 0 || value > 2) return PURLIN_ERR_INVALID_ARG;
            break;
        case PURLIN_OPT_AR_MODE:
            if (value < 0 || value > 3) return PURLIN_ERR_INVALID_ARG;
            break;
        case PURLIN_OPT_CHUNK_BYTES:
            if (value < 0 || (value > 0 && (value < 16 || value % 16 != 0 || value > (1 << 20))))
                return PURLIN_ERR_INVALID_ARG;
            break;
        case PURLIN_OPT_STAGES:
            if (value < 0 || value == 1 || value > 32) return PURLIN_ERR_INVALID_ARG;
            break;
        case PURLIN_OPT_DROP_NOTIFY:
            if (value < -1) return PURLIN_ERR_INVALID_ARG;
            break;
        case PURLIN_OPT_LAT_BLOCK:
            if (value < 0 || value > 256 || value % 32 != 0) return PURLIN_ERR_INVALID_ARG;
            break;
        case PURLIN_OPT_CONSUMER_WARPS:
            if (value < 0 || value > 14) return PURLIN_ERR_INVALID_ARG;
            break;
        case PURLIN_OPT_COPY_STORES:
            if (value < 0 || value > 2) return PURLIN_ERR_INVALID_ARG;
            break;
        default:
            if (value < 0) return PURLIN_ERR_INVALID_ARG;
    }
    ctx->opt[opt] = value;
    return PURLIN_OK;
}

purlin_status purlin_get_option(purlin_ctx *ctx, purlin_option opt, int64_t *value) {
    if (ctx == nullptr || value == nullptr || (int)opt < 0 || (int)opt >= kNumOptions)
        return PURLIN_ERR_INVALID_ARG;
    *value = ctx->opt[opt];
    return PURLIN_OK;
}

purlin_status purlin_last_launch(const purlin_ctx *ctx, purlin_launch_info *info) {
    if (ctx == nullptr || info == nullptr) return PURLIN_ERR_INVALID_ARG;
    *info = ctx->last;
    return PURLIN_OK;
}

purlin_status purlin_plan_inspect(purlin_collective coll, int R, const void *const src[],
                                  void *const dst[], size_t n, const size_t counts[],
                                  purlin_dtype dtype, purlin_op op, purlin_layout layout,
                                  int variant, int ar_mode, uint64_t chunk_bytes,
                                  purlin_segment *segs, size_t cap, size_t *nseg,
                                  uint64_t *nchunks, uint64_t *nunits) {
    if ((int)coll < 0 || (int)coll > (int)PURLIN_COLL_ALL_TO_ALL_V) return PURLIN_ERR_INVALID_ARG;
    if (variant != kVariantLatency && variant != kVariantThroughput) return PURLIN_ERR_INVALID_ARG;
    CallDesc c = make_desc(coll, R, n, counts, dtype, op, layout);
    purlin_status st = validate_call(c, src, dst);
    if (st != PURLIN_OK) return st;
    const uint32_t copy_chunk = (uint32_t)(chunk_bytes ? chunk_bytes : kInspectChunkBytes);
    const uint32_t red_slot =
        (uint32_t)(chunk_bytes ? chunk_bytes * (uint64_t)R : kInspectChunkBytes);
    Plan p;
    st = compile_plan(c, variant, ar_mode, red_slot, copy_chunk, &p);
    if (st != PURLIN_OK) return st;
    if (nseg) *nseg = p.segs.size();
    if (nchunks) *nchunks = p.nchunks;
    if (nunits) *nunits = p.nunits;
    for (size_t i = 0; i < p.segs.size() && i < cap && segs; ++i) {
        const Seg &s = p.segs[i];
        purlin_segment &o = segs[i];
        o.src_off = s.src_off;
        o.dst_off = s.dst_off;
        o.bytes = s.bytes;
        o.src_rank = s.src_rank;
        o.dst_rank = s.dst_rank;
        o.skip_rank = s.skip_rank;
        o.src_is_dst = s.src_is_dst;
        o.sync = s.sync;
        o.tma = s.tma;
        o.shift = s.shift;
        o.head_bytes = s.head;
        o.tail_bytes = s.tail;
        o.chunk_begin = s.chunk_begin;
        o.chunk_bytes = s.chunk_bytes;
        o.unit_begin = s.unit_begin;
    }
    return PURLIN_OK;
}

purlin_status purlin_device_prepare(purlin_ctx *ctx, purlin_collective coll,
                                    const void *const src[], void *const dst[], size_t n,
                                    const size_t counts[], purlin_dtype dtype, purlin_op op,
                                    purlin_layout layout, int blocks,
                                    uint32_t max_workspace_bytes, purlin_device_coll *out) {
    if (ctx == nullptr || out == nullptr) return PURLIN_ERR_INVALID_ARG;
    if ((int)coll < 0 || (int)coll > (int)PURLIN_COLL_ALL_TO_ALL_V) return PURLIN_ERR_INVALID_ARG;
    if (blocks < 1 || blocks > 65535) return PURLIN_ERR_INVALID_ARG;
    const bool is_v = coll == PURLIN_COLL_ALL_GATHER_V || coll == PURLIN_COLL_REDUCE_SCATTER_V ||
                      coll == PURLIN_COLL_ALL_TO_ALL_V;
    const CallDesc c = make_desc(coll, ctx->R, is_v ? 0 : n, is_v ? counts : nullptr, dtype, op,
                                 layout);
    purlin_status st = validate_call(c, src, dst);
    if (st != PURLIN_OK) return st;

    // The launch's CTA budget for the workspace: the caller's cap, else the
    // device maximum less room for the kernel's own static shared memory.
    const uint32_t dev_limit = (uint32_t)ctx->max_smem - 4096u;
    const uint32_t limit = max_workspace_bytes ? std::min(max_workspace_bytes, dev_limit) : dev_limit;
    const uint32_t ctl_bytes = 128;   // snac::Ctl, padded to the workspace alignment
    if (limit <= ctl_bytes) return PURLIN_ERR_UNSUPPORTED;

    const Policy shape = call_policy(ctx, c);
    const int64_t chunk_opt = ctx->opt[PURLIN_OPT_CHUNK_BYTES];
    uint32_t chunk = (uint32_t)(chunk_opt > 0 ? chunk_opt : shape.chunk);
    Plan pl;
    RingShape rs;
    for (;;) {   // halve the chunk until the ring fits the cap
        st = compile_plan(c, kVariantThroughput, ring_ar_mode(ctx), chunk * (uint32_t)c.R, chunk,
                          &pl);
        if (st != PURLIN_OK) return st;
        st = ring_shape(ctx, c, shape, pl, limit - ctl_bytes, &rs);
        if (st == PURLIN_OK) break;
        if (st != PURLIN_ERR_UNSUPPORTED || chunk <= 256) return st;
        chunk = std::max<uint32_t>(256, (chunk / 2) & ~15u);
    }
    if (pl.composed && pl.notify_chunks > (uint64_t)kFlagSlots * 0xFFFFull)
        return PURLIN_ERR_INVALID_ARG;

    purlin_device_coll d;
    std::memset(&d, 0, sizeof d);
    for (int r = 0; r < c.R; ++r) {
        d.src[r] = src[r];
        d.dst[r] = dst[r];
    }
    d.nchunks = pl.nchunks;
    d.nunits = pl.nunits;
    d.epoch_inc = 1;
    d.timeout_ns = ctx->opt[PURLIN_OPT_SPIN_TIMEOUT_NS] > 0 ? ctx->opt[PURLIN_OPT_SPIN_TIMEOUT_NS]
                                                            : kDefaultTimeoutNs;
    d.drop_notify = ctx->opt[PURLIN_OPT_DROP_NOTIFY];
    d.flag_slots = 1;
    d.stages = rs.stages;
    d.slot_stride = rs.slot_stride;
    d.workspace_bytes = rs.smem + ctl_bytes;
    d.nseg = (int32_t)pl.segs.size();
    d.R = c.R;
    d.dtype = dtype;
    d.vector_copies = rs.vector_copies ? 1 : 0;
    d.blocks = blocks;
    d.threads = 32 * (2 + rs.consumer_warps);
    d.composed = pl.composed ? 1 : 0;
    d.coll = coll;

    DeviceCollMem m;
    auto fail = [&](purlin_status s) {
        free_device_coll(m);
        return s;
    };
    const size_t seg_bytes = std::max<size_t>(1, pl.segs.size()) * sizeof(Seg);
    if (cudaMalloc(&m.segs, seg_bytes) != cudaSuccess ||
        cudaMalloc(&m.epochs, (size_t)blocks * sizeof(unsigned long long)) != cudaSuccess ||
        cudaMalloc(&m.err, sizeof(unsigned long long)) != cudaSuccess)
        return fail(PURLIN_ERR_OOM);
    if (pl.composed) {
        flag_geometry(pl.notify_chunks, blocks, &d.flag_slots, &d.epoch_inc);
        if (cudaMalloc(&m.flags, 2 * (size_t)d.flag_slots * sizeof(unsigned long long)) !=
            cudaSuccess)
            return fail(PURLIN_ERR_OOM);
        if (cudaMemset(m.flags, 0, 2 * (size_t)d.flag_slots * sizeof(unsigned long long)) !=
            cudaSuccess)
            return fail(PURLIN_ERR_CUDA);
    }
    // Every CTA starts at epoch 1: flags start at 0, below any epoch.
    std::vector<unsigned long long> ep((size_t)blocks, 1ull);
    if ((!pl.segs.empty() &&
         cudaMemcpy(m.segs, pl.segs.data(), pl.segs.size() * sizeof(Seg),
                    cudaMemcpyHostToDevice) != cudaSuccess) ||
        cudaMemcpy(m.epochs, ep.data(), ep.size() * sizeof(unsigned long long),
                   cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemset(m.err, 0, sizeof(unsigned long long)) != cudaSuccess)
        return fail(PURLIN_ERR_CUDA);
    d.segs = m.segs;
    d.flags = m.flags;
    d.epochs = m.epochs;
    d.err = m.err;
    ctx->device_colls.push_back(m);
    d.owner = &ctx->device_colls.back();
    *out = d;
    return PURLIN_OK;
}

purlin_status purlin_device_check(const purlin_device_coll *coll, purlin_stream stream) {
    if (coll == nullptr || coll->err == nullptr) return PURLIN_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PURLIN_ERR_CUDA;
    unsigned long long word = 0;
    if (cudaMemcpy(&word, coll->err, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return PURLIN_ERR_CUDA;
    if (word == 0) return PURLIN_OK;
    if (cudaMemset(coll->err, 0, sizeof word) != cudaSuccess) return PURLIN_ERR_CUDA;
    return static_cast<purlin_status>(word & 0xFF);
}

purlin_status purlin_device_release(purlin_ctx *ctx, purlin_device_coll *coll) {
    if (ctx == nullptr || coll == nullptr) return PURLIN_ERR_INVALID_ARG;
    if (coll->owner == nullptr) return PURLIN_OK;
    for (auto it = ctx->device_colls.begin(); it != ctx->device_colls.end(); ++it) {
        if (&*it != coll->owner) continue;
        free_device_coll(*it);
        ctx->device_colls.erase(it);
        std::memset(coll, 0, sizeof *coll);
        return PURLIN_OK;
    }
    return PURLIN_ERR_INVALID_ARG;
}

size_t purlin_device_coll_size(void) { return sizeof(purlin_device_coll); }

}  // extern "C"
