// api.cpp -- the C ABI declared in include/purlin.h.
//
// Host side of one call: validate (no partial work on error), compile the
// layout into a plan (cached by its key), pick the variant by message size
// (codesign policy, "Purlin: Separating Orchestration from the Datapath of
// Collectives" §4.2; push/latency vs pull/throughput, §3.2), size the
// launch (CTAs, ring depth: in-flight capacity near the bandwidth-delay
// product with few CTAs, §3.3) and enqueue one kernel.  Notifying launches
// advance the epoch (§4.3) themselves, in device memory.  The device-side
// API's host calls are in device_api.cpp, the device-count V collectives'
// in vcounts_api.cpp; what they share with this file is in host.h.  Nothing here synchronises with the device
// except purlin_check, purlin_finalize and purlin_set_stream.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <list>
#include <new>
#include <string>
#include <unordered_map>

#include "host.h"
#include "launch.h"
#include "plan.h"

using namespace purlin;
using namespace purlin::host;

// ---- shared with the other host translation units (host.h)

namespace purlin {
namespace host {

Policy policy_for(purlin_collective coll, int R) {
    auto clamp16 = [](uint64_t v, uint64_t lo, uint64_t hi) {
        return (uint32_t)(std::min(hi, std::max(lo, v)) & ~uint64_t(15));
    };
    // Crossovers: the largest per-rank input the vector kernel wins at,
    // measured with each variant forced (host.h).  kVectorAlways: it won at
    // every size measured, up to 256 MiB per rank.
    switch (coll) {
        case PURLIN_COLL_REDUCE_SCATTER:
            return {clamp16(98304 / (uint64_t)R, 1024, 16384), 2, kVectorAlways, false, 0, 1};
        case PURLIN_COLL_REDUCE_SCATTER_V:   // both paths read ragged blocks aligned
            return {clamp16(98304 / (uint64_t)R, 1024, 16384), 2, kVectorAlways, false, 0, 1};
        case PURLIN_COLL_ALL_REDUCE:
            // (composed mode: the gather chunks are stored by the consumer warps)
            return {clamp16(32768 / (uint64_t)R, 512, 8192), 4, kVectorAlways, true, 0, 1};
        case PURLIN_COLL_ALL_GATHER:
            return {16384, 2, kVectorAlways, true, 8, 1};
        case PURLIN_COLL_ALL_GATHER_V:
            return {16384, 2, kVectorAlways, true, 8, 1};
        case PURLIN_COLL_ALL_TO_ALL:   // two CTAs per SM
            return {16384, 3, 2ull << 20, false, 0, 2};
        default:   // AllToAllV: two CTAs per SM
            return {16384, 3, 512ull << 10, false, 0, 2};
    }
}

// Composed AllReduce (reducing CTAs notify, gathering CTAs wait): each
// gather chunk covers R reduce chunks and acquires R flags, so large chunks
// pay off: 96 KiB stages (12 KiB per source at R = 8), 2 stages, 12 consumer
// warps, one CTA per SM.  At 256 MiB per rank this measured 5.53 TB/s
// against 4.07 TB/s with the fused AllReduce's 4 KiB x 3-stage ring.
Policy composed_all_reduce_policy(int R) {
    const uint32_t chunk = (uint32_t)std::max<uint64_t>(512, (98304 / (uint64_t)R) & ~uint64_t(15));
    return {chunk, 2, 8ull << 20, true, 12, 1};
}

void free_device_coll(DeviceCollMem &m) {
    if (m.segs) cudaFree(m.segs);
    if (m.flags) cudaFree(m.flags);
    if (m.epochs) cudaFree(m.epochs);
    if (m.err) cudaFree(m.err);
    m = DeviceCollMem{};
}

bool capturing(cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    return cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs != cudaStreamCaptureStatusNone;
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

purlin_status ring_shape(const purlin_ctx *ctx, const CallDesc &c, const Policy &shape,
                         const Plan &pl, uint32_t limit, RingShape *out) {
    RingShape r;
    r.slot_stride = (pl.slot_bytes + 127u) & ~127u;
    // Point-to-point copies at other 16-byte phases (ragged AllToAllV) go
    // through the consumer warps: 6 warps keep two CTAs per SM (measured +35%
    // over 8 warps).  They keep the policy's 3 stages: 4 measured 5-6% slower
    // from 16 to 256 MiB per rank, 2 slower still.
    const bool shifted_p2p = pl.has_shifted_copies && !shape.vector_copies &&
                             (c.coll == PURLIN_COLL_ALL_TO_ALL ||
                              c.coll == PURLIN_COLL_ALL_TO_ALL_V);
    uint32_t stages = (uint32_t)(ctx->opt[PURLIN_OPT_STAGES] > 0 ? ctx->opt[PURLIN_OPT_STAGES]
                                                                 : shape.stages);
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

// Per-parity flag slots for a grid of `grid` CTAs and the odd epoch
// increment that keeps every generation of a call distinct.  The slots are a
// multiple of the grid: when a call reuses them, notifying chunks number
// their flags by walk position (flag_at in plan.h), and positions pos and
// pos + slots then belong to the same CTA.  Those positions stay below the
// call's chunk count.
void flag_geometry(uint64_t notify_chunks, uint64_t nchunks, int64_t grid, uint32_t *slots,
                   uint64_t *epoch_inc) {
    *slots = (kFlagSlots / (uint32_t)grid) * (uint32_t)grid;
    uint64_t gens = notify_chunks <= *slots ? 1 : (nchunks + *slots - 1) / *slots;
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

}  // namespace host
}  // namespace purlin

namespace {

constexpr size_t kPlanCacheCap = 64;

// Built-in policy.
constexpr int64_t kInspectChunkBytes = 32 * 1024;        // plan_inspect default chunk
constexpr int kLatBlock = 256;
constexpr int64_t kMaxLatGrid = 1 << 24;   // CTAs of a vector-kernel launch
// Small plans whose every unit stores to all R ranks: see the latency launch.
constexpr uint64_t kSpreadUnits = 16384;
constexpr uint64_t kSpreadCtas = 16;
constexpr uint64_t kSpreadVectors = 2048;

int64_t env_or(const char *name, int64_t dflt) {
    const char *v = std::getenv(name);
    if (!v || !*v) return dflt;
    return std::strtoll(v, nullptr, 0);
}

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
        // One unit a thread: the block scheduler hands out the CTAs as SMs
        // free up, which balances the tail better than a persistent grid of 4
        // CTAs per SM looping over the units (6-11% faster for AllGather at 1-8
        // MiB per rank, 5% for AllReduce at 16-32 MiB); the loop only covers
        // plans past kMaxLatGrid CTAs.
        const int64_t cap = ctx->opt[PURLIN_OPT_LAT_CTAS] > 0
                                ? std::min<int64_t>(ctx->opt[PURLIN_OPT_LAT_CTAS], kMaxLatGrid)
                                : kMaxLatGrid;
        const int max_block = ctx->opt[PURLIN_OPT_LAT_BLOCK] > 0
                                  ? (int)ctx->opt[PURLIN_OPT_LAT_BLOCK] : kLatBlock;
        int block = (int)std::min<uint64_t>(max_block, (pl.nunits + 31) / 32 * 32);
        // A small plan whose every unit stores to all R ranks (AllReduce,
        // AllGather(V)) writes R times what it reads: spread it over about
        // 16 CTAs of 32-128 threads so more SMs drain the stores.  Per call
        // in a CUDA graph (R = 8, bf16, alternating builds on one box):
        // AllReduce 2-256 KiB per rank 1.58-2.08 -> 1.39-1.76 us, AllGather
        // 512 B-16 KiB 1.84-1.96 -> 1.71-1.75 us.  Plans that move fewer
        // than kSpreadVectors 16-byte vectors (loads + stores) or hold more
        // than kSpreadUnits units were slower spread, and so were
        // ReduceScatter and AllToAll (one store per unit): they keep blocks
        // of up to 256.
        if (ctx->opt[PURLIN_OPT_LAT_BLOCK] <= 0 && pl.nunits <= kSpreadUnits && !pl.segs.empty() &&
            std::all_of(pl.segs.begin(), pl.segs.end(),
                        [](const Seg &sg) { return sg.dst_rank == kRankAll; })) {
            const bool red = pl.segs.front().src_rank == kRankAll;
            const uint64_t vectors = pl.nunits * (uint64_t)(red ? 2 * c.R : 1 + c.R);
            if (vectors >= kSpreadVectors) {
                const uint64_t per = (pl.nunits + kSpreadCtas - 1) / kSpreadCtas;
                block = (int)std::min<uint64_t>(128, std::max<uint64_t>(32, (per + 31) / 32 * 32));
            }
        }
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
        const bool ragged = ragged_ring(pl);
        if (throughput_occupancy(c.dtype, pclass, ragged, block, smem, &per_sm) != cudaSuccess ||
            per_sm < 1)
            return PURLIN_ERR_UNSUPPORTED;
        // the policy's CTAs per SM, or the option's grid; never more than fit at once
        int64_t grid = ctx->opt[PURLIN_OPT_CTAS] > 0
                           ? std::min<int64_t>(ctx->opt[PURLIN_OPT_CTAS], (int64_t)ctx->sms * per_sm)
                           : (int64_t)ctx->sms * std::min(per_sm, std::max(1, shape.ctas_per_sm));
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
            // A reused flag slot is numbered by walk position, which keeps it
            // on one CTA (slots a multiple of the grid), so a later
            // generation of a slot implies the earlier one landed.
            flag_geometry(pl.notify_chunks, pl.nchunks, grid, &a.flag_slots, &epoch_inc);
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
    for (ChannelMem &m : ctx->channels) {
        if (m.staging) cudaFree(m.staging);
        if (m.state) cudaFree(m.state);
    }
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

purlin_status purlin_empty_launch(purlin_stream stream) {
    return launch_empty(static_cast<cudaStream_t>(stream)) == cudaSuccess ? PURLIN_OK
                                                                          : PURLIN_ERR_CUDA;
}

purlin_status purlin_touch_launch(const void *src, void *dst, purlin_stream stream) {
    if (src == nullptr || dst == nullptr) return PURLIN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u)
        return PURLIN_ERR_ALIGNMENT;
    return launch_touch(src, dst, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PURLIN_OK
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

}  // extern "C"
