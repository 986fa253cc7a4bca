// vcounts_api.cpp -- host side of the V collectives whose counts are in
// device memory (include/purlin.h, purlin_*_v_device_counts; the kernel is
// in vcounts.cu).
#include <cuda_runtime.h>

#include <algorithm>
#include <vector>

#include "host.h"
#include "launch.h"
#include "plan.h"

using namespace purlin;
using namespace purlin::host;

namespace {

// Per-rank input bytes up to which the device-count kernel takes its vector
// path.  That path runs inside the ring's grid (one or two CTAs per SM,
// looping over the units), not as the host calls' vector kernel with a CTA
// for every 256 units, so it keeps the crossovers measured for a vector
// kernel of that size: AllGatherV 3 MiB, ReduceScatterV 24 MiB, AllToAllV
// 256 KiB.
uint64_t device_count_crossover(purlin_collective coll) {
    switch (coll) {
        case PURLIN_COLL_ALL_GATHER_V: return 3ull << 20;
        case PURLIN_COLL_REDUCE_SCATTER_V: return 24ull << 20;
        default: return 256ull << 10;
    }
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
    // Any count may put a copy's source at another 16-byte phase: room for its
    // hull.  A reduce stages its sources on their own grid.
    const uint32_t slot = reduce ? chunk * (uint32_t)c.R : chunk + 16u;
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
    if (vcounts_occupancy(dtype, c.R, coll, block, smem, &per_sm) != cudaSuccess || per_sm < 1)
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
                      : device_count_crossover(coll);
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
    // the policy's CTAs per SM, or the option's grid; never more than fit at once
    int64_t grid = ctx->opt[PURLIN_OPT_CTAS] > 0
                       ? std::min<int64_t>(ctx->opt[PURLIN_OPT_CTAS], (int64_t)ctx->sms * per_sm)
                       : (int64_t)ctx->sms * std::min(per_sm, std::max(1, shape.ctas_per_sm));
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

}  // namespace

extern "C" {

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

}  // extern "C"
