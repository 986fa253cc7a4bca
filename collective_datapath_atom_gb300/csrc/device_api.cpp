// device_api.cpp -- host side of the device-side API (include/purlin.h,
// purlin_device_*): compile a collective for kernels that run it themselves
// ("Purlin" project README, "Device-side").  The plan compiler, policy and
// ring shaping are the host calls'; this file adds the descriptor and the
// device memory it names (segment table, per-CTA epochs, flags, error word).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <vector>

#include "host.h"
#include "launch.h"
#include "plan.h"

using namespace purlin;
using namespace purlin::host;

extern "C" {

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
    d.ragged = ragged_ring(pl) ? 1 : 0;

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
        flag_geometry(pl.notify_chunks, pl.nchunks, blocks, &d.flag_slots, &d.epoch_inc);
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
