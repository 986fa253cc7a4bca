// channel_api.cpp -- host side of the packet channel (include/purlin.h,
// purlin_packet_channel_*): the staging buffers and state a producer/consumer
// pair of CTAs exchange 16-byte payload+flag packets through ("Purlin:
// Separating Orchestration from the Datapath of Collectives" §3.2 latency
// path, §4.1 two staging buffers, §4.3 epoch parity).  The device side is
// purlin::device::channel_* in include/purlin_device.cuh.
#include <cuda_runtime.h>

#include <cstring>

#include "host.h"

using namespace purlin::host;

namespace {

constexpr uint64_t kMaxChannelBytes = 1ull << 34;
constexpr int64_t kDefaultChannelTimeoutNs = 100 * 1000 * 1000;

}  // namespace

extern "C" {

purlin_status purlin_packet_channel_create(purlin_ctx *ctx, size_t capacity_bytes, int ctas,
                                           purlin_packet_channel *out) {
    if (ctx == nullptr || out == nullptr) return PURLIN_ERR_INVALID_ARG;
    if (capacity_bytes == 0 || capacity_bytes > kMaxChannelBytes || ctas < 1 || ctas > 65535)
        return PURLIN_ERR_INVALID_ARG;
    const uint64_t units = (capacity_bytes + 7) / 8;
    ChannelMem m;
    // two packet sets (one per epoch parity), 16 bytes per unit
    if (cudaMalloc(&m.staging, 2 * 16 * units) != cudaSuccess) return PURLIN_ERR_OOM;
    if (cudaMalloc(&m.state, 4 * sizeof(unsigned long long)) != cudaSuccess) {
        cudaFree(m.staging);
        return PURLIN_ERR_OOM;
    }
    // Packets start at flag 0 and the epoch at 1, so no zeroed packet ever
    // carries a launch's flag.
    const unsigned long long init[4] = {0ull, 0ull, 1ull, 0ull};
    if (cudaMemset(m.staging, 0, 2 * 16 * units) != cudaSuccess ||
        cudaMemcpy(m.state, init, sizeof init, cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaFree(m.staging);
        cudaFree(m.state);
        return PURLIN_ERR_CUDA;
    }
    purlin_packet_channel ch;
    std::memset(&ch, 0, sizeof ch);
    ch.staging = m.staging;
    ch.state = m.state;
    ch.capacity = units;
    ch.timeout_ns = ctx->opt[PURLIN_OPT_SPIN_TIMEOUT_NS] > 0 ? ctx->opt[PURLIN_OPT_SPIN_TIMEOUT_NS]
                                                             : kDefaultChannelTimeoutNs;
    ch.drop_unit = ctx->opt[PURLIN_OPT_DROP_NOTIFY];
    ch.ctas = ctas;
    ctx->channels.push_back(m);
    ch.owner = &ctx->channels.back();
    *out = ch;
    return PURLIN_OK;
}

purlin_status purlin_packet_channel_check(const purlin_packet_channel *ch, purlin_stream stream) {
    if (ch == nullptr || ch->state == nullptr) return PURLIN_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PURLIN_ERR_CUDA;
    unsigned long long word = 0;
    if (cudaMemcpy(&word, ch->state, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return PURLIN_ERR_CUDA;
    if (word == 0) return PURLIN_OK;
    if (cudaMemset(ch->state, 0, sizeof word) != cudaSuccess) return PURLIN_ERR_CUDA;
    return static_cast<purlin_status>(word & 0xFF);
}

purlin_status purlin_packet_channel_release(purlin_ctx *ctx, purlin_packet_channel *ch) {
    if (ctx == nullptr || ch == nullptr) return PURLIN_ERR_INVALID_ARG;
    if (ch->owner == nullptr) return PURLIN_OK;
    for (auto it = ctx->channels.begin(); it != ctx->channels.end(); ++it) {
        if (&*it != ch->owner) continue;
        cudaFree(it->staging);   // (cudaFree waits for the device)
        cudaFree(it->state);
        ctx->channels.erase(it);
        std::memset(ch, 0, sizeof *ch);
        return PURLIN_OK;
    }
    return PURLIN_ERR_INVALID_ARG;
}

}  // extern "C"
