// host.h -- what the host-side translation units of the C ABI share: the
// context, the plan cache entry, the codesign policy and the ring shaping.
// Internal to the library (not part of include/).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <list>
#include <string>
#include <unordered_map>

#include "launch.h"
#include "plan.h"

namespace purlin {
namespace host {

constexpr int kNumOptions = 12;
constexpr int64_t kDefaultTimeoutNs = 100 * 1000 * 1000;   // 100 ms
constexpr int kCopyConsumerWarps = 4;
constexpr int kReduceConsumerWarps = 8;
constexpr int kShiftedCopyConsumerWarps = 6;

// Policy per collective (codesign policy, "Purlin: Separating Orchestration
// from the Datapath of Collectives" §4.2), measured on GB300 over 256 B..64
// MiB per rank and at the workloads' sizes.
// Crossover: per-rank message bytes up to which the one-shot vector kernel
// beats the staged ring (both forced, single launches and graph replays
// with the L2 flushed, 256 KiB..256 MiB per rank at R = 8, confirmed on a
// second box).  With one 16-byte window a thread and as many CTAs as that
// takes, the vector kernel won at every size for AllGather(V), AllReduce
// and ReduceScatter(V): at 256 MiB per rank AllReduce 628.7 against 657.4
// us, ReduceScatter 350.2 against 367.6 us; AllGather at 128 MiB 1433.6
// against 1540.8 us (kVectorAlways).  AllToAll 2 MiB (13.9 against 14.8 us
// there; the ring leads at 4 MiB in a graph), AllToAllV 512 KiB (the ring
// leads from 1 MiB).  The composed AllReduce has its own (api.cpp), and so
// do the device-count calls, whose vector path runs inside the ring's grid
// (vcounts_api.cpp).
// Ring shape:
//   ReduceScatter(V)  one destination per reduced chunk: large per-source
//                     chunks (96 KiB per stage), 2 stages;
//   AllReduce         R stores per reduced vector: 32 KiB per stage, 4 stages
//                     (0.8-0.9% faster than 3 at 64 and 256 MiB per rank);
//   AllGather(V)      one staged tile written to R destinations: 16 KiB
//                     chunks, 2 stages, and the 8 consumer warps store the
//                     tile with 128-bit stores (0.956 of the copy peak versus
//                     0.92 with bulk stores from one warp).  2 stages against
//                     4: AllGather 2.6% faster at 16 MiB per rank and 5.8-6.7%
//                     at 64-128 MiB, level at 4-8 MiB; AllGatherV level to
//                     0.6% faster;
//   AllToAll(V)       one load, one store per chunk: 16 KiB chunks, 3 stages,
//                     bulk stores (0.98).
constexpr uint64_t kVectorAlways = ~0ull;   // crossover: the vector kernel at every size

struct Policy {
    uint32_t chunk;         // bytes per source per chunk
    uint32_t stages;
    uint64_t crossover;     // latency kernel at or below this many bytes per rank
    bool vector_copies;     // aligned copies stored by the consumer warps
    int consumer_warps;     // 0: by plan (8 with reductions or shifted copies, else 4)
    int ctas_per_sm;        // the ring's CTAs per SM the shape was tuned at (the
                            // occupancy limit when lower)
};

Policy policy_for(purlin_collective coll, int R);

// Composed AllReduce's ring shape (see api.cpp).
Policy composed_all_reduce_policy(int R);

// Device memory behind one purlin_device_coll.
struct DeviceCollMem {
    Seg *segs = nullptr;
    unsigned long long *flags = nullptr;
    unsigned long long *epochs = nullptr;
    unsigned long long *err = nullptr;
};

void free_device_coll(DeviceCollMem &m);

// Device memory of one packet channel (purlin_packet_channel_create).
struct ChannelMem {
    unsigned char *staging = nullptr;
    unsigned long long *state = nullptr;
};

struct CacheEntry {
    std::string key;
    Plan plan;
    Seg *segs_dev = nullptr;
    bool pinned = false;   // used while a CUDA graph was captured: kept until finalize
};

// True while a CUDA graph is being captured from stream s.
bool capturing(cudaStream_t s);

CallDesc make_desc(purlin_collective coll, int R, size_t n, const size_t *counts, int dtype,
                   int op, purlin_layout layout);

// Ring shape of a throughput launch: stages (reduced until the shared
// memory fits `limit`), stage stride, consumer warps and copy stores.
struct RingShape {
    uint32_t stages = 0;
    uint32_t slot_stride = 0;
    uint32_t smem = 0;
    int consumer_warps = 0;
    bool vector_copies = false;
};

}  // namespace host
}  // namespace purlin

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
    int64_t opt[purlin::host::kNumOptions] = {};
    purlin_launch_info last = {};
    std::list<purlin::host::CacheEntry> lru;
    std::unordered_map<std::string, std::list<purlin::host::CacheEntry>::iterator> index;
    std::list<purlin::host::DeviceCollMem> device_colls;   // memory of purlin_device_prepare descriptors
    std::list<purlin::host::ChannelMem> channels;          // memory of packet channels
};

namespace purlin {
namespace host {

purlin_status ring_shape(const purlin_ctx *ctx, const CallDesc &c, const Policy &shape,
                         const Plan &pl, uint32_t limit, RingShape *out);
void flag_geometry(uint64_t notify_chunks, uint64_t nchunks, int64_t grid, uint32_t *slots,
                   uint64_t *epoch_inc);
int ring_ar_mode(const purlin_ctx *ctx);
Policy call_policy(const purlin_ctx *ctx, const CallDesc &c);

}  // namespace host
}  // namespace purlin
