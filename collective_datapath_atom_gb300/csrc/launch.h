// launch.h -- host-side interface to the two kernel families.
#pragma once

#include <cuda_runtime_api.h>

#include "plan.h"

namespace purlin {

constexpr uint32_t kFlagSlots = 65536;      // per parity
constexpr int kSmallMaxR = 8;               // parameter block sizes: small ...
constexpr int kSmallMaxSeg = 16;
constexpr int kBigMaxR = PURLIN_MAX_RANKS;  // ... and big
constexpr int kBigMaxSeg = 64;

struct LaunchArgs {
    const Plan *plan = nullptr;
    const Seg *segs_dev = nullptr;   // device copy of plan->segs, or null (inline)
    const void *const *src = nullptr;
    void *const *dst = nullptr;
    int R = 0;
    int dtype = 0;
    unsigned long long *flags = nullptr;   // both parity sets, flag_slots each (composed)
    uint32_t flag_slots = kFlagSlots;
    unsigned long long *dev_epoch = nullptr;   // {epoch, done} in device memory (composed)
    uint64_t epoch_inc = 1;                    // odd
    unsigned long long *err = nullptr;
    int64_t timeout_ns = 0;
    int64_t drop_notify = -1;
    int grid = 0;
    int block = 0;
    uint32_t smem = 0;
    uint32_t stages = 0;
    uint32_t slot_stride = 0;
    bool cooperative = false;
    bool vector_copies = false;   // aligned copy chunks stored by the consumer warps
    cudaStream_t stream = nullptr;
};

// V collectives with device-resident counts (vcounts.cu).
constexpr int kVcMaxRanks = 16;   // R*R <= 256 segments per CTA's table

struct VcLaunch {
    const void *const *src = nullptr;
    void *const *dst = nullptr;
    const unsigned long long *counts = nullptr;   // device
    unsigned long long *err = nullptr;
    uint64_t in_cap = 0;      // elements
    uint64_t out_cap = 0;     // elements
    uint64_t crossover = 0;   // bytes: largest per-rank input run by vector units alone
    int64_t timeout_ns = 0;
    uint32_t red_chunk = 0;
    uint32_t copy_chunk = 0;
    uint32_t stages = 0;
    uint32_t slot_stride = 0;
    int R = 0;
    int coll = 0;
    int dtype = 0;
    bool vector_copies = false;
    int grid = 0;
    int block = 0;
    uint32_t smem = 0;
    cudaStream_t stream = nullptr;
};

uint32_t vcounts_smem(int coll, int R, uint32_t stages, uint32_t slot_stride);
cudaError_t launch_vcounts(const VcLaunch &a);
cudaError_t configure_vcounts(int max_dyn_smem);
cudaError_t vcounts_occupancy(int dtype, int R, int coll, int block, size_t smem, int *per_sm);

// Composed AllReduce on the latency path (packets.cu).
constexpr uint64_t kPacketStagingBytes = 2ull << 20;   // per parity: 16-byte packets
constexpr uint64_t kPacketPayloadBytes = kPacketStagingBytes / 2;   // 8 payload bytes per packet

struct PktLaunch {
    const void *const *src = nullptr;
    void *const *dst = nullptr;
    unsigned char *staging = nullptr;   // both parities, kPacketStagingBytes each
    unsigned long long *dev_epoch = nullptr;   // {epoch, done}: selects the parity, gives the flag
    unsigned long long *err = nullptr;
    uint64_t nbytes = 0;
    int64_t timeout_ns = 0;
    int64_t drop_unit = -1;
    int R = 0;
    int dtype = 0;
    int G = 0;                          // reducing CTAs; as many gather
    cudaStream_t stream = nullptr;
};

int packet_threads();
cudaError_t launch_packet_all_reduce(const PktLaunch &a);

// Kernel parameter blocks ("launch classes"): the segment table inline in
// the parameters (small: R <= 8 and up to 16 segments; big: up to 64), or in
// device memory with only the rank pointers inline (R <= 8, or up to 64).
enum LaunchClass : int {
    kClassSmall = 0,
    kClassBig = 1,
    kClassDev8 = 2,
    kClassDev64 = 3,
};

// The inline class a plan fits (small or big), -1 if none.
int param_class(int R, size_t nseg);

// The class a launch uses: a device table's class, else param_class.
int launch_class(int R, size_t nseg, bool device_table);

cudaError_t launch_latency(const LaunchArgs &a);
cudaError_t launch_empty(cudaStream_t stream);
cudaError_t launch_touch(const void *src, void *dst, cudaStream_t stream);
cudaError_t launch_throughput(const LaunchArgs &a);

// Largest dynamic shared memory the throughput kernels may use; set once.
cudaError_t configure_kernels(int max_dyn_smem);

// ragged: the plan has ring chunks at another 16-byte phase than their
// destination (ragged_ring), which a separate build of the ring kernel runs.
cudaError_t throughput_occupancy(int dtype, int pclass, bool ragged, int block, size_t smem,
                                 int *per_sm);

// The ring kernel's RAGGED build (kernels_ragged.cu), behind
// launch_throughput, configure_kernels and throughput_occupancy.
cudaError_t launch_throughput_ragged(const LaunchArgs &a);
cudaError_t configure_kernels_ragged(int max_dyn_smem);
cudaError_t throughput_occupancy_ragged(int dtype, int pclass, int block, size_t smem, int *per_sm);

// Shared-memory bytes a throughput launch needs for `stages` ring slots of
// `slot_stride` bytes, their mbarriers and the staged segment table.
uint32_t throughput_smem(uint32_t stages, uint32_t slot_stride);

}  // namespace purlin
