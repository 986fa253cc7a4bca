// kernels.cu -- the library's two kernel families over the device-side
// SNAC functions of snac.cuh.
//
// "Purlin: Separating Orchestration from the Datapath of Collectives",
// §2.1: prefill payloads are throughput-bound and decode messages
// latency-bound, and a high-bandwidth path's setup dominates small messages.
// §3.2: push for latency, pull for bandwidth.  On one GPU these become the
// vector kernel and the staged ring.
//
// Latency kernel: one thread per 16-byte destination window ("unit"); no
//   flags, since every output has one owner.
// Throughput kernel: persistent CTAs running the ring (snac::run_ring) over
//   the launch's whole grid.
#include <cuda_runtime.h>

#include "atom.cuh"
#include "launch.h"
#include "snac.cuh"

namespace purlin {

namespace {

using namespace snac;

constexpr int kTputMaxThreads = 512;

template <int MAXR, int MAXSEG>
struct KParams {
    const void *src[MAXR];
    void *dst[MAXR];
    Seg segs[MAXSEG];
    const Seg *segs_dev;
    unsigned long long *flags;   // both parities' flag sets (flag_slots each), or null
    unsigned long long *err;
    DevEpoch *dev_epoch;         // the device epoch, when chunks notify one another
    uint64_t epoch_inc;          // odd: added to the device epoch by the launch
    uint64_t nchunks;
    uint64_t nunits;
    int64_t timeout_ns;
    int64_t drop_notify;
    uint32_t flag_slots;
    uint32_t stages;
    uint32_t slot_stride;
    int32_t nseg;
    int32_t R;
    int32_t vector_copies;   // aligned copy chunks are stored by the consumer warps too
};

// ---------------------------------------------------------- latency kernel --

// Four CTAs of 256 threads per SM (the host's grid cap) leave 64 registers
// a thread; the instantiations for more than 8 ranks take two.
template <int DT, int MAXR, int MAXSEG>
__global__ void __launch_bounds__(256, MAXR > 8 ? 2 : 4) purlin_latency_kernel(
    const __grid_constant__ KParams<MAXR, MAXSEG> p) {
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    const uint64_t u0 = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    // An inline table whose segments are long (16 or more units each on
    // average, or a single segment) is read straight from the parameter bank:
    // the threads of a warp then look at one or two segments, nearly a
    // broadcast, and the CTA skips the staging and its barrier (measured in
    // graph replays: 2.49 -> 2.08 us for a 2 KiB AllReduce, 2.41 -> 2.15 us
    // for a 2 KiB AllGather).  Short segments would make a warp read many
    // addresses, so those tables are staged in shared memory.
    if (MAXSEG > 1 && (p.nseg == 1 || p.nunits >= 16ull * (uint64_t)p.nseg)) {
        units_loop<DT, MAXR, false>(p, p.segs, u0, stride);
        return;
    }
    // an inline table of MAXSEG segments, or up to kSmemSegs of a device table
    constexpr int kStage = MAXSEG > 1 ? MAXSEG : kSmemSegs;
    __shared__ Seg s_segs[kStage];
    const Seg *segs = stage_segs(p, s_segs, kStage);
    __syncthreads();
    units_loop<DT, MAXR, false>(p, segs, u0, stride);
}

// ------------------------------------------------------- throughput kernel --

template <int DT, int MAXR, int MAXSEG>
__global__ void __launch_bounds__(kTputMaxThreads, 1) purlin_throughput_kernel(
    const __grid_constant__ KParams<MAXR, MAXSEG> p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ Ctl ctl;
    if (p.dev_epoch == nullptr) {
        run_ring<DT, MAXR>(p, smem, &ctl, blockIdx.x, gridDim.x, nullptr, 0);
        return;
    }
    // chunks notify one another: the launch's epoch comes from device memory
    epoch_enter(p.dev_epoch, &ctl);
    __syncthreads();
    const uint64_t epoch = ctl.epoch;
    run_ring<DT, MAXR>(p, smem, &ctl, blockIdx.x, gridDim.x,
                       p.flags + (epoch & 1ull) * p.flag_slots, epoch);
    epoch_leave(p.dev_epoch, p.epoch_inc, gridDim.x);   // run_ring ended with a CTA barrier
}

template <int MAXR, int MAXSEG>
void fill_params(KParams<MAXR, MAXSEG> &p, const LaunchArgs &a) {
    for (int r = 0; r < MAXR; ++r) {
        p.src[r] = r < a.R ? a.src[r] : nullptr;
        p.dst[r] = r < a.R ? a.dst[r] : nullptr;
    }
    const Plan &pl = *a.plan;
    const size_t nseg = pl.segs.size();
    for (size_t i = 0; i < (size_t)MAXSEG; ++i) p.segs[i] = i < nseg && !a.segs_dev ? pl.segs[i] : Seg{};
    p.segs_dev = a.segs_dev;
    p.flags = a.flags;
    p.dev_epoch = reinterpret_cast<DevEpoch *>(a.dev_epoch);
    p.epoch_inc = a.epoch_inc;
    p.err = a.err;
    p.nchunks = pl.nchunks;
    p.nunits = pl.nunits;
    p.timeout_ns = a.timeout_ns;
    p.drop_notify = a.drop_notify;
    p.flag_slots = a.flag_slots;
    p.stages = a.stages;
    p.slot_stride = a.slot_stride;
    p.nseg = (int32_t)nseg;
    p.R = a.R;
    p.vector_copies = a.vector_copies ? 1 : 0;
}

template <int DT, int MAXR, int MAXSEG>
cudaError_t launch_lat_t(const LaunchArgs &a) {
    KParams<MAXR, MAXSEG> p;
    fill_params(p, a);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.grid);
    cfg.blockDim = dim3((unsigned)a.block);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = a.stream;
    return cudaLaunchKernelEx(&cfg, purlin_latency_kernel<DT, MAXR, MAXSEG>, p);
}

template <int DT, int MAXR, int MAXSEG>
cudaError_t launch_tput_t(const LaunchArgs &a) {
    KParams<MAXR, MAXSEG> p;
    fill_params(p, a);
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.grid);
    cfg.blockDim = dim3((unsigned)a.block);
    cfg.dynamicSmemBytes = a.smem;
    cfg.stream = a.stream;
    if (a.cooperative) {
        // CTAs that wait on one another's flags must all be resident.
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, purlin_throughput_kernel<DT, MAXR, MAXSEG>, p);
}

__global__ void purlin_empty_kernel() {}

}  // namespace

cudaError_t launch_empty(cudaStream_t stream) {
    purlin_empty_kernel<<<1, 32, 0, stream>>>();
    return cudaGetLastError();
}

int param_class(int R, size_t nseg) {
    if (R <= kSmallMaxR && nseg <= (size_t)kSmallMaxSeg) return kClassSmall;
    if (nseg <= (size_t)kBigMaxSeg) return kClassBig;
    return -1;
}

int launch_class(int R, size_t nseg, bool device_table) {
    if (device_table) return R <= kSmallMaxR ? kClassDev8 : kClassDev64;
    return param_class(R, nseg);
}

uint32_t throughput_smem(uint32_t stages, uint32_t slot_stride) {
    return ring_workspace_bytes(stages, slot_stride);
}

namespace {

// Calls f.template run<DT, MAXR, MAXSEG>() for a launch class and dtype.
template <class F>
cudaError_t by_class(int pc, int dtype, F &&f) {
    const bool f32 = dtype == PURLIN_F32;
    switch (pc) {
        case kClassSmall:
            return f32 ? f.template run<PURLIN_F32, kSmallMaxR, kSmallMaxSeg>()
                       : f.template run<PURLIN_BF16, kSmallMaxR, kSmallMaxSeg>();
        case kClassBig:
            return f32 ? f.template run<PURLIN_F32, kBigMaxR, kBigMaxSeg>()
                       : f.template run<PURLIN_BF16, kBigMaxR, kBigMaxSeg>();
        case kClassDev8:
            return f32 ? f.template run<PURLIN_F32, kSmallMaxR, 1>()
                       : f.template run<PURLIN_BF16, kSmallMaxR, 1>();
        case kClassDev64:
            return f32 ? f.template run<PURLIN_F32, kBigMaxR, 1>()
                       : f.template run<PURLIN_BF16, kBigMaxR, 1>();
    }
    return cudaErrorInvalidValue;
}

struct LatLaunch {
    const LaunchArgs &a;
    template <int DT, int MR, int MS>
    cudaError_t run() { return launch_lat_t<DT, MR, MS>(a); }
};
struct TputLaunch {
    const LaunchArgs &a;
    template <int DT, int MR, int MS>
    cudaError_t run() { return launch_tput_t<DT, MR, MS>(a); }
};
struct TputConfigure {
    int max_dyn_smem;
    template <int DT, int MR, int MS>
    cudaError_t run() {
        return cudaFuncSetAttribute(purlin_throughput_kernel<DT, MR, MS>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn_smem);
    }
};
struct TputOccupancy {
    int block;
    size_t smem;
    int *per_sm;
    template <int DT, int MR, int MS>
    cudaError_t run() {
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            per_sm, purlin_throughput_kernel<DT, MR, MS>, block, smem);
    }
};

int class_of(const LaunchArgs &a) {
    return launch_class(a.R, a.plan->segs.size(), a.segs_dev != nullptr);
}

}  // namespace

cudaError_t launch_latency(const LaunchArgs &a) { return by_class(class_of(a), a.dtype, LatLaunch{a}); }

cudaError_t launch_throughput(const LaunchArgs &a) {
    return by_class(class_of(a), a.dtype, TputLaunch{a});
}

cudaError_t configure_kernels(int max_dyn_smem) {
    for (int pc : {kClassSmall, kClassBig, kClassDev8, kClassDev64})
        for (int dt : {PURLIN_F32, PURLIN_BF16}) {
            const cudaError_t e = by_class(pc, dt, TputConfigure{max_dyn_smem});
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}

cudaError_t throughput_occupancy(int dtype, int pclass, int block, size_t smem, int *per_sm) {
    return by_class(pclass, dtype, TputOccupancy{block, smem, per_sm});
}

}  // namespace purlin
