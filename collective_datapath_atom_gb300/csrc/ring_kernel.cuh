// ring_kernel.cuh -- the ring kernel (snac::run_ring over the launch's
// whole grid), its parameter block and its launch, shared by the two
// translation units that build it: kernels.cu (plans whose ring chunks share
// their destination's 16-byte phase) and kernels_ragged.cu (plans with
// chunks at another phase, RAGGED).  Internal to the library.
#pragma once

#include <cuda_runtime.h>

#include "atom.cuh"
#include "launch.h"
#include "snac.cuh"

namespace purlin {
namespace ringk {

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

// ------------------------------------------------------- throughput kernel --

// RAGGED: built for plans with ring chunks at another 16-byte phase than their
// destination (ragged_ring).
template <int DT, int MAXR, int MAXSEG, bool RAGGED>
__global__ void __launch_bounds__(kTputMaxThreads, 1) purlin_throughput_kernel(
    const __grid_constant__ KParams<MAXR, MAXSEG> p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ Ctl ctl;
    if (p.dev_epoch == nullptr) {
        run_ring<DT, MAXR, RAGGED>(p, smem, &ctl, blockIdx.x, gridDim.x, nullptr, 0);
        return;
    }
    // chunks notify one another: the launch's epoch comes from device memory
    epoch_enter(p.dev_epoch, &ctl);
    __syncthreads();
    const uint64_t epoch = ctl.epoch;
    run_ring<DT, MAXR, RAGGED>(p, smem, &ctl, blockIdx.x, gridDim.x,
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

template <int DT, int MAXR, int MAXSEG, bool RAGGED>
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
    return cudaLaunchKernelEx(&cfg, purlin_throughput_kernel<DT, MAXR, MAXSEG, RAGGED>, p);
}

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

inline int class_of(const LaunchArgs &a) {
    return launch_class(a.R, a.plan->segs.size(), a.segs_dev != nullptr);
}

template <bool RAGGED>
struct TputLaunch {
    const LaunchArgs &a;
    template <int DT, int MR, int MS>
    cudaError_t run() { return launch_tput_t<DT, MR, MS, RAGGED>(a); }
};
template <bool RAGGED>
struct TputConfigure {
    int max_dyn_smem;
    template <int DT, int MR, int MS>
    cudaError_t run() {
        return cudaFuncSetAttribute(purlin_throughput_kernel<DT, MR, MS, RAGGED>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn_smem);
    }
};
template <bool RAGGED>
struct TputOccupancy {
    int block;
    size_t smem;
    int *per_sm;
    template <int DT, int MR, int MS>
    cudaError_t run() {
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            per_sm, purlin_throughput_kernel<DT, MR, MS, RAGGED>, block, smem);
    }
};

// The ring kernels of one build (RAGGED or not) for every launch class and dtype.
template <bool RAGGED>
cudaError_t configure_ring(int max_dyn_smem) {
    for (int pc : {kClassSmall, kClassBig, kClassDev8, kClassDev64})
        for (int dt : {PURLIN_F32, PURLIN_BF16}) {
            const cudaError_t e = by_class(pc, dt, TputConfigure<RAGGED>{max_dyn_smem});
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}

}  // namespace ringk
}  // namespace purlin
