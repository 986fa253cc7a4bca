// kernels.cu -- the library's two kernel families over the device-side
// SNAC functions of snac.cuh.
//
// "Purlin: Separating Orchestration from the Datapath of Collectives",
// §2.1: prefill payloads are throughput-bound and decode messages
// latency-bound, and a high-bandwidth path's setup dominates small messages.
// §3.2: push for latency, pull for bandwidth.  On one GPU these become the
// vector kernel and the staged ring; measured on GB300 the vector kernel,
// one window a thread and a CTA per 256 windows, also wins at every size for
// AllGather(V), AllReduce and ReduceScatter(V) (the host's policy).
//
// Latency (vector) kernel: one thread per 16-byte window ("unit"); no flags,
//   since every output has one owner.
// Throughput kernel: persistent CTAs running the ring (snac::run_ring) over
//   the launch's whole grid (ring_kernel.cuh); this unit builds it for
//   plans whose ring chunks share their destination's 16-byte phase, and
//   kernels_ragged.cu for plans with chunks at another phase.
#include "ring_kernel.cuh"

namespace purlin {

namespace {

using namespace snac;
using ringk::KParams;
using ringk::by_class;
using ringk::class_of;
using ringk::fill_params;

// ---------------------------------------------------------- latency kernel --

// Launch bounds of four CTAs of 256 threads per SM leave 64 registers a
// thread; the instantiations for more than 8 ranks take two (the whole-window
// copy builds use 30 and fit eight).  The host launches a CTA per 256 units,
// so the loop below normally runs once a thread.  WHOLE: a
// build for plans whose segments are all made of whole aligned 16-byte
// windows and all copies (1) or all reductions (2) (Plan::whole_op), with
// only the short unit path for that operation (whole_unit); 3, a uniform
// AllToAll, reads no segment table at all (transposed_unit).
template <int DT, int MAXR, int MAXSEG, int WHOLE = 0>
__global__ void __launch_bounds__(256, MAXR > 8 ? 2 : 4) purlin_latency_kernel(
    const __grid_constant__ KParams<MAXR, MAXSEG> p) {
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    const uint64_t u0 = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if constexpr (WHOLE == 3) {   // uniform AllToAll: addresses from the unit index alone
        const uint32_t W = (uint32_t)(p.nunits / (uint64_t)(p.R * p.R));
        for (uint64_t u = u0; u < p.nunits; u += stride) transposed_unit<MAXR>(p, (uint32_t)u, W);
        return;
    }
    // An inline table whose segments are long (16 or more units each on
    // average, or a single segment) is read straight from the parameter bank:
    // the threads of a warp then look at one or two segments, nearly a
    // broadcast, and the CTA skips the staging and its barrier (measured in
    // graph replays: 2.49 -> 2.08 us for a 2 KiB AllReduce, 2.41 -> 2.15 us
    // for a 2 KiB AllGather).  Short segments would make a warp read many
    // addresses, so those tables are staged in shared memory.
    if (MAXSEG > 1 && (p.nseg == 1 || p.nunits >= 16ull * (uint64_t)p.nseg)) {
        units_loop<DT, MAXR, false, WHOLE>(p, p.segs, u0, stride);
        return;
    }
    // an inline table of MAXSEG segments, or up to kSmemSegs of a device table
    constexpr int kStage = MAXSEG > 1 ? MAXSEG : kSmemSegs;
    __shared__ Seg s_segs[kStage];
    const Seg *segs = stage_segs(p, s_segs, kStage);
    __syncthreads();
    units_loop<DT, MAXR, false, WHOLE>(p, segs, u0, stride);
}

template <int DT, int MAXR, int MAXSEG, int WHOLE = 0>
cudaError_t launch_lat_t(const LaunchArgs &a) {
    KParams<MAXR, MAXSEG> p;
    fill_params(p, a);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.grid);
    cfg.blockDim = dim3((unsigned)a.block);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = a.stream;
    return cudaLaunchKernelEx(&cfg, purlin_latency_kernel<DT, MAXR, MAXSEG, WHOLE>, p);
}

__global__ void purlin_empty_kernel() {}

// One 16-byte load and one 16-byte store by one thread: the least a kernel
// that touches memory does (the memory-touch floor of small messages).
__global__ void purlin_touch_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst) {
    if (threadIdx.x == 0) *dst = *src;
}

struct LatLaunch {
    const LaunchArgs &a;
    template <int DT, int MR, int MS>
    cudaError_t run() { return launch_lat_t<DT, MR, MS>(a); }
};

}  // namespace

cudaError_t launch_empty(cudaStream_t stream) {
    purlin_empty_kernel<<<1, 32, 0, stream>>>();
    return cudaGetLastError();
}

cudaError_t launch_touch(const void *src, void *dst, cudaStream_t stream) {
    purlin_touch_kernel<<<1, 32, 0, stream>>>(static_cast<const uint4 *>(src),
                                              static_cast<uint4 *>(dst));
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

cudaError_t launch_latency(const LaunchArgs &a) {
    if (a.plan->whole_op == 3 && a.R <= kSmallMaxR)   // bytes only: one build serves both dtypes
        return launch_lat_t<PURLIN_BF16, kSmallMaxR, 1, 3>(a);
    const int pc = class_of(a);
    if (a.plan->whole_op != 0 && (pc == kClassSmall || pc == kClassDev8)) {
        const bool f32 = a.dtype == PURLIN_F32;
        const bool red = a.plan->whole_op == 2;
        if (pc == kClassSmall) {
            if (red) return f32 ? launch_lat_t<PURLIN_F32, kSmallMaxR, kSmallMaxSeg, 2>(a)
                                : launch_lat_t<PURLIN_BF16, kSmallMaxR, kSmallMaxSeg, 2>(a);
            return f32 ? launch_lat_t<PURLIN_F32, kSmallMaxR, kSmallMaxSeg, 1>(a)
                       : launch_lat_t<PURLIN_BF16, kSmallMaxR, kSmallMaxSeg, 1>(a);
        }
        if (red) return f32 ? launch_lat_t<PURLIN_F32, kSmallMaxR, 1, 2>(a)
                            : launch_lat_t<PURLIN_BF16, kSmallMaxR, 1, 2>(a);
        return f32 ? launch_lat_t<PURLIN_F32, kSmallMaxR, 1, 1>(a)
                   : launch_lat_t<PURLIN_BF16, kSmallMaxR, 1, 1>(a);
    }
    return by_class(pc, a.dtype, LatLaunch{a});
}

cudaError_t launch_throughput(const LaunchArgs &a) {
    if (ragged_ring(*a.plan)) return launch_throughput_ragged(a);
    return by_class(class_of(a), a.dtype, ringk::TputLaunch<false>{a});
}

cudaError_t configure_kernels(int max_dyn_smem) {
    const cudaError_t e = ringk::configure_ring<false>(max_dyn_smem);
    return e != cudaSuccess ? e : configure_kernels_ragged(max_dyn_smem);
}

cudaError_t throughput_occupancy(int dtype, int pclass, bool ragged, int block, size_t smem,
                                 int *per_sm) {
    if (ragged) return throughput_occupancy_ragged(dtype, pclass, block, smem, per_sm);
    return by_class(pclass, dtype, ringk::TputOccupancy<false>{block, smem, per_sm});
}

}  // namespace purlin
