// kernels_phase.cu -- the ring kernel (ring_kernel.cuh) built for plans
// with reduce chunks stored at another 16-byte phase than their sources
// (a ragged ReduceScatter(V): each block's sources are staged on their own
// grid and the sums stored at the destination's phase).  A unit of its own,
// compiled beside kernels.cu, so that neither build waits on the other.
#include "ring_kernel.cuh"

namespace purlin {

cudaError_t launch_throughput_phase(const LaunchArgs &a) {
    return ringk::by_class(ringk::class_of(a), a.dtype, ringk::TputLaunch<true>{a});
}

cudaError_t configure_kernels_phase(int max_dyn_smem) {
    return ringk::configure_ring<true>(max_dyn_smem);
}

cudaError_t throughput_occupancy_phase(int dtype, int pclass, int block, size_t smem, int *per_sm) {
    return ringk::by_class(pclass, dtype, ringk::TputOccupancy<true>{block, smem, per_sm});
}

}  // namespace purlin
