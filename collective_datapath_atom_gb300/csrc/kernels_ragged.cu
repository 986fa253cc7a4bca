// kernels_ragged.cu -- the ring kernel (ring_kernel.cuh) built for plans
// with ring chunks at another 16-byte phase than their destination: the
// blocks of a ragged ReduceScatter(V) (sources staged on their own grid, sums
// stored at the destination's phase) and ragged copies (AllToAllV,
// AllGatherV: hulls shifted into place with the word offset fixed at compile
// time).  A unit of its own, compiled beside kernels.cu.
#include "ring_kernel.cuh"

namespace purlin {

cudaError_t launch_throughput_ragged(const LaunchArgs &a) {
    return ringk::by_class(ringk::class_of(a), a.dtype, ringk::TputLaunch<true>{a});
}

cudaError_t configure_kernels_ragged(int max_dyn_smem) {
    return ringk::configure_ring<true>(max_dyn_smem);
}

cudaError_t throughput_occupancy_ragged(int dtype, int pclass, int block, size_t smem, int *per_sm) {
    return ringk::by_class(pclass, dtype, ringk::TputOccupancy<true>{block, smem, per_sm});
}

}  // namespace purlin
