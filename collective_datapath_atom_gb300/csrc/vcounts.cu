// vcounts.cu -- the variable-length collectives with their counts in device
// memory.
//
// "Purlin: Separating Orchestration from the Datapath of Collectives", §C.4
// (the V variants) and the same page's §4 note that the implementation
// takes prefix sums on the device; here the counts come from a kernel (an
// MoE router, say) and never travel to the host.  One kernel does it all:
// every CTA loads the counts, checks them against the capacities the caller
// declared, derives the displacements (exclusive prefix sums of the counts,
// or of the count matrix's rows and columns), builds the segment table
// with the same cut as the host plan compiler (cut_transfer), and runs the
// ring of snac.cuh on it; when the largest per-rank input is at most the
// crossover it runs the vector units alone.  Every CTA derives the same
// table from the same counts, so the CTAs need no communication; the cost
// is a few hundred nanoseconds of shared-memory work per CTA, against a
// host round trip and a second launch.
#include <cuda_runtime.h>

#include "atom.cuh"
#include "launch.h"
#include "snac.cuh"

namespace purlin {

namespace {

using namespace snac;

constexpr int kVcThreadsMax = 512;
constexpr uint64_t kVcMaxCount = 1ull << 40;   // elements in one count

template <int MAXR>
struct VcParams {
    const void *src[MAXR];
    void *dst[MAXR];
    const unsigned long long *counts;   // R (AGV, RSV) or R*R (A2AV) element counts, device
    unsigned long long *err;
    uint64_t in_cap;      // elements each input buffer holds
    uint64_t out_cap;     // elements each output buffer holds
    uint64_t crossover;   // largest per-rank input bytes run by the vector units alone
    int64_t timeout_ns;
    uint32_t red_chunk;   // bytes per source per reduce chunk
    uint32_t copy_chunk;  // bytes per copy chunk
    uint32_t stages;
    uint32_t slot_stride;
    int32_t R;
    int32_t coll;         // purlin_collective: AGV, RSV or A2AV
    int32_t es;           // element bytes
    int32_t vector_copies;
};

// What the ring reads (snac.cuh, class P).
struct VcView {
    const void *const *src;
    void *const *dst;
    const Seg *segs;
    const Seg *segs_dev;
    unsigned long long *err;
    uint64_t nchunks;
    uint64_t nunits;
    int64_t timeout_ns;
    int64_t drop_notify;
    uint32_t flag_slots;
    uint32_t stages;
    uint32_t slot_stride;
    int32_t nseg;
    int32_t R;
    int32_t vector_copies;
};

struct VcHeader {
    unsigned long long nchunks;
    unsigned long long nunits;
    unsigned long long max_in_bytes;
    int invalid;
    int pad;
};

__host__ __device__ constexpr int vc_nseg(int coll, int R) {
    return coll == PURLIN_COLL_ALL_TO_ALL_V ? R * R : R;
}

}  // namespace

// Shared memory of one CTA: ring | 4*S barriers | segment table | counts |
// per-segment chunk and unit counts | header | ring control.
uint32_t vcounts_smem(int coll, int R, uint32_t stages, uint32_t slot_stride) {
    const uint32_t nseg = (uint32_t)vc_nseg(coll, R);
    return stages * slot_stride + 4 * stages * 8 + nseg * (uint32_t)sizeof(Seg) + nseg * 8 +
           2 * nseg * 8 + (uint32_t)sizeof(VcHeader) + (uint32_t)sizeof(Ctl);
}

namespace {

// RAGGED: built for ReduceScatterV, whose ragged blocks put reduce chunks at
// another 16-byte phase than their destination (snac::run_ring).  The copies
// (AllGatherV, AllToAllV) take the other build, whose generic shifted-copy
// path serves any phase.
template <int DT, int MAXR, bool RAGGED>
__global__ void __launch_bounds__(kVcThreadsMax, 1)
    purlin_vcounts_kernel(const __grid_constant__ VcParams<MAXR> p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const int R = p.R;
    const int nseg = vc_nseg(p.coll, R);
    const uint32_t S = p.stages;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)S * p.slot_stride);
    Seg *segs = reinterpret_cast<Seg *>(bars + 4 * S);   // where the ring stages its table
    unsigned long long *cnt = reinterpret_cast<unsigned long long *>(segs + nseg);
    unsigned long long *nch = cnt + nseg;
    unsigned long long *nun = nch + nseg;
    VcHeader *hdr = reinterpret_cast<VcHeader *>(nun + nseg);
    Ctl *ctl = reinterpret_cast<Ctl *>(hdr + 1);
    const uint64_t es = (uint64_t)p.es;

    // ---- the counts
    for (int i = threadIdx.x; i < nseg; i += blockDim.x) cnt[i] = p.counts[i];
    if (threadIdx.x == 0) {
        hdr->max_in_bytes = 0;
        hdr->invalid = 0;
    }
    __syncthreads();

    // ---- per rank: input and output extents against the capacities; the
    // largest input (the crossover decision)
    for (int r = threadIdx.x; r < R; r += blockDim.x) {
        uint64_t in_e = 0, out_e = 0;
        bool bad = false;
        if (p.coll == PURLIN_COLL_ALL_TO_ALL_V) {
            for (int j = 0; j < R; ++j) {
                const uint64_t row = cnt[r * R + j], col = cnt[j * R + r];
                bad |= row >= kVcMaxCount || col >= kVcMaxCount;
                in_e += row;
                out_e += col;
            }
        } else {
            uint64_t total = 0;
            for (int j = 0; j < R; ++j) {
                bad |= cnt[j] >= kVcMaxCount;
                total += cnt[j];
            }
            if (p.coll == PURLIN_COLL_ALL_GATHER_V) {
                in_e = cnt[r];
                out_e = total;
            } else {   // ReduceScatterV
                in_e = total;
                out_e = cnt[r];
            }
        }
        if (bad || in_e > p.in_cap || out_e > p.out_cap) atomicOr(&hdr->invalid, 1);
        atomicMax(&hdr->max_in_bytes, (unsigned long long)(in_e * es));
    }
    __syncthreads();
    if (hdr->invalid) {
        if (blockIdx.x == 0 && threadIdx.x == 0)
            record_error(p.err, PURLIN_ERR_INVALID_ARG, kSiteDeviceCounts, 0);
        return;   // uniform: every CTA read the same counts
    }
    const bool ring = hdr->max_in_bytes > p.crossover;

    // ---- per segment: displacements, the transfer, its cut
    for (int i = threadIdx.x; i < nseg; i += blockDim.x) {
        Seg sg = {};
        sg.skip_rank = -1;
        uint64_t so = 0, dof = 0, bytes = 0;
        if (p.coll == PURLIN_COLL_ALL_TO_ALL_V) {
            // input of s packed by destination, output of d packed by source
            const int s = i / R, d = i % R;
            uint64_t S_sd = 0, Q_ds = 0;
            for (int j = 0; j < d; ++j) S_sd += cnt[s * R + j];
            for (int j = 0; j < s; ++j) Q_ds += cnt[j * R + d];
            so = S_sd * es;
            dof = Q_ds * es;
            bytes = cnt[i] * es;
            sg.src_rank = (int8_t)s;
            sg.dst_rank = (int8_t)d;
        } else {
            uint64_t D = 0;
            for (int j = 0; j < i; ++j) D += cnt[j];
            bytes = cnt[i] * es;
            if (p.coll == PURLIN_COLL_ALL_GATHER_V) {   // block i of every output
                so = 0;
                dof = D * es;
                sg.src_rank = (int8_t)i;
                sg.dst_rank = (int8_t)kRankAll;
            } else {                                    // reduce block i into output i
                so = D * es;
                dof = 0;
                sg.src_rank = (int8_t)kRankAll;
                sg.dst_rank = (int8_t)i;
            }
        }
        sg.src_off = so;
        sg.dst_off = dof;
        sg.bytes = bytes;
        sg.chunk_bytes = sg.src_rank < 0 ? p.red_chunk : p.copy_chunk;
        uint64_t chunks = 0, units = units_in(unit_grid(so, dof, sg.src_rank < 0), 0, bytes);
        if (ring) {
            const Cut cut = cut_transfer(so, dof, bytes, sg.src_rank < 0);
            if (cut.body > 0) {
                sg.tma = 1;
                sg.head = (uint8_t)cut.head;
                sg.tail = (uint8_t)cut.tail;
                sg.shift = (uint8_t)cut.shift;
                chunks = (cut.body + sg.chunk_bytes - 1) / sg.chunk_bytes;
                units = (cut.head ? 1u : 0u) + (cut.tail ? 1u : 0u);
            }
        }
        segs[i] = sg;
        nch[i] = chunks;
        nun[i] = units;
    }
    __syncthreads();

    // ---- exclusive prefix sums of the chunk and unit counts (warp 0: each
    // lane a run of consecutive segments, then a shuffle scan over lanes)
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int per = (nseg + 31) / 32;
        const int a = lane * per < nseg ? lane * per : nseg;
        const int b = a + per < nseg ? a + per : nseg;
        unsigned long long sc = 0, su = 0;
        for (int i = a; i < b; ++i) {
            sc += nch[i];
            su += nun[i];
        }
        unsigned long long ic = sc, iu = su;   // inclusive scan over lanes
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long tc = __shfl_up_sync(0xFFFFFFFFu, ic, o);
            const unsigned long long tu = __shfl_up_sync(0xFFFFFFFFu, iu, o);
            if (lane >= o) {
                ic += tc;
                iu += tu;
            }
        }
        unsigned long long c0 = ic - sc, u0 = iu - su;
        for (int i = a; i < b; ++i) {
            segs[i].chunk_begin = (uint32_t)c0;
            segs[i].unit_begin = u0;
            c0 += nch[i];
            u0 += nun[i];
        }
        if (lane == 31) {
            hdr->nchunks = ic;
            hdr->nunits = iu;
        }
    }
    __syncthreads();

    const VcView v{p.src,        p.dst,         nullptr,      segs, p.err,
                   hdr->nchunks, hdr->nunits,   p.timeout_ns, -1,   1u,
                   S,            p.slot_stride, nseg,         R,    p.vector_copies};
    if (hdr->nchunks > 0xFFFFFFF0ull) {
        if (blockIdx.x == 0 && threadIdx.x == 0)
            record_error(p.err, PURLIN_ERR_INVALID_ARG, kSiteDeviceCounts, 1);
        return;
    }
    if (!ring) {
        // one-shot vector units over every thread of the grid
        const uint64_t nt = blockDim.x;
        units_loop<DT, MAXR, false>(v, segs, (uint64_t)blockIdx.x * nt + threadIdx.x,
                                    (uint64_t)gridDim.x * nt);
        return;
    }
    run_ring<DT, MAXR, RAGGED>(v, smem, ctl, blockIdx.x, gridDim.x, nullptr, 0);
}

template <int DT, int MAXR, bool RAGGED>
cudaError_t launch_vc_t(const VcLaunch &a) {
    VcParams<MAXR> p;
    for (int r = 0; r < MAXR; ++r) {
        p.src[r] = r < a.R ? a.src[r] : nullptr;
        p.dst[r] = r < a.R ? a.dst[r] : nullptr;
    }
    p.counts = a.counts;
    p.err = a.err;
    p.in_cap = a.in_cap;
    p.out_cap = a.out_cap;
    p.crossover = a.crossover;
    p.timeout_ns = a.timeout_ns;
    p.red_chunk = a.red_chunk;
    p.copy_chunk = a.copy_chunk;
    p.stages = a.stages;
    p.slot_stride = a.slot_stride;
    p.R = a.R;
    p.coll = a.coll;
    p.es = elem_bytes(a.dtype);
    p.vector_copies = a.vector_copies ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.grid);
    cfg.blockDim = dim3((unsigned)a.block);
    cfg.dynamicSmemBytes = a.smem;
    cfg.stream = a.stream;
    return cudaLaunchKernelEx(&cfg, purlin_vcounts_kernel<DT, MAXR, RAGGED>, p);
}

// Calls f(kernel) with the device-count kernel for a dtype, R and collective.
template <class F>
cudaError_t with_vc_kernel(int dtype, int R, int coll, F &&f) {
    const bool phase = coll == PURLIN_COLL_REDUCE_SCATTER_V;
    const bool f32 = dtype == PURLIN_F32, small = R <= 8;
    if (phase) {
        if (f32) return small ? f(purlin_vcounts_kernel<PURLIN_F32, 8, true>)
                              : f(purlin_vcounts_kernel<PURLIN_F32, kVcMaxRanks, true>);
        return small ? f(purlin_vcounts_kernel<PURLIN_BF16, 8, true>)
                     : f(purlin_vcounts_kernel<PURLIN_BF16, kVcMaxRanks, true>);
    }
    if (f32) return small ? f(purlin_vcounts_kernel<PURLIN_F32, 8, false>)
                          : f(purlin_vcounts_kernel<PURLIN_F32, kVcMaxRanks, false>);
    return small ? f(purlin_vcounts_kernel<PURLIN_BF16, 8, false>)
                 : f(purlin_vcounts_kernel<PURLIN_BF16, kVcMaxRanks, false>);
}

}  // namespace

cudaError_t launch_vcounts(const VcLaunch &a) {
    const bool phase = a.coll == PURLIN_COLL_REDUCE_SCATTER_V;
    if (a.dtype == PURLIN_F32) {
        if (phase)
            return a.R <= 8 ? launch_vc_t<PURLIN_F32, 8, true>(a)
                            : launch_vc_t<PURLIN_F32, kVcMaxRanks, true>(a);
        return a.R <= 8 ? launch_vc_t<PURLIN_F32, 8, false>(a)
                        : launch_vc_t<PURLIN_F32, kVcMaxRanks, false>(a);
    }
    if (phase)
        return a.R <= 8 ? launch_vc_t<PURLIN_BF16, 8, true>(a)
                        : launch_vc_t<PURLIN_BF16, kVcMaxRanks, true>(a);
    return a.R <= 8 ? launch_vc_t<PURLIN_BF16, 8, false>(a)
                    : launch_vc_t<PURLIN_BF16, kVcMaxRanks, false>(a);
}

cudaError_t configure_vcounts(int max_dyn_smem) {
    for (int coll : {PURLIN_COLL_ALL_TO_ALL_V, PURLIN_COLL_REDUCE_SCATTER_V})
        for (int dtype : {PURLIN_F32, PURLIN_BF16})
            for (int R : {8, kVcMaxRanks}) {
                const cudaError_t e = with_vc_kernel(dtype, R, coll, [&](auto kernel) {
                    return cudaFuncSetAttribute(
                        kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn_smem);
                });
                if (e != cudaSuccess) return e;
            }
    return cudaSuccess;
}

cudaError_t vcounts_occupancy(int dtype, int R, int coll, int block, size_t smem, int *per_sm) {
    return with_vc_kernel(dtype, R, coll, [&](auto kernel) {
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, kernel, block, smem);
    });
}

}  // namespace purlin
