// packets.cu -- the composed AllReduce on the latency path: payload and
// notification travel together in 16-byte packets.
//
// "Purlin: Separating Orchestration from the Datapath of Collectives":
//   §3.2  the latency path joins payload and notification in one 16-byte
//         packet (twice the bytes, no separate flag round trip); SCORE on
//         the latency path: each output is computed once, by one thread, in
//         source order;
//   §4.1  two staging buffers of 2 MiB for latency-bound execution;
//   §4.3  the epoch's parity selects the buffer and the epoch is the
//         notification value.
//
// One cooperative launch of 2G CTAs.  CTAs [0, G) reduce: thread t of CTA b
// owns the 8-byte payload units u = b*T + t, + G*T, ...; it adds the R
// sources of unit u in rank order in binary32, rounds once, and stores the
// packet of u into the staging buffer.  CTAs [G, 2G) gather: the same units
// in the same order, each polled (bounded) until its packet carries this
// call's flag, then its payload is written to all R outputs.  A unit is
// reduced exactly once and every output gets the same bits, as in the
// ring's composed AllReduce; what changes is the notification, which costs
// no fence and no flag store here.
#include <cuda_runtime.h>

#include "atom.cuh"
#include "launch.h"
#include "snac.cuh"

namespace purlin {

namespace {

using namespace snac;

constexpr int kPktThreads = 256;

template <int MAXR>
struct PktParams {
    const void *src[MAXR];
    void *dst[MAXR];
    unsigned char *staging;   // both parities, kPacketStagingBytes each: 16 bytes per unit
    DevEpoch *dev_epoch;      // the launch's epoch: parity and flag
    unsigned long long *err;
    uint64_t nbytes;          // bytes per rank buffer
    uint64_t units;           // ceil(nbytes / 8)
    int64_t timeout_ns;
    int64_t drop_unit;        // fault injection: a unit whose packet is never stored, or -1
    int32_t R;
    int32_t G;                // reducing CTAs (as many gather)
};

// 8 payload bytes of source s at byte offset off: `valid` bytes (the rest 0).
template <int DT>
__device__ __forceinline__ uint64_t load_unit(const char *base, uint64_t off, uint32_t valid) {
    if (valid == 8) return *reinterpret_cast<const uint64_t *>(base + off);
    uint64_t v = 0;
    constexpr uint32_t ES = DT == PURLIN_F32 ? 4 : 2;
    for (uint32_t j = 0; j < valid; j += ES) {
        const uint64_t e = ES == 4 ? *reinterpret_cast<const uint32_t *>(base + off + j)
                                   : *reinterpret_cast<const uint16_t *>(base + off + j);
        v |= e << (8 * j);
    }
    return v;
}

template <int DT>
__device__ __forceinline__ void store_unit(char *base, uint64_t off, uint32_t valid, uint64_t v) {
    if (valid == 8) {
        *reinterpret_cast<uint64_t *>(base + off) = v;
        return;
    }
    constexpr uint32_t ES = DT == PURLIN_F32 ? 4 : 2;
    for (uint32_t j = 0; j < valid; j += ES) {
        if (ES == 4) *reinterpret_cast<uint32_t *>(base + off + j) = (uint32_t)(v >> (8 * j));
        else *reinterpret_cast<uint16_t *>(base + off + j) = (uint16_t)(v >> (8 * j));
    }
}

// SCORE over one unit: binary32 from source 0, sources added in rank order,
// one rounding at the end.
template <int DT, int MAXR>
__device__ __forceinline__ uint64_t reduce_unit(const PktParams<MAXR> &p, uint64_t off,
                                                uint32_t valid) {
    if (DT == PURLIN_F32) {
        const uint64_t w0 = load_unit<DT>(static_cast<const char *>(p.src[0]), off, valid);
        float a0 = __uint_as_float((uint32_t)w0), a1 = __uint_as_float((uint32_t)(w0 >> 32));
        for (int s = 1; s < p.R; ++s) {
            const uint64_t w = load_unit<DT>(static_cast<const char *>(p.src[s]), off, valid);
            a0 = __fadd_rn(a0, __uint_as_float((uint32_t)w));
            a1 = __fadd_rn(a1, __uint_as_float((uint32_t)(w >> 32)));
        }
        return (uint64_t)__float_as_uint(a0) | ((uint64_t)__float_as_uint(a1) << 32);
    }
    const uint64_t w0 = load_unit<DT>(static_cast<const char *>(p.src[0]), off, valid);
    float a[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) a[j] = __uint_as_float((uint32_t)((w0 >> (16 * j)) & 0xFFFFu) << 16);
    for (int s = 1; s < p.R; ++s) {
        const uint64_t w = load_unit<DT>(static_cast<const char *>(p.src[s]), off, valid);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            a[j] = __fadd_rn(a[j], __uint_as_float((uint32_t)((w >> (16 * j)) & 0xFFFFu) << 16));
    }
    return (uint64_t)atom::pack_bf16x2(a[0], a[1]) | ((uint64_t)atom::pack_bf16x2(a[2], a[3]) << 32);
}

template <int DT, int MAXR>
__global__ void __launch_bounds__(kPktThreads) purlin_packet_ar_kernel(
    const __grid_constant__ PktParams<MAXR> p) {
    // The epoch comes from device memory, so a launch replayed from a graph
    // still uses a new flag and the other staging buffer.
    __shared__ Ctl ctl;
    epoch_enter(p.dev_epoch, &ctl);
    __syncthreads();
    const uint64_t epoch = ctl.epoch;
    const uint32_t flag = (uint32_t)epoch;
    unsigned char *const staging = p.staging + (epoch & 1ull) * kPacketStagingBytes;

    const bool reducer = (int)blockIdx.x < p.G;
    const uint64_t b = reducer ? blockIdx.x : blockIdx.x - (unsigned)p.G;
    const uint64_t stride = (uint64_t)p.G * blockDim.x;
    for (uint64_t u = b * blockDim.x + threadIdx.x; u < p.units; u += stride) {
        const uint64_t off = 8 * u;
        const uint32_t valid = (uint32_t)(p.nbytes - off < 8 ? p.nbytes - off : 8);
        unsigned char *pk = staging + 16 * u;
        if (reducer) {
            const uint64_t v = reduce_unit<DT>(p, off, valid);
            if ((int64_t)u != p.drop_unit) atom::packet_store(pk, v, flag);
            continue;
        }
        uint64_t v;
        if (!packet_wait(pk, flag, p.timeout_ns, p.err, u, &v)) break;
        for (int d = 0; d < p.R; ++d) store_unit<DT>(static_cast<char *>(p.dst[d]), off, valid, v);
    }
    __syncthreads();
    epoch_leave(p.dev_epoch, 1, gridDim.x);
}

template <int DT, int MAXR>
cudaError_t launch_pkt_t(const PktLaunch &a) {
    PktParams<MAXR> p;
    for (int r = 0; r < MAXR; ++r) {
        p.src[r] = r < a.R ? a.src[r] : nullptr;
        p.dst[r] = r < a.R ? a.dst[r] : nullptr;
    }
    p.staging = a.staging;
    p.dev_epoch = reinterpret_cast<DevEpoch *>(a.dev_epoch);
    p.err = a.err;
    p.nbytes = a.nbytes;
    p.units = (a.nbytes + 7) / 8;
    p.timeout_ns = a.timeout_ns;
    p.drop_unit = a.drop_unit;
    p.R = a.R;
    p.G = a.G;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // gathering CTAs wait on reducing ones
    attr[0].val.cooperative = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * a.G));
    cfg.blockDim = dim3(kPktThreads);
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, purlin_packet_ar_kernel<DT, MAXR>, p);
}

}  // namespace

int packet_threads() { return kPktThreads; }

cudaError_t launch_packet_all_reduce(const PktLaunch &a) {
    if (a.dtype == PURLIN_F32)
        return a.R <= kSmallMaxR ? launch_pkt_t<PURLIN_F32, kSmallMaxR>(a)
                                 : launch_pkt_t<PURLIN_F32, kBigMaxR>(a);
    return a.R <= kSmallMaxR ? launch_pkt_t<PURLIN_BF16, kSmallMaxR>(a)
                             : launch_pkt_t<PURLIN_BF16, kBigMaxR>(a);
}

}  // namespace purlin
