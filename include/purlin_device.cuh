/*
 * purlin_device.cuh -- device-side API: collectives and Atoms called from
 * inside a user's kernel (CUDA C++, sm_103a).
 *
 * "Purlin" project README, "Device-side" and "Samples": a kernel hands some
 * of its CTAs to a collective, or has a CTA copy one aligned slice through
 * the Atom, and does its own work before and after.  Exactly `blocks` CTAs
 * enter a collective, each with the Atom's thread count and pipeline
 * shared memory.  Paper summary §3: applications invoke the Atom directly
 * and tune its pipeline; §3.2 SNAC; §3.3 the Atom's staged pipeline and
 * SCORE reductions.
 *
 * The code that runs is the library's own: the same ring (stage warp,
 * write-back warp, consumer warps; bounded waits; per-chunk flags for the
 * composed AllReduce) that purlin_all_reduce and the other host calls
 * launch, entered here with the caller's CTA index and count.
 *
 * Collectives.  Prepare a purlin_device_coll on the host with
 * purlin_device_prepare (include/purlin.h), pass it to the kernel, and in
 * each of its coll.blocks CTAs call
 *
 *     purlin::device::collective(coll, {workspace, coll.blocks, index});
 *
 * with `workspace` = coll.workspace_bytes of shared memory, 128-byte
 * aligned, and `index` in [0, coll.blocks), each index entered exactly once
 * per call.  Every thread of the CTA must make the call (it synchronises the
 * CTA).  When it returns, this CTA's share of the collective is stored; the
 * rest of the outputs are stored once every entering CTA has returned (order
 * a read of other CTAs' outputs after a grid-wide barrier).  Data that this
 * CTA or others wrote before the call (ordered by such a barrier) is what
 * the collective reads.  Errors (a mismatched argument, an expired wait)
 * are recorded in the descriptor's error word: purlin_device_check.  Two
 * calls in one kernel must be separated by a grid-wide barrier over the
 * entering CTAs, so that no CTA starts a call while another is still in the
 * one before (the flags of calls two apart share a parity set).
 *
 * Atoms.  purlin::device::Atom<STAGES, CHUNK, CONSUMER_WARPS> moves data
 * through one CTA's ring without any host preparation:
 *   Atom::copy(dst, src, bytes, workspace)            bitwise copy
 *   Atom::reduce<DT>(dst, srcs, nsrc, elems, workspace)
 *       dst[i] = sum over s = 0..nsrc-1, in order, of srcs[s][i], in
 *       binary32 from srcs[0][i], rounded once to DT (SCORE)
 * Launch with Atom::THREADS threads per block and give each call
 * Atom::PIPELINE_SMEM_BYTES of 128-byte aligned shared memory.  All threads
 * of the CTA make the call.  copy: dst and src 2-byte aligned, bytes even;
 * any 16-byte phases (a source at another phase than its destination is
 * shifted into place).  reduce: dst and every srcs[s] 16-byte aligned,
 * 1 <= nsrc <= 64, `srcs` readable by the device (e.g. a kernel parameter).
 * Both return PURLIN_OK, PURLIN_ERR_ALIGNMENT / PURLIN_ERR_INVALID_ARG
 * (nothing moved), or PURLIN_ERR_TIMEOUT (a ring wait expired), the same
 * value in every thread.
 *
 * Packet channels.  purlin_packet_channel (include/purlin.h) carries 8-byte
 * payload units between CTAs of one launch as 16-byte payload+flag packets
 * (paper summary §3.2, the latency path).  In each of the channel's `ctas`
 * CTAs, every thread calls
 *
 *     purlin::device::Packets pk = purlin::device::channel_open(ch);
 *     ... send(ch, pk, u, payload) / recv(ch, pk, u, &payload) ...
 *     purlin::device::channel_close(ch);
 *
 * send() stores unit u's packet (one thread, one 16-byte store, no fence);
 * recv() waits, bounded by ch.timeout_ns, until unit u's packet of this
 * launch has arrived and returns its payload, or returns false (TIMEOUT in
 * the channel's error word: purlin_packet_channel_check).  Each unit is sent
 * once and may be received by any number of threads.  Producers and
 * consumers must be resident together (a cooperative launch).
 */
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "purlin.h"
#include "../collective_datapath_atom_gb300/csrc/snac.cuh"

namespace purlin {
namespace device {

// The pages' SnacArgs, with the buffers carried by the descriptor.
struct SnacArgs {
    void *workspace;   // coll.workspace_bytes of shared memory, 128-byte aligned
    int blocks;        // CTAs entering this call: must equal coll.blocks
    int bIdx;          // this CTA's index among them
};

namespace detail {

// The ring's parameter view of a descriptor (snac.cuh, class P).
struct CollView {
    const void *const *src;
    void *const *dst;
    const Seg *segs;       // no inline table
    const Seg *segs_dev;   // the descriptor's device table
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

__device__ __forceinline__ bool block_shape_ok() {
    return (blockDim.x & 31u) == 0 && blockDim.x >= 96 && blockDim.y == 1 && blockDim.z == 1;
}

}  // namespace detail

// Run a prepared collective with the calling CTA as CTA `a.bIdx` of
// `a.blocks`.  DT and MAXR must cover the descriptor (dtype == DT, R <= MAXR);
// collective() below picks them.
template <int DT, int MAXR>
__device__ purlin_status collective_t(const purlin_device_coll &c, const SnacArgs &a) {
    unsigned char *ws = static_cast<unsigned char *>(a.workspace);
    const bool bad = a.blocks != c.blocks || a.bIdx < 0 || a.bIdx >= a.blocks ||
                     !detail::block_shape_ok() || (reinterpret_cast<uintptr_t>(ws) & 127u) != 0 ||
                     c.R > MAXR || c.dtype != DT || c.err == nullptr;
    if (bad) {
        if (threadIdx.x == 0 && c.err != nullptr)
            snac::record_error(c.err, PURLIN_ERR_INVALID_ARG, snac::kSiteDeviceArgs, blockIdx.x);
        return PURLIN_ERR_INVALID_ARG;
    }
    snac::Ctl *ctl =
        reinterpret_cast<snac::Ctl *>(ws + snac::ring_workspace_bytes(c.stages, c.slot_stride));
    __syncthreads();   // the caller is done with the workspace
    if (threadIdx.x == 0) ctl->epoch = *reinterpret_cast<volatile unsigned long long *>(&c.epochs[a.bIdx]);
    __syncthreads();
    const uint64_t epoch = ctl->epoch;
    const detail::CollView v{c.src,
                             c.dst,
                             nullptr,
                             static_cast<const Seg *>(c.segs),
                             c.err,
                             c.nchunks,
                             c.nunits,
                             c.timeout_ns,
                             c.drop_notify,
                             c.flag_slots,
                             c.stages,
                             c.slot_stride,
                             c.nseg,
                             c.R,
                             c.vector_copies};
    unsigned long long *flags = c.flags ? c.flags + (epoch & 1ull) * c.flag_slots : nullptr;
    // Ragged blocks (chunks at another 16-byte phase than their
    // destination): that build of the ring, for descriptors that need it only.
    if (c.ragged)
        snac::run_ring<DT, MAXR, true>(v, ws, ctl, (uint32_t)a.bIdx, (uint32_t)a.blocks, flags,
                                       epoch);
    else
        snac::run_ring<DT, MAXR, false>(v, ws, ctl, (uint32_t)a.bIdx, (uint32_t)a.blocks, flags,
                                        epoch);
    // (run_ring ends with a CTA barrier.)  One thread reads the error word
    // so that every thread returns the same status.
    if (threadIdx.x == 0) {
        c.epochs[a.bIdx] = epoch + c.epoch_inc;
        ctl->epoch = *reinterpret_cast<volatile unsigned long long *>(c.err);
    }
    __syncthreads();
    const unsigned long long word = ctl->epoch;
    __syncthreads();   // the workspace is the caller's again
    return static_cast<purlin_status>(word & 0xFFull);
}

// Run a prepared collective (dtype and R taken from the descriptor).  A
// kernel that calls it holds eight builds of the ring (two dtypes, two rank
// bounds, plain and ragged) and compiles for tens of seconds; kernels that
// call it from several places can share one out-of-line wrapper (at a few
// percent of bandwidth, measured on the library's examples).
__device__ inline purlin_status collective(const purlin_device_coll &c, const SnacArgs &a) {
    if (c.dtype == PURLIN_F32)
        return c.R <= 8 ? collective_t<PURLIN_F32, 8>(c, a)
                        : collective_t<PURLIN_F32, PURLIN_MAX_RANKS>(c, a);
    return c.R <= 8 ? collective_t<PURLIN_BF16, 8>(c, a)
                    : collective_t<PURLIN_BF16, PURLIN_MAX_RANKS>(c, a);
}

// ----------------------------------------------------------- packets --

// One launch's view of a packet channel: its packet set and flag.
struct Packets {
    unsigned char *set;   // the launch's packet set (16 bytes per unit)
    uint32_t flag;        // the launch's notification value
};

// Every thread of each of the channel's ch.ctas CTAs, before its first send
// or receive.  The epoch only moves once all of them have closed, so every
// thread of the launch reads the same value.
__device__ __forceinline__ Packets channel_open(const purlin_packet_channel &ch) {
    const unsigned long long e = *reinterpret_cast<const volatile unsigned long long *>(ch.state + 2);
    return Packets{ch.staging + (e & 1ull) * ch.capacity * 16ull, (uint32_t)e};
}

// Unit u's payload, from one thread: one 16-byte packet store.  A unit past
// the capacity is skipped and recorded (INVALID_ARG).
__device__ __forceinline__ void send(const purlin_packet_channel &ch, const Packets &pk, uint64_t u,
                                     uint64_t payload) {
    if (u >= ch.capacity) {
        snac::record_error(ch.state, PURLIN_ERR_INVALID_ARG, snac::kSiteChannelArgs, u);
        return;
    }
    if ((int64_t)u == ch.drop_unit) return;   // host-side fault injection
    atom::packet_store(pk.set + 16ull * u, payload, pk.flag);
}

// Unit u's payload of this launch, waiting for it (bounded).  False when the
// wait expired (TIMEOUT recorded), when an earlier wait of the launch gave
// up, or for a unit past the capacity (INVALID_ARG recorded).
__device__ __forceinline__ bool recv(const purlin_packet_channel &ch, const Packets &pk, uint64_t u,
                                     uint64_t *payload) {
    if (u >= ch.capacity) {
        snac::record_error(ch.state, PURLIN_ERR_INVALID_ARG, snac::kSiteChannelArgs, u);
        return false;
    }
    return snac::packet_wait(pk.set + 16ull * u, pk.flag, ch.timeout_ns, ch.state, u, payload);
}

// Every thread of each entering CTA, after its last send or receive.  The
// last CTA of the launch to close advances the epoch: the next launch uses
// the other packet set and the next flag.
__device__ __forceinline__ void channel_close(const purlin_packet_channel &ch) {
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long *epoch = ch.state + 2, *done = ch.state + 3;
        if (atomicAdd(done, 1ull) == (unsigned long long)ch.ctas - 1ull) {
            *done = 0;
            atomicAdd(epoch, 1ull);
        }
    }
}

// One CTA's ring over a single transfer.
//   STAGES          ring depth (>= 2)
//   CHUNK           bytes per stage (a multiple of 128); a copy stages
//                   CHUNK - 16 bytes per chunk (room for a shifted hull), a
//                   reduce of nsrc sources CHUNK / nsrc bytes per source
//   CONSUMER_WARPS  warps that reduce, shift or store vectors (>= 1)
template <int STAGES = 4, int CHUNK = 16384, int CONSUMER_WARPS = 8>
struct Atom {
    static_assert(STAGES >= 2 && STAGES <= 32, "ring depth");
    static_assert(CHUNK >= 256 && CHUNK % 128 == 0, "stage size");
    static_assert(CONSUMER_WARPS >= 1 && CONSUMER_WARPS <= 30, "consumer warps");

    static constexpr int THREADS = 32 * (2 + CONSUMER_WARPS);

  private:
    // workspace: ring | staged table (one segment) and barriers | the
    // transfer's segment | two rank pointers | control | error word
    static constexpr uint32_t kRing = (uint32_t)STAGES * CHUNK + 4u * STAGES * 8u;
    static constexpr uint32_t kTable = kRing;   // run_ring stages the table after the barriers
    static constexpr uint32_t kSeg = kTable + (uint32_t)sizeof(Seg);
    static constexpr uint32_t kPtrs = (kSeg + (uint32_t)sizeof(Seg) + 15u) & ~15u;
    static constexpr uint32_t kCtl = kPtrs + 16u;
    static constexpr uint32_t kErr = kCtl + (uint32_t)sizeof(snac::Ctl);

    struct View {
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

    // One segment from offsets relative to 16-byte aligned bases, cut as the
    // host plan compiler cuts a transfer; chunk counts and units returned.
    __device__ static Seg make_seg(uint64_t src_off, uint64_t dst_off, uint64_t bytes,
                                   int src_rank, uint32_t chunk, uint64_t *nchunks,
                                   uint64_t *nunits) {
        Seg s = {};
        s.src_off = src_off;
        s.dst_off = dst_off;
        s.bytes = bytes;
        s.src_rank = (int8_t)src_rank;
        s.dst_rank = 0;
        s.skip_rank = -1;
        s.chunk_bytes = chunk;
        const Cut cut = cut_transfer(src_off, dst_off, bytes, src_rank < 0);
        if (cut.body > 0) {
            s.tma = 1;
            s.head = (uint8_t)cut.head;
            s.tail = (uint8_t)cut.tail;
            s.shift = (uint8_t)cut.shift;
            *nchunks = (cut.body + chunk - 1) / chunk;
            *nunits = (cut.head ? 1u : 0u) + (cut.tail ? 1u : 0u);
        } else {
            *nchunks = 0;
            *nunits = units_in(unit_grid(src_off, dst_off, src_rank < 0), 0, bytes);
        }
        return s;
    }

    template <int DT, int MAXR>
    __device__ static purlin_status run(unsigned char *ws, const void *const *src, int nsrc,
                                        uint64_t nchunks, uint64_t nunits) {
        const View v{src,
                     reinterpret_cast<void *const *>(ws + kPtrs + 8),
                     nullptr,
                     reinterpret_cast<const Seg *>(ws + kSeg),
                     reinterpret_cast<unsigned long long *>(ws + kErr),
                     nchunks,
                     nunits,
                     0,
                     -1,
                     1,
                     (uint32_t)STAGES,
                     (uint32_t)CHUNK,
                     1,
                     nsrc,
                     0};
        // One transfer whose reduce sources and destination share a phase
        // (reduce() requires 16-byte aligned buffers).
        snac::run_ring<DT, MAXR, false>(v, ws, reinterpret_cast<snac::Ctl *>(ws + kCtl), 0u, 1u,
                                        nullptr, 0);
        return *reinterpret_cast<volatile unsigned long long *>(ws + kErr) != 0ull
                   ? PURLIN_ERR_TIMEOUT
                   : PURLIN_OK;
    }

  public:
    static constexpr uint32_t PIPELINE_SMEM_BYTES = (kErr + 8u + 127u) & ~127u;
    static constexpr uint32_t COPY_PIPELINE_SMEM_BYTES = PIPELINE_SMEM_BYTES;
    static constexpr uint32_t REDUCE_PIPELINE_SMEM_BYTES = PIPELINE_SMEM_BYTES;

    // Bitwise copy of `bytes` bytes (see the header comment for alignment).
    __device__ static purlin_status copy(void *dst, const void *src, size_t bytes,
                                         void *workspace) {
        unsigned char *ws = static_cast<unsigned char *>(workspace);
        const uintptr_t s = reinterpret_cast<uintptr_t>(src), d = reinterpret_cast<uintptr_t>(dst);
        if (!detail::block_shape_ok() || (reinterpret_cast<uintptr_t>(ws) & 127u) != 0)
            return PURLIN_ERR_INVALID_ARG;
        if (((s | d | bytes) & 1u) != 0) return PURLIN_ERR_ALIGNMENT;
        if (bytes == 0) return PURLIN_OK;
        uint64_t nchunks = 0, nunits = 0;
        const Seg seg = make_seg(s & 15u, d & 15u, bytes, 0, (uint32_t)CHUNK - 16u, &nchunks, &nunits);
        __syncthreads();   // the caller is done with the workspace
        if (threadIdx.x == 0) {
            *reinterpret_cast<Seg *>(ws + kSeg) = seg;
            reinterpret_cast<const void **>(ws + kPtrs)[0] = reinterpret_cast<const void *>(s & ~uintptr_t(15));
            reinterpret_cast<void **>(ws + kPtrs)[1] = reinterpret_cast<void *>(d & ~uintptr_t(15));
            *reinterpret_cast<unsigned long long *>(ws + kErr) = 0ull;
        }
        __syncthreads();
        // 2-byte elements: the ragged path moves whole 16-bit words.
        return run<PURLIN_BF16, 8>(ws, reinterpret_cast<const void *const *>(ws + kPtrs), 1,
                                   nchunks, nunits);
    }

    // SCORE reduction of nsrc sources into dst (see the header comment).
    template <int DT>
    __device__ static purlin_status reduce(void *dst, const void *const *srcs, int nsrc,
                                           size_t elems, void *workspace) {
        static_assert(DT == PURLIN_F32 || DT == PURLIN_BF16, "dtype");
        constexpr uint64_t ES = DT == PURLIN_F32 ? 4 : 2;
        unsigned char *ws = static_cast<unsigned char *>(workspace);
        if (!detail::block_shape_ok() || (reinterpret_cast<uintptr_t>(ws) & 127u) != 0 ||
            nsrc < 1 || nsrc > PURLIN_MAX_RANKS || srcs == nullptr)
            return PURLIN_ERR_INVALID_ARG;
        uintptr_t bits = reinterpret_cast<uintptr_t>(dst);
        for (int i = 0; i < nsrc; ++i) bits |= reinterpret_cast<uintptr_t>(srcs[i]);
        if ((bits & 15u) != 0) return PURLIN_ERR_ALIGNMENT;
        if (elems == 0) return PURLIN_OK;
        const uint32_t chunk = ((uint32_t)CHUNK / (uint32_t)nsrc) & ~15u;
        if (chunk < 16u) return PURLIN_ERR_INVALID_ARG;
        uint64_t nchunks = 0, nunits = 0;
        const Seg seg = make_seg(0, 0, elems * ES, kRankAll, chunk, &nchunks, &nunits);
        __syncthreads();   // the caller is done with the workspace
        if (threadIdx.x == 0) {
            *reinterpret_cast<Seg *>(ws + kSeg) = seg;
            reinterpret_cast<void **>(ws + kPtrs)[1] = dst;
            *reinterpret_cast<unsigned long long *>(ws + kErr) = 0ull;
        }
        __syncthreads();
        return nsrc <= 8 ? run<DT, 8>(ws, srcs, nsrc, nchunks, nunits)
                         : run<DT, PURLIN_MAX_RANKS>(ws, srcs, nsrc, nchunks, nunits);
    }
};

}  // namespace device
}  // namespace purlin
