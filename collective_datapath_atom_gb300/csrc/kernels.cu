// kernels.cu -- the two kernel families of the single-GPU Purlin datapath.
//
// "Purlin: Separating Orchestration from the Datapath of Collectives":
//   §2.1  prefill payloads are throughput-bound, decode messages latency-
//         bound; a high-bandwidth path's setup dominates small messages.
//   §3.2  SNAC: chunks are staged, their readiness is notified, consumers
//         then copy or reduce them; composed AllReduce overlaps staging,
//         reduction and gathering on chunks; push for latency, pull for
//         bandwidth (one GPU: the vector kernel vs the staged ring).
//   §3.3  the Atom pipeline stages data in CTA-local shared memory so
//         fetches overlap with processing; SCORE reductions; in-flight
//         capacity near the bandwidth-delay product with few CTAs.
//   §4.3  a monotonic 64-bit epoch is the notification value and its
//         parity selects the buffer set.
//
// Latency kernel: one thread per 16-byte destination window ("unit");
//   128-bit loads of every source, ordered binary32 accumulation, 128-bit
//   stores to every destination.  No flags: each output has one owner.
// Throughput kernel: persistent CTAs with three warp roles over a ring of
//   shared-memory stages.
//   warp 0 (one lane)  Stage: cp.async.bulk global -> shared for the chunk
//                      (R tiles for a reduce, one for a copy), completion on
//                      the stage's mbarrier.  For a chunk that depends on
//                      another CTA's chunk it first acquires that chunk's
//                      flag (bounded spin).
//   warps 2..          Consume (reduce): SCORE over the R tiles into an
//                      output tile; also the ragged head/tail units.
//   warp 1 (one lane)  Consume (copy) / write-back: cp.async.bulk shared ->
//                      global to one or all destinations; then Notify:
//                      once a chunk's stores have completed, release-store
//                      epoch + generation into its flag.
// Every wait is bounded; an expired wait records PURLIN_ERR_TIMEOUT in the
// error word and the CTA winds down (its own bulk copies are waited for).
#include <cuda_runtime.h>

#include "atom.cuh"
#include "launch.h"

namespace purlin {

namespace {

constexpr int kNotifyLag = 4;      // bulk groups kept in flight before notifying
constexpr int kNotifyQueue = 16;
constexpr int kTputMaxThreads = 512;
constexpr uint64_t kRingWaitNs = 2000000000ull;   // 2 s bound on a ring wait

template <int MAXR, int MAXSEG>
struct KParams {
    const void *src[MAXR];
    void *dst[MAXR];
    Seg segs[MAXSEG];
    const Seg *segs_dev;
    unsigned long long *flags;
    unsigned long long *err;
    uint64_t nchunks;
    uint64_t nunits;
    uint64_t epoch;
    int64_t timeout_ns;
    int64_t drop_notify;
    uint32_t flag_slots;
    uint32_t stages;
    uint32_t slot_stride;
    uint32_t out_tile;
    int32_t nseg;
    int32_t R;
};

template <class P>
__device__ __forceinline__ const Seg *seg_table(const P &p) {
    return p.segs_dev != nullptr ? p.segs_dev : p.segs;
}

// Last segment whose first chunk (unit) index is <= x: the one holding x.
__device__ __forceinline__ int seg_of_chunk(const Seg *segs, int nseg, uint64_t x) {
    int lo = 0, hi = nseg;   // answer in [lo, hi)
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if ((uint64_t)segs[mid].chunk_begin <= x) lo = mid;
        else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ int seg_of_unit(const Seg *segs, int nseg, uint64_t x) {
    int lo = 0, hi = nseg;
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (segs[mid].unit_begin <= x) lo = mid;
        else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ void record_error(unsigned long long *err, uint64_t code, uint64_t site,
                                             uint64_t where) {
    unsigned long long v = (unsigned long long)((code & 0xFF) | ((site & 0xFF) << 8) |
                                                ((where & 0xFFFFFFFFFFFFull) << 16));
    atomicCAS(err, 0ull, v);
}

__device__ __forceinline__ bool error_set(const unsigned long long *err) {
    return *reinterpret_cast<const volatile unsigned long long *>(err) != 0ull;
}

// ------------------------------------------------------------ vector unit --

// One 16-byte destination window of a segment: copy or reduce it to every
// destination.  A full window whose source is 16-byte aligned uses 128-bit
// accesses; anything else goes element by element.
template <int DT, int MAXR, class P>
__device__ void do_unit(const P &p, const Seg &sg, uint64_t k) {
    using V = atom::Vec<DT>;
    constexpr int ES = DT == PURLIN_F32 ? 4 : 2;
    uint64_t lo, hi;
    if (sg.tma) {
        if (k == 0 && sg.head) {
            lo = 0;
            hi = sg.head;
        } else {
            lo = sg.bytes - sg.tail;
            hi = sg.bytes;
        }
    } else {
        const uint64_t a = (sg.dst_off / 16 + k) * 16;
        lo = (a > sg.dst_off ? a : sg.dst_off) - sg.dst_off;
        const uint64_t b = a + 16, e = sg.dst_off + sg.bytes;
        hi = (b < e ? b : e) - sg.dst_off;
    }
    const int R = p.R;
    const bool vec = (hi - lo == 16) && (((sg.src_off + lo) & 15u) == 0);
    const uint64_t doff = sg.dst_off + lo;

    if (sg.src_rank >= 0) {   // copy, bitwise
        const char *s = static_cast<const char *>(sg.src_is_dst ? p.dst[sg.src_rank]
                                                                : p.src[sg.src_rank]) +
                        sg.src_off + lo;
        auto put = [&](char *d) {
            if (d == s) return;   // in-place AllGather: the block is already there
            if (vec) {
                atom::st_v4(d, atom::ld_v4(s));
            } else {
                for (uint64_t j = 0; j < hi - lo; j += ES) {
                    if (ES == 4)
                        *reinterpret_cast<uint32_t *>(d + j) =
                            *reinterpret_cast<const uint32_t *>(s + j);
                    else
                        *reinterpret_cast<uint16_t *>(d + j) =
                            *reinterpret_cast<const uint16_t *>(s + j);
                }
            }
        };
        if (sg.dst_rank >= 0) {
            put(static_cast<char *>(p.dst[sg.dst_rank]) + doff);
        } else {
            for (int d = 0; d < R; ++d)
                if (d != sg.skip_rank) put(static_cast<char *>(p.dst[d]) + doff);
        }
        return;
    }

    // reduce (SCORE): rank order 0..R-1, binary32, one rounding at the end
    const uint64_t soff = sg.src_off + lo;
    if (vec) {
        float acc[V::VE];
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < R) v[j] = atom::ld_v4(static_cast<const char *>(p.src[j]) + soff);
        V::init(acc, v[0]);
#pragma unroll
        for (int j = 1; j < 8; ++j)
            if (j < R) V::add(acc, v[j]);
        if (MAXR > 8) {
            for (int s0 = 8; s0 < R; s0 += 8) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (s0 + j < R)
                        v[j] = atom::ld_v4(static_cast<const char *>(p.src[s0 + j]) + soff);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (s0 + j < R) V::add(acc, v[j]);
            }
        }
        const uint4 out = V::pack(acc);
        if (sg.dst_rank >= 0) {
            atom::st_v4(static_cast<char *>(p.dst[sg.dst_rank]) + doff, out);
        } else {
            for (int d = 0; d < R; ++d)
                if (d != sg.skip_rank) atom::st_v4(static_cast<char *>(p.dst[d]) + doff, out);
        }
        return;
    }
    for (uint64_t j = 0; j < hi - lo; j += ES) {
        float acc = atom::load_elem<DT>(static_cast<const char *>(p.src[0]) + soff + j);
        for (int s = 1; s < R; ++s)
            acc = __fadd_rn(acc, atom::load_elem<DT>(static_cast<const char *>(p.src[s]) + soff + j));
        if (sg.dst_rank >= 0) {
            atom::store_elem<DT>(static_cast<char *>(p.dst[sg.dst_rank]) + doff + j, acc);
        } else {
            for (int d = 0; d < R; ++d)
                if (d != sg.skip_rank)
                    atom::store_elem<DT>(static_cast<char *>(p.dst[d]) + doff + j, acc);
        }
    }
}

// ---------------------------------------------------------- latency kernel --

template <int DT, int MAXR, int MAXSEG>
__global__ void __launch_bounds__(256) purlin_latency_kernel(
    const __grid_constant__ KParams<MAXR, MAXSEG> p) {
    const Seg *segs = seg_table(p);
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t u = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; u < p.nunits; u += stride) {
        const Seg &sg = segs[seg_of_unit(segs, p.nseg, u)];
        do_unit<DT, MAXR>(p, sg, u - sg.unit_begin);
    }
}

// ------------------------------------------------------- throughput kernel --

struct ChunkGeo {
    const Seg *sg;
    uint64_t ci;      // chunk index within the segment
    uint64_t off;     // byte offset of the chunk within the segment
    uint32_t bytes;   // bytes per source
};

__device__ __forceinline__ ChunkGeo chunk_geo(const Seg *segs, int nseg, uint64_t c) {
    ChunkGeo g;
    g.sg = &segs[seg_of_chunk(segs, nseg, c)];
    const Seg &sg = *g.sg;
    g.ci = c - sg.chunk_begin;
    const uint64_t body = sg.bytes - sg.head - sg.tail;
    const uint64_t done = g.ci * sg.chunk_bytes;
    g.off = sg.head + done;
    const uint64_t rem = body - done;
    g.bytes = (uint32_t)(rem < sg.chunk_bytes ? rem : sg.chunk_bytes);
    return g;
}

struct Ctl {
    int abort;
};

// Bounded wait on an mbarrier phase.  `abortable`: give up as soon as
// another role of the CTA has given up.
__device__ __forceinline__ bool ring_wait(uint64_t *bar, uint32_t parity, volatile Ctl *ctl,
                                          unsigned long long *err, uint64_t site, bool abortable) {
    if (atom::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = atom::globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (atom::mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 0) {
            if (abortable && ctl->abort) return false;
            if (atom::globaltimer_ns() - t0 > kRingWaitNs) {
                record_error(err, PURLIN_ERR_TIMEOUT, site, blockIdx.x);
                ctl->abort = 1;
                return false;
            }
        }
    }
}

// SNAC consume-side acquire: wait until the producing chunk's flag holds at
// least this call's value for it.  Bounded; on expiry the error word is set
// and later waits of the launch are skipped.
template <class P>
__device__ void acquire_chunk(const P &p, uint64_t dep) {
    if (error_set(p.err)) return;
    const unsigned long long *f = p.flags + (dep % p.flag_slots);
    const unsigned long long want = p.epoch + dep / p.flag_slots;
    if (atom::flag_acquire(f) < want) {
        const uint64_t t0 = atom::globaltimer_ns();
        uint32_t ns = 32;
        while (atom::flag_acquire(f) < want) {
            if ((int64_t)(atom::globaltimer_ns() - t0) > p.timeout_ns) {
                record_error(p.err, PURLIN_ERR_TIMEOUT, kSiteFlagWait, dep);
                return;
            }
            __nanosleep(ns);
            if (ns < 1024) ns <<= 1;
        }
    }
    atom::fence_async_global();   // the staged reads below are async-proxy reads
}

// SNAC notify: publish a completed chunk (its stores are complete and
// ordered before this store by the caller).
template <class P>
__device__ __forceinline__ void notify_chunk(const P &p, uint64_t c) {
    if ((int64_t)c == p.drop_notify) return;   // host-side fault injection
    atom::flag_release(p.flags + (c % p.flag_slots), p.epoch + c / p.flag_slots);
}

template <int DT, int MAXR, int MAXSEG>
__global__ void __launch_bounds__(kTputMaxThreads, 1) purlin_throughput_kernel(
    const __grid_constant__ KParams<MAXR, MAXSEG> p) {
    using V = atom::Vec<DT>;
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ Ctl ctl;

    const Seg *segs = seg_table(p);
    const uint32_t S = p.stages;
    const int R = p.R;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ncw = (int)(blockDim.x >> 5) - 2;   // consumer warps

    unsigned char *ring = smem;
    unsigned char *outt = smem + (size_t)S * p.slot_stride;
    uint64_t *bars = reinterpret_cast<uint64_t *>(outt + 2 * (size_t)p.out_tile);
    uint64_t *full = bars;             // S: producer arrive + transaction bytes
    uint64_t *empty = bars + S;        // S: ncw arrivals (consumer warps, or the writer)
    uint64_t *ofull = bars + 2 * S;    // 2: ncw arrivals (consumer warps)
    uint64_t *ofree = bars + 2 * S + 2;// 2: writer arrival

    if (threadIdx.x == 0) {
        for (uint32_t i = 0; i < S; ++i) {
            atom::mbar_init(&full[i], 1);
            atom::mbar_init(&empty[i], (uint32_t)ncw);
        }
        for (int i = 0; i < 2; ++i) {
            atom::mbar_init(&ofull[i], (uint32_t)ncw);
            atom::mbar_init(&ofree[i], 1);
        }
        ctl.abort = 0;
        atom::mbar_init_fence();
    }
    __syncthreads();

    if (warp == 0) {
        // ---------------------------------------------------------- Stage --
        if (lane == 0) {
            const uint64_t pol = atom::policy_evict_first();
            uint32_t k = 0;
            for (uint64_t c = blockIdx.x; c < p.nchunks; c += gridDim.x, ++k) {
                const uint32_t slot = k % S;
                if (k >= S && !ring_wait(&empty[slot], ((k / S) & 1u) ^ 1u, &ctl, p.err,
                                         kSiteRingEmpty, true))
                    break;
                const ChunkGeo g = chunk_geo(segs, p.nseg, c);
                const Seg &sg = *g.sg;
                if (sg.sync == kSyncWait) acquire_chunk(p, sg.dep_chunk + g.ci);
                unsigned char *sp = ring + (size_t)slot * p.slot_stride;
                if (sg.src_rank < 0) {
                    atom::mbar_arrive_expect_tx(&full[slot], g.bytes * (uint32_t)R);
                    for (int s = 0; s < R; ++s)
                        atom::bulk_load(sp + (size_t)s * sg.chunk_bytes,
                                        static_cast<const char *>(p.src[s]) + sg.src_off + g.off,
                                        g.bytes, &full[slot], pol);
                } else {
                    const char *base = static_cast<const char *>(
                        sg.src_is_dst ? p.dst[sg.src_rank] : p.src[sg.src_rank]);
                    atom::mbar_arrive_expect_tx(&full[slot], g.bytes);
                    atom::bulk_load(sp, base + sg.src_off + g.off, g.bytes, &full[slot], pol);
                }
            }
            // Every load this thread issued must land before the CTA exits.
            const uint32_t issued = k;
            for (uint32_t j = issued > S ? issued - S : 0; j < issued; ++j)
                ring_wait(&full[j % S], (j / S) & 1u, &ctl, p.err, kSiteRingFull, false);
        }
    } else if (warp == 1) {
        // ----------------------------------------- write-back and Notify --
        if (lane == 0) {
            const uint64_t pol = atom::policy_evict_first();
            uint32_t k = 0, kr = 0;
            int owed_kind = 0;          // staging owed back for the newest group: 1 out tile, 2 slot
            uint32_t owed_idx = 0;
            uint64_t q_chunk[kNotifyQueue] = {}, q_group[kNotifyQueue] = {};
            uint32_t q_head = 0, q_tail = 0;
            uint64_t group = 0;
            auto settle = [&]() {
                if (owed_kind == 1) atom::mbar_arrive(&ofree[owed_idx]);
                else if (owed_kind == 2) atom::mbar_arrive_count(&empty[owed_idx], (uint32_t)ncw);
                owed_kind = 0;
            };
            auto retire = [&](uint64_t upto) {
                while (q_head != q_tail && q_group[q_head % kNotifyQueue] <= upto) {
                    notify_chunk(p, q_chunk[q_head % kNotifyQueue]);
                    ++q_head;
                }
            };
            for (uint64_t c = blockIdx.x; c < p.nchunks; c += gridDim.x, ++k) {
                const ChunkGeo g = chunk_geo(segs, p.nseg, c);
                const Seg &sg = *g.sg;
                const unsigned char *from;
                const char *self = nullptr;
                int kind;
                uint32_t idx;
                if (sg.src_rank < 0) {
                    idx = kr & 1u;
                    if (!ring_wait(&ofull[idx], (kr >> 1) & 1u, &ctl, p.err, kSiteOutFull, true))
                        break;
                    from = outt + (size_t)idx * p.out_tile;
                    kind = 1;
                    ++kr;
                } else {
                    if (sg.sync == kSyncWait && q_head != q_tail) {
                        // Publish everything before possibly waiting on others.
                        atom::bulk_wait_all<0>();
                        settle();
                        atom::fence_async_global();
                        retire(group);
                    }
                    idx = k % S;
                    if (!ring_wait(&full[idx], (k / S) & 1u, &ctl, p.err, kSiteRingFull, true))
                        break;
                    from = ring + (size_t)idx * p.slot_stride;
                    kind = 2;
                    self = static_cast<const char *>(sg.src_is_dst ? p.dst[sg.src_rank]
                                                                   : p.src[sg.src_rank]) +
                           sg.src_off + g.off;
                }
                const uint64_t doff = sg.dst_off + g.off;
                if (sg.dst_rank >= 0) {
                    char *d = static_cast<char *>(p.dst[sg.dst_rank]) + doff;
                    if (d != self) atom::bulk_store(d, from, g.bytes, pol);
                } else {
                    for (int d = 0; d < R; ++d) {
                        if (d == sg.skip_rank) continue;
                        char *dp = static_cast<char *>(p.dst[d]) + doff;
                        if (dp != self) atom::bulk_store(dp, from, g.bytes, pol);
                    }
                }
                atom::bulk_commit();
                ++group;
                if (sg.sync == kSyncNotify) {
                    q_chunk[q_tail % kNotifyQueue] = c;
                    q_group[q_tail % kNotifyQueue] = group;
                    ++q_tail;
                }
                // The previous group has finished reading its staging: hand it back.
                atom::bulk_wait_read<1>();
                settle();
                owed_kind = kind;
                owed_idx = idx;
                if (q_head != q_tail && q_group[q_head % kNotifyQueue] + kNotifyLag <= group) {
                    atom::bulk_wait_all<kNotifyLag>();
                    atom::fence_async_global();
                    retire(group - kNotifyLag);
                }
            }
            atom::bulk_wait_all<0>();
            settle();
            atom::fence_async_global();
            retire(group);
        }
    } else {
        // --------------------------------------------- Consume (reduce) --
        const int ctid = (int)threadIdx.x - 64;
        const int nct = (int)blockDim.x - 64;
        const uint64_t ustride = (uint64_t)gridDim.x * nct;
        for (uint64_t u = (uint64_t)blockIdx.x * nct + ctid; u < p.nunits; u += ustride) {
            const Seg &sg = segs[seg_of_unit(segs, p.nseg, u)];
            do_unit<DT, MAXR>(p, sg, u - sg.unit_begin);
        }
        uint32_t k = 0, kr = 0;
        for (uint64_t c = blockIdx.x; c < p.nchunks; c += gridDim.x, ++k) {
            const ChunkGeo g = chunk_geo(segs, p.nseg, c);
            const Seg &sg = *g.sg;
            if (sg.src_rank >= 0) continue;
            const uint32_t slot = k % S;
            const uint32_t b = kr & 1u;
            // Every lane waits (bounded) and the warp leaves together.
            bool ok = ring_wait(&full[slot], (k / S) & 1u, &ctl, p.err, kSiteRingFull, true);
            if (ok && kr >= 2)
                ok = ring_wait(&ofree[b], ((kr >> 1) & 1u) ^ 1u, &ctl, p.err, kSiteOutFree, true);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            const unsigned char *sp = ring + (size_t)slot * p.slot_stride;
            unsigned char *op = outt + (size_t)b * p.out_tile;
            const uint32_t cb = sg.chunk_bytes;
            const int nvec = (int)(g.bytes >> 4);
            for (int v = ctid; v < nvec; v += nct) {
                float acc[V::VE];
                const unsigned char *t = sp + 16 * (size_t)v;
                V::init(acc, atom::lds_v4(t));
                if (MAXR <= 8) {
#pragma unroll
                    for (int s = 1; s < MAXR; ++s)
                        if (s < R) V::add(acc, atom::lds_v4(t + (size_t)s * cb));
                } else {
#pragma unroll 8
                    for (int s = 1; s < R; ++s) V::add(acc, atom::lds_v4(t + (size_t)s * cb));
                }
                atom::sts_v4(op + 16 * (size_t)v, V::pack(acc));
            }
            atom::fence_async_shared();
            __syncwarp();
            if (lane == 0) {
                atom::mbar_arrive(&empty[slot]);
                atom::mbar_arrive(&ofull[b]);
            }
            ++kr;
        }
    }
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
    p.err = a.err;
    p.nchunks = pl.nchunks;
    p.nunits = pl.nunits;
    p.epoch = a.epoch;
    p.timeout_ns = a.timeout_ns;
    p.drop_notify = a.drop_notify;
    p.flag_slots = a.flag_slots;
    p.stages = a.stages;
    p.slot_stride = a.slot_stride;
    p.out_tile = pl.has_reduce ? pl.red_chunk : 0;
    p.nseg = (int32_t)nseg;
    p.R = a.R;
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

template <template <int, int, int> class F>
struct Dispatch;

}  // namespace

int param_class(int R, size_t nseg) {
    if (R <= kSmallMaxR && nseg <= (size_t)kSmallMaxSeg) return 0;
    if (nseg <= (size_t)kBigMaxSeg) return 1;
    return -1;
}

uint32_t throughput_smem(uint32_t stages, uint32_t slot_stride, uint32_t out_tile) {
    return stages * slot_stride + 2 * out_tile + (2 * stages + 4) * 8;
}

cudaError_t launch_latency(const LaunchArgs &a) {
    const int pc = a.segs_dev ? 1 : param_class(a.R, a.plan->segs.size());
    if (a.dtype == PURLIN_F32)
        return pc == 0 ? launch_lat_t<PURLIN_F32, kSmallMaxR, kSmallMaxSeg>(a)
                       : launch_lat_t<PURLIN_F32, kBigMaxR, kBigMaxSeg>(a);
    return pc == 0 ? launch_lat_t<PURLIN_BF16, kSmallMaxR, kSmallMaxSeg>(a)
                   : launch_lat_t<PURLIN_BF16, kBigMaxR, kBigMaxSeg>(a);
}

cudaError_t launch_throughput(const LaunchArgs &a) {
    const int pc = a.segs_dev ? 1 : param_class(a.R, a.plan->segs.size());
    if (a.dtype == PURLIN_F32)
        return pc == 0 ? launch_tput_t<PURLIN_F32, kSmallMaxR, kSmallMaxSeg>(a)
                       : launch_tput_t<PURLIN_F32, kBigMaxR, kBigMaxSeg>(a);
    return pc == 0 ? launch_tput_t<PURLIN_BF16, kSmallMaxR, kSmallMaxSeg>(a)
                   : launch_tput_t<PURLIN_BF16, kBigMaxR, kBigMaxSeg>(a);
}

cudaError_t configure_kernels(int max_dyn_smem) {
    cudaError_t e;
#define PURLIN_SET(DT, MR, MS)                                                                \
    e = cudaFuncSetAttribute(purlin_throughput_kernel<DT, MR, MS>,                           \
                             cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn_smem);     \
    if (e != cudaSuccess) return e;
    PURLIN_SET(PURLIN_F32, kSmallMaxR, kSmallMaxSeg)
    PURLIN_SET(PURLIN_F32, kBigMaxR, kBigMaxSeg)
    PURLIN_SET(PURLIN_BF16, kSmallMaxR, kSmallMaxSeg)
    PURLIN_SET(PURLIN_BF16, kBigMaxR, kBigMaxSeg)
#undef PURLIN_SET
    return cudaSuccess;
}

cudaError_t throughput_occupancy(int dtype, int pclass, int block, size_t smem, int *per_sm) {
    if (dtype == PURLIN_F32)
        return pclass == 0 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                 per_sm, purlin_throughput_kernel<PURLIN_F32, kSmallMaxR, kSmallMaxSeg>,
                                 block, smem)
                           : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                 per_sm, purlin_throughput_kernel<PURLIN_F32, kBigMaxR, kBigMaxSeg>,
                                 block, smem);
    return pclass == 0 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                             per_sm, purlin_throughput_kernel<PURLIN_BF16, kSmallMaxR, kSmallMaxSeg>,
                             block, smem)
                       : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                             per_sm, purlin_throughput_kernel<PURLIN_BF16, kBigMaxR, kBigMaxSeg>,
                             block, smem);
}

}  // namespace purlin
