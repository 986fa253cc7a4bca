// atom.cuh -- sm_103a datapath primitives (the "Atom").
//
// "Purlin: Separating Orchestration from the Datapath of Collectives":
//   §3.3  the Atom offers copy and reduce through a pipeline that stages
//         data in CTA-local shared memory so asynchronous fetches overlap
//         with processing; SCORE: each output element belongs to one
//         thread, which accumulates the sources in a fixed order, with
//         several independent accumulators and pipelined source fetches.
//   §3.2  SNAC: stage, notify (a flag carrying the epoch, §4.3), consume.
// "Purlin" project README, "Atom implementations": a generic vectorised
// load/store Atom plus per-generation ones (here: the Blackwell bulk-copy
// engine driven from one elected thread, with mbarrier completion).
//
// Everything here is hand-written inline PTX for sm_103a.
#pragma once

#include <cstdint>

#include "../../include/purlin.h"

namespace purlin {
namespace atom {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------- mbarrier --

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Retire a barrier whose every phase has completed, before its shared
// memory is used for anything else (including a new mbarrier).
__device__ __forceinline__ void mbar_inval(uint64_t *bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Make barrier initialisation visible to the bulk-copy engine.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_count(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Arrive once and add `bytes` to the transaction count of the current phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// True once the phase with parity `parity` has completed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// ------------------------------------------------------ bulk async copies --

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Global -> shared, completion counted on `bar` (bytes: multiple of 16,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gsrc, uint32_t bytes,
                                          uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Shared -> global, tracked by the issuing thread's bulk async-groups.
__device__ __forceinline__ void bulk_store(void *gdst, const void *smem_src, uint32_t bytes,
                                           uint64_t policy) {
    asm volatile(
        "cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(
            gdst),
        "r"(smem_u32(smem_src)), "r"(bytes), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's bulk groups still READ shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N of this thread's bulk groups are incomplete (writes
// performed and visible to this thread).
template <int N>
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The same ordering for global memory (between bulk copies and flags).
__device__ __forceinline__ void fence_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ---------------------------------------------------------------- flags --

// Acquire-release fence at GPU scope (lighter than a sequentially consistent
// one): orders everything this thread has observed before the stores after it.
__device__ __forceinline__ void fence_acq_rel_gpu() {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

__device__ __forceinline__ void flag_release(unsigned long long *f, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(f), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long flag_acquire(const unsigned long long *f) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(f) : "memory");
    return v;
}

// ------------------------------------------------------------- packets --
//
// The latency path's payload+notification packet ("Purlin: Separating Orchestration from the Datapath of Collectives"
// §3.2): 16
// bytes holding 8 payload bytes and the call's 32-bit flag twice, as two
// 8-byte lines {payload word, flag}.  The store is one v2.u64 access whose
// two 64-bit elements are each single-copy atomic (aligned 64-bit accesses),
// so a reader that sees a line's flag sees that line's payload: no fence
// and no separate flag store.  Half of every packet is flag, which doubles
// the bytes moved, as the pages say of their packets.

__device__ __forceinline__ void packet_store(void *p, uint64_t payload, uint32_t flag) {
    const uint64_t a = (payload & 0xFFFFFFFFull) | ((uint64_t)flag << 32);
    const uint64_t b = (payload >> 32) | ((uint64_t)flag << 32);
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b)
                 : "memory");
}

// True, with the payload, once both lines of the packet carry `flag`.
__device__ __forceinline__ bool packet_load(const void *p, uint32_t flag, uint64_t *payload) {
    uint64_t a, b;
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p)
                 : "memory");
    if ((uint32_t)(a >> 32) != flag || (uint32_t)(b >> 32) != flag) return false;
    *payload = (a & 0xFFFFFFFFull) | (b << 32);
    return true;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------- 128-bit vector access --

__device__ __forceinline__ uint4 ld_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 128-bit load that may allocate in L1: the shifted path reads each source
// vector from two neighbouring threads.
__device__ __forceinline__ uint4 ld_v4_l1(const void *p) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Bytes [sh, sh + 16) of the 32-byte pair (a, b), 0 <= sh < 16.
__device__ __forceinline__ uint4 shift_pair(uint4 a, uint4 b, uint32_t sh) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    const uint32_t k = sh >> 2, r = (sh & 3u) * 8u;
    uint32_t o[5];
#pragma unroll
    for (int i = 0; i < 5; ++i)
        o[i] = k == 0 ? w[i] : k == 1 ? w[i + 1] : k == 2 ? w[i + 2] : w[i + 3];
    return make_uint4(__funnelshift_r(o[0], o[1], r), __funnelshift_r(o[1], o[2], r),
                      __funnelshift_r(o[2], o[3], r), __funnelshift_r(o[3], o[4], r));
}

__device__ __forceinline__ void st_v4(void *p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint4 lds_v4(const void *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}

__device__ __forceinline__ uint32_t lds_u32(const void *p) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)));
    return v;
}

// 16 bytes of shared memory starting at p + sh (p 16-byte aligned, sh < 16
// and even): five aligned 32-bit words, funnel-shifted into place.
__device__ __forceinline__ uint4 lds_v4_shifted(const unsigned char *p, uint32_t sh) {
    const unsigned char *q = p + (sh & ~3u);
    const uint32_t r = (sh & 3u) * 8u;
    const uint32_t w0 = lds_u32(q), w1 = lds_u32(q + 4), w2 = lds_u32(q + 8),
                   w3 = lds_u32(q + 12), w4 = lds_u32(q + 16);
    return make_uint4(__funnelshift_r(w0, w1, r), __funnelshift_r(w1, w2, r),
                      __funnelshift_r(w2, w3, r), __funnelshift_r(w3, w4, r));
}

__device__ __forceinline__ void sts_v4(void *p, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(p)), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// ------------------------------------------------ SCORE accumulate (§3.3) --
//
// A 16-byte vector holds VE elements: 4 fp32 or 8 bf16.  Accumulation is
// binary32 with explicit round-to-nearest adds (no contraction), in the
// order the caller feeds the sources; the accumulator starts from the first
// source's value; conversion to bf16 happens once, at the end.

template <int DT>
struct Vec;

template <>
struct Vec<PURLIN_F32> {
    static constexpr int VE = 4;
    __device__ __forceinline__ static void init(float (&a)[4], uint4 v) {
        a[0] = __uint_as_float(v.x);
        a[1] = __uint_as_float(v.y);
        a[2] = __uint_as_float(v.z);
        a[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static void add(float (&a)[4], uint4 v) {
        a[0] = __fadd_rn(a[0], __uint_as_float(v.x));
        a[1] = __fadd_rn(a[1], __uint_as_float(v.y));
        a[2] = __fadd_rn(a[2], __uint_as_float(v.z));
        a[3] = __fadd_rn(a[3], __uint_as_float(v.w));
    }
    __device__ __forceinline__ static uint4 pack(const float (&a)[4]) {
        return make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                          __float_as_uint(a[3]));
    }
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two binary32 values -> one word of two bf16 (round to nearest even);
// `lo` lands in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

template <>
struct Vec<PURLIN_BF16> {
    static constexpr int VE = 8;
    __device__ __forceinline__ static void init(float (&a)[8], uint4 v) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            a[2 * j] = bf16_lo(w[j]);
            a[2 * j + 1] = bf16_hi(w[j]);
        }
    }
    __device__ __forceinline__ static void add(float (&a)[8], uint4 v) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            a[2 * j] = __fadd_rn(a[2 * j], bf16_lo(w[j]));
            a[2 * j + 1] = __fadd_rn(a[2 * j + 1], bf16_hi(w[j]));
        }
    }
    __device__ __forceinline__ static uint4 pack(const float (&a)[8]) {
        return make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]),
                          pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7]));
    }
};

// Scalar element access for the ragged path.
template <int DT>
__device__ __forceinline__ float load_elem(const char *p);
template <>
__device__ __forceinline__ float load_elem<PURLIN_F32>(const char *p) {
    return __uint_as_float(*reinterpret_cast<const uint32_t *>(p));
}
template <>
__device__ __forceinline__ float load_elem<PURLIN_BF16>(const char *p) {
    return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(p)) << 16);
}

template <int DT>
__device__ __forceinline__ void store_elem(char *p, float v);
template <>
__device__ __forceinline__ void store_elem<PURLIN_F32>(char *p, float v) {
    *reinterpret_cast<uint32_t *>(p) = __float_as_uint(v);
}
template <>
__device__ __forceinline__ void store_elem<PURLIN_BF16>(char *p, float v) {
    *reinterpret_cast<uint16_t *>(p) = static_cast<uint16_t>(pack_bf16x2(v, 0.0f) & 0xFFFFu);
}

}  // namespace atom
}  // namespace purlin
