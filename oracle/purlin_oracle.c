/*
 * purlin_oracle.c -- plain, slow, obviously correct CPU oracle for the seven
 * non-rooted collectives of Purlin (AllGather, AllGatherV, ReduceScatter,
 * ReduceScatterV, AllReduce, AllToAll, AllToAllV) over R rank buffers held in
 * one address space.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this file's library.  The product
 * library never links, loads or calls it, and this file includes nothing from
 * the product (no shared headers, tables or helpers).
 *
 * Sources (page title, then section):
 *   [P2] "Purlin: Separating Orchestration from the Datapath of Collectives"
 *        §2.1: collective contracts are fixed independently of
 *        the communication steps; variable-length variants let contributions
 *        or partitions differ in size.  §3.1 layouts: packed, scattered,
 *        transposed; AllReduce is ReduceScatter followed by AllGather.  §3.3
 *        SCORE: one thread owns each output element and accumulates the
 *        sources in a fixed order, which makes the reduction deterministic.
 *        §C.4 variable-length collectives: AllGatherV contributes each rank's
 *        share, ReduceScatterV outputs that share, AllToAllV sends/receives
 *        per-pair partitions.
 *   [P4] "Purlin" (project README): "Understanding totalBytes" (AllGather
 *        output is all contributions, per-rank input otherwise);
 *        "Deterministic Reduction" (bit-wise repeatable results for the same
 *        inputs and operator).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - Accumulation is binary32, in rank order 0..R-1, starting from the
 *     value of rank 0 (not from +0.0), rounded once to the output type.
 *   - bf16 rounding is round-to-nearest-even; a NaN becomes the quiet NaN
 *     0x7FC0.  Copies are bitwise (NaN payloads and -0.0 survive).
 *   - ReduceScatter and AllToAll need n divisible by R; the V variants cover
 *     ragged splits.
 *   - AllToAllV input of rank s is packed by destination in destination
 *     order; output of rank d is packed by source in source order.
 *
 * Build: gcc -O2 -fno-fast-math -ffp-contract=off -std=c99 -shared -fPIC.
 * Each float addition below is one IEEE binary32 addition (FLT_EVAL_METHOD
 * 0 on both x86-64 SSE and AArch64), so the result is fixed by the order.
 *
 * The same source is also built with -fopenmp, for the CPU baseline leg of
 * the benchmark over all host cores.  Only the element loops are split
 * across threads (PARALLEL_ELEMENTS); each element is still computed by one
 * thread with the same operations in the same order, so both builds give
 * the same bits.  Without -fopenmp the macro is empty.
 */
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#define PARALLEL_ELEMENTS _Pragma("omp parallel for schedule(static)")
#else
#define PARALLEL_ELEMENTS
#endif

#define ORACLE_F32 0
#define ORACLE_BF16 1

/* Threads the element loops use: sets the count first when k > 0.  The
 * single-threaded build ignores k and returns 1. */
int oracle_threads(int k) {
#ifdef _OPENMP
    if (k > 0) omp_set_num_threads(k);
    return omp_get_max_threads();
#else
    (void)k;
    return 1;
#endif
}

/* ------------------------------------------------------------------ */
/* bf16 codec, written from the definition of the formats.             */
/* ------------------------------------------------------------------ */

/* bf16 is the top 16 bits of a binary32, so widening is exact. */
uint32_t oracle_bf16_to_f32_bits(uint16_t b) { return ((uint32_t)b) << 16; }

/* Round a binary32 bit pattern to bf16, nearest with ties to even.
 * Adding 0x7FFF plus the lowest kept bit carries into bit 16 exactly when
 * the dropped half is above one half, or equal to one half with an odd kept
 * part.  A carry out of the mantissa moves into the exponent, which is the
 * right result (including rounding the largest finite value up to inf). */
uint16_t oracle_f32_bits_to_bf16(uint32_t u) {
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u) {
        return (uint16_t)0x7FC0u;
    }
    uint32_t kept_lsb = (u >> 16) & 1u;
    u += 0x7FFFu + kept_lsb;
    return (uint16_t)(u >> 16);
}

/* The same rounding over an array (lets the tests sweep millions of patterns). */
void oracle_f32_bits_to_bf16_n(const uint32_t *in, uint16_t *out, size_t n) {
    for (size_t i = 0; i < n; ++i) out[i] = oracle_f32_bits_to_bf16(in[i]);
}

static float bits_to_f32(uint32_t u) {
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t f32_to_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

static int elem_size(int dtype) {
    if (dtype == ORACLE_F32) return 4;
    if (dtype == ORACLE_BF16) return 2;
    return 0;
}

static float load_as_f32(int dtype, const void *buf, size_t i) {
    if (dtype == ORACLE_F32) {
        float f;
        memcpy(&f, (const char *)buf + 4 * i, 4);
        return f;
    }
    uint16_t b;
    memcpy(&b, (const char *)buf + 2 * i, 2);
    return bits_to_f32(oracle_bf16_to_f32_bits(b));
}

static void store_rounded(int dtype, void *buf, size_t i, float v) {
    if (dtype == ORACLE_F32) {
        memcpy((char *)buf + 4 * i, &v, 4);
        return;
    }
    uint16_t b = oracle_f32_bits_to_bf16(f32_to_bits(v));
    memcpy((char *)buf + 2 * i, &b, 2);
}

/* Bitwise copy of one element of es bytes. */
static void copy_elem(void *dst, size_t di, const void *src, size_t si, int es) {
    memcpy((char *)dst + (size_t)es * di, (const char *)src + (size_t)es * si, (size_t)es);
}

/* SCORE ([P2] §3.3): the value of one output element is the binary32 sum of
 * the R sources at the same index, taken in rank order 0..R-1 starting from
 * rank 0's value, rounded once to the output type. */
static float ordered_sum(int R, int dtype, const void *const *in, size_t idx) {
    float acc = load_as_f32(dtype, in[0], idx);
    for (int s = 1; s < R; ++s) {
        acc = acc + load_as_f32(dtype, in[s], idx);
    }
    return acc;
}

/* Exclusive prefix sum (the displacement arrays of the V variants). */
static void exclusive_scan(int k, const size_t *x, size_t stride, size_t *out) {
    size_t run = 0;
    for (int j = 0; j < k; ++j) {
        out[j] = run;
        run += x[(size_t)j * stride];
    }
}

/* ------------------------------------------------------------------ */
/* Collectives.  in[s] / out[d] are R separate host buffers.  Counts are */
/* in elements.  Return 0, or -1 for an argument the contract rejects.   */
/* ------------------------------------------------------------------ */

/* AllGather ([P2] §2.1, §3.1 packed -> scattered, copy; [P4] totalBytes):
 * every output holds the R inputs of n elements concatenated in rank order,
 *   out_d[s*n + i] = in_s[i]. */
int oracle_all_gather(int R, size_t n, int dtype, const void *const *in, void *const *out) {
    int es = elem_size(dtype);
    if (R < 1 || es == 0) return -1;
    for (int d = 0; d < R; ++d)
        for (int s = 0; s < R; ++s)
            PARALLEL_ELEMENTS
            for (size_t i = 0; i < n; ++i)
                copy_elem(out[d], (size_t)s * n + i, in[s], i, es);
    return 0;
}

/* AllGatherV ([P2] §2.1, §C.4): rank s contributes counts[s] elements;
 *   out_d[D_s + i] = in_s[i],  D_s = sum_{t<s} counts[t]. */
int oracle_all_gather_v(int R, const size_t *counts, int dtype, const void *const *in,
                        void *const *out) {
    int es = elem_size(dtype);
    if (R < 1 || R > 1024 || es == 0) return -1;
    size_t D[1024];
    exclusive_scan(R, counts, 1, D);
    for (int d = 0; d < R; ++d)
        for (int s = 0; s < R; ++s)
            PARALLEL_ELEMENTS
            for (size_t i = 0; i < counts[s]; ++i)
                copy_elem(out[d], D[s] + i, in[s], i, es);
    return 0;
}

/* ReduceScatter ([P2] §2.1, §3.1 scattered -> packed, reduce; §3.3 SCORE):
 * each input has n = R*M elements; rank r receives the ordered sum of slice r,
 *   out_r[i] = rnd(sum_s in_s[r*M + i]). */
int oracle_reduce_scatter(int R, size_t n, int dtype, const void *const *in, void *const *out) {
    if (R < 1 || elem_size(dtype) == 0 || n % (size_t)R != 0) return -1;
    size_t M = n / (size_t)R;
    for (int r = 0; r < R; ++r)
        PARALLEL_ELEMENTS
        for (size_t i = 0; i < M; ++i)
            store_rounded(dtype, out[r], i, ordered_sum(R, dtype, in, (size_t)r * M + i));
    return 0;
}

/* ReduceScatterV ([P2] §C.4: the output of rank r is its assigned share):
 * every input has T = sum(counts) elements;
 *   out_r[i] = rnd(sum_s in_s[D_r + i]),  i < counts[r]. */
int oracle_reduce_scatter_v(int R, const size_t *counts, int dtype, const void *const *in,
                            void *const *out) {
    if (R < 1 || R > 1024 || elem_size(dtype) == 0) return -1;
    size_t D[1024];
    exclusive_scan(R, counts, 1, D);
    for (int r = 0; r < R; ++r)
        PARALLEL_ELEMENTS
        for (size_t i = 0; i < counts[r]; ++i)
            store_rounded(dtype, out[r], i, ordered_sum(R, dtype, in, D[r] + i));
    return 0;
}

/* AllReduce ([P2] §2.1; §3.1 scattered -> scattered, ReduceScatter then
 * AllGather; §3.3 SCORE): every output is the ordered, once-rounded sum,
 *   out_d[i] = rnd(sum_s in_s[i]).
 * Written per destination so each output is its own definition. */
int oracle_all_reduce(int R, size_t n, int dtype, const void *const *in, void *const *out) {
    if (R < 1 || elem_size(dtype) == 0) return -1;
    for (int d = 0; d < R; ++d)
        PARALLEL_ELEMENTS
        for (size_t i = 0; i < n; ++i)
            store_rounded(dtype, out[d], i, ordered_sum(R, dtype, in, i));
    return 0;
}

/* One AllReduce output: every destination holds the same values by the
 * contract above, out[i] = rnd(sum_s in_s[i]), so a test of a large call
 * needs this array only once. */
int oracle_all_reduce_one(int R, size_t n, int dtype, const void *const *in, void *out) {
    if (R < 1 || elem_size(dtype) == 0) return -1;
    PARALLEL_ELEMENTS
    for (size_t i = 0; i < n; ++i) store_rounded(dtype, out, i, ordered_sum(R, dtype, in, i));
    return 0;
}

/* AllToAll ([P2] §2.1; §3.1 scattered -> transposed, copy): each input has
 * n = R*M elements, slice d goes to rank d, landing in slot s:
 *   out_d[s*M + i] = in_s[d*M + i]. */
int oracle_all_to_all(int R, size_t n, int dtype, const void *const *in, void *const *out) {
    int es = elem_size(dtype);
    if (R < 1 || es == 0 || n % (size_t)R != 0) return -1;
    size_t M = n / (size_t)R;
    for (int d = 0; d < R; ++d)
        for (int s = 0; s < R; ++s)
            PARALLEL_ELEMENTS
            for (size_t i = 0; i < M; ++i)
                copy_elem(out[d], (size_t)s * M + i, in[s], (size_t)d * M + i, es);
    return 0;
}

/* AllToAllV ([P2] §2.1, §C.4): C[s*R + d] elements go from rank s to rank d.
 * Send displacement S_s[d] = sum_{d'<d} C[s][d'] (row prefix);
 * receive displacement Q_d[s] = sum_{s'<s} C[s'][d] (column prefix);
 *   out_d[Q_d[s] + i] = in_s[S_s[d] + i],  i < C[s][d]. */
int oracle_all_to_all_v(int R, const size_t *C, int dtype, const void *const *in,
                        void *const *out) {
    int es = elem_size(dtype);
    if (R < 1 || R > 1024 || es == 0) return -1;
    size_t S[1024], Q[1024];
    for (int d = 0; d < R; ++d) {
        exclusive_scan(R, C + d, (size_t)R, Q); /* column d: C[0][d], C[1][d], ... */
        for (int s = 0; s < R; ++s) {
            exclusive_scan(R, C + (size_t)s * R, 1, S); /* row s */
            PARALLEL_ELEMENTS
            for (size_t i = 0; i < C[(size_t)s * R + d]; ++i)
                copy_elem(out[d], Q[s] + i, in[s], S[d] + i, es);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Point evaluation, for sampled checks of full-size outputs.            */
/* ------------------------------------------------------------------ */

/* One reduced element: rnd(sum_s in_s[idx]) written to *out_elem.  Serves
 * AllReduce (idx = i), ReduceScatter (idx = r*M + i) and ReduceScatterV
 * (idx = D_r + i). */
int oracle_reduce_at(int R, int dtype, const void *const *in, size_t idx, void *out_elem) {
    if (R < 1 || elem_size(dtype) == 0) return -1;
    store_rounded(dtype, out_elem, 0, ordered_sum(R, dtype, in, idx));
    return 0;
}

/* Source of output element out_d[j] of AllToAllV: writes the source rank and
 * the source element index.  Returns -1 if j is past the end of out_d. */
int oracle_all_to_all_v_source(int R, const size_t *C, int d, size_t j, int *src_rank,
                               size_t *src_index) {
    if (R < 1 || R > 1024 || d < 0 || d >= R) return -1;
    size_t S[1024], Q[1024];
    exclusive_scan(R, C + d, (size_t)R, Q);
    for (int s = 0; s < R; ++s) {
        size_t c = C[(size_t)s * R + d];
        if (j >= Q[s] && j < Q[s] + c) {
            exclusive_scan(R, C + (size_t)s * R, 1, S);
            *src_rank = s;
            *src_index = S[d] + (j - Q[s]);
            return 0;
        }
    }
    return -1;
}
