/*
 * purlin.h -- C ABI of the single-GPU Purlin collective datapath (sm_103a).
 *
 * What the library computes.  The seven non-rooted collectives of
 * "Purlin: Separating Orchestration from the Datapath of Collectives"
 * (§2.1 collective contracts; §3.1 layouts) over R "rank
 * buffers" that all live in ONE GPU's memory: rank r's input is src[r] and
 * its output is dst[r].  Each call is a single kernel: a layout compiler turns
 * (input layout, output layout, copy-or-reduce op, counts) into a chunk
 * schedule (§3.1); chunks are staged into shared memory, their readiness is
 * published (an mbarrier inside a CTA, or a release-store to a per-chunk
 * flag in global memory between CTAs) and consumers copy or reduce them
 * (§3.2, Stage / Notify / And Consume); the datapath ("Atom", §3.3) is a
 * 128-bit vector load/store kernel (one 16-byte window a thread) and a
 * cp.async.bulk (TMA) multi-stage shared-memory ring.  Which one runs is
 * chosen per collective and message size from GB300 measurements: the vector
 * kernel for AllGather(V), AllReduce and ReduceScatter(V) at every size and
 * for small AllToAll(V), the ring for larger AllToAll(V) and the composed
 * AllReduce (PURLIN_OPT_VARIANT overrides the choice).
 *
 * Reductions (SCORE, §3.3): every output element is owned by one thread,
 * which adds the R sources in rank order 0..R-1 in binary32, starting from
 * rank 0's value, and rounds once to the output type (bf16: round to
 * nearest even).  Results are therefore bit-wise repeatable, as in the
 * deterministic mode of the "Purlin" project README ("Deterministic
 * Reduction"); no other mode exists on one GPU.
 *
 * Conventions shared by every call below.
 *   Pointers.  src and dst are HOST arrays of R DEVICE pointers, read during
 *     the call only.  Every device pointer must be 16-byte aligned.  The
 *     caller allocates and owns all device buffers and must keep them alive
 *     until the enqueued work has finished.  The library owns the context,
 *     its flag array, error word and plan cache.
 *   Counts.  In ELEMENTS of the dtype (the README's C++ API counts bytes).
 *   Streams.  Calls enqueue one kernel on the context's stream and return
 *     without waiting.  Argument errors return before anything is enqueued.
 *   Layout.  Each collective has exactly one legal layout pair (below);
 *     any other pair returns PURLIN_ERR_UNSUPPORTED, as does a wrong op.
 *   Aliasing.  Outputs must not overlap each other.  An input may not
 *     overlap any output, except in-place AllReduce (src[r] == dst[r]) and
 *     in-place AllGather (src[r] == dst[r] + r*n elements).  Violations
 *     return PURLIN_ERR_ALIAS.
 *   Sizes.  1 <= R <= PURLIN_MAX_RANKS.  A call with no elements to move is
 *     a valid no-op.
 *   Device faults.  A bounded wait that expires inside a kernel records
 *     PURLIN_ERR_TIMEOUT in the context's error word; purlin_check reports it.
 *   CUDA graphs.  Calls may be captured from the context's stream and the
 *     graph replayed any number of times (launches whose CTAs notify one
 *     another keep their epoch in device memory).  The first call of a call
 *     shape (collective, sizes, counts, options) compiles its plan; when the
 *     plan's segment table is too large for the kernel parameters
 *     (AllToAll(V) and the composed AllReduce at R = 8, for example) it is
 *     uploaded to device memory, which cannot happen during capture: make
 *     that first call before capturing, or it returns
 *     PURLIN_ERR_UNSUPPORTED.  Plans used during a capture are kept until
 *     purlin_finalize; a graph must not be replayed after it.
 */
#ifndef PURLIN_H
#define PURLIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PURLIN_MAX_RANKS 64

typedef struct purlin_ctx purlin_ctx;   /* opaque; created by purlin_init */
typedef void *purlin_stream;            /* a cudaStream_t (NULL = legacy default stream) */

typedef enum { PURLIN_F32 = 0, PURLIN_BF16 = 1 } purlin_dtype;

/* The consume operation of a collective (§3.1): copy or reduce (sum). */
typedef enum { PURLIN_COPY = 0, PURLIN_SUM = 1 } purlin_op;

/* Rank-relative layouts (§3.1).
 *   PACKED      a rank buffer holds one contiguous region: the rank's own.
 *   SCATTERED   a rank buffer holds R regions, region k belonging to rank k.
 *   TRANSPOSED  a rank buffer holds R regions, region k coming from rank k
 *               (the per-pair blocks of the input transposed across ranks). */
typedef enum {
    PURLIN_PACKED = 0,
    PURLIN_SCATTERED = 1,
    PURLIN_TRANSPOSED = 2
} purlin_layout_kind;

typedef struct {
    int32_t in;   /* purlin_layout_kind of the inputs */
    int32_t out;  /* purlin_layout_kind of the outputs */
} purlin_layout;

typedef enum {
    PURLIN_OK = 0,
    PURLIN_ERR_INVALID_ARG = 1,   /* null pointer, bad R, count not divisible, ... */
    PURLIN_ERR_ALIGNMENT = 2,     /* a device pointer is not 16-byte aligned */
    PURLIN_ERR_UNSUPPORTED = 3,   /* wrong op or layout pair for the collective */
    PURLIN_ERR_ALIAS = 4,         /* forbidden overlap between buffers */
    PURLIN_ERR_OOM = 5,           /* host or device allocation failed */
    PURLIN_ERR_CUDA = 6,          /* a CUDA runtime call failed */
    PURLIN_ERR_TIMEOUT = 7        /* a bounded device-side wait expired */
} purlin_status;

/* ---------------------------------------------------------------- context */

/* Create a context for R rank buffers whose work is enqueued on `stream`
 * (the pages' `initialize(rank, world, stream, memory)`, project README,
 * "Host-side", reshaped for one process holding all R ranks).  Allocates the
 * device flag array (2 parities x 65536 u64, zeroed once here), the
 * latency path's packet staging (2 parities x 2 MiB, zeroed once here;
 * "Purlin: Separating Orchestration from the Datapath of Collectives" §4.1) and a device
 * error word on the current CUDA device,
 * and reads the device's SM count and shared-memory limit.  The epoch
 * ("Purlin: Separating Orchestration from the Datapath of Collectives" §4.3) starts at 1.
 * Errors: INVALID_ARG (R out of range, out == NULL), CUDA, OOM. */
purlin_status purlin_init(int R, purlin_stream stream, purlin_ctx **out);

/* Wait for the context's stream, free the context's device memory and the
 * context itself (README "finalize").  NULL is a no-op. */
purlin_status purlin_finalize(purlin_ctx *ctx);

/* Switch the stream later calls enqueue on.  Waits for the old stream first,
 * so plan memory freed later is never still in use there. */
purlin_status purlin_set_stream(purlin_ctx *ctx, purlin_stream stream);

/* ------------------------------------------------------------ collectives */

/* AllReduce (§2.1; §3.1: ReduceScatter then AllGather, composed as one
 * SCATTERED -> SCATTERED reduction).  src[r], dst[r]: n elements each.
 * dst[d][i] = round(sum_{s=0..R-1} src[s][i]) for every d, summed in rank
 * order in binary32.  op must be SUM, layout {SCATTERED, SCATTERED}.
 * In-place (src[r] == dst[r] for every r) is allowed. */
purlin_status purlin_all_reduce(purlin_ctx *ctx, const void *const src[], void *const dst[],
                                size_t n, purlin_dtype dtype, purlin_op op,
                                purlin_layout layout);

/* ReduceScatter (§2.1; §3.1 SCATTERED -> PACKED reduction).  src[s]: n
 * elements, n divisible by R (else INVALID_ARG), M = n / R.  dst[r]: M
 * elements, dst[r][i] = round(sum_s src[s][r*M + i]).  op SUM. */
purlin_status purlin_reduce_scatter(purlin_ctx *ctx, const void *const src[], void *const dst[],
                                    size_t n, purlin_dtype dtype, purlin_op op,
                                    purlin_layout layout);

/* AllGather (§2.1; §3.1 PACKED -> SCATTERED copy; README "Understanding
 * totalBytes": the output holds every contribution).  src[s]: n elements;
 * dst[d]: R*n elements, dst[d][s*n + i] = src[s][i], bitwise.  op COPY.
 * In-place (src[r] == dst[r] + r*n elements for every r) is allowed. */
purlin_status purlin_all_gather(purlin_ctx *ctx, const void *const src[], void *const dst[],
                                size_t n, purlin_dtype dtype, purlin_op op,
                                purlin_layout layout);

/* AllToAll (§2.1; §3.1 SCATTERED -> TRANSPOSED copy).  src[s], dst[d]: n
 * elements, n divisible by R, M = n / R.  dst[d][s*M + i] = src[s][d*M + i],
 * bitwise.  op COPY. */
purlin_status purlin_all_to_all(purlin_ctx *ctx, const void *const src[], void *const dst[],
                                size_t n, purlin_dtype dtype, purlin_op op,
                                purlin_layout layout);

/* AllGatherV (§2.1 variable-length variants; §C.4: each rank contributes
 * its share).  counts: host array of R element counts; src[s] holds
 * counts[s] elements; dst[d] holds T = sum(counts) elements and
 * dst[d][D_s + i] = src[s][i] with D_s = sum_{t<s} counts[t].  op COPY,
 * layout {PACKED, SCATTERED}. */
purlin_status purlin_all_gather_v(purlin_ctx *ctx, const void *const src[], void *const dst[],
                                  const size_t counts[], purlin_dtype dtype, purlin_op op,
                                  purlin_layout layout);

/* ReduceScatterV (§C.4: the output of rank r is its share).  Every src[s]
 * holds T = sum(counts) elements; dst[r] holds counts[r] elements,
 * dst[r][i] = round(sum_s src[s][D_r + i]).  op SUM, layout
 * {SCATTERED, PACKED}. */
purlin_status purlin_reduce_scatter_v(purlin_ctx *ctx, const void *const src[],
                                      void *const dst[], const size_t counts[],
                                      purlin_dtype dtype, purlin_op op, purlin_layout layout);

/* AllToAllV (§2.1, §C.4).  counts: host array of R*R element counts, row s
 * = source, column d = destination.  src[s] holds sum_d C[s][d] elements
 * packed by destination in destination order; dst[d] holds sum_s C[s][d]
 * elements packed by source in source order:
 * dst[d][Q_d[s] + i] = src[s][S_s[d] + i], S_s[d] = sum_{d'<d} C[s][d'],
 * Q_d[s] = sum_{s'<s} C[s'][d].  op COPY, layout {SCATTERED, TRANSPOSED}. */
purlin_status purlin_all_to_all_v(purlin_ctx *ctx, const void *const src[], void *const dst[],
                                  const size_t counts[], purlin_dtype dtype, purlin_op op,
                                  purlin_layout layout);

/* The three V collectives with their counts in DEVICE memory, e.g. written
 * by an MoE router kernel earlier on the context's stream (§C.4; the paper
 * summary notes the prefix sums are taken on the device).  No host round
 * trip: one kernel reads the counts, derives the displacements (exclusive
 * prefix sums, as in the host calls above), checks them and runs the
 * collective.  counts: device array of size_t, R entries (AllGatherV,
 * ReduceScatterV) or R*R (AllToAllV, row = source), 8-byte aligned, read
 * by the kernel in stream order.  The buffers' extents are declared
 * instead of derived: every src[r] holds in_capacity elements and every
 * dst[r] out_capacity elements (pointers, alignment and overlaps are
 * checked on the host against these extents, as for the host-count calls;
 * no in-place form).  The kernel checks that the counts fit: each rank's
 * input extent (AGV: counts[r]; RSV: the total; A2AV: row r's sum) at most
 * in_capacity, each output extent (AGV: the total; RSV: counts[r]; A2AV:
 * column r's sum) at most out_capacity, and every count below 2^40;
 * otherwise it writes nothing and records INVALID_ARG in the context's
 * error word (purlin_check).  The variant is decided on the device from
 * the largest per-rank input against the crossover (PURLIN_OPT_VARIANT and
 * PURLIN_OPT_CROSSOVER_BYTES apply).  R <= 16, else UNSUPPORTED. */
purlin_status purlin_all_gather_v_device_counts(purlin_ctx *ctx, const void *const src[],
                                                void *const dst[], const size_t counts[],
                                                size_t in_capacity, size_t out_capacity,
                                                purlin_dtype dtype, purlin_op op,
                                                purlin_layout layout);
purlin_status purlin_reduce_scatter_v_device_counts(purlin_ctx *ctx, const void *const src[],
                                                    void *const dst[], const size_t counts[],
                                                    size_t in_capacity, size_t out_capacity,
                                                    purlin_dtype dtype, purlin_op op,
                                                    purlin_layout layout);
purlin_status purlin_all_to_all_v_device_counts(purlin_ctx *ctx, const void *const src[],
                                                void *const dst[], const size_t counts[],
                                                size_t in_capacity, size_t out_capacity,
                                                purlin_dtype dtype, purlin_op op,
                                                purlin_layout layout);

/* AllReduce without any device allocation.  The pages have no counterpart
 * to this entry point; it is an addition of this library for callers that
 * cannot call cudaMalloc at the time they reduce: code running while a CUDA
 * graph is being captured, and engines that give all free device memory to
 * their own pool and let no library take more.  Same contract and result
 * (bit for bit) as purlin_all_reduce with PURLIN_OPT_AR_MODE = composed,
 * without a context: R (1..31) rank buffers, n elements each, enqueued on
 * `stream`.  Its scratch (per-chunk flags, an error word and the device
 * epoch, 128 KiB + 32 bytes) is a fixed device array inside the library,
 * held by every GPU that loads it until the process exits.  The epoch is
 * kept on the device, so a call captured into a CUDA graph stays correct at
 * every replay.  Limit: at most 8192 reduce chunks of
 * 96 KiB / R bytes per source (rounded down to a multiple of 16), i.e.
 * n * element size <= 8192 * (98304 / R) bytes per rank (96 MiB at R = 8);
 * larger calls and R > 31 return
 * INVALID_ARG.  The first call on a device looks up the array's address,
 * sets kernel attributes and zeroes the array with a blocking cudaMemset:
 * make it before any stream capture.  Every call shares the array (it keeps
 * the previous call's contents; the error word is cleared per call), so
 * calls that overlap on the GPU race: order them on one stream.  A device-
 * side wait that expires (100 ms bound per wait; the launch then ends early
 * and that call's outputs are unspecified) is recorded in the array's error
 * word, which the next call clears: read it before then with
 * purlin_noalloc_check.  Needs about 193 KiB of dynamic shared memory per
 * CTA (two 96 KiB stages); a device with less returns UNSUPPORTED.  Errors
 * as for purlin_all_reduce, plus CUDA if the set-up or the launch fails. */
purlin_status purlin_all_reduce_noalloc(int R, const void *const src[], void *const dst[],
                                        size_t n, purlin_dtype dtype, purlin_op op,
                                        purlin_layout layout, purlin_stream stream);

/* Status of the allocation-free AllReduce calls on the current device that
 * `stream` has run: synchronizes `stream`, reads the scratch array's error
 * word and clears it.  OK if no device-side wait expired since the word was
 * last cleared (or no call ran on this device yet); TIMEOUT if one did, and
 * the outputs of the calls since then are unspecified; CUDA if the
 * synchronize or the 8-byte copy fails (a device fault).  Not during stream
 * capture.  Allocates nothing. */
purlin_status purlin_noalloc_check(purlin_stream stream);

/* ------------------------------------------------------------ measurement */

/* Enqueue one empty kernel (<<<1, 32>>>, no parameters) on `stream`: the
 * launch floor that small-message latency is compared against, timed the
 * same way as a collective.  Returns CUDA if the launch fails. */
purlin_status purlin_empty_launch(purlin_stream stream);

/* Enqueue one kernel (<<<1, 32>>>) in which one thread copies the 16 bytes
 * at device address `src` to `dst`: the least a kernel that touches memory
 * does (one load round trip and one store), the second floor small-message
 * latency is compared against.  Both pointers 16-byte aligned (ALIGNMENT
 * otherwise), non-NULL (INVALID_ARG); CUDA if the launch fails. */
purlin_status purlin_touch_launch(const void *src, void *dst, purlin_stream stream);

/* ----------------------------------------------------------------- status */

/* Wait for the context's stream, then read and clear the device error word.
 * Returns PURLIN_ERR_TIMEOUT if a bounded wait expired in any earlier call
 * (the outputs of that call are then unspecified), CUDA if the stream
 * reported an error, else OK. */
purlin_status purlin_check(purlin_ctx *ctx);

/* Static English name of a status code; never NULL. */
const char *purlin_status_string(purlin_status status);

/* ---------------------------------------------------------------- policy */

/* Codesign policy knobs ("Purlin: Separating Orchestration from the Datapath of Collectives"
 * §4.2: crossover, chunk sizes, CTA
 * allocation, pipeline depth, tuned per collective and GPU; applications
 * may override).  0 means "the built-in policy" for every knob.
 * purlin_init also reads PURLIN_VARIANT, PURLIN_CROSSOVER_BYTES,
 * PURLIN_STAGES, PURLIN_CHUNK_BYTES, PURLIN_CTAS and PURLIN_AR_MODE from the
 * environment as initial values of the matching knobs. */
typedef enum {
    PURLIN_OPT_VARIANT = 0,          /* 0 auto, 1 latency (vector ld/st), 2 throughput (TMA ring) */
    PURLIN_OPT_CROSSOVER_BYTES = 1,  /* per-rank message bytes at or below which auto picks latency */
    PURLIN_OPT_AR_MODE = 2,          /* AllReduce: 0 auto, 1 fused, 2 composed (RS CTAs notify, AG CTAs consume),
                                        3 composed on the latency path: 16-byte payload+flag packets
                                        (messages up to 1 MiB per rank; larger ones run mode 2) */
    PURLIN_OPT_CHUNK_BYTES = 3,      /* bytes per source per chunk in the TMA ring */
    PURLIN_OPT_STAGES = 4,           /* TMA ring depth */
    PURLIN_OPT_CTAS = 5,             /* CTAs of a throughput launch (0: the policy's; at most what fits at once) */
    PURLIN_OPT_SPIN_TIMEOUT_NS = 6,  /* bound on a cross-CTA flag wait (default 100 ms) */
    PURLIN_OPT_DROP_NOTIFY = 7,      /* host-side fault injection: chunk whose notify is skipped; -1 off */
    PURLIN_OPT_LAT_CTAS = 8,         /* max CTAs of a latency launch (0: a CTA per block of units, up to 2^24) */
    PURLIN_OPT_LAT_BLOCK = 9,        /* threads per CTA of a latency launch (32..256, multiple of 32) */
    PURLIN_OPT_CONSUMER_WARPS = 10,  /* consumer warps of a throughput CTA (1..14) */
    PURLIN_OPT_COPY_STORES = 11      /* aligned copies in the ring: 0 auto, 1 bulk stores (TMA), 2 vector stores */
} purlin_option;

/* Set one knob; INVALID_ARG for an unknown knob or a value out of range. */
purlin_status purlin_set_option(purlin_ctx *ctx, purlin_option opt, int64_t value);
purlin_status purlin_get_option(purlin_ctx *ctx, purlin_option opt, int64_t *value);

/* What the last collective call of this context enqueued. */
typedef struct {
    int32_t variant;      /* 0 nothing launched, 1 latency, 2 throughput, 3 throughput composed AllReduce, 4 decided on the device (device counts), 5 composed AllReduce with packets */
    int32_t grid;         /* CTAs */
    int32_t block;        /* threads per CTA */
    int32_t stages;       /* TMA ring depth (throughput) */
    int64_t chunk_bytes;  /* bytes per source per chunk (throughput) */
    int64_t chunks;       /* TMA chunks */
    int64_t units;        /* 16-byte vector units outside the TMA ring */
    int64_t segments;     /* segments in the compiled plan */
    int64_t smem_bytes;   /* dynamic shared memory per CTA */
    uint64_t epoch;       /* epoch the launch used (§4.3) */
    uint64_t epoch_next;  /* epoch of the next call */
} purlin_launch_info;

purlin_status purlin_last_launch(const purlin_ctx *ctx, purlin_launch_info *info);

/* --------------------------------------------------- host-side inspection */

typedef enum {
    PURLIN_COLL_ALL_REDUCE = 0,
    PURLIN_COLL_REDUCE_SCATTER = 1,
    PURLIN_COLL_ALL_GATHER = 2,
    PURLIN_COLL_ALL_TO_ALL = 3,
    PURLIN_COLL_ALL_GATHER_V = 4,
    PURLIN_COLL_REDUCE_SCATTER_V = 5,
    PURLIN_COLL_ALL_TO_ALL_V = 6
} purlin_collective;

/* One contiguous transfer of a compiled plan (the layout compiler's output). */
typedef struct {
    uint64_t src_off;      /* byte offset into the source buffer(s) */
    uint64_t dst_off;      /* byte offset into the destination buffer(s) */
    uint64_t bytes;        /* bytes moved per source */
    int32_t src_rank;      /* source rank, or -1: reduce over every rank at src_off */
    int32_t dst_rank;      /* destination rank, or -1: every rank at dst_off */
    int32_t skip_rank;     /* with dst_rank -1: a rank left out, or -1 */
    int32_t src_is_dst;    /* 1: the source buffers are the destination array */
    int32_t sync;          /* 0 none, 1 notify a flag after writing, 2 wait on a flag before reading */
    int32_t tma;           /* 1 if the 16-byte-aligned body goes through the TMA ring */
    int32_t shift;         /* tma: 16-byte phase of the source relative to the destination */
    uint64_t head_bytes;   /* bytes before the aligned body (vector path); the body is aligned
                              on the sources for a reduce, on the destination for a copy */
    uint64_t tail_bytes;   /* bytes after it (vector path) */
    uint64_t chunk_begin;  /* index of the segment's first TMA chunk */
    uint64_t chunk_bytes;  /* bytes per source per TMA chunk */
    uint64_t unit_begin;   /* index of the segment's first vector unit */
} purlin_segment;

/* Run the argument checks and the layout compiler of one call without a
 * GPU: pointer values are compared, never dereferenced.  `counts` is NULL
 * for the uniform collectives (then `n` is used), R entries for AGV/RSV and
 * R*R for AllToAllV.  variant: 1 latency, 2 throughput; ar_mode as for
 * PURLIN_OPT_AR_MODE; chunk_bytes 0 = default.  Writes up to `cap`
 * segments, the segment count, the TMA chunk count and the unit count.
 * Returns the status the real call would return for these arguments. */
purlin_status purlin_plan_inspect(purlin_collective coll, int R, const void *const src[],
                                  void *const dst[], size_t n, const size_t counts[],
                                  purlin_dtype dtype, purlin_op op, purlin_layout layout,
                                  int variant, int ar_mode, uint64_t chunk_bytes,
                                  purlin_segment *segs, size_t cap, size_t *nseg,
                                  uint64_t *nchunks, uint64_t *nunits);

/* ----------------------------------------------------- device-side API */

/* A collective compiled for kernels that run it themselves (the "Purlin"
 * project README, "Device-side": a user kernel calls a collective, or an
 * Atom, from inside itself, so communication fuses with its other work;
 * "Purlin: Separating Orchestration from the Datapath of Collectives" §3: applications
 * invoke the Atom directly).
 *
 * purlin_device_prepare fills one of these for one call shape: the
 * collective, its R rank buffers, counts and dtype, and the number of CTAs
 * (`blocks`) that will enter it.  The user kernel receives it by value
 * (a __grid_constant__ parameter) or through a pointer to device memory and
 * calls purlin::device::collective(coll, args) from include/purlin_device.cuh
 * in exactly `blocks` CTAs, each with:
 *   - a 1-D block whose size is a multiple of 32 and at least 96 (warp 0
 *     stages, warp 1 writes back and publishes, the rest consume; `threads`
 *     is the size the library's policy would pick);
 *   - `workspace_bytes` of shared memory, 128-byte aligned, that the
 *     collective may overwrite (the kernel's dynamic shared memory, usually).
 * Every call through the same descriptor runs the same collective on the
 * same buffers; the data may change between calls.  Any number of calls may
 * follow one another (one per kernel, or several in one kernel): each CTA
 * keeps its epoch in device memory and advances it by `epoch_inc` per call,
 * so the CTAs agree as long as all `blocks` of them enter every call.
 * When `composed` is 1 (AllReduce with PURLIN_OPT_AR_MODE = composed), CTAs
 * wait on one another's chunk flags: all `blocks` CTAs must be resident at
 * once (launch cooperatively), or the waits expire and report TIMEOUT.
 * Pointers in it name device memory that the library owns (segment table,
 * flags, per-CTA epochs, error word) until purlin_device_release or
 * purlin_finalize; the caller must not write them. */
typedef struct purlin_device_coll {
    const void *src[PURLIN_MAX_RANKS];   /* rank input buffers (device), R used */
    void *dst[PURLIN_MAX_RANKS];         /* rank output buffers (device), R used */
    const void *segs;                    /* compiled segment table (device) */
    unsigned long long *flags;           /* 2 x flag_slots chunk flags, or NULL (not composed) */
    unsigned long long *epochs;          /* `blocks` per-CTA epochs (device) */
    unsigned long long *err;             /* error word (device): see purlin_device_check */
    uint64_t nchunks;                    /* ring chunks of the plan */
    uint64_t nunits;                     /* vector units of the plan */
    uint64_t epoch_inc;                  /* odd; added to each CTA's epoch per call */
    int64_t timeout_ns;                  /* bound on one flag wait */
    int64_t drop_notify;                 /* PURLIN_OPT_DROP_NOTIFY at prepare time (testing), else -1 */
    uint32_t flag_slots;                 /* flags per parity (a multiple of blocks) */
    uint32_t stages;                     /* ring stages */
    uint32_t slot_stride;                /* bytes per ring stage */
    uint32_t workspace_bytes;            /* shared memory each entering CTA provides */
    int32_t nseg;                        /* segments in the table */
    int32_t R;                           /* rank buffers */
    int32_t dtype;                       /* purlin_dtype */
    int32_t vector_copies;               /* aligned copies stored by the consumer warps */
    int32_t blocks;                      /* CTAs that enter every call */
    int32_t threads;                     /* suggested block size */
    int32_t composed;                    /* 1: CTAs wait on one another (all must be resident) */
    int32_t coll;                        /* purlin_collective */
    int32_t ragged;                      /* 1: ring chunks at another 16-byte phase than their
                                            destination (ragged blocks) */
    void *owner;                         /* library bookkeeping (host address) */
} purlin_device_coll;

/* Compile a device-side collective for the context's R.  Arguments as for
 * the matching host call: `n` for the uniform collectives, `counts` (R or
 * R*R entries, host memory) for the V ones, NULL otherwise.  `blocks` >= 1
 * CTAs will enter it.  `max_workspace_bytes` caps the shared memory it may
 * ask of each CTA (0: the device's opt-in maximum less 4 KiB); the ring
 * shape follows the host call's policy and the context's options, reduced
 * to fit.  Allocates device memory and copies the plan there with blocking
 * calls (not during graph capture).  Errors: those of the host call, plus
 * INVALID_ARG (blocks < 1 or > 65535, or too many notifying chunks for the
 * flag array), UNSUPPORTED (no ring fits the cap), OOM and CUDA. */
purlin_status purlin_device_prepare(purlin_ctx *ctx, purlin_collective coll,
                                    const void *const src[], void *const dst[], size_t n,
                                    const size_t counts[], purlin_dtype dtype, purlin_op op,
                                    purlin_layout layout, int blocks,
                                    uint32_t max_workspace_bytes, purlin_device_coll *out);

/* Wait for `stream`, then read and clear the descriptor's error word.
 * Returns OK, INVALID_ARG (a kernel entered with a CTA count, index, block
 * shape, workspace alignment or dtype that does not match the descriptor),
 * TIMEOUT (a bounded device wait expired) or CUDA. */
purlin_status purlin_device_check(const purlin_device_coll *coll, purlin_stream stream);

/* Free the device memory of a descriptor (synchronises the device) and
 * clear it.  Releasing a cleared descriptor is a no-op.  INVALID_ARG if it
 * was not prepared on this context. */
purlin_status purlin_device_release(purlin_ctx *ctx, purlin_device_coll *coll);

/* sizeof(purlin_device_coll) as this library was built (for bindings). */
size_t purlin_device_coll_size(void);

/* A payload+flag packet channel between the CTAs of one kernel launch
 * ("Purlin: Separating Orchestration from the Datapath of Collectives" §3.2:
 * the latency path puts payload and notification in one 16-byte packet, so
 * a consumer sees data and readiness in one access, with no separate flag
 * store and no fence, at twice the bytes; §4.1: two staging buffers; §4.3:
 * the epoch is the notification value and its parity picks the buffer).
 * It serves a producer that is not the owner of the chunks its consumers
 * read, e.g. CTAs of a compute kernel that stream each result to consumer
 * CTAs as soon as it exists, instead of writing all of it, passing a grid
 * barrier and starting a collective.
 *
 * The unit of transfer is 8 payload bytes: unit u of a launch travels as
 * the packet at staging + 16 u of the launch's packet set, two 8-byte lines
 * {4 payload bytes, 32-bit flag}, each written and read as one single-copy
 * atomic access; a consumer takes a packet once both lines carry the
 * launch's flag.  In a kernel, exactly `ctas` CTAs call
 * purlin::device::channel_open (include/purlin_device.cuh) before their
 * first send or receive and channel_close after their last (every thread of
 * those CTAs); producers call send(u, payload) once per unit and consumers
 * recv(u) (a bounded wait).  The launch must keep producers and consumers
 * resident together (a cooperative launch).  One round per launch: the flag
 * is the low 32 bits of the channel's epoch, which the last CTA to close
 * advances by one, so the next launch uses the other packet set and a new
 * flag (no reset between launches, and a launch replayed from a CUDA graph
 * is correct too).  Fields other than timeout_ns and drop_unit name device
 * memory the library owns until purlin_packet_channel_release or
 * purlin_finalize; the caller must not write it. */
typedef struct purlin_packet_channel {
    unsigned char *staging;    /* device: 2 packet sets of `capacity` 16-byte packets */
    unsigned long long *state; /* device: [0] error word, [2] epoch, [3] CTAs closed */
    uint64_t capacity;         /* 8-byte payload units per launch */
    int64_t timeout_ns;        /* bound on one packet wait (PURLIN_OPT_SPIN_TIMEOUT_NS) */
    int64_t drop_unit;         /* fault injection: the unit whose packet send() skips, or -1
                                  (PURLIN_OPT_DROP_NOTIFY at creation) */
    int32_t ctas;              /* CTAs that open and close the channel in every launch */
    int32_t pad;
    void *owner;               /* library bookkeeping (host address) */
} purlin_packet_channel;

/* Allocate a channel of capacity_bytes payload bytes per launch (rounded up
 * to 8; 2 x 2 x that many bytes of staging) for `ctas` CTAs per launch, and
 * zero it (blocking calls; not during graph capture).  INVALID_ARG for
 * capacity 0 or above 2^34 bytes, ctas < 1 or > 65535; OOM, CUDA. */
purlin_status purlin_packet_channel_create(purlin_ctx *ctx, size_t capacity_bytes, int ctas,
                                           purlin_packet_channel *out);

/* Wait for `stream`, then read and clear the channel's error word.  OK,
 * TIMEOUT (a receive gave up: that launch's outputs are unspecified),
 * INVALID_ARG (a unit past the capacity was sent or received; it was
 * skipped) or CUDA. */
purlin_status purlin_packet_channel_check(const purlin_packet_channel *ch, purlin_stream stream);

/* Free a channel's device memory (synchronises the device) and clear it.
 * Releasing a cleared channel is a no-op; INVALID_ARG if it was not created
 * on this context. */
purlin_status purlin_packet_channel_release(purlin_ctx *ctx, purlin_packet_channel *ch);

#ifdef __cplusplus
}
#endif

#endif /* PURLIN_H */
