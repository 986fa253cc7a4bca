/*
 * purlin_bench.c -- collective latency / bandwidth sweep through the C ABI.
 *
 * The command line follows the benchmark binaries of the "Purlin" project
 * README ("C++ benchmarks"): a collective, then
 *   [minBytes] [maxBytes] [graphLaunches] [runs] [warmup] [seed]
 * with sizes doubling from minBytes to maxBytes.  A size is the input bytes
 * per rank ("Understanding totalBytes": the reported totalBytes is the
 * output size for AllGather and the per-rank input size otherwise; the
 * bandwidth column divides it by the time).  All R = 8 ranks live on the
 * current GPU.
 *
 * Per size it prints one JSON line with:
 *   single_us   median over `runs` of events around ONE call (includes the
 *               library's host-side cost, as a user sees it);
 *   graph_us    device time per call from a CUDA graph of `graphLaunches`
 *               calls, replayed `runs` times (0 = skipped);
 *   floor_*     the same two measurements of an empty <<<1,32>>> kernel;
 *   touch_*     and of a kernel whose one thread loads 16 bytes and stores
 *               them (the least a kernel that touches memory does);
 *   algbw_gbs   totalBytes / graph time (or single time without graphs);
 *   eff_gbs     bytes every rank buffer reads plus writes / the same time.
 * The V collectives split the size with the Zipf(s = 0.125) partition of the
 * "Purlin: Separating Orchestration from the Datapath of Collectives" §C.4
 * (uniform at 1 and 2 KiB; AllToAllV rotates the
 * partition so every rank sends and receives the full size).
 * Inputs are seeded pseudo-random bf16 values; their values do not change
 * the work.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "../../include/purlin.h"

#define R 8
#define CK(x)                                                                       \
    do {                                                                            \
        cudaError_t e_ = (x);                                                       \
        if (e_ != cudaSuccess) {                                                    \
            fprintf(stderr, "%s:%d %s\n", __FILE__, __LINE__, cudaGetErrorString(e_)); \
            exit(2);                                                                \
        }                                                                           \
    } while (0)
#define PK(x)                                                                       \
    do {                                                                            \
        purlin_status s_ = (x);                                                     \
        if (s_ != PURLIN_OK) {                                                      \
            fprintf(stderr, "%s:%d %s\n", __FILE__, __LINE__, purlin_status_string(s_)); \
            exit(3);                                                                \
        }                                                                           \
    } while (0)

enum { C_AR, C_RS, C_AG, C_A2A, C_AGV, C_RSV, C_A2AV };

static uint64_t rng_state;
static uint64_t next_u64(void) { /* splitmix64 */
    uint64_t z = (rng_state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static size_t parse_size(const char *s) {
    char *end;
    double v = strtod(s, &end);
    if (*end == 'K' || *end == 'k') v *= 1024;
    if (*end == 'M' || *end == 'm') v *= 1024 * 1024;
    if (*end == 'G' || *end == 'g') v *= 1024.0 * 1024 * 1024;
    return (size_t)v;
}

static int cmp_f(const void *a, const void *b) {
    float x = *(const float *)a, y = *(const float *)b;
    return (x > y) - (x < y);
}

/* Zipf(s) split of `total` elements over R ranks, preserving the total. */
static void zipf_split(size_t total, double s, size_t *out) {
    double w[R], sum = 0;
    for (int k = 0; k < R; ++k) sum += (w[k] = pow((double)(k + 1), -s));
    size_t acc = 0;
    for (int k = 0; k < R; ++k) {
        out[k] = (size_t)floor(total * (w[k] / sum));
        acc += out[k];
    }
    out[0] += total - acc;
}

typedef struct {
    int coll;
    size_t n;                /* elements per rank input (uniform collectives) */
    size_t counts[R * R];
    size_t in_elems[R], out_elems[R];
    void *src[R], *dst[R];
} Call;

static purlin_ctx *ctx;
static cudaStream_t stream;

static void call_once(const Call *c) {
    const purlin_layout ss = {PURLIN_SCATTERED, PURLIN_SCATTERED};
    const purlin_layout sp = {PURLIN_SCATTERED, PURLIN_PACKED};
    const purlin_layout ps = {PURLIN_PACKED, PURLIN_SCATTERED};
    const purlin_layout st = {PURLIN_SCATTERED, PURLIN_TRANSPOSED};
    const void *const *s = (const void *const *)c->src;
    switch (c->coll) {
        case C_AR: PK(purlin_all_reduce(ctx, s, c->dst, c->n, PURLIN_BF16, PURLIN_SUM, ss)); break;
        case C_RS: PK(purlin_reduce_scatter(ctx, s, c->dst, c->n, PURLIN_BF16, PURLIN_SUM, sp)); break;
        case C_AG: PK(purlin_all_gather(ctx, s, c->dst, c->n, PURLIN_BF16, PURLIN_COPY, ps)); break;
        case C_A2A: PK(purlin_all_to_all(ctx, s, c->dst, c->n, PURLIN_BF16, PURLIN_COPY, st)); break;
        case C_AGV: PK(purlin_all_gather_v(ctx, s, c->dst, c->counts, PURLIN_BF16, PURLIN_COPY, ps)); break;
        case C_RSV: PK(purlin_reduce_scatter_v(ctx, s, c->dst, c->counts, PURLIN_BF16, PURLIN_SUM, sp)); break;
        case C_A2AV: PK(purlin_all_to_all_v(ctx, s, c->dst, c->counts, PURLIN_BF16, PURLIN_COPY, st)); break;
    }
}

static void *touch_buf;   /* 32 bytes: the touch kernel copies the first 16 to the last 16 */

/* empty: 1 = the empty kernel, 2 = the one-load-one-store kernel */
static void empty_once(int kind) {
    if (kind == 2)
        PK(purlin_touch_launch(touch_buf, (char *)touch_buf + 16, stream));
    else
        PK(purlin_empty_launch(stream));
}

static float single_us(void (*fn)(const Call *), const Call *c, int runs, int empty) {
    cudaEvent_t e0, e1;
    CK(cudaEventCreate(&e0));
    CK(cudaEventCreate(&e1));
    float *t = (float *)malloc(sizeof(float) * (size_t)runs);
    for (int i = 0; i < runs; ++i) {
        CK(cudaEventRecord(e0, stream));
        if (empty) empty_once(empty); else fn(c);
        CK(cudaEventRecord(e1, stream));
        CK(cudaEventSynchronize(e1));
        CK(cudaEventElapsedTime(&t[i], e0, e1));
    }
    qsort(t, (size_t)runs, sizeof(float), cmp_f);
    float med = t[runs / 2] * 1000.0f;
    free(t);
    CK(cudaEventDestroy(e0));
    CK(cudaEventDestroy(e1));
    return med;
}

static float graph_us(const Call *c, int launches, int runs, int empty) {
    cudaGraph_t g;
    cudaGraphExec_t ge;
    CK(cudaStreamBeginCapture(stream, cudaStreamCaptureModeThreadLocal));
    for (int i = 0; i < launches; ++i) {
        if (empty) empty_once(empty); else call_once(c);
    }
    CK(cudaStreamEndCapture(stream, &g));
    CK(cudaGraphInstantiate(&ge, g, 0));
    CK(cudaGraphLaunch(ge, stream));
    CK(cudaStreamSynchronize(stream));
    cudaEvent_t e0, e1;
    CK(cudaEventCreate(&e0));
    CK(cudaEventCreate(&e1));
    float *t = (float *)malloc(sizeof(float) * (size_t)runs);
    for (int i = 0; i < runs; ++i) {
        CK(cudaEventRecord(e0, stream));
        CK(cudaGraphLaunch(ge, stream));
        CK(cudaEventRecord(e1, stream));
        CK(cudaEventSynchronize(e1));
        CK(cudaEventElapsedTime(&t[i], e0, e1));
    }
    qsort(t, (size_t)runs, sizeof(float), cmp_f);
    float med = t[runs / 2] * 1000.0f / (float)launches;
    free(t);
    CK(cudaEventDestroy(e0));
    CK(cudaEventDestroy(e1));
    CK(cudaGraphExecDestroy(ge));
    CK(cudaGraphDestroy(g));
    return med;
}

static int parse_coll(const char *s) {
    const char *names[] = {"AR", "RS", "AG", "A2A", "AGV", "RSV", "A2AV"};
    for (int i = 0; i < 7; ++i)
        if (!strcmp(s, names[i])) return i;
    return -1;
}

static void shape(Call *c, size_t bytes) {
    const size_t n = bytes / 2;   /* bf16 elements per rank input */
    memset(c->counts, 0, sizeof c->counts);
    c->n = n;
    switch (c->coll) {
        case C_AR:
        case C_A2A:
            c->n = n - n % R;
            for (int r = 0; r < R; ++r) c->in_elems[r] = c->out_elems[r] = c->n;
            break;
        case C_RS:
            c->n = n - n % R;
            for (int r = 0; r < R; ++r) {
                c->in_elems[r] = c->n;
                c->out_elems[r] = c->n / R;
            }
            break;
        case C_AG:
            for (int r = 0; r < R; ++r) {
                c->in_elems[r] = n;
                c->out_elems[r] = (size_t)R * n;
            }
            break;
        default: {
            size_t part[R];
            if (bytes <= 2048) {
                for (int k = 0; k < R; ++k) part[k] = n / R;
                part[0] += n - (n / R) * R;
            } else {
                zipf_split(n, 0.125, part);
            }
            if (c->coll == C_AGV) {   /* rank r contributes part[r]; n is the total */
                size_t T = 0;
                for (int r = 0; r < R; ++r) T += (c->counts[r] = part[r]);
                for (int r = 0; r < R; ++r) {
                    c->in_elems[r] = part[r];
                    c->out_elems[r] = T;
                }
            } else if (c->coll == C_RSV) {   /* every input is the total, rank r keeps part[r] */
                for (int r = 0; r < R; ++r) {
                    c->counts[r] = part[r];
                    c->in_elems[r] = n;
                    c->out_elems[r] = part[r];
                }
            } else {   /* A2AV: rotated partition, every rank sends and receives n */
                for (int s = 0; s < R; ++s)
                    for (int d = 0; d < R; ++d) c->counts[s * R + d] = part[(d - s + R) % R];
                for (int r = 0; r < R; ++r) c->in_elems[r] = c->out_elems[r] = n;
            }
        }
    }
}

int main(int argc, char **argv) {
    if (argc < 2 || parse_coll(argv[1]) < 0) {
        fprintf(stderr,
                "usage: %s AR|RS|AG|A2A|AGV|RSV|A2AV [minBytes] [maxBytes] [graphLaunches] "
                "[runs] [warmup] [seed]\n",
                argv[0]);
        return 1;
    }
    Call c;
    memset(&c, 0, sizeof c);
    c.coll = parse_coll(argv[1]);
    size_t min_b = argc > 2 ? parse_size(argv[2]) : 1024;
    size_t max_b = argc > 3 ? parse_size(argv[3]) : (1u << 20);
    int graph_launches = argc > 4 ? atoi(argv[4]) : 100;
    int runs = argc > 5 ? atoi(argv[5]) : 50;
    int warmup = argc > 6 ? atoi(argv[6]) : 5;
    rng_state = argc > 7 ? strtoull(argv[7], NULL, 0) : 42;
    if (runs < 1) runs = 1;
    if (min_b < 16) min_b = 16;

    CK(cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking));
    PK(purlin_init(R, stream, &ctx));
    CK(cudaMalloc(&touch_buf, 32));
    CK(cudaMemset(touch_buf, 0, 32));
    const float floor_single = single_us(NULL, NULL, runs * 4, 1);
    const float floor_graph = graph_launches > 0 ? graph_us(NULL, 1000, runs, 1) : 0.0f;
    const float touch_single = single_us(NULL, NULL, runs * 4, 2);
    const float touch_graph = graph_launches > 0 ? graph_us(NULL, 1000, runs, 2) : 0.0f;

    for (size_t bytes = min_b; bytes <= max_b; bytes *= 2) {
        shape(&c, bytes);
        uint64_t traffic = 0;
        size_t max_elems = 0;
        for (int r = 0; r < R; ++r) {
            size_t ib = c.in_elems[r] * 2, ob = c.out_elems[r] * 2;
            traffic += ib + ob;
            if (c.in_elems[r] > max_elems) max_elems = c.in_elems[r];
            CK(cudaMalloc(&c.src[r], ib ? ib : 16));
            CK(cudaMalloc(&c.dst[r], ob ? ob : 16));
            uint16_t *h = (uint16_t *)malloc(ib ? ib : 16);
            for (size_t i = 0; i < c.in_elems[r]; ++i)
                h[i] = (uint16_t)(0x3C00u + (next_u64() & 0x7FFu)) ^ (uint16_t)((next_u64() & 1u) << 15);
            CK(cudaMemcpy(c.src[r], h, ib, cudaMemcpyHostToDevice));
            free(h);
        }
        /* totalBytes as the README defines it */
        uint64_t total = c.coll == C_AG || c.coll == C_AGV ? c.out_elems[0] * 2 : c.in_elems[0] * 2;
        for (int i = 0; i < warmup; ++i) call_once(&c);
        CK(cudaStreamSynchronize(stream));
        PK(purlin_check(ctx));
        purlin_launch_info info;
        PK(purlin_last_launch(ctx, &info));
        const float s_us = single_us(call_once, &c, runs, 0);
        const float g_us = graph_launches > 0 ? graph_us(&c, graph_launches, runs, 0) : 0.0f;
        PK(purlin_check(ctx));
        const float t = g_us > 0 ? g_us : s_us;
        printf("{\"coll\": \"%s\", \"bytes_per_rank\": %zu, \"total_bytes\": %llu, "
               "\"variant\": %d, \"grid\": %d, \"single_us\": %.3f, \"graph_us\": %.3f, "
               "\"floor_single_us\": %.3f, \"floor_graph_us\": %.3f, "
               "\"x_floor_single\": %.3f, \"x_floor_graph\": %.3f, "
               "\"touch_single_us\": %.3f, \"touch_graph_us\": %.3f, "
               "\"x_touch_single\": %.3f, \"x_touch_graph\": %.3f, "
               "\"algbw_gbs\": %.2f, \"eff_gbs\": %.2f}\n",
               argv[1], bytes, (unsigned long long)total, info.variant, info.grid, s_us, g_us,
               floor_single, floor_graph, s_us / floor_single,
               floor_graph > 0 ? g_us / floor_graph : 0.0, touch_single, touch_graph,
               s_us / touch_single, touch_graph > 0 ? g_us / touch_graph : 0.0,
               total / (t * 1e-6) / 1e9, traffic / (t * 1e-6) / 1e9);
        fflush(stdout);
        for (int r = 0; r < R; ++r) {
            CK(cudaFree(c.src[r]));
            CK(cudaFree(c.dst[r]));
        }
        (void)max_elems;
    }
    PK(purlin_finalize(ctx));
    CK(cudaFree(touch_buf));
    CK(cudaStreamDestroy(stream));
    return 0;
}
