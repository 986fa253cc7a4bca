/*
 * device_examples.h -- C entry points of the example kernels that use the
 * device-side API (include/purlin_device.cuh).  Built as
 * libpurlin_examples.so next to the library.  Each launches one kernel on
 * `stream` and returns without waiting; launch failures return
 * PURLIN_ERR_CUDA, and errors inside the collective are read with
 * purlin_device_check.
 */
#ifndef PURLIN_DEVICE_EXAMPLES_H
#define PURLIN_DEVICE_EXAMPLES_H

#include "../../include/purlin.h"

#ifdef __cplusplus
extern "C" {
#endif

/* A kernel whose coll->blocks CTAs all call purlin::device::collective with
 * the descriptor (threads 0: coll->threads; at most 512).  Launched
 * cooperatively when the descriptor is composed. */
purlin_status purlin_example_collective(const purlin_device_coll *coll, int threads,
                                        purlin_stream stream);

/* A fused kernel: ReLU in place on the first n elements of every rank input
 * (max(x, 0), with -0 and negatives to +0 and NaN kept), a grid barrier, then
 * the collective on the result.  Always a cooperative launch. */
purlin_status purlin_example_relu_collective(const purlin_device_coll *coll, size_t n,
                                             int threads, purlin_stream stream);

/* coll->blocks + extra_blocks CTAs: the first coll->blocks run the
 * collective, the others write fill[i] = i * 2654435761 mod 2^32 for i < words. */
purlin_status purlin_example_subset(const purlin_device_coll *coll, int extra_blocks,
                                    unsigned int *fill, size_t words, int threads,
                                    purlin_stream stream);

/* A compute kernel that streams its results through a packet channel:
 * ch->ctas / 2 producer CTAs compute, for every 8-byte unit of the n-element
 * rank buffers, the rank-order binary32 sum of relu(src[s]) (or of src[s]
 * when relu is 0; relu as above) rounded once to dtype, and send it as a
 * packet; the other ch->ctas / 2 CTAs receive each unit and write it to all
 * R outputs.  The outputs equal the AllReduce of the computed inputs; the
 * inputs are not modified.  ch->ctas even and at least 2, the units within
 * the channel's capacity, buffers 8-byte aligned; a cooperative launch of
 * ch->ctas CTAs of purlin_example_packet_stream_threads() threads.  Packet
 * errors are read with purlin_packet_channel_check. */
purlin_status purlin_example_packet_stream(const purlin_packet_channel *ch,
                                          const void *const src[], void *const dst[], int R,
                                          size_t n, purlin_dtype dtype, int relu,
                                          purlin_stream stream);
int purlin_example_packet_stream_threads(void);

/* The README's sample: CTA b copies bytes [b*per_block, (b+1)*per_block) of
 * src to dst with the Atom (4 stages of 16 KiB, 320 threads).  dst and src
 * 2-byte aligned, bytes even; the first non-OK Atom status lands in *status
 * (device memory, zeroed by the caller). */
purlin_status purlin_example_atom_copy(void *dst, const void *src, size_t bytes,
                                       size_t bytes_per_block, int *status,
                                       purlin_stream stream);

/* CTA b reduces elements [b*per_block, (b+1)*per_block) of the nsrc sources
 * (host array of device pointers, 16-byte aligned) into dst with the Atom. */
purlin_status purlin_example_atom_reduce(void *dst, const void *const srcs[], int nsrc,
                                         size_t elems, size_t elems_per_block,
                                         purlin_dtype dtype, int *status,
                                         purlin_stream stream);

/* The shared memory the example Atom asks of each CTA. */
size_t purlin_example_atom_smem_bytes(void);

#ifdef __cplusplus
}
#endif

#endif /* PURLIN_DEVICE_EXAMPLES_H */
