// device_examples.cu -- kernels written against the device-side API
// (include/purlin_device.cuh), the way an application would write them,
// with C entry points that launch them.  They show the "Purlin" project
// README's device-side uses:
//   * "Samples": each CTA copies one aligned slice with the Atom;
//   * a collective called from inside a kernel by exactly `blocks` CTAs;
//   * fusing with computation: a kernel that computes its inputs, passes a
//     grid barrier and then runs the collective on them;
//   * a collective entered by some of the grid's CTAs while the others do
//     unrelated work.
// The tests drive these entry points and compare with the CPU oracle.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/purlin_device.cuh"
#include "device_examples.h"

namespace cg = cooperative_groups;
using purlin::device::Atom;
using purlin::device::SnacArgs;

namespace {

constexpr int kMaxThreads = 512;
using CopyAtom = Atom<4, 16384, 8>;   // 4 stages of 16 KiB, 320 threads

// ---------------------------------------------------------------- kernels --

__global__ void __launch_bounds__(kMaxThreads, 1)
    collective_kernel(const __grid_constant__ purlin_device_coll c) {
    extern __shared__ __align__(128) unsigned char ws[];
    purlin::device::collective(c, SnacArgs{ws, (int)gridDim.x, (int)blockIdx.x});
}

// The two kernels below enter the collective after work of their own; they
// share one out-of-line copy of it, which keeps this file's build short (the
// collective carries two builds of the ring for every dtype and rank bound).
// collective_kernel above inlines it, which measured 2-3% faster.
__device__ __noinline__ purlin_status shared_collective(const purlin_device_coll &c,
                                                        const SnacArgs &a) {
    return purlin::device::collective(c, a);
}

// The computation: y = max(x, 0) elementwise, in place on every rank input
// (+0 for negative values and for -0; NaN stays NaN).
__device__ __forceinline__ uint32_t relu_f32(uint32_t b) {
    return (b & 0x80000000u) && (b & 0x7FFFFFFFu) <= 0x7F800000u ? 0u : b;
}
__device__ __forceinline__ uint16_t relu_bf16(uint16_t b) {
    return (b & 0x8000u) && (b & 0x7FFFu) <= 0x7F80u ? (uint16_t)0 : b;
}

__global__ void __launch_bounds__(kMaxThreads, 1)
    relu_then_collective_kernel(const __grid_constant__ purlin_device_coll c, size_t n) {
    extern __shared__ __align__(128) unsigned char ws[];
    const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (int r = 0; r < c.R; ++r) {
        // The descriptor holds the inputs as read-only pointers; the kernel
        // owns these buffers and updates them before the collective reads.
        if (c.dtype == PURLIN_F32) {
            uint32_t *x = static_cast<uint32_t *>(const_cast<void *>(c.src[r]));
            for (size_t i = tid; i < n; i += stride) x[i] = relu_f32(x[i]);
        } else {
            uint16_t *x = static_cast<uint16_t *>(const_cast<void *>(c.src[r]));
            for (size_t i = tid; i < n; i += stride) x[i] = relu_bf16(x[i]);
        }
    }
    cg::this_grid().sync();   // every CTA's inputs are written
    shared_collective(c, SnacArgs{ws, (int)gridDim.x, (int)blockIdx.x});
}

// CTAs [0, c.blocks) run the collective; the others fill `fill` with
// fill[i] = i * 2654435761 (mod 2^32).
__global__ void __launch_bounds__(kMaxThreads, 1)
    subset_kernel(const __grid_constant__ purlin_device_coll c, uint32_t *fill, size_t words) {
    extern __shared__ __align__(128) unsigned char ws[];
    if ((int)blockIdx.x < c.blocks) {
        shared_collective(c, SnacArgs{ws, c.blocks, (int)blockIdx.x});
        return;
    }
    const size_t others = gridDim.x - (unsigned)c.blocks;
    const size_t tid = (size_t)(blockIdx.x - (unsigned)c.blocks) * blockDim.x + threadIdx.x;
    for (size_t i = tid; i < words; i += others * blockDim.x) fill[i] = (uint32_t)(i * 2654435761ull);
}

// ---------------------------------------------------- packet streaming --
//
// A compute kernel that streams its results to consumer CTAs through a
// packet channel, with no grid barrier between computing and moving: CTAs
// [0, G) compute y = relu(x) (or x) of every rank input for their 8-byte
// units, add the R results in rank order in binary32 from rank 0's value,
// round once, and send each unit's sum as a packet; CTAs [G, 2G) receive
// every unit as soon as its packet lands and write it to all R outputs.  The
// result is the AllReduce of the computed inputs, and the inputs are never
// rewritten.

struct StreamArgs {
    const void *src[PURLIN_MAX_RANKS];
    void *dst[PURLIN_MAX_RANKS];
    purlin_packet_channel ch;
    uint64_t nbytes;   // bytes per rank buffer
    int32_t R;
    int32_t G;         // producer CTAs; as many consume
    int32_t relu;
};

constexpr int kStreamThreads = 256;

// `valid` bytes (2, 4, 6 or 8) of a buffer at byte `off`, zero above.
template <int ES>
__device__ __forceinline__ uint64_t load8(const void *base, uint64_t off, uint32_t valid) {
    const char *p = static_cast<const char *>(base) + off;
    if (valid == 8) return *reinterpret_cast<const uint64_t *>(p);
    uint64_t v = 0;
    for (uint32_t j = 0; j < valid; j += ES)
        v |= (ES == 4 ? (uint64_t)*reinterpret_cast<const uint32_t *>(p + j)
                      : (uint64_t)*reinterpret_cast<const uint16_t *>(p + j)) << (8 * j);
    return v;
}

template <int ES>
__device__ __forceinline__ void store8(void *base, uint64_t off, uint32_t valid, uint64_t v) {
    char *p = static_cast<char *>(base) + off;
    if (valid == 8) {
        *reinterpret_cast<uint64_t *>(p) = v;
        return;
    }
    for (uint32_t j = 0; j < valid; j += ES) {
        if (ES == 4) *reinterpret_cast<uint32_t *>(p + j) = (uint32_t)(v >> (8 * j));
        else *reinterpret_cast<uint16_t *>(p + j) = (uint16_t)(v >> (8 * j));
    }
}

// The producer's work for one unit: relu (optional) of each rank's elements,
// summed in rank order in binary32 and rounded once.
template <int DT>
__device__ __forceinline__ uint64_t compute_unit(const StreamArgs &a, uint64_t off,
                                                 uint32_t valid) {
    constexpr int ES = DT == PURLIN_F32 ? 4 : 2;
    constexpr int N = 8 / ES;   // elements per unit
    float acc[N];
    for (int s = 0; s < a.R; ++s) {
        const uint64_t w = load8<ES>(a.src[s], off, valid);
#pragma unroll
        for (int j = 0; j < N; ++j) {
            uint32_t bits;
            if (DT == PURLIN_F32) {
                bits = (uint32_t)(w >> (32 * j));
                if (a.relu) bits = relu_f32(bits);
            } else {
                uint16_t h = (uint16_t)(w >> (16 * j));
                if (a.relu) h = relu_bf16(h);
                bits = (uint32_t)h << 16;
            }
            const float x = __uint_as_float(bits);
            acc[j] = s == 0 ? x : __fadd_rn(acc[j], x);
        }
    }
    uint64_t out = 0;
#pragma unroll
    for (int j = 0; j < N; ++j) {
        if (DT == PURLIN_F32) {
            out |= (uint64_t)__float_as_uint(acc[j]) << (32 * j);
        } else {
            const __nv_bfloat16 h = __float2bfloat16_rn(acc[j]);
            out |= (uint64_t)__bfloat16_as_ushort(h) << (16 * j);
        }
    }
    return out;
}

template <int DT>
__global__ void __launch_bounds__(kStreamThreads)
    packet_stream_kernel(const __grid_constant__ StreamArgs a) {
    constexpr int ES = DT == PURLIN_F32 ? 4 : 2;
    const purlin::device::Packets pk = purlin::device::channel_open(a.ch);
    const bool producer = (int)blockIdx.x < a.G;
    const uint64_t b = producer ? blockIdx.x : blockIdx.x - (unsigned)a.G;
    const uint64_t units = (a.nbytes + 7) / 8;
    const uint64_t stride = (uint64_t)a.G * blockDim.x;
    for (uint64_t u = b * blockDim.x + threadIdx.x; u < units; u += stride) {
        const uint64_t off = 8 * u;
        const uint32_t valid = (uint32_t)(a.nbytes - off < 8 ? a.nbytes - off : 8);
        if (producer) {
            purlin::device::send(a.ch, pk, u, compute_unit<DT>(a, off, valid));
            continue;
        }
        uint64_t v;
        if (!purlin::device::recv(a.ch, pk, u, &v)) break;
        for (int d = 0; d < a.R; ++d) store8<ES>(a.dst[d], off, valid, v);
    }
    purlin::device::channel_close(a.ch);
}

// The README's sample: each CTA copies its slice of `total` bytes.
__global__ void __launch_bounds__(CopyAtom::THREADS, 1)
    atom_copy_kernel(char *dst, const char *src, size_t total, size_t per_block,
                     int *status) {
    extern __shared__ __align__(128) unsigned char ws[];
    const size_t off = (size_t)blockIdx.x * per_block;
    if (off >= total) return;
    const size_t len = total - off < per_block ? total - off : per_block;
    const purlin_status st = CopyAtom::copy(dst + off, src + off, len, ws);
    if (threadIdx.x == 0 && st != PURLIN_OK) atomicCAS(status, 0, (int)st);
}

struct SrcList {
    const void *p[PURLIN_MAX_RANKS];
};

// Each CTA reduces its slice of the nsrc sources into dst.
template <int DT>
__global__ void __launch_bounds__(CopyAtom::THREADS, 1)
    atom_reduce_kernel(char *dst, const __grid_constant__ SrcList s, int nsrc, size_t elems,
                       size_t per_block, int *status) {
    extern __shared__ __align__(128) unsigned char ws[];
    constexpr size_t ES = DT == PURLIN_F32 ? 4 : 2;
    const size_t e0 = (size_t)blockIdx.x * per_block;
    if (e0 >= elems) return;
    const size_t len = elems - e0 < per_block ? elems - e0 : per_block;
    // This CTA's source pointers, offset to its slice (shared memory).
    __shared__ const void *mine[PURLIN_MAX_RANKS];
    for (int i = threadIdx.x; i < nsrc; i += blockDim.x)
        mine[i] = static_cast<const char *>(s.p[i]) + e0 * ES;
    __syncthreads();
    const purlin_status st = CopyAtom::reduce<DT>(dst + e0 * ES, mine, nsrc, len, ws);
    if (threadIdx.x == 0 && st != PURLIN_OK) atomicCAS(status, 0, (int)st);
}

// ----------------------------------------------------------------- helpers --

template <class K>
cudaError_t allow_smem(K kernel, size_t smem) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

int block_for(const purlin_device_coll *c, int threads) {
    return threads > 0 ? threads : c->threads;
}

// Launch a descriptor's kernel; cooperatively when its CTAs wait on one
// another (or when the kernel itself has a grid barrier).
template <class... A>
cudaError_t launch(void (*kernel)(A...), int grid, int block, size_t smem, cudaStream_t stream,
                   bool cooperative, A... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (cooperative) {
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

purlin_status status_of(cudaError_t e) { return e == cudaSuccess ? PURLIN_OK : PURLIN_ERR_CUDA; }

}  // namespace

extern "C" {

purlin_status purlin_example_collective(const purlin_device_coll *c, int threads,
                                        purlin_stream stream) {
    if (c == nullptr || c->blocks < 1) return PURLIN_ERR_INVALID_ARG;
    const int block = block_for(c, threads);
    if (block > kMaxThreads) return PURLIN_ERR_INVALID_ARG;
    if (allow_smem(collective_kernel, c->workspace_bytes) != cudaSuccess) return PURLIN_ERR_CUDA;
    return status_of(launch(collective_kernel, c->blocks, block, c->workspace_bytes,
                            static_cast<cudaStream_t>(stream), c->composed != 0, *c));
}

purlin_status purlin_example_relu_collective(const purlin_device_coll *c, size_t n, int threads,
                                             purlin_stream stream) {
    if (c == nullptr || c->blocks < 1) return PURLIN_ERR_INVALID_ARG;
    const int block = block_for(c, threads);
    if (block > kMaxThreads) return PURLIN_ERR_INVALID_ARG;
    if (allow_smem(relu_then_collective_kernel, c->workspace_bytes) != cudaSuccess)
        return PURLIN_ERR_CUDA;
    return status_of(launch(relu_then_collective_kernel, c->blocks, block, c->workspace_bytes,
                            static_cast<cudaStream_t>(stream), true, *c, n));
}

purlin_status purlin_example_subset(const purlin_device_coll *c, int extra_blocks,
                                    unsigned int *fill, size_t words, int threads,
                                    purlin_stream stream) {
    if (c == nullptr || c->blocks < 1 || extra_blocks < 1 || fill == nullptr)
        return PURLIN_ERR_INVALID_ARG;
    const int block = block_for(c, threads);
    if (block > kMaxThreads) return PURLIN_ERR_INVALID_ARG;
    if (allow_smem(subset_kernel, c->workspace_bytes) != cudaSuccess) return PURLIN_ERR_CUDA;
    return status_of(launch(subset_kernel, c->blocks + extra_blocks, block, c->workspace_bytes,
                            static_cast<cudaStream_t>(stream), c->composed != 0, *c,
                            static_cast<uint32_t *>(fill), words));
}

purlin_status purlin_example_packet_stream(const purlin_packet_channel *ch,
                                          const void *const src[], void *const dst[], int R,
                                          size_t n, purlin_dtype dtype, int relu,
                                          purlin_stream stream) {
    if (ch == nullptr || ch->state == nullptr || src == nullptr || dst == nullptr)
        return PURLIN_ERR_INVALID_ARG;
    if (R < 1 || R > PURLIN_MAX_RANKS || ch->ctas < 2 || (ch->ctas & 1) != 0)
        return PURLIN_ERR_INVALID_ARG;
    if (dtype != PURLIN_F32 && dtype != PURLIN_BF16) return PURLIN_ERR_INVALID_ARG;
    const uint64_t es = dtype == PURLIN_F32 ? 4 : 2;
    const uint64_t nbytes = (uint64_t)n * es;
    if ((nbytes + 7) / 8 > ch->capacity) return PURLIN_ERR_INVALID_ARG;
    StreamArgs a = {};
    for (int r = 0; r < R; ++r) {
        if (src[r] == nullptr || dst[r] == nullptr) return PURLIN_ERR_INVALID_ARG;
        if (((reinterpret_cast<uintptr_t>(src[r]) | reinterpret_cast<uintptr_t>(dst[r])) & 7u) != 0)
            return PURLIN_ERR_ALIGNMENT;
        a.src[r] = src[r];
        a.dst[r] = dst[r];
    }
    a.ch = *ch;
    a.nbytes = nbytes;
    a.R = R;
    a.G = ch->ctas / 2;
    a.relu = relu;
    if (n == 0) return PURLIN_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // producers and consumers wait on one another: a cooperative launch
    if (dtype == PURLIN_F32)
        return status_of(launch(packet_stream_kernel<PURLIN_F32>, ch->ctas, kStreamThreads, 0, st,
                                true, a));
    return status_of(launch(packet_stream_kernel<PURLIN_BF16>, ch->ctas, kStreamThreads, 0, st,
                            true, a));
}

int purlin_example_packet_stream_threads(void) { return kStreamThreads; }

purlin_status purlin_example_atom_copy(void *dst, const void *src, size_t bytes,
                                       size_t bytes_per_block, int *status,
                                       purlin_stream stream) {
    if (bytes_per_block == 0 || status == nullptr) return PURLIN_ERR_INVALID_ARG;
    const size_t grid = (bytes + bytes_per_block - 1) / bytes_per_block;
    if (grid == 0) return PURLIN_OK;
    if (grid > 0x7FFFFFFFu) return PURLIN_ERR_INVALID_ARG;
    if (allow_smem(atom_copy_kernel, CopyAtom::PIPELINE_SMEM_BYTES) != cudaSuccess)
        return PURLIN_ERR_CUDA;
    return status_of(launch(atom_copy_kernel, (int)grid, CopyAtom::THREADS,
                            CopyAtom::PIPELINE_SMEM_BYTES, static_cast<cudaStream_t>(stream),
                            false, static_cast<char *>(dst), static_cast<const char *>(src), bytes,
                            bytes_per_block, status));
}

purlin_status purlin_example_atom_reduce(void *dst, const void *const srcs[], int nsrc,
                                         size_t elems, size_t elems_per_block,
                                         purlin_dtype dtype, int *status,
                                         purlin_stream stream) {
    if (nsrc < 1 || nsrc > PURLIN_MAX_RANKS || srcs == nullptr || elems_per_block == 0 ||
        status == nullptr)
        return PURLIN_ERR_INVALID_ARG;
    if (dtype != PURLIN_F32 && dtype != PURLIN_BF16) return PURLIN_ERR_INVALID_ARG;
    SrcList s = {};
    for (int i = 0; i < nsrc; ++i) s.p[i] = srcs[i];
    const size_t grid = (elems + elems_per_block - 1) / elems_per_block;
    if (grid == 0) return PURLIN_OK;
    if (grid > 0x7FFFFFFFu) return PURLIN_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dtype == PURLIN_F32) {
        if (allow_smem(atom_reduce_kernel<PURLIN_F32>, CopyAtom::PIPELINE_SMEM_BYTES) != cudaSuccess)
            return PURLIN_ERR_CUDA;
        return status_of(launch(atom_reduce_kernel<PURLIN_F32>, (int)grid, CopyAtom::THREADS,
                                CopyAtom::PIPELINE_SMEM_BYTES, st, false,
                                static_cast<char *>(dst), s, nsrc, elems, elems_per_block, status));
    }
    if (allow_smem(atom_reduce_kernel<PURLIN_BF16>, CopyAtom::PIPELINE_SMEM_BYTES) != cudaSuccess)
        return PURLIN_ERR_CUDA;
    return status_of(launch(atom_reduce_kernel<PURLIN_BF16>, (int)grid, CopyAtom::THREADS,
                            CopyAtom::PIPELINE_SMEM_BYTES, st, false, static_cast<char *>(dst), s,
                            nsrc, elems, elems_per_block, status));
}

size_t purlin_example_atom_smem_bytes(void) { return CopyAtom::PIPELINE_SMEM_BYTES; }

}  // extern "C"
