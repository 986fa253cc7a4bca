// noalloc.cu -- an AllReduce entry point that allocates no device memory.
//
// Who needs it: callers that must not call cudaMalloc (or any allocating
// routine) when they reduce.  Examples: code that runs while a CUDA graph is
// being captured (allocation is not a capturable operation), and serving
// engines that hand all free HBM to their own pool at start-up and cannot
// let a library take more.  The context API (purlin_init) allocates its flag
// array and error word with cudaMalloc; this entry point uses a fixed,
// file-scope device array instead.
//
// It runs the same composed AllReduce as purlin_all_reduce with the
// composed mode selected (reducing CTAs publish per-chunk flags, gathering
// CTAs acquire them), so its outputs are bit-identical to that call's.  The
// pages describe no such entry point; it is an addition of this library.
//
// The scratch array:
//   g_noalloc_scratch holds 2 x kStaticFlagSlots u64 flags (one set per
//   epoch parity), one u64 error word and the device epoch (epoch and a
//   completion count): 128 KiB + 32 bytes, kept by every GPU that loads the
//   library until the process exits.  The epoch lives on the device, so a
//   call captured into a CUDA graph gets a new epoch at every replay.  The largest call
//   therefore has at most kStaticFlagSlots reduce chunks of 96 KiB / R bytes
//   per source (rounded down to 16): n * element_size <= 8192 * (98304 / R)
//   bytes per rank (96 MiB per rank at R = 8).  Larger calls return
//   PURLIN_ERR_INVALID_ARG.
//   R is limited to 31 so the compiled plan fits the kernel parameters.
//
// First call on a device: with that device current it looks up the array's
// device address (cudaGetSymbolAddress), sets the kernel attributes and
// zeroes the array with a blocking cudaMemset.  Make that first call before
// any stream capture.  Later calls only clear the error word
// (cudaMemsetAsync on the caller's stream) and launch one kernel.
//
// All calls on a device share the array and it keeps the previous call's
// contents.  Flags need no clearing (each call publishes a larger epoch
// than any value already stored); the error word is cleared per call.
// Calls whose kernels overlap on the GPU (e.g. issued on two streams
// without ordering) race on the flags and give wrong results: order them.
// A device-side wait that expires (100 ms bound) is recorded in the error
// word, and that call's outputs are then unspecified.  The next call clears
// the word, so a caller that wants to know reads it first with
// purlin_noalloc_check (a stream synchronize and one 8-byte copy to the
// host; not during stream capture).
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "launch.h"
#include "plan.h"

namespace {

using namespace purlin;

constexpr uint32_t kStaticFlagSlots = 8192;   // per parity
constexpr int kMaxDevices = 64;
constexpr int kMaxStaticRanks = 31;           // 2R + 1 segments fit the big parameter block
constexpr uint32_t kSlotBytes = 96 * 1024;   // R reduce tiles per stage, as in composed mode
constexpr uint32_t kStages = 2;
constexpr int64_t kTimeoutNs = 100 * 1000 * 1000;
constexpr int kConsumerWarps = 12;

}  // namespace

// flags parity 0 | flags parity 1 | error word | pad | device epoch {epoch, done}
static __device__ __align__(256) unsigned long long g_noalloc_scratch[2 * 8192 + 4];

namespace {

static_assert(sizeof(g_noalloc_scratch) == (2 * kStaticFlagSlots + 4) * 8, "scratch layout");
constexpr size_t kErrWord = 2 * kStaticFlagSlots;
constexpr size_t kEpochWords = 2 * kStaticFlagSlots + 2;   // 16-byte aligned

struct DeviceState {
    bool ready = false;
    unsigned long long *scratch = nullptr;   // device address of g_noalloc_scratch
    int sms = 0;
    int max_smem = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

purlin_status setup_device(int dev, DeviceState &st) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
        return PURLIN_ERR_CUDA;
    if (cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&st.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
        return PURLIN_ERR_CUDA;
    if (configure_kernels(st.max_smem - 1024) != cudaSuccess) return PURLIN_ERR_CUDA;
    if (cudaMemset(p, 0, sizeof(g_noalloc_scratch)) != cudaSuccess) return PURLIN_ERR_CUDA;
    st.scratch = static_cast<unsigned long long *>(p);
    static const unsigned long long kFirstEpoch = 1;   // flags start at 0, below any epoch
    if (cudaMemcpy(st.scratch + kEpochWords, &kFirstEpoch, sizeof kFirstEpoch,
                   cudaMemcpyHostToDevice) != cudaSuccess)
        return PURLIN_ERR_CUDA;
    st.ready = true;
    return PURLIN_OK;
}

}  // namespace

extern "C" purlin_status purlin_all_reduce_noalloc(int R, const void *const src[],
                                                   void *const dst[], size_t n,
                                                   purlin_dtype dtype, purlin_op op,
                                                   purlin_layout layout,
                                                   purlin_stream stream) {
    if (R < 1 || R > kMaxStaticRanks) return PURLIN_ERR_INVALID_ARG;
    CallDesc c;
    c.coll = PURLIN_COLL_ALL_REDUCE;
    c.R = R;
    c.dtype = dtype;
    c.n = n;
    c.counts = nullptr;
    c.op = op;
    c.layout = layout;
    purlin_status st = validate_call(c, src, dst);
    if (st != PURLIN_OK) return st;

    Plan pl;
    st = compile_plan(c, kVariantThroughput, /*ar_mode composed*/ 2, kSlotBytes, kSlotBytes, &pl);
    if (st != PURLIN_OK) return st;
    if (pl.notify_chunks > kStaticFlagSlots) return PURLIN_ERR_INVALID_ARG;   // past the array
    if (param_class(R, pl.segs.size()) < 0) return PURLIN_ERR_INVALID_ARG;
    if (pl.nchunks == 0 && pl.nunits == 0) return PURLIN_OK;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return PURLIN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &ds = g_dev[dev];
    if (!ds.ready) {
        st = setup_device(dev, ds);
        if (st != PURLIN_OK) return st;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned long long *err = ds.scratch + kErrWord;
    if (cudaMemsetAsync(err, 0, sizeof(unsigned long long), s) != cudaSuccess)
        return PURLIN_ERR_CUDA;

    const uint32_t slot_stride = (pl.slot_bytes + 127u) & ~127u;
    const uint32_t limit = (uint32_t)ds.max_smem - 1024;
    const uint32_t stages = kStages;
    // Two 96 KiB stages and the ring's barriers and table: about 193 KiB of
    // dynamic shared memory per CTA.  A device with less returns UNSUPPORTED.
    const uint32_t smem = throughput_smem(stages, slot_stride);
    if (smem > limit) return PURLIN_ERR_UNSUPPORTED;
    const int block = 32 * (2 + kConsumerWarps);
    int per_sm = 0;
    const int pc = param_class(R, pl.segs.size());
    if (throughput_occupancy(dtype, pc, ragged_ring(pl), block, smem, &per_sm) != cudaSuccess ||
        per_sm < 1)
        return PURLIN_ERR_UNSUPPORTED;
    int64_t grid = (int64_t)ds.sms * per_sm;
    const int64_t work = (int64_t)std::max<uint64_t>(pl.nchunks, (pl.nunits + 255) / 256);
    grid = std::max<int64_t>(1, std::min<int64_t>(grid, work));

    LaunchArgs a;
    a.plan = &pl;
    a.segs_dev = nullptr;
    a.src = src;
    a.dst = dst;
    a.R = R;
    a.dtype = dtype;
    a.flags = ds.scratch;              // both parities; the device epoch selects one
    a.flag_slots = kStaticFlagSlots;   // one flag per chunk: no slot is reused within a call
    a.dev_epoch = ds.scratch + kEpochWords;
    a.epoch_inc = 1;                   // odd: the parity flips every call
    a.err = err;
    a.timeout_ns = kTimeoutNs;
    a.drop_notify = -1;
    a.grid = (int)grid;
    a.block = block;
    a.smem = smem;
    a.stages = stages;
    a.slot_stride = slot_stride;
    a.cooperative = pl.composed;
    a.stream = s;
    if (launch_throughput(a) != cudaSuccess) return PURLIN_ERR_CUDA;
    return PURLIN_OK;
}

extern "C" purlin_status purlin_noalloc_check(purlin_stream stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return PURLIN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    const DeviceState &ds = g_dev[dev];
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return PURLIN_ERR_CUDA;
    if (!ds.ready) return PURLIN_OK;   // no call on this device yet
    unsigned long long word = 0;
    unsigned long long *err = ds.scratch + kErrWord;
    if (cudaMemcpyAsync(&word, err, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return PURLIN_ERR_CUDA;
    if (word == 0) return PURLIN_OK;
    if (cudaMemsetAsync(err, 0, sizeof word, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return PURLIN_ERR_CUDA;
    return PURLIN_ERR_TIMEOUT;
}
