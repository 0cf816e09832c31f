// noalloc.cu -- an all-reduce entry point that allocates no device memory.
//
// Some callers may not allocate device memory when they reduce:
//   - a host program whose device memory belongs to another allocator (a
//     framework's caching allocator, a pre-planned arena with a fixed
//     budget), where a stray cudaMalloc would go around that allocator;
//   - a caller that cannot pay for cudaMalloc/cudaFree at call time: both
//     can block, and cudaFree synchronises the device.
// rar_init allocates the ring executor's scratch.  This file offers the
// same ring executor without a handle: its scratch -- one progress word per
// warp, one receive counter per CTA, the status word and the abort word -- lives
// in one file-scope device array of fixed size, so the library allocates
// nothing.  The caller still passes the rank buffers, which hold inputs and
// outputs.
//
// Limits (checked on every call; anything beyond them is rejected):
//   p <= 64 ranks (rank pointers travel in the kernel parameters), and
//   p * channels <= 1024 CTAs (the array holds a progress word for each of
//   their warps).
// The array is about 80 KB and stays resident on every GPU that loads the
// library until the process exits.
//
// Set-up: every call takes the array's device address on the current device
// with cudaGetSymbolAddress (cheap; it allocates nothing).  The first call
// on a device, and the first after the array moved (the module is loaded
// again after cudaDeviceReset), also clears the array once, synchronously;
// make that first call before any stream capture.
// Tuning, fixed: 256 threads per CTA, every co-resident CTA up to 1024 in
// all (p * channels), slices of 128 KB, one slice position at a time through
// every step.  The results do not depend on it.
// Every call shares the array: progress words carry the launch's epoch (kept
// in the array itself), so no per-call clearing is needed, but two calls
// that overlap on the GPU (on two streams, or from two threads) race on the
// same words.  Order them.
#include <mutex>
#include <string>

#include "rar_internal.h"

namespace rar {
void set_handleless_error(const std::string &msg);  // defined in rar_api.cu
}

namespace {

using namespace rar;

constexpr int kNoAllocMaxCtas = 1024;
constexpr int kNoAllocMaxDevices = 64;
constexpr int kNoAllocThreads = 256;
constexpr long long kNoAllocSliceBytes = 128 << 10;
constexpr unsigned long long kNoAllocTimeoutNs = 2000000000ull;

// Layout of the scratch array.
struct NoAllocScratch {
    unsigned long long flags[kNoAllocMaxCtas * (kNoAllocThreads / 32)];  // one per warp
    unsigned long long recv_counts[kNoAllocMaxCtas];
    RingStatus status;
    unsigned abort_word;
    unsigned epoch_word;    // the last finished launch's epoch
    unsigned finish_count;  // CTAs of the running launch that finished
};
constexpr size_t kScratchWords = (sizeof(NoAllocScratch) + 7) / 8;

static __device__ __align__(256) unsigned long long g_noalloc_scratch[kScratchWords];

struct DeviceSlot {
    void *cleared = nullptr;  // the array's device address when it was last cleared
};

std::mutex g_mutex;
DeviceSlot g_slots[kNoAllocMaxDevices];

int reject(int code, const std::string &msg) {
    set_handleless_error("rar_allreduce_noalloc: " + msg);
    return code;
}

}  // namespace

extern "C" int rar_allreduce_noalloc(void *const *bufs, int p, size_t n, int dtype, int op, void *stream) {
    set_handleless_error("");
    if (!bufs) return reject(RAR_EINVAL, "bufs is NULL");
    if (p < 1 || p > kInlineP) return reject(RAR_EINVAL, "p must be in [1, 64] (limit of this entry point)");
    if (dtype < RAR_INT32 || dtype > RAR_FLOAT16) return reject(RAR_EINVAL, "unknown dtype");
    if (op < RAR_SUM || op > RAR_AVG_PREDIV) return reject(RAR_EINVAL, "unknown op");
    if ((op == RAR_AVG || op == RAR_AVG_PREDIV) && dtype == RAR_INT32) return reject(RAR_EUNSUPPORTED, "avg is not offered for int32");
    const size_t e = (size_t)elem_bytes(dtype);
    if (n > (size_t)(1ull << 62) / e) return reject(RAR_EINVAL, "n * element size overflows");
    if (n == 0) return RAR_OK;
    for (int r = 0; r < p; r++)
        if (!bufs[r]) return reject(RAR_EINVAL, "rank buffer " + std::to_string(r) + " is NULL");
    if (p == 1) return RAR_OK;
    const size_t bytes = n * e;
    for (int a = 0; a < p; a++)
        for (int b = a + 1; b < p; b++) {
            const uintptr_t x = (uintptr_t)bufs[a], y = (uintptr_t)bufs[b];
            if (x < y + bytes && y < x + bytes)
                return reject(RAR_EINVAL, "rank buffers " + std::to_string(a) + " and " + std::to_string(b) +
                                              " overlap");
        }
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return reject(RAR_ECUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(ce));
    if (dev < 0 || dev >= kNoAllocMaxDevices) return reject(RAR_EUNSUPPORTED, "device ordinal above 63");
    for (int r = 0; r < p; r++) {
        cudaPointerAttributes at{};
        ce = cudaPointerGetAttributes(&at, bufs[r]);
        if (ce != cudaSuccess) {
            cudaGetLastError();
            return reject(RAR_EINVAL, "rank buffer " + std::to_string(r) + " is not CUDA memory");
        }
        if ((at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) || at.device != dev)
            return reject(RAR_EINVAL, "rank buffer " + std::to_string(r) + " is not memory of the current device");
    }
    bool vec16 = true;
    for (int r = 0; r < p; r++)
        if ((uintptr_t)bufs[r] % 16) vec16 = false;

    // channels: all co-resident CTAs, within the scratch array's capacity
    int per_sm = 0;
    int max_ctas = ring_max_coresident_ctas(dtype, op, vec16, kNoAllocThreads, &per_sm);
    if (max_ctas > kNoAllocMaxCtas) max_ctas = kNoAllocMaxCtas;
    const int G = max_ctas / p;
    if (G < 1) return reject(RAR_EUNSUPPORTED, "p rank groups cannot be co-resident");

    // The array's address on this device.  In host code the symbol is only a
    // host-side stand-in; the kernel must be given this address.
    void *addr = nullptr;
    ce = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
    if (ce != cudaSuccess) {
        cudaGetLastError();
        return reject(RAR_ECUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(ce));
    }
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        DeviceSlot &slot = g_slots[dev];
        if (slot.cleared != addr) {
            // first use of this copy of the array: start from zero (epoch,
            // finish count, abort word, progress words)
            ce = cudaMemset(addr, 0, sizeof(g_noalloc_scratch));
            if (ce == cudaSuccess) ce = cudaDeviceSynchronize();
            if (ce != cudaSuccess)
                return reject(RAR_ECUDA, std::string("clearing the scratch array: ") + cudaGetErrorString(ce));
            slot.cleared = addr;
        }
    }
    NoAllocScratch *scratch = static_cast<NoAllocScratch *>(addr);

    // slices: at most 128 KB, and at most 2^20 - 2 slice positions per
    // channel and step (the progress words count 32-bit items)
    long long slice = kNoAllocSliceBytes / (long long)e;
    const long long maxchunk = ((long long)n + p - 1) / p;
    while ((maxchunk + slice - 1) / slice / G > (1ll << 20) - 2) slice *= 2;

    RingArgs a;
    for (int r = 0; r < kInlineP; r++) a.bufs.inl[r] = r < p ? bufs[r] : nullptr;
    a.bufs.table = nullptr;
    a.n = (long long)n;
    a.first = 0;
    a.n_total = (long long)n;
    a.p = p;
    a.layout = RING_FLAT;
    a.group = p;
    a.channels = G;
    a.fwd_channels = G;
    a.split = (long long)n;
    a.slice = slice;
    a.block = 1;  // one slice position at a time through every step, as the handle's default
    a.tree_scale = 0;
    a.first_step = 0;
    a.n_steps = 2 * (p - 1);
    a.inv_p = 1.0f / (float)p;
    a.epoch_word = &scratch->epoch_word;
    a.finish_count = &scratch->finish_count;
    a.flag_capacity = kNoAllocMaxCtas * (kNoAllocThreads / 32);
    a.flags = scratch->flags;
    a.mailbox = nullptr;
    a.mailbox_words = 0;
    a.slot_words = 0;
    a.recv_counts = scratch->recv_counts;
    a.status = &scratch->status;
    a.abort_word = &scratch->abort_word;
    a.timeout_ns = kNoAllocTimeoutNs;
    a.fault_mode = RAR_FAULT_NONE;
    a.fault_rank = 0;
    a.fault_delay_ns = 0;
    a.trace = nullptr;
    a.trace_steps = 0;
    ce = launch_ring(a, dtype, op, vec16, kNoAllocThreads, (cudaStream_t)stream);
    if (ce != cudaSuccess) return reject(RAR_ECUDA, std::string("launching the ring executor: ") + cudaGetErrorString(ce));
    return RAR_OK;
}
