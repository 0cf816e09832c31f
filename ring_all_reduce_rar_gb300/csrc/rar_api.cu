// rar_api.cu -- the C-ABI of the ring all-reduce library: argument checks,
// the handle and its scratch, engine planning and launch, status and send
// accounting.  Declarations and the contract are in include/rar.h.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <string>
#include <utility>
#include <vector>

#include "rar_internal.h"

namespace {

using namespace rar;

constexpr int kMaxRingCtas = 8192;           // counters capacity; CTAs of a ring or tree launch
// progress words: one per warp of a ring launch, one per (rank, slice, warp)
// of a tree launch (32 MB)
constexpr int kFlagWords = 1 << 22;
static_assert(kFlagWords >= kMaxRingCtas * kRingMaxWarps, "a progress word per ring warp");
constexpr int kRingPhases = 3;               // counter arrays: one per ring launch of a call
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;
// Shortest accepted rar_options.timeout_ns: a bound on waits of a few
// microseconds (a hand-off, a bulk load) that still leaves headroom for a
// preempted or briefly stalled CTA; shorter values would report timeouts of
// healthy launches.
constexpr unsigned long long kMinTimeoutNs = 1000000ull;
constexpr long long kMaxSlicesPerChannelStep = (1ll << 20) - 2;  // slice positions per channel and step
constexpr long long kRingMaxSliceBytes = 128 << 10;
constexpr long long kLLMailboxWords = (long long)RAR_LL_MAILBOX_BYTES / 8;
// protocol auto: the low-latency ring up to this many bytes per rank (p = 16
// sweep on GB300: 31 us against 72 us at 4 KB per rank, 68 against 80 at 1 MB)
constexpr size_t kLLAutoMaxBytes = (size_t)1 << 20;
// protocol auto for the tree engine: from p = 16 (below that the
// progress-word tree is as fast: its per-call cost is lower), up to this
// many bytes per rank (p = 16: 20.5 us against 22.5 at 64 KB per rank,
// 41 against 27 at 256 KB, where a thread carries several batches of words
// through the whole tree one after the other)
constexpr int kLLTreeAutoMinP = 16;
constexpr size_t kLLTreeAutoMaxBytes = (size_t)64 << 10;

thread_local std::string g_init_error;  // errors before a handle exists
// step trace: {work, wait} per (rank, step)
constexpr size_t kTraceWords = 2 * (size_t)RAR_MAX_P * RAR_TRACE_MAX_STEPS;

}  // namespace

struct rar_ctx {
    int device = 0;
    rar_options opt{};
    std::string err;
    int sm_count = 0;
    // scratch owned by the handle (ring engines; table for p > kInlineP)
    unsigned long long *flags = nullptr;
    unsigned long long *recv_counts = nullptr;
    RingStatus *status = nullptr;
    unsigned *abort_word = nullptr;
    unsigned *epoch_words = nullptr;  // [0] last finished launch's epoch, [1] finish counter
    void **ptr_table = nullptr;
    unsigned long long *ll_box = nullptr;  // low-latency mailbox, kLLMailboxWords
    unsigned long long *trace = nullptr;   // step trace (rar_options.trace), kTraceWords
    bool last_traced = false;              // the last call filled the trace
    int last_trace_steps = 0;
    unsigned acked_seq = 0;           // status failures already reported
    // last call, for rar_status / rar_send_counts
    bool have_last = false;
    cudaStream_t last_stream = nullptr;
    bool last_ring = false;
    int last_p = 0;
    // ring launches of the last call (the hierarchical schedule makes three)
    int last_phases = 0;
    int last_layout[3] = {0, 0, 0};
    int last_channels[3] = {0, 0, 0};
    int last_fwd_channels[3] = {0, 0, 0};
    int last_group = 0;
};

namespace {

int fail(rar_ctx *h, int code, const std::string &msg) {
    if (h) h->err = msg;
    else g_init_error = msg;
    return code;
}

int cuda_fail(rar_ctx *h, cudaError_t e, const char *what) {
    return fail(h, RAR_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// Make `dev` current for the scope of a call and restore the caller's device.
struct DeviceGuard {
    int prev = -1;
    bool changed = false;
    cudaError_t err = cudaSuccess;
    explicit DeviceGuard(int dev) {
        err = cudaGetDevice(&prev);
        if (err == cudaSuccess && prev != dev) {
            err = cudaSetDevice(dev);
            changed = err == cudaSuccess;
        }
    }
    ~DeviceGuard() {
        if (changed) cudaSetDevice(prev);
    }
};

int check_options(rar_ctx *h, const rar_options &o) {
    if (o.engine < RAR_ENGINE_FUSED || o.engine > RAR_ENGINE_TREE)
        return fail(h, RAR_EINVAL, "unknown engine");
    if (o.channels < 0 || o.slice_elems < 0 || o.block_threads < 0)
        return fail(h, RAR_EINVAL, "negative channels, slice_elems or block_threads");
    if (o.block_threads && (o.block_threads % 32 || o.block_threads > 1024))
        return fail(h, RAR_EINVAL, "block_threads must be a multiple of 32, at most 1024");
    if (o.fault_mode < RAR_FAULT_NONE || o.fault_mode > RAR_FAULT_DELAY)
        return fail(h, RAR_EINVAL, "unknown fault_mode");
    if (o.fused_path < 0 || o.fused_path > 2) return fail(h, RAR_EINVAL, "unknown fused_path");
    if (o.hier_group < 0 || o.hier_group > RAR_MAX_P) return fail(h, RAR_EINVAL, "hier_group out of range");
    if (o.protocol < 0 || o.protocol > 2) return fail(h, RAR_EINVAL, "unknown protocol");
    if (o.slice_block < 0) return fail(h, RAR_EINVAL, "negative slice_block");
    if (o.timeout_ns != 0 && o.timeout_ns < kMinTimeoutNs)
        return fail(h, RAR_EINVAL, "timeout_ns must be 0 (2 s) or at least 1 ms (1000000)");
    return RAR_OK;
}

// Argument checks shared by every collective (include/rar.h, rar_allreduce).
// host_mapped: the pointers are device aliases of page-locked host memory.
int check_call(rar_ctx *h, void *const *bufs, int p, size_t n, int dtype, int op, bool host_mapped = false) {
    if (!bufs) return fail(h, RAR_EINVAL, "bufs is NULL");
    if (p < 1 || p > RAR_MAX_P) return fail(h, RAR_EINVAL, "p must be in [1, RAR_MAX_P]");
    if (dtype < RAR_INT32 || dtype > RAR_FLOAT16) return fail(h, RAR_EINVAL, "unknown dtype");
    if (op < RAR_SUM || op > RAR_AVG_PREDIV) return fail(h, RAR_EINVAL, "unknown op");
    if ((op == RAR_AVG || op == RAR_AVG_PREDIV) && dtype == RAR_INT32) return fail(h, RAR_EUNSUPPORTED, "avg is not offered for int32");
    const size_t e = (size_t)elem_bytes(dtype);
    if (n > (size_t)(1ull << 62) / e) return fail(h, RAR_EINVAL, "n * element size overflows");
    if (n == 0) return RAR_OK;  // nothing is accessed: NULL buffers are fine
    for (int r = 0; r < p; r++)
        if (!bufs[r]) return fail(h, RAR_EINVAL, "rank buffer " + std::to_string(r) + " is NULL");
    if (p == 1) return RAR_OK;
    const size_t bytes = n * e;
    std::vector<std::pair<uintptr_t, int>> spans;
    spans.reserve((size_t)p);
    for (int r = 0; r < p; r++) spans.emplace_back((uintptr_t)bufs[r], r);
    std::sort(spans.begin(), spans.end());
    for (int k = 1; k < p; k++)
        if (spans[k].first < spans[k - 1].first + bytes)
            return fail(h, RAR_EINVAL, "rank buffers " + std::to_string(spans[k - 1].second) + " and " +
                                           std::to_string(spans[k].second) + " overlap");
    if (!h->opt.skip_pointer_check && !host_mapped) {
        for (int r = 0; r < p; r++) {
            cudaPointerAttributes at{};
            cudaError_t ce = cudaPointerGetAttributes(&at, bufs[r]);
            if (ce != cudaSuccess) {
                cudaGetLastError();
                return fail(h, RAR_EINVAL, "rank buffer " + std::to_string(r) + " is not CUDA memory");
            }
            if ((at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) || at.device != h->device)
                return fail(h, RAR_EINVAL, "rank buffer " + std::to_string(r) + " is not device memory of device " +
                                               std::to_string(h->device));
        }
    }
    return RAR_OK;
}

// Fill the pointer part of the launch arguments (table copy for large p).
int fill_ptrs(rar_ctx *h, RankPtrs &rp, void *const *bufs, int p, cudaStream_t stream) {
    std::memset(&rp, 0, sizeof(rp));
    if (p <= kInlineP) {
        for (int r = 0; r < p; r++) rp.inl[r] = bufs[r];
        return RAR_OK;
    }
    // pageable source: staged by the runtime before the call returns
    cudaError_t ce = cudaMemcpyAsync(h->ptr_table, bufs, sizeof(void *) * (size_t)p, cudaMemcpyHostToDevice, stream);
    if (ce != cudaSuccess) return cuda_fail(h, ce, "copying the rank pointer table");
    rp.table = h->ptr_table;
    return RAR_OK;
}

bool all_aligned16(void *const *bufs, int p) {
    for (int r = 0; r < p; r++)
        if ((uintptr_t)bufs[r] % 16) return false;
    return true;
}

// Record a ring or tree launch of the current call, for rar_send_counts:
// launch `idx` of the call (the hierarchical schedule makes three).
void note_ring_launch(rar_ctx *h, int idx, int layout, int channels, int fwd_channels, int group) {
    h->last_ring = true;
    h->last_layout[idx] = layout;
    h->last_channels[idx] = channels;
    h->last_fwd_channels[idx] = fwd_channels;
    h->last_group = group;
    h->last_phases = idx + 1;
}

// Launch arguments shared by every ring and tree launch of a handle: the
// rank pointers, sizes, the handle's scratch (epoch, progress words,
// mailbox, counters, status) and its timeout and fault options.  The caller
// sets the schedule fields (layout, channels, slices, steps).
RingArgs handle_ring_args(const rar_ctx *h, const RankPtrs &ptrs, int p, size_t n, long long g_first,
                          long long n_total) {
    RingArgs a;
    a.bufs = ptrs;
    a.n = (long long)n;
    a.first = g_first;
    a.n_total = n_total;
    a.p = p;
    a.layout = RING_FLAT;
    a.group = p;
    a.channels = 1;
    a.fwd_channels = 1;
    a.split = n_total;
    a.slice = 0;
    a.block = 0;
    a.tree_scale = 0;
    a.first_step = 0;
    a.n_steps = 0;
    a.inv_p = 1.0f / (float)p;
    a.epoch_word = h->epoch_words;
    a.finish_count = h->epoch_words + 1;
    a.flag_capacity = kFlagWords;
    a.flags = h->flags;
    a.mailbox = h->ll_box;
    a.mailbox_words = kLLMailboxWords;
    a.slot_words = 0;
    a.recv_counts = h->recv_counts;
    a.status = h->status;
    a.abort_word = h->abort_word;
    a.timeout_ns = h->opt.timeout_ns ? h->opt.timeout_ns : kDefaultTimeoutNs;
    a.fault_mode = h->opt.fault_mode;
    a.fault_rank = h->opt.fault_rank;
    a.fault_delay_ns = h->opt.fault_delay_ns;
    a.trace = nullptr;
    a.trace_steps = 0;
    return a;
}

// Arm the step trace for a launch of `steps` schedule steps per rank: clear
// the record (stream-ordered) and point the launch at it.
int arm_trace(rar_ctx *h, RingArgs &a, int p, int steps, cudaStream_t stream) {
    if (!h->opt.trace || !h->trace) return RAR_OK;
    cudaError_t ce = cudaMemsetAsync(h->trace, 0, sizeof(unsigned long long) * 2 * (size_t)p * (size_t)steps, stream);
    if (ce != cudaSuccess) return cuda_fail(h, ce, "clearing the step trace");
    a.trace = h->trace;
    a.trace_steps = steps;
    h->last_traced = true;
    h->last_trace_steps = steps;
    return RAR_OK;
}

// One ring launch: `layout` picks the rings (flat; inside nodes of `group`;
// across nodes), steps [first, first + steps) of that ring size, counters in
// array `phase_idx`.  Channels and slices follow the tuned defaults unless
// the options set them.
int launch_ring_phase(rar_ctx *h, const RankPtrs &ptrs, int p, size_t n, long long g_first, long long n_total,
                      int dtype, int op, bool vec16, bool bidir, int layout, int group, int first, int steps,
                      int phase_idx, cudaStream_t stream) {
    const int threads = h->opt.block_threads ? h->opt.block_threads : 512;
    if (threads > 512) return fail(h, RAR_EINVAL, "ring engines run at most 512 threads per CTA");
    int per_sm = 0;
    const int max_ctas = std::min(ring_max_coresident_ctas(dtype, op, vec16, threads, &per_sm), kMaxRingCtas);
    // Defaults (from slice x channel x block sweeps on GB300): use every
    // co-resident CTA, and give each channel slices of up to 128 KB, since
    // each slice hand-off costs a couple of microseconds.
    int G = h->opt.channels;
    if (G == 0) G = std::max(1, max_ctas / p);
    if (bidir && G < 2) G = 2;
    if ((long long)G * p > max_ctas) {
        if (h->opt.channels) return fail(h, RAR_EUNSUPPORTED, "p * channels CTAs cannot be co-resident on this GPU");
        G = max_ctas / p;
        if (G < (bidir ? 2 : 1))
            return fail(h, RAR_EUNSUPPORTED, "p = " + std::to_string(p) + " rank groups cannot be co-resident");
    }
    const long long split = bidir ? n_total - n_total / 2 : n_total;  // chunk_bounds(n_total, 2)
    int fwd_channels = bidir ? (G + 1) / 2 : G;
    int min_g = bidir ? std::min(fwd_channels, G - fwd_channels) : G;
    // the longest chunk piece any ring of this launch moves
    const int rp = layout == RING_FLAT ? p : layout == RING_INTRA ? group : p / group;
    const long long seg = layout == RING_INTER ? (n_total + group - 1) / group : std::max(split, n_total - split);
    const long long maxchunk = std::min((seg + rp - 1) / rp, (long long)n);
    // small buffers: no more channels than slices of at least 1024
    // elements (an idle CTA still costs its launch and its finish count)
    if (!h->opt.channels) {
        const long long per_ring = std::max<long long>(1, (maxchunk + 1023) / 1024);
        const long long needed = bidir ? 2 * per_ring : per_ring;
        if (needed < G) {
            G = (int)needed;
            fwd_channels = bidir ? G / 2 : G;
            min_g = bidir ? G / 2 : G;
        }
    }
    // slices: a channel's share of the longest chunk, at most 128 KB
    // (GB300, p = 4 ... 16 fp32/int32 at 1-4 GiB: 1.18-1.21 of the roofline
    // with 128 KB slices, 1.03-1.07 with 256 KB)
    long long slice = h->opt.slice_elems;
    if (slice == 0) {
        slice = (maxchunk + min_g - 1) / min_g;
        slice = (slice + 1023) / 1024 * 1024;
        slice = std::min<long long>(std::max<long long>(slice, 1024), kRingMaxSliceBytes / elem_bytes(dtype));
    }
    slice = std::max<long long>(16, (slice + 15) / 16 * 16);
    while ((maxchunk + slice - 1) / slice / min_g > kMaxSlicesPerChannelStep) slice *= 2;

    RingArgs a = handle_ring_args(h, ptrs, p, n, g_first, n_total);
    a.layout = layout;
    a.group = group;
    a.channels = G;
    a.fwd_channels = fwd_channels;
    a.split = split;
    a.slice = slice;
    // slice order: one slice position at a time through every step (p = 8,
    // 16 GiB bf16 on GB300: 9.3 ms, against 11.2 ms step by step; the
    // neighbour's reads of fresh partials then hit L2)
    a.block = h->opt.slice_block ? h->opt.slice_block : 1;
    a.first_step = first;
    a.n_steps = steps;
    a.recv_counts = h->recv_counts + (size_t)phase_idx * kMaxRingCtas;
    if (layout == RING_FLAT) {  // (the hierarchical schedule's launches are not traced)
        int rc = arm_trace(h, a, p, 2 * (p - 1), stream);
        if (rc != RAR_OK) return rc;
    }
    cudaError_t ce = launch_ring(a, dtype, op, vec16, threads, stream);
    if (ce != cudaSuccess) {
        if (ce == cudaErrorCooperativeLaunchTooLarge) return fail(h, RAR_EUNSUPPORTED, "ring grid cannot be co-resident");
        return cuda_fail(h, ce, "launching the ring executor");
    }
    note_ring_launch(h, phase_idx, layout, G, fwd_channels, group);
    return RAR_OK;
}

// Words per mailbox slot for the low-latency ring: the longest chunk part
// of the launch, in 32-bit words; 0 if the mailbox cannot hold
// p * 2 (p - 1) such slots.
long long ll_slot_words(int p, size_t n, long long n_total, int dtype) {
    const long long maxchunk = std::min((n_total + p - 1) / p, (long long)n);
    const long long epw = 4 / elem_bytes(dtype);
    const long long words = std::max<long long>(1, (maxchunk + epw - 1) / epw);
    if ((long long)p * 2 * (p - 1) * words > kLLMailboxWords) return 0;
    return words;
}

// The low-latency ring (full all-reduce, flat forward ring): enough CTAs per
// rank for one word per thread and step, within the co-resident grid.
int launch_ring_ll_phase(rar_ctx *h, const RankPtrs &ptrs, int p, size_t n, long long g_first, long long n_total,
                         int dtype, int op, long long slot_words, cudaStream_t stream) {
    const int threads = ring_ll_threads();
    const int max_ctas = std::min(ll_max_coresident_ctas(false, dtype, op), kMaxRingCtas);
    if (max_ctas < p) return fail(h, RAR_EUNSUPPORTED, "p = " + std::to_string(p) + " rank groups cannot be co-resident");
    int G = h->opt.channels;
    if (G == 0) G = (int)std::min<long long>(max_ctas / p, (slot_words + threads - 1) / threads);
    if ((long long)G * p > max_ctas) return fail(h, RAR_EUNSUPPORTED, "p * channels CTAs cannot be co-resident on this GPU");
    RingArgs a = handle_ring_args(h, ptrs, p, n, g_first, n_total);
    a.channels = G;
    a.fwd_channels = G;
    a.n_steps = 2 * (p - 1);
    a.slot_words = slot_words;
    cudaError_t ce = launch_ring_ll(a, dtype, op, stream);
    if (ce != cudaSuccess) {
        if (ce == cudaErrorCooperativeLaunchTooLarge) return fail(h, RAR_EUNSUPPORTED, "ring grid cannot be co-resident");
        return cuda_fail(h, ce, "launching the low-latency ring");
    }
    note_ring_launch(h, 0, RING_FLAT, G, G, p);
    return RAR_OK;
}

// Words per mailbox slot for the low-latency tree: the whole buffer, in
// 32-bit words; 0 if p * (ceil(log2 p) + 1) such slots do not fit.
long long tree_ll_slot_words(int p, size_t n, int dtype) {
    int L = 0;
    while ((1 << L) < p) L++;
    const long long epw = 4 / elem_bytes(dtype);
    const long long words = std::max<long long>(1, ((long long)n + epw - 1) / epw);
    if ((long long)p * (L + 1) * words > kLLMailboxWords) return 0;
    return words;
}

// The low-latency tree: one word per thread where the co-resident grid
// allows it.
int launch_tree_ll_phase(rar_ctx *h, const RankPtrs &ptrs, int p, size_t n, int dtype, int op, long long slot_words,
                         cudaStream_t stream) {
    const int threads = ring_ll_threads();
    const int max_ctas = std::min(ll_max_coresident_ctas(true, dtype, op), kMaxRingCtas);
    if (max_ctas < p) return fail(h, RAR_EUNSUPPORTED, "p = " + std::to_string(p) + " rank groups cannot be co-resident");
    int G = h->opt.channels;
    if (G == 0) G = (int)std::min<long long>(max_ctas / p, (slot_words + threads - 1) / threads);
    if ((long long)G * p > max_ctas) return fail(h, RAR_EUNSUPPORTED, "p * channels CTAs cannot be co-resident on this GPU");
    cudaError_t ce = cudaMemsetAsync(h->recv_counts, 0, sizeof(unsigned long long) * (size_t)p, stream);
    if (ce != cudaSuccess) return cuda_fail(h, ce, "clearing the send counters");
    RingArgs a = handle_ring_args(h, ptrs, p, n, 0, (long long)n);  // the tree's order ignores the index
    a.layout = TREE;
    a.channels = G;
    a.fwd_channels = G;
    a.slot_words = slot_words;
    ce = launch_tree_ll(a, dtype, op, stream);
    if (ce != cudaSuccess) {
        if (ce == cudaErrorCooperativeLaunchTooLarge) return fail(h, RAR_EUNSUPPORTED, "tree grid cannot be co-resident");
        return cuda_fail(h, ce, "launching the low-latency tree");
    }
    note_ring_launch(h, 0, TREE, G, G, p);
    return RAR_OK;
}

// The tree executor.  CTAs: rank r gets scale * w_r of them (w_r: the steps
// it takes part in, 2 (p - 1) in all), with the largest scale that fits the
// co-resident grid, so that every CTA carries about the same work; when even
// scale 1 does not fit, or `channels` is set, every rank gets the same
// number.  Slices: up to 128 KB, with one progress word per (rank, slice,
// warp).
int launch_tree_schedule(rar_ctx *h, const RankPtrs &ptrs, int p, size_t n, int dtype, int op, bool vec16,
                         cudaStream_t stream) {
    const int threads = h->opt.block_threads ? h->opt.block_threads : 512;
    if (threads > 512) return fail(h, RAR_EINVAL, "the tree executor runs at most 512 threads per CTA");
    const int max_ctas = std::min(tree_max_coresident_ctas(dtype, op, vec16, threads), kMaxRingCtas);
    int scale = 0, G = 0;
    if (h->opt.channels) {
        G = h->opt.channels;
        if ((long long)G * p > max_ctas) return fail(h, RAR_EUNSUPPORTED, "p * channels CTAs cannot be co-resident on this GPU");
    } else {
        scale = max_ctas / (2 * (p - 1));
        if (scale < 1) {
            G = max_ctas / p;
            if (G < 1) return fail(h, RAR_EUNSUPPORTED, "p = " + std::to_string(p) + " rank groups cannot be co-resident");
        }
    }
    // the CTAs of the rank with the least work (odd ranks: one step)
    const long long g_min = scale > 0 ? scale : G;
    long long slice = h->opt.slice_elems;
    if (slice == 0) {
        slice = ((long long)n + g_min - 1) / g_min;
        slice = std::min<long long>(std::max<long long>((slice + 1023) / 1024 * 1024, 1024),
                                    kRingMaxSliceBytes / elem_bytes(dtype));
    }
    slice = std::max<long long>(16, (slice + 15) / 16 * 16);
    // one progress word per (rank, slice, warp)
    while ((long long)p * (((long long)n + slice - 1) / slice) * (threads / 32) > kFlagWords) slice *= 2;
    cudaError_t ce = cudaMemsetAsync(h->recv_counts, 0, sizeof(unsigned long long) * (size_t)p, stream);
    if (ce != cudaSuccess) return cuda_fail(h, ce, "clearing the send counters");
    RingArgs a = handle_ring_args(h, ptrs, p, n, 0, (long long)n);  // the tree's order ignores the index
    a.layout = TREE;
    a.channels = G;
    a.fwd_channels = G;
    a.tree_scale = scale;
    a.slice = slice;
    // slice groups of the wavefront: slice_block slices per CTA of the
    // least-loaded ranks.  Default (GB300, bf16/int32): 1 when that gives at
    // least 128 groups, 2 below (p = 8 x 2^30 bf16: 9.07 / 9.72 ms for 1 / 2;
    // p = 16 x 4^13 int32: 2.56 / 2.66 ms; p = 64 x 2^24 bf16, 85 groups:
    // 1.81 / 1.55 ms; p = 8 x 6.5 M fp32, 6 groups: 166 / 154 us)
    const long long nsl = ((long long)n + slice - 1) / slice;
    const int block = h->opt.slice_block ? h->opt.slice_block : (nsl >= 128 * g_min ? 1 : 2);
    a.block = (long long)block * g_min;
    int L = 0;
    while ((1 << L) < p) L++;
    int rc = arm_trace(h, a, p, 2 * L, stream);
    if (rc != RAR_OK) return rc;
    ce = launch_tree(a, dtype, op, vec16, threads, stream);
    if (ce != cudaSuccess) {
        if (ce == cudaErrorCooperativeLaunchTooLarge) return fail(h, RAR_EUNSUPPORTED, "tree grid cannot be co-resident");
        return cuda_fail(h, ce, "launching the tree executor");
    }
    note_ring_launch(h, 0, TREE, G, G, p);
    return RAR_OK;
}

// n elements behind each pointer; they are global indices
// [g_first, g_first + n) of rank buffers of n_total elements (g_first = 0,
// n_total = n for a whole-buffer call).
int run(rar_ctx *h, void *const *bufs, int p, size_t n, int dtype, int op, int phase, void *stream_v,
        bool host_mapped = false, long long g_first = 0, long long n_total = -1) {
    if (!h) return fail(nullptr, RAR_EINVAL, "handle is NULL");
    h->err.clear();
    if (n_total < 0) n_total = (long long)n;
    int rc = check_call(h, bufs, p, n, dtype, op, host_mapped);
    if (rc != RAR_OK) return rc;
    cudaStream_t stream = (cudaStream_t)stream_v;
    h->have_last = true;
    h->last_stream = stream;
    h->last_ring = false;
    h->last_phases = 0;
    h->last_p = p;
    h->last_traced = false;
    if (n == 0 || p == 1) return RAR_OK;

    DeviceGuard dg(h->device);
    if (dg.err != cudaSuccess) return cuda_fail(h, dg.err, "selecting the device");
    const bool vec16 = all_aligned16(bufs, p);
    const float inv_p = 1.0f / (float)p;
    const int engine = h->opt.engine;
    // hierarchical 2D schedule: nodes of `group` ranks (1 and p are the flat ring)
    const int group = h->opt.hier_group;
    const bool hier = group > 1 && group < p;
    if (hier && p % group != 0) return fail(h, RAR_EINVAL, "hier_group must divide p");

    if (engine == RAR_ENGINE_FUSED || engine == RAR_ENGINE_FUSED_TREE) {
        FusedArgs a;
        rc = fill_ptrs(h, a.bufs, bufs, p, stream);
        if (rc != RAR_OK) return rc;
        a.n = (long long)n;
        a.first = g_first;
        a.n_total = n_total;
        a.p = p;
        a.phase = phase;
        a.inv_p = inv_p;
        a.status = h->status;
        a.timeout_ns = h->opt.timeout_ns ? h->opt.timeout_ns : kDefaultTimeoutNs;
        a.fault_mode = h->opt.fault_mode;
        a.fault_rank = h->opt.fault_rank;
        const bool tree = engine == RAR_ENGINE_FUSED_TREE && phase != PHASE_AG;
        if (hier) {
            if (engine != RAR_ENGINE_FUSED || phase != PHASE_ALL || h->opt.fused_path == 2)
                return fail(h, RAR_EUNSUPPORTED,
                            "the hierarchical order is offered for the full all-reduce on the fused engine's "
                            "per-thread path and on the ring engine");
            cudaError_t ce = launch_fused_hier(a, dtype, op, group, vec16, 256, stream);
            if (ce != cudaSuccess) return cuda_fail(h, ce, "launching the hierarchical fused kernel");
            return RAR_OK;
        }
        // data path: per-thread 128-bit loads ("registers") or the
        // rank-sequential bulk-copy streaming path.  Auto (measured on GB300):
        // streaming from 256 MB over all ranks and 8 MB per rank, registers
        // below.  Registers / streaming, fraction of the roofline or time:
        // p = 8 fp32, 25 MB per rank 0.90 / 0.88, 48 MB 0.92 / 0.95; p = 16,
        // 16 MB per rank: tied; p = 64 bf16, 4 MB per rank 162 / 195 us,
        // 8 MB 289 / 231 us.  Small buffers are latency-bound, and the
        // streaming path walks the p ranks one bulk copy after another.
        const size_t bytes = n * (size_t)elem_bytes(dtype);
        const bool stream_ok = engine == RAR_ENGINE_FUSED && phase == PHASE_ALL && vec16;
        int path = h->opt.fused_path;
        if (path == 2 && !stream_ok)
            return fail(h, RAR_EUNSUPPORTED,
                        "the streaming path needs engine fused, a full all-reduce and 16-byte aligned rank buffers");
        if (path == 0)
            path = (stream_ok && (size_t)p * bytes >= (size_t)256 << 20 && bytes >= (size_t)8 << 20) ? 2 : 1;
        if (path == 2) {
            // tile per rank: slice_elems (up to 32 KB), else the largest tile
            // up to 28 KB (a multiple of 512 bytes) that cuts the buffer into
            // k rounds of one tile per CTA (one CTA per SM), k >= 4, with the
            // last round nearly full; stages: channels, else 3.  (28 KB
            // against 32 KB tiles on GB300: p = 8 bf16 at 16 GiB 5.10 / 5.20
            // ms, p = 16 int32 at 256 MB per rank 1.27 / 1.31 ms, p = 4 and
            // p = 64 equal; 24 KB fell to 0.93 of the roofline at p = 4.)
            size_t tb;
            if (h->opt.slice_elems) {
                tb = (size_t)h->opt.slice_elems * (size_t)elem_bytes(dtype);
                tb = std::min<size_t>(std::max<size_t>(tb / 512 * 512, 512), 32768);
            } else {
                constexpr size_t kAutoTile = 28672;
                const size_t sms = (size_t)h->sm_count;
                const size_t rounds = std::max<size_t>(4, (bytes + kAutoTile * sms - 1) / (kAutoTile * sms));
                tb = (bytes + rounds * sms - 1) / (rounds * sms);
                tb = std::min<size_t>(std::max<size_t>((tb + 511) / 512 * 512, 512), kAutoTile);
            }
            const int stages = h->opt.channels ? h->opt.channels : 3;
            if (stages < 2 || stages > 8 || (size_t)(stages + 2) * tb > 227 * 1024)
                return fail(h, RAR_EINVAL, "streaming path: stages (channels) must be in [2, 8] and fit in 227 KB");
            cudaError_t ce = launch_fused_stream(a, dtype, op, (int)tb, stages, stream);
            if (ce != cudaSuccess) return cuda_fail(h, ce, "launching the streaming fused kernel");
            return RAR_OK;
        }
        const int threads = 256;  // the fused kernels are compiled for 256 threads
        cudaError_t ce = launch_fused(a, dtype, op, tree, vec16, threads, stream);
        if (ce != cudaSuccess) return cuda_fail(h, ce, "launching the fused kernel");
        return RAR_OK;
    }

    if (engine == RAR_ENGINE_TREE) {
        if (phase != PHASE_ALL || hier || op == RAR_AVG_PREDIV)
            return fail(h, RAR_EUNSUPPORTED, "the tree executor runs the full all-reduce with sum, max or avg");
        RankPtrs ptrs;
        rc = fill_ptrs(h, ptrs, bufs, p, stream);
        if (rc != RAR_OK) return rc;
        // hand-off protocol (rar_options.protocol), as for the ring
        const int proto = h->opt.protocol;
        if (proto != 1) {
            const long long slot_words = tree_ll_slot_words(p, n, dtype);
            if (proto == 2 && slot_words == 0)
                return fail(h, RAR_EUNSUPPORTED, "the buffers are too large for the low-latency mailbox");
            const bool fits = slot_words > 0 && ll_max_coresident_ctas(true, dtype, op) >= p;
            if (proto == 2 || (fits && p >= kLLTreeAutoMinP && n * (size_t)elem_bytes(dtype) <= kLLTreeAutoMaxBytes))
                return launch_tree_ll_phase(h, ptrs, p, n, dtype, op, slot_words, stream);
        }
        return launch_tree_schedule(h, ptrs, p, n, dtype, op, vec16, stream);
    }

    // ---- ring engines
    const bool bidir = engine == RAR_ENGINE_RING_BIDIR;
    if (hier && (bidir || phase != PHASE_ALL))
        return fail(h, RAR_EUNSUPPORTED, "the hierarchical ring runs the full all-reduce on the forward ring only");
    if (h->opt.protocol == 2 && (hier || bidir || phase != PHASE_ALL))
        return fail(h, RAR_EUNSUPPORTED, "the low-latency protocol runs the full all-reduce on the flat forward ring");
    RankPtrs ptrs;
    rc = fill_ptrs(h, ptrs, bufs, p, stream);
    if (rc != RAR_OK) return rc;
    if (!hier) {
        // hand-off protocol of the flat forward ring (rar_options.protocol)
        const int proto = h->opt.protocol;
        if (engine == RAR_ENGINE_RING && phase == PHASE_ALL && proto != 1) {
            const long long slot_words = ll_slot_words(p, n, n_total, dtype);
            if (proto == 2 && slot_words == 0)
                return fail(h, RAR_EUNSUPPORTED, "the buffers are too large for the low-latency mailbox");
            const bool fits = slot_words > 0 && ll_max_coresident_ctas(false, dtype, op) >= p;
            if (proto == 2 || (fits && n * (size_t)elem_bytes(dtype) <= kLLAutoMaxBytes))
                return launch_ring_ll_phase(h, ptrs, p, n, g_first, n_total, dtype, op, slot_words, stream);
        }
        const int first = phase == PHASE_AG ? p - 1 : 0;
        const int steps = phase == PHASE_ALL ? 2 * (p - 1) : p - 1;
        return launch_ring_phase(h, ptrs, p, n, g_first, n_total, dtype, op, vec16, bidir, RING_FLAT, p, first, steps,
                                 0, stream);
    }
    // "Ring All-Reduce, in depth", "Hierarchy": reduce-scatter inside the
    // nodes, all-reduce of each shard across the nodes, all-gather inside the
    // nodes -- three launches in stream order
    const int m = p / group;
    rc = launch_ring_phase(h, ptrs, p, n, g_first, n_total, dtype, op, vec16, false, RING_INTRA, group, 0, group - 1,
                           0, stream);
    if (rc == RAR_OK)
        rc = launch_ring_phase(h, ptrs, p, n, g_first, n_total, dtype, op, vec16, false, RING_INTER, group, 0,
                               2 * (m - 1), 1, stream);
    if (rc == RAR_OK)
        rc = launch_ring_phase(h, ptrs, p, n, g_first, n_total, dtype, op, vec16, false, RING_INTRA, group, group - 1,
                               group - 1, 2, stream);
    return rc;
}

}  // namespace

namespace rar {
// Message returned by rar_last_error(NULL) for entry points without a handle.
void set_handleless_error(const std::string &msg) { g_init_error = msg; }
}  // namespace rar

extern "C" {

int rar_version(void) { return RAR_VERSION; }

int rar_init(rar_handle *out, int device, const rar_options *opt) {
    g_init_error.clear();
    if (!out) return fail(nullptr, RAR_EINVAL, "out is NULL");
    *out = nullptr;
    rar_options o{};
    if (opt) o = *opt;
    if (check_options(nullptr, o) != RAR_OK) return RAR_EINVAL;
    int ndev = 0;
    cudaError_t ce = cudaGetDeviceCount(&ndev);
    if (ce != cudaSuccess) {
        cudaGetLastError();
        return fail(nullptr, RAR_ECUDA, std::string("cudaGetDeviceCount: ") + cudaGetErrorString(ce));
    }
    if (device < 0 || device >= ndev) return fail(nullptr, RAR_EINVAL, "no such device");

    rar_ctx *h = new rar_ctx();
    h->device = device;
    h->opt = o;
    DeviceGuard dg(device);
    if (dg.err != cudaSuccess) {
        delete h;
        return fail(nullptr, RAR_ECUDA, std::string("cudaSetDevice: ") + cudaGetErrorString(dg.err));
    }
    h->sm_count = current_device_sm_count();
    if (h->sm_count < 1) {
        delete h;
        return fail(nullptr, RAR_ECUDA, "querying the device's SM count failed");
    }
    bool ok = cudaMalloc((void **)&h->flags, sizeof(unsigned long long) * kFlagWords) == cudaSuccess &&
              cudaMalloc((void **)&h->recv_counts, sizeof(unsigned long long) * kMaxRingCtas * kRingPhases) == cudaSuccess &&
              cudaMalloc((void **)&h->status, sizeof(RingStatus)) == cudaSuccess &&
              cudaMalloc((void **)&h->abort_word, sizeof(unsigned)) == cudaSuccess &&
              cudaMalloc((void **)&h->epoch_words, 2 * sizeof(unsigned)) == cudaSuccess &&
              cudaMalloc((void **)&h->ptr_table, sizeof(void *) * RAR_MAX_P) == cudaSuccess &&
              cudaMalloc((void **)&h->ll_box, sizeof(unsigned long long) * kLLMailboxWords) == cudaSuccess &&
              (!o.trace || cudaMalloc((void **)&h->trace, sizeof(unsigned long long) * kTraceWords) == cudaSuccess);
    if (ok) {
        ok = cudaMemset(h->flags, 0, sizeof(unsigned long long) * kFlagWords) == cudaSuccess &&
             cudaMemset(h->recv_counts, 0, sizeof(unsigned long long) * kMaxRingCtas * kRingPhases) == cudaSuccess &&
             cudaMemset(h->status, 0, sizeof(RingStatus)) == cudaSuccess &&
             cudaMemset(h->abort_word, 0, sizeof(unsigned)) == cudaSuccess &&
             cudaMemset(h->epoch_words, 0, 2 * sizeof(unsigned)) == cudaSuccess &&
             cudaMemset(h->ll_box, 0, sizeof(unsigned long long) * kLLMailboxWords) == cudaSuccess &&
             cudaDeviceSynchronize() == cudaSuccess;
    }
    if (!ok) {
        cudaGetLastError();
        cudaFree(h->flags);
        cudaFree(h->recv_counts);
        cudaFree(h->status);
        cudaFree(h->abort_word);
        cudaFree(h->epoch_words);
        cudaFree(h->ptr_table);
        cudaFree(h->ll_box);
        cudaFree(h->trace);
        delete h;
        return fail(nullptr, RAR_ENOMEM, "allocating the handle's scratch failed");
    }
    *out = h;
    return RAR_OK;
}

int rar_set_options(rar_handle h, const rar_options *opt) {
    if (!h) return fail(nullptr, RAR_EINVAL, "handle is NULL");
    rar_options o{};
    if (opt) o = *opt;
    int rc = check_options(h, o);
    if (rc != RAR_OK) return rc;
    if (o.trace && !h->trace) {
        DeviceGuard dg(h->device);
        if (dg.err != cudaSuccess) return cuda_fail(h, dg.err, "selecting the device");
        if (cudaMalloc((void **)&h->trace, sizeof(unsigned long long) * kTraceWords) != cudaSuccess) {
            cudaGetLastError();
            h->trace = nullptr;
            return fail(h, RAR_ENOMEM, "allocating the step trace failed");
        }
    }
    h->opt = o;
    return RAR_OK;
}

int rar_trace(rar_handle h, unsigned long long *work_ns, unsigned long long *wait_ns, int p, int max_steps,
              int *steps) {
    if (!h) return fail(nullptr, RAR_EINVAL, "handle is NULL");
    if (!work_ns || !wait_ns || !steps) return fail(h, RAR_EINVAL, "NULL output");
    if (!h->have_last || p != h->last_p) return fail(h, RAR_EINVAL, "p differs from the last call's p");
    if (!h->last_traced)
        return fail(h, RAR_EINVAL, "the last call was not traced (rar_options.trace, ring or tree executor with "
                                   "progress words)");
    const int S = h->last_trace_steps;
    *steps = S;
    if (max_steps < S) return fail(h, RAR_EINVAL, "max_steps is below the last call's step count");
    int rc = rar_status(h);
    if (rc != RAR_OK && rc != RAR_ETIMEOUT) return rc;
    DeviceGuard dg(h->device);
    std::vector<unsigned long long> rec(2 * (size_t)p * (size_t)S);
    cudaError_t ce = cudaMemcpy(rec.data(), h->trace, sizeof(unsigned long long) * rec.size(), cudaMemcpyDeviceToHost);
    if (ce != cudaSuccess) return cuda_fail(h, ce, "reading the step trace");
    for (int r = 0; r < p; r++)
        for (int s = 0; s < S; s++) {
            work_ns[(size_t)r * max_steps + s] = rec[2 * ((size_t)r * S + s)];
            wait_ns[(size_t)r * max_steps + s] = rec[2 * ((size_t)r * S + s) + 1];
        }
    return RAR_OK;
}

int rar_allreduce(rar_handle h, void *const *bufs, int p, size_t n, int dtype, int op, void *stream) {
    return run(h, bufs, p, n, dtype, op, PHASE_ALL, stream);
}

int rar_reduce_scatter(rar_handle h, void *const *bufs, int p, size_t n, int dtype, int op, void *stream) {
    return run(h, bufs, p, n, dtype, op, PHASE_RS, stream);
}

int rar_all_gather(rar_handle h, void *const *bufs, int p, size_t n, int dtype, void *stream) {
    return run(h, bufs, p, n, dtype, RAR_SUM, PHASE_AG, stream);
}

int rar_allreduce_range(rar_handle h, void *const *bufs, int p, size_t n_total, size_t lo, size_t hi, int dtype,
                        int op, void *stream) {
    if (!h) return fail(nullptr, RAR_EINVAL, "handle is NULL");
    if (lo > hi || hi > n_total) return fail(h, RAR_EINVAL, "the range needs lo <= hi <= n_total");
    if (dtype >= RAR_INT32 && dtype <= RAR_FLOAT16 && n_total > (size_t)(1ull << 62) / (size_t)elem_bytes(dtype))
        return fail(h, RAR_EINVAL, "n_total * element size overflows");
    return run(h, bufs, p, hi - lo, dtype, op, PHASE_ALL, stream, false, (long long)lo, (long long)n_total);
}

int rar_allreduce_host(rar_handle h, void *const *host_bufs, void *const *dev_bufs, int p, size_t n, int dtype,
                       int op, void *stream) {
    if (!h) return fail(nullptr, RAR_EINVAL, "handle is NULL");
    h->err.clear();
    if (!host_bufs) return fail(h, RAR_EINVAL, "host_bufs is NULL");
    if (p < 1 || p > RAR_MAX_P) return fail(h, RAR_EINVAL, "p must be in [1, RAR_MAX_P]");
    if (n == 0) return run(h, host_bufs, p, n, dtype, op, PHASE_ALL, stream, true);
    for (int r = 0; r < p; r++)
        if (!host_bufs[r]) return fail(h, RAR_EINVAL, "host buffer " + std::to_string(r) + " is NULL");
    DeviceGuard dg(h->device);
    if (dg.err != cudaSuccess) return cuda_fail(h, dg.err, "selecting the device");
    // Zero copy: page-locked host memory mapped for this device is read and
    // written by the kernel itself over the host link, in one pass.
    std::vector<void *> mapped((size_t)p, nullptr);
    bool zero_copy = true;
    for (int r = 0; r < p && zero_copy; r++) {
        cudaPointerAttributes at{};
        if (cudaPointerGetAttributes(&at, host_bufs[r]) != cudaSuccess) {
            cudaGetLastError();
            zero_copy = false;
        } else if (at.type == cudaMemoryTypeHost && at.devicePointer) {
            mapped[(size_t)r] = at.devicePointer;
        } else {
            zero_copy = false;
        }
    }
    if (zero_copy) return run(h, mapped.data(), p, n, dtype, op, PHASE_ALL, stream, true);

    // Staged: pageable host memory goes through the caller's device buffers.
    if (!dev_bufs) return fail(h, RAR_EINVAL, "host buffers are not page-locked and dev_bufs is NULL");
    int rc = check_call(h, dev_bufs, p, n, dtype, op);
    if (rc != RAR_OK) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t bytes = n * (size_t)elem_bytes(dtype);
    for (int r = 0; r < p; r++) {
        cudaError_t ce = cudaMemcpyAsync(dev_bufs[r], host_bufs[r], bytes, cudaMemcpyHostToDevice, s);
        if (ce != cudaSuccess) return cuda_fail(h, ce, "copying a rank buffer to the device");
    }
    rc = run(h, dev_bufs, p, n, dtype, op, PHASE_ALL, stream);
    if (rc != RAR_OK) return rc;
    for (int r = 0; r < p; r++) {
        cudaError_t ce = cudaMemcpyAsync(host_bufs[r], dev_bufs[r], bytes, cudaMemcpyDeviceToHost, s);
        if (ce != cudaSuccess) return cuda_fail(h, ce, "copying a result back to the host");
    }
    return RAR_OK;
}

int rar_status(rar_handle h) {
    if (!h) return fail(nullptr, RAR_EINVAL, "handle is NULL");
    if (!h->have_last) return RAR_OK;
    DeviceGuard dg(h->device);
    cudaError_t ce = cudaStreamSynchronize(h->last_stream);
    if (ce != cudaSuccess) return cuda_fail(h, ce, "synchronising the last call's stream");
    RingStatus st{};
    ce = cudaMemcpy(&st, h->status, sizeof(st), cudaMemcpyDeviceToHost);
    if (ce != cudaSuccess) return cuda_fail(h, ce, "reading the status word");
    if (st.seq != h->acked_seq) {
        // a wait ran out since the last report (this call, or a replay of a
        // captured one)
        h->acked_seq = st.seq;
        char buf[256];
        if (st.rank >= 0)
            std::snprintf(buf, sizeof(buf),
                          "ring wait timed out: rank %d, step %d, slice %d, waiting on rank %d "
                          "(progress word 0x%llx, wanted 0x%llx)",
                          st.rank, st.step, st.slice, st.waited_on, st.flag_seen, st.flag_wanted);
        else
            std::snprintf(buf, sizeof(buf),
                          "bulk-copy wait timed out: tile %d, step %d, waiting for rank %d's tile (fused streaming "
                          "path)",
                          st.slice, st.step, st.waited_on);
        h->err = buf;
        return st.code ? (int)st.code : RAR_ETIMEOUT;
    }
    return RAR_OK;
}

int rar_send_counts(rar_handle h, unsigned long long *out, int p) {
    if (!h) return fail(nullptr, RAR_EINVAL, "handle is NULL");
    if (!out) return fail(h, RAR_EINVAL, "out is NULL");
    if (!h->have_last || p != h->last_p) return fail(h, RAR_EINVAL, "p differs from the last call's p");
    for (int r = 0; r < p; r++) out[r] = 0;
    int rc = rar_status(h);
    if (rc != RAR_OK && rc != RAR_ETIMEOUT) return rc;
    if (!h->last_ring) return RAR_OK;
    DeviceGuard dg(h->device);
    if (h->last_layout[0] == TREE) {
        // the tree executor counts per sender directly
        std::vector<unsigned long long> counts((size_t)p);
        cudaError_t ce =
            cudaMemcpy(counts.data(), h->recv_counts, sizeof(unsigned long long) * (size_t)p, cudaMemcpyDeviceToHost);
        if (ce != cudaSuccess) return cuda_fail(h, ce, "reading the send counters");
        for (int r = 0; r < p; r++) out[r] = counts[(size_t)r];
        return RAR_OK;
    }
    for (int ph = 0; ph < h->last_phases; ph++) {
        const int G = h->last_channels[ph];
        std::vector<unsigned long long> counts((size_t)p * (size_t)G);
        cudaError_t ce = cudaMemcpy(counts.data(), h->recv_counts + (size_t)ph * kMaxRingCtas,
                                    sizeof(unsigned long long) * counts.size(), cudaMemcpyDeviceToHost);
        if (ce != cudaSuccess) return cuda_fail(h, ce, "reading the send counters");
        // a CTA counts what it received; the sender is its ring neighbour
        const int g = h->last_group;
        for (int r = 0; r < p; r++)
            for (int j = 0; j < G; j++) {
                int sender;
                if (h->last_layout[ph] == RING_INTRA) {
                    sender = r - r % g + (r % g + g - 1) % g;
                } else if (h->last_layout[ph] == RING_INTER) {
                    const int m = p / g;
                    sender = ((r / g + m - 1) % m) * g + r % g;
                } else {
                    sender = j < h->last_fwd_channels[ph] ? (r + p - 1) % p : (r + 1) % p;
                }
                out[sender] += counts[(size_t)r * G + j];
            }
    }
    return RAR_OK;
}

const char *rar_last_error(rar_handle h) {
    if (!h) return g_init_error.c_str();
    return h->err.c_str();
}

int rar_debug_set_epoch(rar_handle h, unsigned epoch) {
    if (!h) return fail(nullptr, RAR_EINVAL, "handle is NULL");
    DeviceGuard dg(h->device);
    cudaError_t ce = cudaDeviceSynchronize();
    if (ce == cudaSuccess) ce = cudaMemcpy(h->epoch_words, &epoch, sizeof(unsigned), cudaMemcpyHostToDevice);
    if (ce != cudaSuccess) return cuda_fail(h, ce, "setting the epoch");
    return RAR_OK;
}

int rar_destroy(rar_handle h) {
    if (!h) return RAR_OK;
    {
        DeviceGuard dg(h->device);
        if (h->have_last) cudaStreamSynchronize(h->last_stream);
        cudaFree(h->flags);
        cudaFree(h->recv_counts);
        cudaFree(h->status);
        cudaFree(h->abort_word);
        cudaFree(h->epoch_words);
        cudaFree(h->ptr_table);
        cudaFree(h->ll_box);
        cudaFree(h->trace);
    }
    delete h;
    return RAR_OK;
}

}  // extern "C"
