// rar_internal.h -- launch arguments shared by the host runtime and the
// kernels of the ring all-reduce library.  Not a public header.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "rar.h"

namespace rar {

// SM count of the current device (cached per device ordinal; 0 if the
// query fails, which callers treat as "nothing can be co-resident").
inline int current_device_sm_count() {
    constexpr int kMaxDevices = 64;
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        int v = 0;
        return cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess ? v : 0;
    }
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        cache[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

// Warps per CTA of the ring executor at most (512 threads): each warp has a
// progress word of its own.
constexpr int kRingMaxWarps = 16;

// Rank pointers travel in the kernel parameters for p <= kInlineP; larger p
// read a device-side table kept in the handle's scratch.
constexpr int kInlineP = 64;

enum Dtype { DT_I32 = RAR_INT32, DT_F32 = RAR_FLOAT32, DT_BF16 = RAR_BFLOAT16, DT_F16 = RAR_FLOAT16 };
enum Op { OP_SUM = RAR_SUM, OP_MAX = RAR_MAX, OP_AVG = RAR_AVG, OP_AVG_PREDIV = RAR_AVG_PREDIV };

// Which part of the schedule a launch runs.
enum Phase { PHASE_ALL = 0, PHASE_RS = 1, PHASE_AG = 2 };

inline int elem_bytes(int dt) { return (dt == DT_BF16 || dt == DT_F16) ? 2 : 4; }

struct RankPtrs {
    void *inl[kInlineP];
    void *const *table;  // device array of p pointers when p > kInlineP
};

// Device-side status: a CTA whose bounded wait runs out fills in the
// details and bumps `seq`; the host reports a failure when `seq` moved.
struct RingStatus {
    unsigned epoch;   // ring/tree: the epoch of the launch that failed (first reporter of a launch)
    unsigned seq;     // number of give-ups so far (never reset)
    unsigned code;    // RAR_ETIMEOUT
    int rank;         // rank whose wait ran out
    int step;         // global schedule step it was waiting to start
    int slice;        // slice index within the chunk
    int waited_on;    // neighbour rank it was waiting for
    unsigned long long flag_seen;
    unsigned long long flag_wanted;
};

// Index ranges: the rank pointers may address element `first` of buffers
// that hold `n_total` elements each; a launch then covers global indices
// [first, first + n), and the chunks are cut from n_total, so the result is
// that of the whole-buffer call on those indices.  first = 0 and
// n_total = n for a whole-buffer call.

// Fused engines: one launch covers [0, n) of every rank pointer.
struct FusedArgs {
    RankPtrs bufs;
    long long n;
    long long first;
    long long n_total;
    int p;
    int phase;     // Phase
    float inv_p;   // binary32 nearest to 1/p
    // streaming path only: where a bounded wait that ran out is recorded,
    // the bound, and the host-requested fault (RAR_FAULT_MUTE: the loads of
    // rank fault_rank are never issued)
    RingStatus *status;
    unsigned long long timeout_ns;
    int fault_mode;
    int fault_rank;
};

// Which rings a ring launch runs (the hierarchical schedule uses 1 and 2).
enum RingLayout {
    RING_FLAT = 0,   // one ring over all p ranks
    RING_INTRA = 1,  // a ring inside each node of `group` consecutive ranks
    RING_INTER = 2,  // a ring across the nodes per local rank, on that rank's shard
    TREE = 3         // the tree executor (tree.cu); its counters are per sender
};

// Ring engines: persistent cooperative launch of p * channels CTAs.
struct RingArgs {
    RankPtrs bufs;
    long long n;         // elements behind each rank pointer
    long long first;     // global index of element 0 (see FusedArgs)
    long long n_total;
    int p;
    int layout;          // RingLayout
    int group;           // ranks per node (RING_INTRA / RING_INTER)
    int channels;        // CTAs per rank
    int fwd_channels;    // bidirectional: channels [0, fwd_channels) run the
                         // forward ring on the first half, the rest the
                         // mirrored ring on the second half; == channels if
                         // not bidirectional
    long long split;     // bidirectional: first global index of the second half (n_total otherwise)
    long long slice;     // elements per slice
    long long block;     // slice positions per block of the processing order (0: all)
    int tree_scale;      // tree executor: rank r runs tree_scale * w_r CTAs (w_r: the
                         // steps it takes part in); 0: `channels` CTAs per rank
    int first_step;      // global schedule steps [first_step, first_step + n_steps)
    int n_steps;
    float inv_p;
    // Device-side epochs: a launch uses *epoch_word + 1; the last CTA to
    // finish (counted in *finish_count) stores it back, so every launch --
    // also every replay of a captured one -- gets a fresh epoch.
    unsigned *epoch_word;
    unsigned *finish_count;
    int flag_capacity;                // progress words to clear when the epoch wraps
    unsigned long long *flags;        // progress words: [p * channels * warps per CTA] for the
                                      // ring executor, [p * slices * warps per CTA] for the tree executor
    // The low-latency mailbox (ll.cu): words tagged with the
    // launch's epoch, so any launch that wraps the epoch clears all of them;
    // slot_words = words per (rank, step) slot.  NULL / 0 where unused.
    unsigned long long *mailbox;
    long long mailbox_words;
    long long slot_words;
    unsigned long long *recv_counts;  // [p * channels] elements received by each CTA
    RingStatus *status;
    unsigned *abort_word;             // == the launch's epoch once any CTA gave up
    unsigned long long timeout_ns;
    int fault_mode;
    int fault_rank;
    unsigned fault_delay_ns;
    // per (rank, global step): {work ns, wait ns} summed over the rank's
    // CTAs (first warp of each), trace_steps steps per rank; NULL: off
    unsigned long long *trace;
    int trace_steps;
};

// Launchers (return cudaError_t of the launch).  `vec16` selects the 128-bit
// path (all rank pointers 16-byte aligned).
cudaError_t launch_fused(const FusedArgs &a, int dtype, int op, bool tree, bool vec16,
                         int threads, cudaStream_t stream);
cudaError_t launch_ring(const RingArgs &a, int dtype, int op, bool vec16, int threads,
                        cudaStream_t stream);
// Rank-sequential streaming fused path (PHASE_ALL, 16-byte aligned ranks);
// tile_bytes per rank in [512, 32768], a multiple of 512; n_stages in [2, 8];
// (n_stages + 2) tiles must fit in 227 KB of shared memory.
cudaError_t launch_fused_stream(const FusedArgs &a, int dtype, int op, int tile_bytes, int n_stages,
                                cudaStream_t stream);
// Hierarchical order (nodes of g ranks, 1 < g < p, g | p), full all-reduce.
cudaError_t launch_fused_hier(const FusedArgs &a, int dtype, int op, int g, bool vec16, int threads,
                              cudaStream_t stream);
// Tree executor (tree.cu): full all-reduce; a.recv_counts holds p per-rank
// send counters, zeroed by the caller before the launch.
cudaError_t launch_tree(const RingArgs &a, int dtype, int op, bool vec16, int threads, cudaStream_t stream);
int tree_max_coresident_ctas(int dtype, int op, bool vec16, int threads);
// CTAs of a tree launch: tree_scale * 2 (p - 1), or p * channels when
// tree_scale is 0.
long long tree_grid_ctas(int p, int tree_scale, int channels);
// Largest co-resident grid for the ring kernel of this dtype/op (per device).
int ring_max_coresident_ctas(int dtype, int op, bool vec16, int threads, int *out_per_sm);
// Low-latency hand-offs (ll.cu), p * channels CTAs of ring_ll_threads()
// threads.  Ring: full all-reduce on the flat forward ring; a.mailbox holds
// p * 2 (p - 1) slots of a.slot_words words (at least the longest chunk
// part, in 32-bit words).  Tree: full all-reduce with sum, max or avg;
// p * (ceil(log2 p) + 1) slots of at least the buffer's words; a.recv_counts
// holds p per-sender counters, zeroed by the caller.
cudaError_t launch_ring_ll(const RingArgs &a, int dtype, int op, cudaStream_t stream);
cudaError_t launch_tree_ll(const RingArgs &a, int dtype, int op, cudaStream_t stream);
int ll_max_coresident_ctas(bool tree, int dtype, int op);
int ring_ll_threads();

}  // namespace rar
