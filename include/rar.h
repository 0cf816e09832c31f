/*
 * rar.h -- ring all-reduce over p virtual ranks held in one GPU's memory.
 *
 * The operation ("Ring All-Reduce, in depth", section "The schedule"):
 * p ranks, each with an n-element buffer cut into p chunks by chunk_bounds
 * (section "An implementation": the first n mod p chunks are one element
 * longer).  Reduce-scatter runs p - 1 steps; at step s rank r sends chunk
 * (r - s) mod p to rank r + 1, which combines it into its own copy, so that
 * afterwards rank r holds the complete reduction of chunk (r + 1) mod p.
 * All-gather runs p - 1 more steps; at step s rank r sends chunk
 * (r + 1 - s) mod p and the receiver overwrites its copy.  Every rank ends
 * with the elementwise reduction ("AllReduce 与 Ring 通信算法详解", section
 * "AllReduce 语义": sum, average or maximum).
 *
 * Arithmetic follows the ring's hop order exactly: element i of chunk c
 * becomes x_c[i] (+) x_(c+1)[i] (+) ... (+) x_(c+p-1)[i] (indices mod p),
 * each (+) rounded to the buffer's dtype ("Derive the cost of a ring
 * all-reduce", last probe: the reduction runs in the buffer's dtype), so the
 * result is bit-identical to the schedule run on real ranks.  avg is that
 * sum times 1/p (rounded to binary32), applied once by the chunk's owner and
 * rounded once to binary32, then to a 16-bit dtype.  max keeps the running
 * value unless the receiver's element is strictly greater.
 *
 * All p rank buffers live in the GPU's HBM; the library moves no data
 * between GPUs.  Engines (rar_options.engine):
 *   RAR_ENGINE_FUSED       one kernel reads every rank's element once, folds
 *                          in hop order and stores the result to every rank
 *                          (2 p n element moves); on the per-thread path with
 *                          p > 8, a second small launch folds the vectors that
 *                          lie across an unaligned chunk start;
 *   RAR_ENGINE_RING        persistent executor: CTA groups play the ranks and
 *                          run the schedule step by step, slice-pipelined,
 *                          handing slices to the right neighbour through
 *                          acquire/release flags (5 (p - 1) n element moves),
 *                          or, for small buffers, through tagged words in a
 *                          mailbox (rar_options.protocol);
 *   RAR_ENGINE_RING_BIDIR  as RING, with the buffer's second half run by a
 *                          ring in the opposite direction ("Bidirectional
 *                          rings" in "Ring All-Reduce, in depth", section
 *                          "What real libraries add");
 *   RAR_ENGINE_FUSED_TREE  one kernel, tree order over the rank index (adjacent
 *                          pairs level by level); not bit-identical to the
 *                          ring, float sums within 4 p 2^-24 sum|x| of exact.
 *   RAR_ENGINE_TREE        persistent executor of the tree all-reduce schedule
 *                          ("Derive the cost of a ring all-reduce": reduce up a
 *                          binary tree, broadcast down, 2 ceil(log2 p) steps);
 *                          same arithmetic as RAR_ENGINE_FUSED_TREE; full
 *                          all-reduce with sum, max or avg; the same two
 *                          hand-offs as RAR_ENGINE_RING.
 *
 * Conventions for every call:
 *   - Return value: RAR_OK or a rar_status_code; rar_last_error(h) gives a
 *     message.  Argument errors are reported synchronously and launch
 *     nothing.  Device-side errors (a ring wait that timed out) surface
 *     through rar_status().
 *   - Buffers: `bufs` is a host array of p device pointers, each to n
 *     contiguous elements on the handle's device, pairwise non-overlapping.
 *     The caller owns them; the operation is in place.  The array itself is
 *     read during the call only.  All pointers 16-byte aligned select the
 *     128-bit path; otherwise a per-element path runs (same results).
 *   - Streams: work is enqueued on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and the call returns without waiting.  One call
 *     in flight per handle: calls on one stream are ordered; calls on several
 *     streams with one handle must be ordered by the caller.
 *   - Ring and tree engines run one cooperative launch of up to every
 *     co-resident CTA of the device; the GPU runs all CTAs of a launch
 *     together, and every wait inside is bounded (rar_options.timeout_ns),
 *     so a launch that cannot make progress ends with RAR_ETIMEOUT rather
 *     than hanging.
 *   - CUDA graphs: rar_allreduce, rar_reduce_scatter and rar_all_gather may
 *     be recorded with stream capture and replayed any number of times; the
 *     ring and tree executors keep their epoch in device memory, so every
 *     replay is a fresh launch.  Create the handle outside the capture.
 *   - Trivial calls: p == 1 or n == 0 return RAR_OK and launch nothing (the
 *     torch ring in "An implementation" returns its tensor when p == 1);
 *     with n == 0 the rank pointers may be NULL.
 */
#ifndef RAR_H
#define RAR_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RAR_VERSION 1
#define RAR_MAX_P 1024

typedef struct rar_ctx *rar_handle;

typedef enum { RAR_INT32 = 0, RAR_FLOAT32 = 1, RAR_BFLOAT16 = 2, RAR_FLOAT16 = 3 } rar_dtype;
typedef enum {
    RAR_SUM = 0,
    RAR_MAX = 1,
    RAR_AVG = 2,        /* ring-order sum, then x 1/p at the chunk's owner */
    RAR_AVG_PREDIV = 3  /* every rank's element x 1/p (rounded to the dtype) as it
                           enters the ring, then the ring-order sum: a 16-bit sum over
                           many ranks cannot overflow ("Ring All-Reduce, in depth",
                           "Failure modes": pre-divide) */
} rar_op;
typedef enum {
    RAR_ENGINE_FUSED = 0,
    RAR_ENGINE_RING = 1,
    RAR_ENGINE_RING_BIDIR = 2,
    RAR_ENGINE_FUSED_TREE = 3,
    RAR_ENGINE_TREE = 4
} rar_engine;

typedef enum {
    RAR_OK = 0,
    RAR_EINVAL = 1,        /* bad argument (null, p out of range, overlap, wrong device) */
    RAR_EUNSUPPORTED = 2,  /* valid but not offered (avg on int32, grid not co-resident) */
    RAR_ENOMEM = 3,        /* scratch allocation failed in rar_init */
    RAR_ECUDA = 4,         /* a CUDA runtime call failed; message in rar_last_error */
    RAR_ETIMEOUT = 5,      /* a bounded wait ran past timeout_ns (from rar_status) */
    RAR_EABORTED = 6       /* the call was abandoned after another CTA timed out */
} rar_status_code;

typedef enum { RAR_FAULT_NONE = 0, RAR_FAULT_MUTE = 1, RAR_FAULT_DELAY = 2 } rar_fault_mode;

/* Options; an all-zero struct means "defaults". */
typedef struct {
    int engine;                    /* rar_engine */
    int channels;                  /* ring engines: CTAs per rank, 0 = chosen from the SM count */
    int slice_elems;               /* ring engines: elements per pipelined slice, 0 = auto */
    int block_threads;             /* threads per CTA (multiple of 32, <= 1024), 0 = auto */
    unsigned long long timeout_ns; /* bound on every wait of the ring and tree engines and
                                      of the fused engine's streaming path (a bulk load
                                      that does not arrive); 0 = 2 s; nonzero values
                                      below 1 ms (1000000) are refused with RAR_EINVAL.
                                      A wait that runs out ends the call with
                                      RAR_ETIMEOUT (rar_status); the streaming path
                                      still waits for every bulk load it issued before
                                      its CTAs finish, whatever this bound */
    int skip_pointer_check;        /* nonzero: skip the per-call device-pointer query */
    int fault_mode;                /* rar_fault_mode (tests): ring and tree engines; and
                                      RAR_FAULT_MUTE on the fused streaming path, where
                                      the loads of rank fault_rank are never issued, as
                                      if that rank had died */
    int fault_rank;                /* rank the fault applies to */
    unsigned fault_delay_ns;       /* RAR_FAULT_DELAY: pause before each slice */
    int fused_path;                /* RAR_ENGINE_FUSED data path, same results on both:
                                      0 auto; 1 per-thread 128-bit loads of all p
                                      ranks and streaming stores; 2 rank-sequential
                                      streaming: bulk copies (TMA) of one rank tile
                                      at a time in hop order into shared memory,
                                      running values in registers, bulk stores of
                                      the result (full all-reduce, 16-byte aligned
                                      ranks; slice_elems = tile elements per rank,
                                      channels = pipeline stages, 0 = auto) */
    int hier_group;                /* 0 (or 1 or p): the flat ring.  g with 1 < g < p, g | p:
                                      the hierarchical 2D schedule over p / g nodes of g
                                      consecutive ranks ("Ring All-Reduce, in depth",
                                      "Hierarchy"): reduce-scatter inside each node,
                                      all-reduce of each 1/g shard across the nodes, all-gather
                                      inside each node.  Full all-reduce only; RAR_ENGINE_RING
                                      runs it as three ring launches, RAR_ENGINE_FUSED folds in
                                      its order on the per-thread path */
    int protocol;                  /* RAR_ENGINE_RING and RAR_ENGINE_TREE hand-off, same
                                      results on both:
                                      0 auto (low latency for small buffers);
                                      1 progress words: a slice is published by a
                                      release store, and the receiver reads it in place
                                      in the sender's buffer;
                                      2 low latency: every 32-bit word travels with a
                                      tag in one 64-bit store through a mailbox in the
                                      handle's scratch.  Ring: full all-reduce on the flat
                                      ring, while p * 2 (p - 1) chunk-sized slots fit in
                                      RAR_LL_MAILBOX_BYTES; tree: while
                                      p * (ceil(log2 p) + 1) buffer-sized slots fit */
    int slice_block;               /* ring and tree executors with progress words.  Ring:
                                      each channel takes its slices in blocks of this many and
                                      runs a block through every step before the next, so that
                                      the reader finds a fresh slice still in L2 (0 = auto: 1;
                                      a value at least the slices per step gives the
                                      step-by-step order).  Tree: slices per CTA of the
                                      least-loaded ranks in one group of the wavefront (0 =
                                      auto: 1 or 2).  Results do not depend on it. */
    int trace;                     /* nonzero: the ring executor (flat and bidirectional)
                                      and the tree executor, with progress words, record per
                                      rank and schedule step the time spent waiting for the
                                      neighbour and the time spent on its slices (rar_trace).
                                      rar_init / rar_set_options allocate the record, 2 x
                                      RAR_MAX_P x RAR_TRACE_MAX_STEPS words (32 MB) */
} rar_options;

/* Schedule steps a trace holds per rank (2 (RAR_MAX_P - 1)). */
#define RAR_TRACE_MAX_STEPS 2046

/* Bytes of the low-latency mailbox each handle allocates in rar_init. */
#define RAR_LL_MAILBOX_BYTES (64u << 20)

/* Create a handle on `device`; allocates the ring and tree engines' progress
 * words, counters and status word there (about 33 MB) and the low-latency mailbox
 * (RAR_LL_MAILBOX_BYTES).  opt may be NULL.
 * Errors: RAR_EINVAL (out NULL, bad device or option), RAR_ENOMEM,
 * RAR_ECUDA. */
int rar_init(rar_handle *out, int device, const rar_options *opt);

/* Replace the handle's options between calls (same validation as rar_init). */
int rar_set_options(rar_handle h, const rar_options *opt);

/* In-place all-reduce of p rank buffers of n elements (the whole schedule:
 * reduce-scatter then all-gather).
 * Errors: RAR_EINVAL (null handle/array/pointer, p < 1 or p > RAR_MAX_P,
 * unknown dtype or op, n * element size overflows, overlapping buffers,
 * pointers not device memory of the handle's device), RAR_EUNSUPPORTED
 * (avg or avg_prediv on int32; ring engine grid cannot be co-resident), RAR_ECUDA. */
int rar_allreduce(rar_handle h, void *const *bufs, int p, size_t n, int dtype, int op,
                  void *stream);

/* The reduce-scatter half alone ("Ring All-Reduce, in depth", section
 * "Trade-offs": the two halves are also used separately).  Afterwards rank r
 * holds the complete reduction of chunk (r + 1) mod p in that chunk's place
 * in its buffer (avg already scaled); its other chunks hold partial values
 * (fused engines: unchanged inputs; ring engines: the schedule's partials).
 * RAR_ENGINE_RING_BIDIR: the first half's chunk (r + 1) and the second
 * half's chunk (r - 1), both by chunk_bounds of that half.
 * Same arguments and errors as rar_allreduce. */
int rar_reduce_scatter(rar_handle h, void *const *bufs, int p, size_t n, int dtype, int op,
                       void *stream);

/* The all-gather half alone: rank r's chunk (r + 1) mod p is copied to every
 * other rank (RAR_ENGINE_RING_BIDIR: by the same split as in
 * rar_reduce_scatter).  After rar_reduce_scatter this completes the
 * all-reduce.  No arithmetic; dtype only sets the element size.
 * Same arguments and errors as rar_allreduce (op is not taken). */
int rar_all_gather(rar_handle h, void *const *bufs, int p, size_t n, int dtype, void *stream);

/* In-place all-reduce of the index range [lo, hi) of p rank buffers of
 * n_total elements each: bufs[r] points at element lo of rank r's buffer
 * (hi - lo elements behind it, owned by the caller).  Chunks are cut from
 * n_total by chunk_bounds, and every element is reduced in its chunk's order,
 * so the range ends up exactly as rar_allreduce over the whole buffers leaves
 * it, bit for bit, with the handle's engine.  The pages have no such call;
 * it rests on each result element depending only on the inputs at its index
 * and on its chunk: disjoint ranges can be reduced by separate calls (on
 * separate streams, or on the GPUs that hold them) without any exchange.
 * Send counts (rar_send_counts) are the elements moved for this range; over
 * ranges that cover [0, n_total) they add up to the whole call's counts.
 * Errors: as rar_allreduce; RAR_EINVAL unless lo <= hi <= n_total.
 * lo == hi is a no-op. */
int rar_allreduce_range(rar_handle h, void *const *bufs, int p, size_t n_total, size_t lo, size_t hi, int dtype,
                        int op, void *stream);

/* All-reduce of host-resident rank buffers, with the handle's engine.
 *   host_bufs  host array of p host pointers, n elements each; the result
 *              replaces the inputs
 *   dev_bufs   host array of p device pointers (n elements each, owned by
 *              the caller), or NULL; used only for pageable host memory
 * If every host buffer is page-locked and mapped for the handle's device
 * (cudaHostAlloc, or torch's pin_memory), the kernel reads the inputs and
 * writes the results over the host link itself, in one pass, and dev_bufs is
 * not touched.  Otherwise the buffers are staged, in stream order: each host
 * buffer is copied into dev_bufs[r], those are all-reduced (as
 * rar_allreduce), and the results are copied back (these copies wait for the
 * host when the memory is pageable).  The library allocates nothing.
 * Errors: as rar_allreduce; RAR_EINVAL if host_bufs or an entry is NULL, or
 * the memory is pageable and dev_bufs is NULL. */
int rar_allreduce_host(rar_handle h, void *const *host_bufs, void *const *dev_bufs, int p, size_t n, int dtype,
                       int op, void *stream);

/* All-reduce for callers that may not allocate device memory: callers whose
 * device memory belongs to another allocator (a framework's caching
 * allocator, a pre-planned arena with a fixed budget), and callers that
 * cannot pay for cudaMalloc/cudaFree at call time (both can block; cudaFree
 * synchronises the device).  The source pages have no counterpart: this is
 * the ring executor (RAR_ENGINE_RING with progress words) without a handle,
 * with its scratch -- progress words, receive counters, the status and the
 * abort word -- in one fixed-size device array inside the library (about
 * 80 KB, resident on every GPU that loads the library until exit).  Its
 * tuning is fixed: 256 threads per CTA, every co-resident CTA up to 1024 in
 * all, 128 KB slices (the handle's ring uses 512 threads and slices of up to
 * 128 KB); the results are the same bits as rar_allreduce's with
 * RAR_ENGINE_RING.
 * Arguments and results are as rar_allreduce's, on the current device.
 * Limits: p <= 64 and p * channels <= 1024 CTAs; larger p returns
 * RAR_EINVAL with a message from rar_last_error(NULL).
 * The first call on a device, with that device current, sets the array up
 * (clears it once, synchronously; so does the first call after
 * cudaDeviceReset, which reloads the array); make that first call before
 * any stream capture.  Every call uses the same array: calls that overlap
 * on the GPU (two streams, two threads) race and must be ordered by the
 * caller.
 * A ring wait that runs out (2 s) ends the kernel early and leaves the
 * buffers partly reduced; without a handle this entry point cannot report
 * it, so callers who need that status use rar_allreduce.
 * Errors: as rar_allreduce, reported through the return value and
 * rar_last_error(NULL). */
int rar_allreduce_noalloc(void *const *bufs, int p, size_t n, int dtype, int op, void *stream);

/* Synchronise the stream of the last call and return the device-side status:
 * RAR_OK, or RAR_ETIMEOUT if a bounded wait ran out since the previous report
 * (in the last call, or in a replay of a captured one); rar_last_error names
 * the rank, step and slice.  Each failure is reported once.  A timed-out call
 * leaves the buffers partly updated; the handle stays usable. */
int rar_status(rar_handle h);

/* Per-rank count of elements each rank sent in the last ring-engine call
 * (the fused engines send nothing; counts are 0).  out has p entries; p must
 * equal the last call's p.  Synchronises like rar_status.  For the full
 * all-reduce, sends_r = 2 n - |C_(r+1)| - |C_(r+2)| ("Ring All-Reduce, in
 * depth", "The schedule": 2 (p - 1)/p x n when p divides n). */
int rar_send_counts(rar_handle h, unsigned long long *out, int p);

/* Message for the handle's last error (never NULL; "" when none).  Valid
 * until the next call on the handle.  h may be NULL for rar_init errors. */
const char *rar_last_error(rar_handle h);

/* Synchronise the device, free the scratch and the handle.  NULL is a no-op. */
int rar_destroy(rar_handle h);

/* RAR_VERSION of the loaded library. */
int rar_version(void);

/* Per-rank step times of the last call, when rar_options.trace was set and
 * the call ran the ring executor (flat or bidirectional) or the tree
 * executor with progress words ("Ring All-Reduce, in depth", "Failure
 * modes": a straggler shows as the rank whose steps take longest, and its
 * right neighbour as the one that waits longest).  For rank r and schedule
 * step s (global step index: 0 .. 2 (p - 1) - 1 for the ring, 0 .. 2L - 1
 * for the tree), work_ns[r * max_steps + s] is the time the rank's CTAs spent on
 * their slices of that step (from the end of the wait to the release of the
 * slice, summed over CTAs; an injected delay counts as work), and
 * wait_ns[r * max_steps + s] the time they spent waiting for the neighbour's
 * progress word; both from the first warp of each CTA, in nanoseconds of
 * %globaltimer.  *steps receives the step count; the arrays hold
 * p * max_steps entries.  Synchronises like rar_status.
 * Errors: RAR_EINVAL (null argument, p differs from the last call's,
 * max_steps too small, or the last call was not traced). */
int rar_trace(rar_handle h, unsigned long long *work_ns, unsigned long long *wait_ns, int p, int max_steps,
              int *steps);

/* Test hook: set the handle's launch epoch counter (device memory; the next
 * ring-engine or tree launch runs with epoch + 1).  The ring engines tag
 * progress words and mailbox words with a 32-bit epoch; the launch that runs
 * with epoch 0xFFFFFFFF clears them all and restarts the count, so no stale
 * tag can match.  This call lets a test reach that launch without 2^32
 * calls.  Synchronises the device; no call may be in flight.
 * Errors: RAR_EINVAL (null handle), RAR_ECUDA. */
int rar_debug_set_epoch(rar_handle h, unsigned epoch);

#ifdef __cplusplus
}
#endif
#endif
