// ring.cu -- engine (b): the schedule-faithful persistent ring executor.
//
// The schedule of "Ring All-Reduce, in depth" ("The schedule"), run as
// written: p rank groups of `channels` CTAs each, all co-resident (one
// cooperative launch).  At reduce-scatter step s rank r receives chunk
// (r - 1 - s) mod p from rank r - 1 and combines it into its own copy; at
// all-gather step s it receives chunk (r - s) mod p and overwrites its copy.
// Data moves through the rank buffers themselves (the receiver reads the
// sender's copy in place), so a reduce-scatter hop costs 3 element moves
// (read incoming, read own, write own) and an all-gather hop 2.  A partial
// that has been handed on is dead until its owner's all-gather step
// overwrites it, so where that overwrite is certain -- a launch of the whole
// flat or cross-node schedule, and the hierarchical reduce-scatter inside
// the nodes, whose all-gather launch follows -- the receiver drops its lines
// from L2 once it has read them: a partial still in L2 never reaches DRAM.
//
// Pipelining ("What real libraries add", "Pipelining"): each chunk is cut
// into slices of `slice` elements; slice k belongs to channel k mod
// channels, and every channel is an independent ring over its slices
// ("Multiple rings, or channels").  A channel takes its slice positions in
// blocks of `block` and runs each block through every step before the next
// (one position at a time by default), so the right neighbour rereads a
// fresh partial while it is still in L2.
//
// Hand-off per warp.  Thread t of a CTA always takes the same vectors and
// elements of a slice (vector v of [vlo, vhi) goes to thread (v - vlo) mod
// blockDim.x, element k of the unaligned ends to thread k mod blockDim.x),
// and every rank cuts a chunk into the same slices, so warp w of the
// receiving CTA reads exactly the part of a slice that warp w of the
// sending CTA wrote at the step before.  Each warp therefore runs its own
// chain: after its part of a slice it publishes its progress with a release
// store of its own 64-bit word
//     (epoch << 32) | (items done in this order),
// and warp w of the right neighbour's CTA of the same channel acquires that
// word before it reads its part at the next step.  No CTA barrier sits
// between slices: a warp that finished its part moves on while the others
// still stream, which keeps the memory pipeline full.  The epoch comes from
// device memory (flag_sync.cuh), so the words need no reset between
// launches and a launch captured in a CUDA graph can be replayed.
//
// In-place safety, per warp's part of a slice of a chunk and so in any
// processing order: rank r - 1 overwrites the part r read at reduce-scatter
// step s only at its all-gather step s, and that write waits on a chain of
// progress words of the same warp index that starts with r's own release
// after the read (the chunk's remaining reduce-scatter hops, its owner, the
// all-gather hops up to r - 1).  The same chain orders that write after r's
// discard of the part's lines, which r issues before its release (PTX
// treats a discard as a write of an indeterminate value).
//
// Bidirectional variant ("Bidirectional rings"): channels
// [fwd_channels, channels) run the mirrored ring (send to r - 1) on the
// second half of the buffer, cut by chunk_bounds(n, 2).
//
// Index ranges: a launch may cover global indices [first, first + n) of
// buffers of n_total elements; chunks are cut from n_total and each hop moves
// the part of its chunk inside the range, so the range gets the whole-buffer
// result and schedule.
//
// Every wait is bounded (globaltimer and an iteration cap).  A CTA that runs
// out records the failure in the status word, raises the abort word and
// returns; the others see the abort word in their next wait and return.
// Nothing traps or spins forever.
#include "flag_sync.cuh"

namespace rar {

constexpr int kRingThreads = 512;
constexpr int kRingUnroll = 4;

// Store of a reduce-scatter partial with the L2 evict-last policy: its reader
// (the right neighbour, one slice step later) should find it in L2, and it
// is dropped there once read, so it never needs to reach DRAM.
__device__ __forceinline__ void st_keep(uint4 *addr, uint4 v) {
    asm volatile("{\n\t.reg .b64 pol;\n\tcreatepolicy.fractional.L2::evict_last.b64 pol, 1.0;\n\t"
                 "st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, pol;\n\t}" ::"l"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// One slice [lo, hi) of one hop: dst = reduce ? op(src, dst) : src, then the
// owner's avg scaling if `scale`; 16-byte vectors where the slice is aligned
// (VEC), single elements at its ends.  `partial`: the result is a
// reduce-scatter partial that the right neighbour reads next (st_keep).
template <int DT, int OP, bool VEC>
__device__ __forceinline__ void ring_slice(const char *src, char *dst, long long lo, long long hi, bool reduce,
                                           bool scale, bool prescale_in, bool prescale_own, bool discard_src,
                                           float inv_p, bool partial = false) {
    constexpr int hop_op = HopOf<OP>::value;
    constexpr bool prediv = OP == OP_AVG_PREDIV;
    constexpr int VE = VEC ? 16 / ElemInfo<DT>::bytes : 1;
    const int T = blockDim.x;
    const long long vlo = (lo + VE - 1) / VE, vhi = hi / VE;
    const bool vec_path = VEC && vlo < vhi;  // otherwise all of it on the element path
    // single elements: [lo, vlo * VE) and [vhi * VE, hi), in one loop.
    // Pre-divided average: a rank's original element enters scaled -- the
    // receiver's own, and the incoming one at reduce-scatter step 0.
    const long long n_head = vec_path ? vlo * VE - lo : hi - lo;
    const long long n_tail = vec_path ? hi - vhi * VE : 0;
    for (long long t = threadIdx.x; t < n_head + n_tail; t += T) {
        const long long i = t < n_head ? lo + t : vhi * VE + (t - n_head);
        uint32_t x = load_elem<DT>(src, i);
        if (reduce) {
            if (prediv && prescale_in) x = scale_word<DT>(x, inv_p);
            uint32_t own = load_elem<DT>(dst, i);
            if (prediv && prescale_own) own = scale_word<DT>(own, inv_p);
            x = hop_word<DT, hop_op>(x, own);
        }
        if (OP == OP_AVG && scale) x = scale_word<DT>(x, inv_p);
        store_elem<DT>(dst, i, x);
    }
    if (!vec_path) return;
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
    // Both reads are the last use of their lines in L2, so both take the
    // evict-first policy (ld.global.cs) and leave L2 to the partials still
    // waiting for their reader: the receiver's own element is an input read
    // once; the incoming one is a partial (dropped below), the sender's
    // original input, or a final value that only this rank reads (the next
    // rank reads this rank's copy).
    for (long long v = vlo + threadIdx.x; v < vhi; v += (long long)T * kRingUnroll) {
        uint4 in[kRingUnroll], own[kRingUnroll];
#pragma unroll
        for (int u = 0; u < kRingUnroll; u++) {
            const long long vv = v + (long long)u * T;
            if (vv < vhi) {
                in[u] = __ldcs(s4 + vv);
                if (reduce) own[u] = __ldcs(d4 + vv);
            }
        }
#pragma unroll
        for (int u = 0; u < kRingUnroll; u++) {
            const long long vv = v + (long long)u * T;
            if (vv < vhi) {
                uint4 x = in[u];
                if (reduce) {
                    if (prediv && prescale_in) x = scale_vec<DT>(x, inv_p);
                    x = hop_vec<DT, hop_op>(x, (prediv && prescale_own) ? scale_vec<DT>(own[u], inv_p) : own[u]);
                }
                if (OP == OP_AVG && scale) x = scale_vec<DT>(x, inv_p);
                if (partial) st_keep(d4 + vv, x); else d4[vv] = x;
            }
        }
    }
    // The incoming partial is dead once read: its owner overwrites it at its
    // all-gather step, and nobody reads it before that.  Drop its lines from
    // L2 so that a partial still there is never written back.
    if (discard_src) discard_read_lines(s4, vlo, vhi, T);
}

// TRACE: record the step trace (RingArgs::trace); a separate instantiation,
// so that the untraced kernel carries none of its code.
template <int DT, int OP, bool VEC, bool TRACE>
__global__ void __launch_bounds__(kRingThreads, 2) ring_executor_kernel(const __grid_constant__ RingArgs a) {
    __shared__ long long s_cs[RAR_MAX_P], s_ce[RAR_MAX_P], s_nsl[RAR_MAX_P];  // per chunk of the ring
    __shared__ unsigned long long s_trace_t0, s_trace_t1;                      // (step trace)
    const int p = a.p;
    const int r = blockIdx.x / a.channels;
    const int j = blockIdx.x % a.channels;
    const bool fwd = j < a.fwd_channels;
    const int jj = fwd ? j : j - a.fwd_channels;
    const int GG = fwd ? a.fwd_channels : a.channels - a.fwd_channels;
    const int W = blockDim.x >> 5;  // warps per CTA: one progress word each
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this rank's ring: its size rp, its position in it, the global rank at
    // a position, and the segment of the buffer the ring works on
    // (segments and chunks in global indices; see the clamp below)
    int rp = p, pos = r, ring_base = 0, ring_step = 1;
    long long seg_lo = fwd ? 0 : a.split;
    long long L = fwd ? a.split : a.n_total - a.split;
    if (a.layout == RING_INTRA) {
        rp = a.group;
        pos = r % a.group;
        ring_base = r - pos;
        seg_lo = 0;
        L = a.n_total;
    } else if (a.layout == RING_INTER) {
        const int local = r % a.group;
        rp = p / a.group;
        pos = r / a.group;
        ring_base = local;
        ring_step = a.group;
        const long long gb = a.n_total / a.group, ge = a.n_total % a.group;
        const int c = local + 1 == a.group ? 0 : local + 1;  // the shard this rank owns after the intra ring
        seg_lo = chunk_start(c, gb, ge);
        L = gb + (c < ge ? 1 : 0);
    }
    const unsigned epoch = launch_epoch_begin(a);
    const int nb_pos = fwd ? mod_p(pos - 1, rp) : mod_p(pos + 1, rp);
    const int nb = ring_base + nb_pos * ring_step;  // the rank this CTA receives from
    // avg scales once, at the final owner; pre-division scales each original
    // contribution once, where it enters the reduction
    const bool scale_here = OP == OP_AVG && a.layout != RING_INTRA;
    const bool prediv_here = OP == OP_AVG_PREDIV && a.layout != RING_INTER;
    // the receiver drops a partial's lines from L2 once read (ring_slice)
    // where the partial is certain to be overwritten before anyone reads it
    // again: a launch of the whole flat or across-node schedule (its own
    // all-gather), and the hierarchical schedule's reduce-scatter inside the
    // nodes (its all-gather launch); not a reduce-scatter call, whose
    // result includes the partials
    const bool discard_partials =
        (a.layout != RING_INTRA && a.first_step == 0 && a.n_steps == 2 * (rp - 1)) ||
        (a.layout == RING_INTRA && a.first_step == 0);
    const char *src = rank_ptr(a.bufs, p, nb);
    char *dst = rank_ptr(a.bufs, p, r);
    unsigned long long *my_flag = a.flags + (long long)blockIdx.x * W + w;
    const unsigned long long *nb_flag = a.flags + ((long long)nb * a.channels + j) * W + w;
    const long long base = L / rp, extra = L % rp;
    unsigned long long received = 0;
    const bool muted = a.fault_mode == RAR_FAULT_MUTE && r == a.fault_rank;
    const bool slow = a.fault_mode == RAR_FAULT_DELAY && r == a.fault_rank;

    // the part of each chunk c of this rank's ring inside this launch's index
    // range, in local indices (empty when the range misses the chunk), and
    // its slice count: computed once per CTA
    const long long gl = a.first, gh = a.first + a.n;
    for (int c = threadIdx.x; c < rp; c += blockDim.x) {
        long long cs = seg_lo + chunk_start(c, base, extra);
        long long ce = seg_lo + chunk_start(c + 1, base, extra);
        cs = (cs < gl ? gl : cs > gh ? gh : cs) - gl;
        ce = (ce < gl ? gl : ce > gh ? gh : ce) - gl;
        s_cs[c] = cs;
        s_ce[c] = ce;
        s_nsl[c] = (ce - cs + a.slice - 1) / a.slice;
    }
    // the chunk this rank receives at a schedule step
    auto chunk_at = [&](int step) {
        const bool rs = step < rp - 1;
        const int s = rs ? step : step - (rp - 1);
        if (fwd) return rs ? mod_p(pos - 1 - s, rp) : mod_p(pos - s, rp);
        return rs ? mod_p(pos + 1 + s, rp) : mod_p(pos + s, rp);
    };
    // Processing order: blocks of K of this channel's slice positions
    // (loc = 0, 1, ...); each block goes through every step before the next
    // block starts.  K >= every step's slice count is the step-by-step order;
    // a small K lets the right neighbour read a partial soon after it was
    // written, while it is still in L2.  Progress words count the items
    // (block, step, k) in this order, so they only grow; the item one step
    // behind (block, step - 1, k) is K items earlier.
    const long long nsl_max = (base + (extra > 0 ? 1 : 0) + a.slice - 1) / a.slice;  // the longest chunk's
    // (at most 2^20 slice positions per channel and step: 32-bit counters)
    const int max_locs = nsl_max > jj ? (int)((nsl_max - jj + GG - 1) / GG) : 0;
    const int K = a.block > 0 && a.block < max_locs ? (int)a.block : (max_locs > 0 ? max_locs : 1);
    const int S = a.n_steps;
    __syncthreads();  // the chunk table

    if (!muted) {
        // items (block, step, k) in processing order: item = (blk * S + t) * K + k
        const unsigned blocks = (unsigned)((max_locs + K - 1) / K);
        const unsigned n_items = blocks * (unsigned)S * (unsigned)K;
        int k = 0, t = 0, loc0 = 0;  // item's k and step, first slice position of its block
        for (unsigned item = 0; item < n_items; item++) {
            // (two equivalent decodes: whichever keeps the vector loop of this
            // element size in registers, as measured with -Xptxas -v)
            if constexpr (ElemInfo<DT>::bytes == 2) {
                k = (int)(item % (unsigned)K);
                const unsigned bt = item / (unsigned)K;
                t = (int)(bt % (unsigned)S);
                loc0 = (int)(bt / (unsigned)S) * K;
            } else if (item > 0 && ++k == K) {  // next (block, step)
                k = 0;
                if (++t == S) {
                    t = 0;
                    loc0 += K;
                }
            }
            const long long sl = jj + (long long)(loc0 + k) * GG;
            const int step = a.first_step + t;
            const int c = chunk_at(step);
            if (sl >= s_nsl[c]) {  // (the same chunk, one step behind, has no such slice either)
                item += (unsigned)(K - 1 - k);  // skip the rest of this (block, step)
                k = K - 1;
                continue;
            }
            const bool rs = step < rp - 1;
            const int s = rs ? step : step - (rp - 1);
            // this warp's part of the slice is ready once the same warp of
            // the left neighbour passed this slice at the step before
            int ok = 1;
            if (lane == 0) {
                if (TRACE && w == 0) s_trace_t0 = global_ns();
                if (t > 0)
                    ok = ring_wait(a, epoch, nb_flag, ((unsigned long long)epoch << 32) | (item - K + 1), r, step, sl,
                                   nb);
                else
                    ok = ld_relaxed_u32(a.abort_word) != epoch;
                if (TRACE && w == 0) s_trace_t1 = global_ns();
                if (ok && slow) ring_delay(a.fault_delay_ns);
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            __syncwarp();  // orders lane 0's acquire before the other lanes' reads
            {
                const long long ce = s_ce[c];
                const long long lo = s_cs[c] + sl * a.slice;
                const long long hi = lo + a.slice < ce ? lo + a.slice : ce;
                // scale: this rank becomes the chunk's owner
                ring_slice<DT, OP, VEC>(src, dst, lo, hi, rs, scale_here && rs && s == rp - 2,
                                        prediv_here && rs && s == 0, prediv_here, discard_partials && rs && s > 0,
                                        a.inv_p, discard_partials && rs && s < rp - 2);
                received += (unsigned long long)(hi - lo);
            }
            // the warp barrier orders the lanes' stores of this part before
            // lane 0's release store of the progress word
            __syncwarp();
            if (lane == 0) {
                st_release_u64(my_flag, ((unsigned long long)epoch << 32) | (item + 1));
                if (TRACE && w == 0) trace_add(a, r, step, s_trace_t0, s_trace_t1);
            }
        }
    }
    if (threadIdx.x == 0) a.recv_counts[blockIdx.x] = received;  // (warp 0 takes part in every slice)
    launch_epoch_end(a, epoch);
}

template <int DT, int OP, bool VEC>
static cudaError_t launch_ring_t(const RingArgs &a, int threads, cudaStream_t stream) {
    void *args[] = {const_cast<RingArgs *>(&a)};
    const void *kernel = a.trace ? (const void *)ring_executor_kernel<DT, OP, VEC, true>
                                 : (const void *)ring_executor_kernel<DT, OP, VEC, false>;
    return cudaLaunchCooperativeKernel(kernel, dim3((unsigned)(a.p * a.channels)), dim3((unsigned)threads), args, 0,
                                       stream);
}

template <int DT, int OP>
static cudaError_t launch_ring_op(const RingArgs &a, bool vec16, int threads, cudaStream_t stream) {
    return vec16 ? launch_ring_t<DT, OP, true>(a, threads, stream) : launch_ring_t<DT, OP, false>(a, threads, stream);
}

cudaError_t launch_ring(const RingArgs &a, int dtype, int op, bool vec16, int threads, cudaStream_t stream) {
    return dispatch_dtype_op<true>(dtype, op, cudaErrorInvalidValue, [&](auto dt, auto o) {
        return launch_ring_op<decltype(dt)::value, decltype(o)::value>(a, vec16, threads, stream);
    });
}

template <typename K>
static int occ_of(K kernel, int threads) {
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, threads, 0) != cudaSuccess) return 0;
    return nb;
}

template <int DT, int OP>
static int ring_occ(bool vec16, int threads) {
    // (the traced instantiation has the same launch bounds)
    return vec16 ? occ_of(ring_executor_kernel<DT, OP, true, false>, threads)
                 : occ_of(ring_executor_kernel<DT, OP, false, false>, threads);
}

int ring_max_coresident_ctas(int dtype, int op, bool vec16, int threads, int *out_per_sm) {
    const int per_sm = dispatch_dtype_op<true>(dtype, op, 0, [&](auto dt, auto o) {
        return ring_occ<decltype(dt)::value, decltype(o)::value>(vec16, threads);
    });
    const int sms = current_device_sm_count();
    if (out_per_sm) *out_per_sm = per_sm;
    return per_sm * sms;
}

}  // namespace rar
