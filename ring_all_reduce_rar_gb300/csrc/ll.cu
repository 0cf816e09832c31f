// ll.cu -- the ring and tree schedules with a low-latency hand-off, for
// small buffers.
//
// The ring and tree executors (ring.cu, tree.cu) hand a slice over through a
// progress word: the sender's release store publishes it after its slice
// stores, and the receiver polls the word and only then reads the data.  A
// hop thus costs several round trips to L2 -- about 2 us on GB300 -- and
// for small buffers the hops are the whole cost ("Derive the cost of a ring
// all-reduce": the latency term grows with the number of steps).
//
// Here every 32-bit word of a message travels with a 32-bit tag, the
// launch's epoch, in one aligned 64-bit store, which a reader sees whole or
// not at all.  The receiver polls the message words themselves: no fence, no
// separate flag, no CTA barrier, so a hop costs about one store-to-load trip.
//
// Messages go through a mailbox in the handle's scratch with one slot per
// (receiving rank, message), so a sender never overwrites a message that its
// receiver has not read yet, and a rank only ever waits for the ranks the
// schedule makes it wait for.  Schedules, fold orders and epilogues are the
// executors' ("Ring All-Reduce, in depth", "The schedule"; the tree of
// "Derive the cost of a ring all-reduce"), so results and send counts are
// identical bit for bit.  Rank buffers are read once (own inputs) and written
// once (final values); partial sums live only in the mailbox, so the traffic
// is about twice the in-place executors': this is a latency path.
//
// Word w holds element w (32-bit types) or elements 2w and 2w + 1 (16-bit
// types) of a chunk (ring) or of the buffer (tree).  Thread
// w mod (channels x blockDim) of every rank handles word w at every step, so
// each thread is an independent chain through the schedule.  Every wait is
// bounded; a wait that runs out records the failure in the status word and
// raises the abort word, like the executors'.
#include "flag_sync.cuh"

namespace rar {

constexpr int kLLThreads = 128;
constexpr int kLLBatch = 4;  // words a thread polls at once

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Wait (bounded) until every word of a batch carries this launch's tag:
// words w0 + b * stride for b < nb, already loaded once into v.  All words
// still missing are re-polled together, so a batch costs one trip per poll,
// not one per word.
static __device__ __forceinline__ bool ll_wait_batch(const RingArgs &a, unsigned epoch, const unsigned long long *slot, long long w0,
                                     long long stride, int nb_words, unsigned long long (&v)[kLLBatch], int rank,
                                     int step, int nb) {
    unsigned pending = 0;
#pragma unroll
    for (int b = 0; b < kLLBatch; b++)
        if (b < nb_words && (unsigned)(v[b] >> 32) != epoch) pending |= 1u << b;
    if (!pending) return true;
    const unsigned long long t0 = global_ns();
    const unsigned long long max_iters = a.timeout_ns / 16ull + (1ull << 20);
    for (unsigned long long it = 0;; it++) {
        if (it >= 64) __nanosleep(32);
#pragma unroll
        for (int b = 0; b < kLLBatch; b++)
            if (pending & (1u << b)) v[b] = ld_relaxed_u64(slot + w0 + b * stride);
#pragma unroll
        for (int b = 0; b < kLLBatch; b++)
            if ((pending & (1u << b)) && (unsigned)(v[b] >> 32) == epoch) pending &= ~(1u << b);
        if (!pending) return true;
        if ((it & 15) == 15) {
            if (ld_relaxed_u32(a.abort_word) == epoch) return false;
            if (it >= max_iters || global_ns() - t0 > a.timeout_ns) {
                const int b = __ffs(pending) - 1;
                ring_give_up(a, epoch, rank, step, w0 + b * stride, nb, v[b], (unsigned long long)epoch << 32);
                return false;
            }
        }
    }
}

// Word w of a chunk part [cs, ce) of a rank buffer (16-bit types: two
// elements, the second lane 0 past the end).
template <int DT>
__device__ __forceinline__ uint32_t ll_load_word(const char *buf, long long e0, long long ce) {
    if constexpr (ElemInfo<DT>::bytes == 4) {
        return load_elem<DT>(buf, e0);
    } else {
        const uint32_t lo = load_elem<DT>(buf, e0);
        const uint32_t hi = e0 + 1 < ce ? load_elem<DT>(buf, e0 + 1) : 0u;
        return lo | (hi << 16);
    }
}
template <int DT>
__device__ __forceinline__ void ll_store_word(char *buf, long long e0, long long ce, uint32_t w) {
    if constexpr (ElemInfo<DT>::bytes == 4) {
        store_elem<DT>(buf, e0, w);
    } else {
        store_elem<DT>(buf, e0, w & 0xFFFFu);
        if (e0 + 1 < ce) store_elem<DT>(buf, e0 + 1, w >> 16);
    }
}

template <int DT, int OP>
__global__ void __launch_bounds__(kLLThreads) ring_ll_kernel(const __grid_constant__ RingArgs a) {
    __shared__ unsigned long long s_recv;
    constexpr int EPW = 4 / ElemInfo<DT>::bytes;  // elements per word
    constexpr int hop_op = HopOf<OP>::value;
    constexpr bool prediv = OP == OP_AVG_PREDIV;
    const int p = a.p;
    const int r = blockIdx.x / a.channels;
    const int j = blockIdx.x % a.channels;
    const long long gt = (long long)j * blockDim.x + threadIdx.x;  // this thread's first word
    const long long GT = (long long)a.channels * blockDim.x;         // threads of the rank
    const int nslots = 2 * (p - 1);
    const int nb = r == 0 ? p - 1 : r - 1;  // receives from
    const int to = r + 1 == p ? 0 : r + 1;  // sends to
    char *own = rank_ptr(a.bufs, p, r);
    const unsigned long long *inbox = a.mailbox + (long long)r * nslots * a.slot_words;
    unsigned long long *outbox = a.mailbox + (long long)to * nslots * a.slot_words;
    // chunk c's part inside this launch's index range, in local indices
    const long long base = a.n_total / p, extra = a.n_total % p;
    const long long gl = a.first, gh = a.first + a.n;
    auto part = [&](int c, long long &cs, long long &ce) {
        cs = chunk_start(c, base, extra);
        ce = chunk_start(c + 1, base, extra);
        cs = (cs < gl ? gl : cs > gh ? gh : cs) - gl;
        ce = (ce < gl ? gl : ce > gh ? gh : ce) - gl;
    };
    if (threadIdx.x == 0) s_recv = 0;
    const unsigned epoch = launch_epoch_begin(a);  // (its barrier also orders s_recv)
    const unsigned long long tag = (unsigned long long)epoch << 32;
    unsigned long long received = 0;
    const bool muted = a.fault_mode == RAR_FAULT_MUTE && r == a.fault_rank;
    const bool slow = a.fault_mode == RAR_FAULT_DELAY && r == a.fault_rank;

    if (!muted) {
        // the first reduce-scatter message: this rank's own chunk r, as is
        {
            long long cs, ce;
            part(r, cs, ce);
            const long long words = (ce - cs + EPW - 1) / EPW;
            for (long long w = gt; w < words; w += GT)
                st_relaxed_u64(outbox + w, tag | ll_load_word<DT>(own, cs + w * EPW, ce));
        }
        for (int s = 0; s < nslots; s++) {
            const bool rs = s < p - 1;
            const int k = rs ? s : s - (p - 1);
            const int c = rs ? mod_p(r - 1 - k, p) : mod_p(r - k, p);
            long long cs, ce;
            part(c, cs, ce);
            const long long words = (ce - cs + EPW - 1) / EPW;
            const bool owner_step = rs && k == p - 2;  // this rank completes chunk c
            const bool forward = s + 1 < nslots;
            const unsigned long long *in_s = inbox + (long long)s * a.slot_words;
            unsigned long long *out_s = outbox + (long long)(s + 1) * a.slot_words;
            if (slow) ring_delay(a.fault_delay_ns);
            for (long long w0 = gt; w0 < words; w0 += GT * kLLBatch) {
                const long long left = (words - w0 + GT - 1) / GT;
                const int nbw = left < kLLBatch ? (int)left : kLLBatch;  // words of this batch
                unsigned long long v[kLLBatch];
                uint32_t ownw[kLLBatch];
                // issue the batch's mailbox and own loads together
#pragma unroll
                for (int b = 0; b < kLLBatch; b++) {
                    if (b < nbw) {
                        const long long w = w0 + b * GT;
                        v[b] = ld_relaxed_u64(in_s + w);
                        if (rs) ownw[b] = ll_load_word<DT>(own, cs + w * EPW, ce);
                    }
                }
                if (!ll_wait_batch(a, epoch, in_s, w0, GT, nbw, v, r, s, nb)) goto done;
#pragma unroll
                for (int b = 0; b < kLLBatch; b++) {
                    if (b >= nbw) break;
                    const long long w = w0 + b * GT;
                    uint32_t y = (uint32_t)v[b];
                    const long long e0 = cs + w * EPW;
                    if (rs) {
                        // pre-divided average: an original contribution
                        // enters scaled (the sender's at step 0, the own)
                        if (prediv && k == 0) y = scale_word<DT>(y, a.inv_p);
                        const uint32_t o = prediv ? scale_word<DT>(ownw[b], a.inv_p) : ownw[b];
                        y = hop_word<DT, hop_op>(y, o);
                        if (OP == OP_AVG && owner_step) y = scale_word<DT>(y, a.inv_p);
                    }
                    if (!rs || owner_step) ll_store_word<DT>(own, e0, ce, y);
                    if (forward) st_relaxed_u64(out_s + w, tag | y);
                    received += (unsigned long long)(ce - e0 < EPW ? ce - e0 : EPW);
                }
            }
        }
    }
done:
    atomicAdd(&s_recv, received);
    __syncthreads();
    if (threadIdx.x == 0) a.recv_counts[blockIdx.x] = s_recv;
    launch_epoch_end(a, epoch);
}

// The tree all-reduce (tree.cu's schedule and order) with tagged words.
// L = ceil(log2 p).  Rank r > 0 sends up at level ls = (lowest set bit of r)
// to its parent r - 2^ls, after folding in its children r + 2^l, l < ls
// (the root: all levels); each partial is acc = op(acc, child), the lower
// ranks on the left.  The root scales avg; then the final value travels
// down: each rank waits for its parent's word and passes it on to its
// children from the highest level down.  Mailbox slots per rank: one per
// up level (0 .. L-1) and one for the down message (L).
template <int DT, int OP>
__global__ void __launch_bounds__(kLLThreads) tree_ll_kernel(const __grid_constant__ RingArgs a) {
    __shared__ unsigned long long s_sent;
    constexpr int EPW = 4 / ElemInfo<DT>::bytes;
    constexpr int hop_op = HopOf<OP>::value;
    const int p = a.p;
    const int r = blockIdx.x / a.channels;
    const int j = blockIdx.x % a.channels;
    const long long gt = (long long)j * blockDim.x + threadIdx.x;
    const long long GT = (long long)a.channels * blockDim.x;
    int L = 0;
    while ((1 << L) < p) L++;
    const int ls = r == 0 ? L : __ffs(r) - 1;  // the level r sends up at (the root: none)
    const int parent = r == 0 ? 0 : r - (1 << ls);
    char *own = rank_ptr(a.bufs, p, r);
    const long long n = a.n;
    const long long words = (n + EPW - 1) / EPW;
    auto slot = [&](int rank, int k) { return a.mailbox + ((long long)rank * (L + 1) + k) * a.slot_words; };
    if (threadIdx.x == 0) s_sent = 0;
    const unsigned epoch = launch_epoch_begin(a);  // (its barrier also orders s_sent)
    const unsigned long long tag = (unsigned long long)epoch << 32;
    unsigned long long sent = 0;
    const bool muted = a.fault_mode == RAR_FAULT_MUTE && r == a.fault_rank;
    const bool slow = a.fault_mode == RAR_FAULT_DELAY && r == a.fault_rank;

    if (!muted) {
        for (long long w0 = gt; w0 < words; w0 += GT * kLLBatch) {
            const long long left = (words - w0 + GT - 1) / GT;
            const int nbw = left < kLLBatch ? (int)left : kLLBatch;  // words of this batch
            uint32_t acc[kLLBatch];
            unsigned long long v[kLLBatch];
            long long elems = 0;  // elements in this batch's words
#pragma unroll
            for (int b = 0; b < kLLBatch; b++) {
                if (b < nbw) {
                    const long long e0 = (w0 + b * GT) * EPW;
                    acc[b] = ll_load_word<DT>(own, e0, n);
                    elems += n - e0 < EPW ? n - e0 : EPW;
                }
            }
            // reduce: fold in each child's partial, lowest level first
            for (int l = 0; l < ls; l++) {
                const int child = r + (1 << l);
                if (child >= p) break;  // higher levels' children are farther still
                if (slow) ring_delay(a.fault_delay_ns);
                const unsigned long long *in = slot(r, l);
#pragma unroll
                for (int b = 0; b < kLLBatch; b++)
                    if (b < nbw) v[b] = ld_relaxed_u64(in + w0 + b * GT);
                if (!ll_wait_batch(a, epoch, in, w0, GT, nbw, v, r, l, child)) goto done;
#pragma unroll
                for (int b = 0; b < kLLBatch; b++)
                    if (b < nbw) acc[b] = hop_word<DT, hop_op>(acc[b], (uint32_t)v[b]);
            }
            if (r == 0) {
                if constexpr (OP == OP_AVG) {
#pragma unroll
                    for (int b = 0; b < kLLBatch; b++)
                        if (b < nbw) acc[b] = scale_word<DT>(acc[b], a.inv_p);
                }
            } else {
                // send the partial up, then wait for the final value
                if (slow) ring_delay(a.fault_delay_ns);
                unsigned long long *up = slot(parent, ls);
#pragma unroll
                for (int b = 0; b < kLLBatch; b++)
                    if (b < nbw) st_relaxed_u64(up + w0 + b * GT, tag | acc[b]);
                sent += (unsigned long long)elems;
                const unsigned long long *in = slot(r, L);
#pragma unroll
                for (int b = 0; b < kLLBatch; b++)
                    if (b < nbw) v[b] = ld_relaxed_u64(in + w0 + b * GT);
                if (!ll_wait_batch(a, epoch, in, w0, GT, nbw, v, r, L, parent)) goto done;
#pragma unroll
                for (int b = 0; b < kLLBatch; b++)
                    if (b < nbw) acc[b] = (uint32_t)v[b];
            }
            // broadcast: to the children, highest level first, then keep it
            for (int l = ls - 1; l >= 0; l--) {
                const int child = r + (1 << l);
                if (child >= p) continue;
                unsigned long long *down = slot(child, L);
#pragma unroll
                for (int b = 0; b < kLLBatch; b++)
                    if (b < nbw) st_relaxed_u64(down + w0 + b * GT, tag | acc[b]);
                sent += (unsigned long long)elems;
            }
#pragma unroll
            for (int b = 0; b < kLLBatch; b++)
                if (b < nbw) ll_store_word<DT>(own, (w0 + b * GT) * EPW, n, acc[b]);
        }
    }
done:
    atomicAdd(&s_sent, sent);
    __syncthreads();
    if (threadIdx.x == 0 && s_sent) atomicAdd(&a.recv_counts[r], s_sent);  // counted per sender
    launch_epoch_end(a, epoch);
}

template <int DT, int OP>
static cudaError_t launch_ll_t(const RingArgs &a, cudaStream_t stream) {
    void *args[] = {const_cast<RingArgs *>(&a)};
    return cudaLaunchCooperativeKernel((const void *)ring_ll_kernel<DT, OP>, dim3((unsigned)(a.p * a.channels)),
                                       dim3((unsigned)kLLThreads), args, 0, stream);
}

cudaError_t launch_ring_ll(const RingArgs &a, int dtype, int op, cudaStream_t stream) {
    return dispatch_dtype_op<true>(dtype, op, cudaErrorInvalidValue, [&](auto dt, auto o) {
        return launch_ll_t<decltype(dt)::value, decltype(o)::value>(a, stream);
    });
}

template <int DT, int OP>
static cudaError_t launch_tree_ll_t(const RingArgs &a, cudaStream_t stream) {
    void *args[] = {const_cast<RingArgs *>(&a)};
    return cudaLaunchCooperativeKernel((const void *)tree_ll_kernel<DT, OP>, dim3((unsigned)(a.p * a.channels)),
                                       dim3((unsigned)kLLThreads), args, 0, stream);
}

cudaError_t launch_tree_ll(const RingArgs &a, int dtype, int op, cudaStream_t stream) {
    return dispatch_dtype_op<false>(dtype, op, cudaErrorInvalidValue, [&](auto dt, auto o) {
        return launch_tree_ll_t<decltype(dt)::value, decltype(o)::value>(a, stream);
    });
}

template <typename K>
static int ll_occ_of(K kernel) {
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, kLLThreads, 0) != cudaSuccess) return 0;
    return nb;
}

int ll_max_coresident_ctas(bool tree, int dtype, int op) {
    const int per_sm =
        tree ? dispatch_dtype_op<false>(dtype, op, 0, [&](auto dt, auto o) {
                   return ll_occ_of(tree_ll_kernel<decltype(dt)::value, decltype(o)::value>);
               })
             : dispatch_dtype_op<true>(dtype, op, 0, [&](auto dt, auto o) {
                   return ll_occ_of(ring_ll_kernel<decltype(dt)::value, decltype(o)::value>);
               });
    const int sms = current_device_sm_count();
    return per_sm * sms;
}

int ring_ll_threads() { return kLLThreads; }

}  // namespace rar
