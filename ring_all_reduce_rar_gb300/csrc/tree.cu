// tree.cu -- the tree all-reduce schedule as a persistent executor.
//
// "Derive the cost of a ring all-reduce" compares the ring with a tree
// all-reduce: a reduce up a binary tree and a broadcast down, about
// 2 log2(n) steps instead of 2(n - 1), so fewer step latencies on small
// buffers.  Here p rank groups of `channels` CTAs (one cooperative launch)
// run L = ceil(log2 p) reduce levels and L broadcast levels over the whole
// buffer, slice-pipelined like the ring executor:
//   reduce level l:    rank r with r mod 2^(l+1) == 0 and r + 2^l < p
//                      combines its child's buffer into its own:
//                      own = op(own, child) (lower rank index on the left);
//   broadcast level l: (from l = L - 1 down to 0) rank c with
//                      c mod 2^(l+1) == 2^l copies its parent c - 2^l.
// The reduce folds in exactly the tree order of the fused tree mode (adjacent
// pairs level by level, an odd last rank carried up), so the result equals
// that order bit for bit.  avg is scaled by the root after its last level.
// Element moves: (p - 1) reduce hops of 3 moves and (p - 1) broadcast hops of
// 2, the same 5 (p - 1) n as the ring.
//
// Hand-offs use the progress words of flag_sync.cuh, counting items (slice
// block, step, slice) in processing order; a rank with nothing to do at a
// step still passes its items so that waiters move on.  Every wait is
// bounded.
#include "flag_sync.cuh"

namespace rar {

constexpr int kTreeThreads = 512;

// One slice [lo, hi): reduce: dst = op(dst, src) (+ the root's avg scaling);
// broadcast: dst = src.  discard_src: src is a child's partial that nobody
// reads again before the broadcast overwrites it; its lines are dropped
// from L2 once read, so that it is not written back.
template <int DT, int OP, bool VEC>
__device__ __forceinline__ void tree_slice(const char *src, char *dst, long long lo, long long hi, bool reduce,
                                           bool scale, bool discard_src, float inv_p) {
    constexpr int hop_op = HopOf<OP>::value;
    constexpr int VE = VEC ? 16 / ElemInfo<DT>::bytes : 1;
    const int T = blockDim.x;
    auto one = [&](long long i) {
        uint32_t x = load_elem<DT>(src, i);
        if (reduce) x = hop_word<DT, hop_op>(load_elem<DT>(dst, i), x);
        if (OP == OP_AVG && scale) x = scale_word<DT>(x, inv_p);
        store_elem<DT>(dst, i, x);
    };
    if constexpr (!VEC) {
        for (long long i = lo + threadIdx.x; i < hi; i += T) one(i);
    } else {
        const long long vlo = (lo + VE - 1) / VE, vhi = hi / VE;
        if (vlo >= vhi) {
            for (long long i = lo + threadIdx.x; i < hi; i += T) one(i);
            return;
        }
        for (long long i = lo + threadIdx.x; i < vlo * VE; i += T) one(i);
        for (long long i = vhi * VE + threadIdx.x; i < hi; i += T) one(i);
        const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
        for (long long v = vlo + threadIdx.x; v < vhi; v += T) {
            uint4 x = __ldcg(s4 + v);
            if (reduce) x = hop_vec<DT, hop_op>(__ldcs(d4 + v), x);
            if (OP == OP_AVG && scale) x = scale_vec<DT>(x, inv_p);
            d4[v] = x;
        }
        if (discard_src) discard_read_lines(s4, vlo, vhi, T);
    }
}

template <int DT, int OP, bool VEC>
__global__ void __launch_bounds__(kTreeThreads, 3) tree_executor_kernel(const __grid_constant__ RingArgs a) {
    __shared__ int s_stop;
    const int p = a.p;
    const int r = blockIdx.x / a.channels;
    const int j = blockIdx.x % a.channels;
    int L = 0;
    while ((1 << L) < p) L++;
    char *mine = rank_ptr(a.bufs, p, r);
    unsigned long long *my_flag = a.flags + blockIdx.x;
    const long long nsl = (a.n + a.slice - 1) / a.slice;
    const bool muted = a.fault_mode == RAR_FAULT_MUTE && r == a.fault_rank;
    const bool slow = a.fault_mode == RAR_FAULT_DELAY && r == a.fault_rank;
    // Processing order, as in the ring executor: this channel's slice
    // positions (loc = 0, 1, ...) in blocks of K, each block through every
    // step before the next, so that a reader finds the slice it waited for
    // still in L2; progress words count the items (block, step, k) in this
    // order, and a rank with nothing to do at a step still passes its items.
    const int max_locs = nsl > j ? (int)((nsl - j + a.channels - 1) / a.channels) : 0;
    const int K = a.block > 0 && a.block < max_locs ? (int)a.block : (max_locs > 0 ? max_locs : 1);
    const int S = 2 * L;
    const unsigned n_items = (unsigned)((max_locs + K - 1) / K) * (unsigned)S * (unsigned)K;
    const unsigned epoch = launch_epoch_begin(a);
    if (muted) goto done;

    {
        int k = 0, t = 0, loc0 = 0;  // item's k and step, first slice position of its block
        for (unsigned item = 0; item < n_items; item++) {
            if (item > 0 && ++k == K) {  // next (block, step)
                k = 0;
                if (++t == S) {
                    t = 0;
                    loc0 += K;
                }
            }
            const long long sl = j + (long long)(loc0 + k) * a.channels;
            if (sl >= nsl) {  // past the last slice: the rest of this (block, step) is empty too
                item += (unsigned)(K - 1 - k);
                k = K - 1;
                continue;
            }
            const bool up = t < L;
            const int l = up ? t : 2 * L - 1 - t;
            const int span = 1 << l;
            int peer = -1;  // the rank read at this step
            if (up) {
                if ((r & (2 * span - 1)) == 0 && r + span < p) peer = r + span;
            } else {
                if ((r & (2 * span - 1)) == span) peer = r - span;
            }
            if (peer < 0) {
                // nothing to do at this step: pass the whole (block, step) at once
                item += (unsigned)(K - 1 - k);
                k = K - 1;
                if (threadIdx.x == 0) st_release_u64(my_flag, ((unsigned long long)epoch << 32) | (item + 1));
                continue;
            }
            {
                const char *src = rank_ptr(a.bufs, p, peer);
                const unsigned long long *peer_flag = a.flags + (long long)peer * a.channels + j;
                if (threadIdx.x == 0) {
                    // the peer's data is final for this slice once it passed
                    // the same slice at step t - 1 (K items earlier)
                    bool ok = t > 0 ? ring_wait(a, epoch, peer_flag, ((unsigned long long)epoch << 32) | (item - K + 1),
                                                r, t, sl, peer)
                                    : ld_relaxed_u32(a.abort_word) != epoch;
                    if (ok && slow) ring_delay(a.fault_delay_ns);
                    s_stop = ok ? 0 : 1;
                }
                __syncthreads();
                if (s_stop) goto done;
                const long long lo = sl * a.slice;
                const long long hi = lo + a.slice < a.n ? lo + a.slice : a.n;
                // from level 1 up the child holds a partial sum of its subtree
                tree_slice<DT, OP, VEC>(src, mine, lo, hi, up, up && r == 0 && l == L - 1, up && l > 0, a.inv_p);
                __syncthreads();
                if (threadIdx.x == 0) atomicAdd(&a.recv_counts[peer], (unsigned long long)(hi - lo));  // the peer sent
            }
            // the release store orders the CTA's slice stores (ordered before
            // it by the barrier) ahead of the progress word
            if (threadIdx.x == 0) st_release_u64(my_flag, ((unsigned long long)epoch << 32) | (item + 1));
        }
    }
done:
    launch_epoch_end(a, epoch);
}

template <int DT, int OP, bool VEC>
static cudaError_t launch_tree_t(const RingArgs &a, int threads, cudaStream_t stream) {
    void *args[] = {const_cast<RingArgs *>(&a)};
    return cudaLaunchCooperativeKernel((const void *)tree_executor_kernel<DT, OP, VEC>,
                                       dim3((unsigned)(a.p * a.channels)), dim3((unsigned)threads), args, 0, stream);
}

template <int DT, int OP>
static cudaError_t launch_tree_op(const RingArgs &a, bool vec16, int threads, cudaStream_t stream) {
    return vec16 ? launch_tree_t<DT, OP, true>(a, threads, stream) : launch_tree_t<DT, OP, false>(a, threads, stream);
}

cudaError_t launch_tree(const RingArgs &a, int dtype, int op, bool vec16, int threads, cudaStream_t stream) {
    return dispatch_dtype_op<false>(dtype, op, cudaErrorInvalidValue, [&](auto dt, auto o) {
        return launch_tree_op<decltype(dt)::value, decltype(o)::value>(a, vec16, threads, stream);
    });
}

template <typename K>
static int tree_occ_of(K kernel, int threads) {
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, threads, 0) != cudaSuccess) return 0;
    return nb;
}

template <int DT, int OP>
static int tree_occ(bool vec16, int threads) {
    return vec16 ? tree_occ_of(tree_executor_kernel<DT, OP, true>, threads)
                 : tree_occ_of(tree_executor_kernel<DT, OP, false>, threads);
}

int tree_max_coresident_ctas(int dtype, int op, bool vec16, int threads) {
    const int per_sm = dispatch_dtype_op<false>(dtype, op, 0, [&](auto dt, auto o) {
        return tree_occ<decltype(dt)::value, decltype(o)::value>(vec16, threads);
    });
    const int sms = current_device_sm_count();
    return per_sm * sms;
}

}  // namespace rar
