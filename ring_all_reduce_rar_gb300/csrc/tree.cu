// tree.cu -- the tree all-reduce schedule as a persistent executor.
//
// "Derive the cost of a ring all-reduce" compares the ring with a tree
// all-reduce: a reduce up a binary tree and a broadcast down, about
// 2 log2(n) steps instead of 2(n - 1), so fewer step latencies on small
// buffers.  Here groups of CTAs (one cooperative launch) play the p ranks and
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
// Work per rank.  Rank r takes part in w_r of the 2L steps: the root in its L
// reduce levels; any other rank in the reduce levels l < ctz(r) where it has
// a child (r + 2^l < p) and in one broadcast level, ctz(r).  The w_r add up
// to 2 (p - 1), but they range from 1 (odd ranks) to L, so equal CTA groups
// would leave most CTAs idle at every step.  Rank r gets tree_scale * w_r
// CTAs instead (or `channels` CTAs each when 2 (p - 1) CTAs do not fit), so
// every CTA carries about the same work: CTA j of rank r takes slices j,
// j + G_r, ... and runs only the rank's active steps.
//
// Hand-offs: one progress word per (rank, slice, warp), holding
// (epoch << 32) | (active steps the rank has completed on that slice).  As
// in the ring executor, every rank cuts the same slices and thread t always
// takes the same vectors and elements of a slice, so warp w only ever reads
// what warp w of the peer wrote, and waits for that warp alone: no CTA
// barrier sits between slices.  A
// parent at reduce level l needs its child c's subtree partial, complete
// once c has done all its reduce levels (w_c - 1 steps); a child at its
// broadcast level needs its parent's final value, complete once the parent
// has done all its w_P steps.  Both conditions also order every overwrite
// after the reads of the old value: a rank's buffer is overwritten by its
// broadcast only after its parent finished, which includes reading it.
// Every wait is bounded.
//
// L2 policies: a reduce level reads the child's data and its own for the
// last time (the child's partial is dropped from L2 once read, its own is
// overwritten), so both reads take the evict-first policy, and a partial
// that the next level reads is stored with the evict-last policy.  A
// broadcast level l >= 1 reads a parent that its other children read again
// at lower levels, so those reads keep the normal policy; level 0 is the
// last read.
#include "flag_sync.cuh"
#include "tree_plan.h"

namespace rar {

constexpr int kTreeThreads = 512;

// Store with the L2 evict-last policy (a partial that the next level reads).
__device__ __forceinline__ void tree_st_keep(uint4 *addr, uint4 v) {
    asm volatile("{\n\t.reg .b64 pol;\n\tcreatepolicy.fractional.L2::evict_last.b64 pol, 1.0;\n\t"
                 "st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, pol;\n\t}" ::"l"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// One slice [lo, hi): reduce: dst = op(dst, src) (+ the root's avg scaling);
// broadcast: dst = src.  discard_src: src is a child's partial that nobody
// reads again before the broadcast overwrites it; its lines are dropped
// from L2 once read, so that it is not written back.
template <int DT, int OP, bool VEC>
__device__ __forceinline__ void tree_slice(const char *src, char *dst, long long lo, long long hi, bool reduce,
                                           bool scale, bool discard_src, bool last_read, bool keep, float inv_p) {
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
            uint4 x = last_read ? __ldcs(s4 + v) : __ldcg(s4 + v);
            if (reduce) x = hop_vec<DT, hop_op>(__ldcs(d4 + v), x);
            if (OP == OP_AVG && scale) x = scale_vec<DT>(x, inv_p);
            if (keep) tree_st_keep(d4 + v, x); else d4[v] = x;
        }
        if (discard_src) discard_read_lines(s4, vlo, vhi, T);
    }
}

template <int DT, int OP, bool VEC>
__global__ void __launch_bounds__(kTreeThreads, 3) tree_executor_kernel(const __grid_constant__ RingArgs a) {
    __shared__ int s_rank, s_j, s_g;
    __shared__ unsigned long long s_trace_t0, s_trace_t1;  // (step trace)
    const int p = a.p;
    const int L = tree_levels(p);
    if (threadIdx.x == 0) {
        // this CTA's rank: the last r whose first CTA is at or before it
        int lo = 0, hi = p - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) / 2;
            if (tree_first_cta(mid, p, L, a.tree_scale, a.channels) <= (long long)blockIdx.x) lo = mid;
            else hi = mid - 1;
        }
        s_rank = lo;
        s_j = (int)(blockIdx.x - tree_first_cta(lo, p, L, a.tree_scale, a.channels));
        s_g = a.tree_scale > 0 ? a.tree_scale * tree_weight(lo, p, L) : a.channels;
    }
    __syncthreads();
    const int r = s_rank, j = s_j, G = s_g;
    char *mine = rank_ptr(a.bufs, p, r);
    const long long nsl = (a.n + a.slice - 1) / a.slice;
    const int W = blockDim.x >> 5;  // warps per CTA: a progress word each, per slice
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned long long *my_flags = a.flags + (long long)r * nsl * W + w;  // [slice * W]
    const bool muted = a.fault_mode == RAR_FAULT_MUTE && r == a.fault_rank;
    const bool slow = a.fault_mode == RAR_FAULT_DELAY && r == a.fault_rank;
    // the rank's active steps: reduce levels 0 .. m - 1, then (not the root)
    // the broadcast at level b = ctz(r)
    const int b = r == 0 ? L : __ffs(r) - 1;
    const int m = tree_reduce_levels(r, p, L);
    const int S = m + (r == 0 ? 0 : 1);
    // Processing order: a wavefront over global slice groups [g B, (g + 1) B)
    // (B = a.block).  At time tau a CTA runs each of the rank's active steps,
    // of schedule step lambda, on its slices of group tau - lambda.  Every
    // wait is for an earlier schedule step on the same group, which its
    // owner runs at an earlier time, so the CTA at the earliest time is never
    // blocked and the launch cannot deadlock, whatever the CTA counts; and
    // a reader usually finds the data produced one time step before, still
    // in L2, while every rank keeps several groups in flight.
    const long long B = a.block > 0 ? a.block : 1;
    const long long ngroups = (nsl + B - 1) / B;
    const unsigned epoch = launch_epoch_begin(a);
    if (muted) goto done;

    for (long long tau = 0; tau < ngroups + 2 * L; tau++) {
        for (int t = S - 1; t >= 0; t--) {  // the oldest group first
            const bool up = t < m;
            const int l = up ? t : b;
            const int step = up ? l : 2 * L - 1 - l;  // lambda
            const long long g = tau - step;
            if (g < 0 || g >= ngroups) continue;
            const long long g0 = g * B, g1 = g0 + B < nsl ? g0 + B : nsl;
            const long long s_first = g0 + (((long long)j - g0 % G) % G + G) % G;  // first s >= g0, s = j (mod G)
            const int peer = up ? r + (1 << l) : r - (1 << l);
            // the peer's active steps that must be complete on the slice
            const int need = up ? tree_weight(peer, p, L) - 1 : tree_weight(peer, p, L);
            const char *src = rank_ptr(a.bufs, p, peer);
            for (long long sl = s_first; sl < g1; sl += G) {
                // this warp's part of the slice: the same warp of the peer
                int ok = 1;
                if (lane == 0) {
                    if (a.trace && w == 0) s_trace_t0 = global_ns();
                    ok = need > 0 ? ring_wait(a, epoch, a.flags + ((long long)peer * nsl + sl) * W + w,
                                              ((unsigned long long)epoch << 32) | (unsigned)need, r, step, sl, peer)
                                  : ld_relaxed_u32(a.abort_word) != epoch;
                    if (a.trace && w == 0) s_trace_t1 = global_ns();
                    if (ok && slow) ring_delay(a.fault_delay_ns);
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) goto done;
                __syncwarp();  // orders lane 0's acquire before the other lanes' reads
                const long long lo = sl * a.slice;
                const long long hi = lo + a.slice < a.n ? lo + a.slice : a.n;
                // from level 1 up the child holds a partial of its subtree;
                // below the root's last level the result is a partial
                const bool root_last = r == 0 && l == L - 1;
                tree_slice<DT, OP, VEC>(src, mine, lo, hi, up, up && root_last, up && l > 0, up || l == 0,
                                        up && !root_last, a.inv_p);
                // the warp barrier orders the lanes' stores of this part
                // before lane 0's release of the warp's word
                __syncwarp();
                if (lane == 0) {
                    st_release_u64(my_flags + sl * W, ((unsigned long long)epoch << 32) | (unsigned)(t + 1));
                    if (w == 0) {
                        atomicAdd(&a.recv_counts[peer], (unsigned long long)(hi - lo));  // the peer sent
                        if (a.trace) trace_add(a, r, step, s_trace_t0, s_trace_t1);
                    }
                }
            }
        }
    }
done:
    launch_epoch_end(a, epoch);
}

template <int DT, int OP, bool VEC>
static cudaError_t launch_tree_t(const RingArgs &a, int threads, cudaStream_t stream) {
    void *args[] = {const_cast<RingArgs *>(&a)};
    return cudaLaunchCooperativeKernel((const void *)tree_executor_kernel<DT, OP, VEC>,
                                       dim3((unsigned)tree_grid_ctas(a.p, a.tree_scale, a.channels)),
                                       dim3((unsigned)threads), args, 0, stream);
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

long long tree_grid_ctas(int p, int tree_scale, int channels) {
    return tree_first_cta(p, p, tree_levels(p), tree_scale, channels) + 0;
}

int tree_max_coresident_ctas(int dtype, int op, bool vec16, int threads) {
    const int per_sm = dispatch_dtype_op<false>(dtype, op, 0, [&](auto dt, auto o) {
        return tree_occ<decltype(dt)::value, decltype(o)::value>(vec16, threads);
    });
    const int sms = current_device_sm_count();
    return per_sm * sms;
}

}  // namespace rar
