// fused_impl.cuh -- engine (a): the fused order-faithful reducer.
//
// The ring's data movement collapses to: every output element of chunk c is
// x_c (+) x_(c+1) (+) ... (+) x_(c+p-1) (indices mod p) in that exact order
// ("Ring All-Reduce, in depth", "The schedule" / "Tracing four GPUs": chunk c
// starts at rank c and collects one contribution per hop), scaled by 1/p at
// the owner for avg, and then copied to every rank by the all-gather.  One
// kernel therefore reads each rank's element once and stores the result once
// per rank: 2 p n element moves, the minimum for an in-place all-reduce.
//
// Work is split into tiles of blockDim.x * U 16-byte vectors, walked by a
// grid-stride loop over a grid sized to the co-resident CTA count.  A tile
// inside a single chunk takes the uniform path (one fold order for the whole
// CTA; for p = 4, 8, 16 all p loads issued before the fold, for other p in
// batches of 4 ranks); tiles that cross a chunk boundary or the ragged tail
// fall back to per-vector and per-element folds, so that no vector lane ever
// mixes two chunks' orders.  For p > 8 the vectors that hold an unaligned
// chunk start go to a warp each in a second launch (fused_straddle_kernel).
#pragma once

#include "elem_ops.cuh"

namespace rar {

constexpr int kFusedThreads = 256;

// Fold order for chunk c over ranks c, c+1, ..., c+p-1 on U vectors at
// v0, v0 + stride, ..., then store per phase.
template <int DT, int OP, int P, int U>
__device__ __forceinline__ void fused_fold_vectors(const FusedArgs &a, int p, int c, long long v0,
                                                   long long stride) {
    uint4 acc[U];
    const int phase = a.phase;
    const int owner = (c == 0) ? p - 1 : c - 1;
    if (phase == PHASE_AG) {
        // all-gather alone: the owner's finished chunk goes to everyone
        const uint4 *src = reinterpret_cast<const uint4 *>(rank_ptr(a.bufs, p, owner));
#pragma unroll
        for (int u = 0; u < U; u++) acc[u] = __ldcs(src + v0 + u * stride);
        for (int r = 0; r < p; r++) {
            if (r == owner) continue;
            uint4 *dst = reinterpret_cast<uint4 *>(rank_ptr(a.bufs, p, r));
#pragma unroll
            for (int u = 0; u < U; u++) __stcs(dst + v0 + u * stride, acc[u]);
        }
        return;
    }
    constexpr int hop = HopOf<OP>::value;
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(rank_ptr(a.bufs, p, c));
#pragma unroll
        for (int u = 0; u < U; u++) acc[u] = contrib_vec<DT, OP>(__ldcs(src + v0 + u * stride), a.inv_p);
    }
    if constexpr (P > 0) {
        uint4 own[P > 1 ? P - 1 : 1][U];
#pragma unroll
        for (int k = 1; k < P; k++) {
            int r = c + k;
            r -= (r >= P) ? P : 0;
            const uint4 *src = reinterpret_cast<const uint4 *>(rank_ptr(a.bufs, P, r));
#pragma unroll
            for (int u = 0; u < U; u++) own[k - 1][u] = __ldcs(src + v0 + u * stride);
        }
#pragma unroll
        for (int k = 1; k < P; k++)
#pragma unroll
            for (int u = 0; u < U; u++) acc[u] = hop_vec<DT, hop>(acc[u], contrib_vec<DT, OP>(own[k - 1][u], a.inv_p));
    } else {
        // loads in batches of G ranks: 4 keeps the kernel at 64-76 registers
        // (4 CTAs per SM; with 8, 128 registers and 2), which measured
        // faster wherever the grid takes more than one wave (p = 40 x 1 M
        // bf16: 62.8 -> 41.1 us) and within 2% elsewhere
        constexpr int G = 4;
        for (int k0 = 1; k0 < p; k0 += G) {
            uint4 own[G][U];
#pragma unroll
            for (int j = 0; j < G; j++) {
                int k = k0 + j;
                if (k < p) {
                    int r = c + k;
                    r -= (r >= p) ? p : 0;
                    const uint4 *src = reinterpret_cast<const uint4 *>(rank_ptr(a.bufs, p, r));
#pragma unroll
                    for (int u = 0; u < U; u++) own[j][u] = __ldcs(src + v0 + u * stride);
                }
            }
#pragma unroll
            for (int j = 0; j < G; j++)
                if (k0 + j < p)
#pragma unroll
                    for (int u = 0; u < U; u++)
                        acc[u] = hop_vec<DT, hop>(acc[u], contrib_vec<DT, OP>(own[j][u], a.inv_p));
        }
    }
    if constexpr (OP == OP_AVG) {
#pragma unroll
        for (int u = 0; u < U; u++) acc[u] = scale_vec<DT>(acc[u], a.inv_p);
    }
    if (phase == PHASE_RS) {
        uint4 *dst = reinterpret_cast<uint4 *>(rank_ptr(a.bufs, p, owner));
#pragma unroll
        for (int u = 0; u < U; u++) __stcs(dst + v0 + u * stride, acc[u]);
        return;
    }
    for (int r = 0; r < p; r++) {
        uint4 *dst = reinterpret_cast<uint4 *>(rank_ptr(a.bufs, p, r));
#pragma unroll
        for (int u = 0; u < U; u++) __stcs(dst + v0 + u * stride, acc[u]);
    }
}

// One element i of chunk c, same order and phases.
template <int DT, int OP>
__device__ __forceinline__ void fused_fold_element(const FusedArgs &a, int p, int c, long long i) {
    const int owner = (c == 0) ? p - 1 : c - 1;
    uint32_t acc;
    if (a.phase == PHASE_AG) {
        acc = load_elem<DT>(rank_ptr(a.bufs, p, owner), i);
        for (int r = 0; r < p; r++)
            if (r != owner) store_elem<DT>(rank_ptr(a.bufs, p, r), i, acc);
        return;
    }
    constexpr int hop = HopOf<OP>::value;
    acc = contrib_word<DT, OP>(load_elem<DT>(rank_ptr(a.bufs, p, c), i), a.inv_p);
    for (int k = 1; k < p; k++) {
        int r = c + k;
        r -= (r >= p) ? p : 0;
        acc = hop_word<DT, hop>(acc, contrib_word<DT, OP>(load_elem<DT>(rank_ptr(a.bufs, p, r), i), a.inv_p));
    }
    if constexpr (OP == OP_AVG) acc = scale_word<DT>(acc, a.inv_p);
    if (a.phase == PHASE_RS) {
        store_elem<DT>(rank_ptr(a.bufs, p, owner), i, acc);
        return;
    }
    for (int r = 0; r < p; r++) store_elem<DT>(rank_ptr(a.bufs, p, r), i, acc);
}

// A 16-byte vector v whose elements lie in more than one chunk, the first of
// them in chunk ca, folded from global memory by a whole warp.  The warp
// passes over the ranks from ca on, lane j loading the whole vector of rank
// (ca + j0 + j) mod p as pass step j0 + j, 32 ranks at a time; lane l < VE
// folds element l, of chunk ca + d_l, taking pass step j as its hop j - d_l
// (the lag of the streaming path's segments), so every element is folded in
// its own chunk's order, as fused_fold_element folds it.  All 32 lanes of a
// converged warp call it with the same v and ca; every lane gets the vector.
template <int DT, int OP>
__device__ __forceinline__ uint4 warp_fold_straddling_vector(const FusedArgs &a, int p, long long base,
                                                             long long extra, long long v, int ca) {
    constexpr int EB = ElemInfo<DT>::bytes;
    constexpr int VE = 16 / EB;
    constexpr int hop = HopOf<OP>::value;
    const int lane = threadIdx.x & 31;
    const int my_l = lane < VE ? lane : VE - 1;  // (lanes >= VE shadow the last element)
    // d_l: the chunks after ca that start at or before element l
    const long long gi = a.first + v * VE + my_l;
    int d = 0;
    while (ca + d + 1 < p && chunk_start(ca + d + 1, base, extra) <= gi) d++;
    const int steps = p + __shfl_sync(0xffffffffu, d, 31);  // (lane 31 holds the last element's d)
    const int wi = (my_l * EB) >> 2;                          // the word holding this lane's element
    uint32_t acc = 0;
    for (int j0 = 0; j0 < steps; j0 += 32) {
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (j0 + lane < steps)
            x = __ldcg(reinterpret_cast<const uint4 *>(rank_ptr(a.bufs, p, (ca + j0 + lane) % p)) + v);
        const int jn = steps - j0 < 32 ? steps - j0 : 32;
        for (int j = 0; j < jn; j++) {
            const uint32_t w0 = __shfl_sync(0xffffffffu, x.x, j), w1 = __shfl_sync(0xffffffffu, x.y, j);
            const uint32_t w2 = __shfl_sync(0xffffffffu, x.z, j), w3 = __shfl_sync(0xffffffffu, x.w, j);
            const uint32_t w = wi == 0 ? w0 : wi == 1 ? w1 : wi == 2 ? w2 : w3;
            const int k = j0 + j - d;
            if (lane < VE && k >= 0 && k < p) {
                // the element in the low half of a word, as load_elem gives it
                const uint32_t e = contrib_word<DT, OP>(EB == 4 ? w : (w >> (16 * (my_l & 1))) & 0xFFFFu, a.inv_p);
                acc = k == 0 ? e : hop_word<DT, hop>(acc, e);
            }
        }
    }
    if constexpr (OP == OP_AVG) acc = scale_word<DT>(acc, a.inv_p);
    uint32_t out[4];
#pragma unroll
    for (int q = 0; q < 4; q++) {
        if constexpr (EB == 4) out[q] = __shfl_sync(0xffffffffu, acc, q);
        else
            out[q] = (__shfl_sync(0xffffffffu, acc, 2 * q) & 0xFFFFu) |
                     ((__shfl_sync(0xffffffffu, acc, 2 * q + 1) & 0xFFFFu) << 16);
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

// The vectors across a chunk boundary of a whole all-reduce on the
// per-thread path (16-byte aligned ranks), which the main kernel left out
// (its straddle_pass): warp w takes the start of chunk w + 1 and, where that
// start is not vector-aligned, folds the vector holding it and stores it to
// every rank; a vector holding several starts goes with the first.  Its own
// launch, so that this rarely used code does not weigh on the main kernel's
// registers; it runs after the main kernel (pdl_wait), like any next kernel.
template <int DT, int OP>
__global__ void __launch_bounds__(kFusedThreads) fused_straddle_kernel(const __grid_constant__ FusedArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    constexpr int VE = 16 / ElemInfo<DT>::bytes;
    const int p = a.p;
    const long long base = a.n_total / p, extra = a.n_total % p;
    const int c = 1 + (int)(((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    if (c >= p) return;  // (the tests below are warp-uniform)
    const long long b = chunk_start(c, base, extra) - a.first;  // chunk c's first element, local index
    if (b <= 0 || b % VE == 0) return;                           // outside the range, or vector-aligned
    const long long sv = b / VE;
    if (sv >= a.n / VE) return;  // the ragged tail: the main kernel folds it element by element
    // Chunk c - 1 starts at bp.  If bp lies inside the same vector (not at
    // its first element), the vector goes with chunk c - 1's start; else
    // bp <= the vector's first element < b, so that element is in chunk
    // c - 1.
    const long long bp = chunk_start(c - 1, base, extra) - a.first;
    if (bp > sv * VE && bp / VE == sv) return;
    const uint4 x = warp_fold_straddling_vector<DT, OP>(a, p, base, extra, sv, c - 1);
    for (int r = threadIdx.x & 31; r < p; r += 32) __stcs(reinterpret_cast<uint4 *>(rank_ptr(a.bufs, p, r)) + sv, x);
}

template <int DT, int OP, int P, int U, bool VEC>
__global__ void __launch_bounds__(kFusedThreads)
    fused_ring_order_kernel(const __grid_constant__ FusedArgs a, int straddle_pass) {
    pdl_wait();
    pdl_launch_dependents();
    const int p = P > 0 ? P : a.p;
    const long long n = a.n;
    const long long base = a.n_total / p, extra = a.n_total % p;
    const long long g0 = a.first;  // global index of local element 0
    constexpr int VE = VEC ? 16 / ElemInfo<DT>::bytes : 1;  // elements per vector
    const long long nvec = (n + VE - 1) / VE;
    const long long nfull = n / VE;
    const long long tv = (long long)blockDim.x * U;
    for (long long t0 = (long long)blockIdx.x * tv; t0 < nvec; t0 += (long long)gridDim.x * tv) {
        const long long t1 = t0 + tv < nvec ? t0 + tv : nvec;
        const int c0 = chunk_of(g0 + t0 * VE, base, extra);
        const long long last = (t1 * VE < n ? t1 * VE : n) - 1;
        const int c1 = chunk_of(g0 + last, base, extra);
        if (VEC && t1 - t0 == tv && t1 <= nfull && c0 == c1) {
            fused_fold_vectors<DT, OP, P, U>(a, p, c0, t0 + threadIdx.x, blockDim.x);
            continue;
        }
#pragma unroll 1
        for (int u = 0; u < U; u++) {
            const long long v = t0 + threadIdx.x + (long long)u * blockDim.x;
            if (v >= t1) break;
            const long long e0 = v * VE;
            if (VEC && v < nfull) {
                const int ca = chunk_of(g0 + e0, base, extra);
                const int cb = chunk_of(g0 + e0 + VE - 1, base, extra);
                if (ca == cb) {
                    fused_fold_vectors<DT, OP, P, 1>(a, p, ca, v, 0);
                    continue;
                }
                if (straddle_pass) continue;  // (fused_straddle_kernel folds it)
            }
            for (int l = 0; l < VE; l++) {
                const long long i = e0 + l;
                if (i >= n) break;
                fused_fold_element<DT, OP>(a, p, chunk_of(g0 + i, base, extra), i);
            }
        }
    }
}

// ---------------------------------------------------------------- tree order
//
// Tree order over the rank index: adjacent pairs level by level, an odd last
// entry carried up.  Streaming form: push ranks 0, 1, ... onto a stack and
// merge the top two while they cover equally many ranks; at the end merge
// from the top down.  (The two forms build the same tree for every p.)
// The order does not depend on the chunk, only the reduce-scatter-only
// phase needs the owner.

template <int DT, int OP, int P>
__device__ __forceinline__ uint4 tree_fold_vector(const FusedArgs &a, int p, long long v) {
    constexpr int kMaxDepth = 12;  // log2(RAR_MAX_P) + 2
    uint4 st[kMaxDepth];
    int sz[kMaxDepth];
    int sp = 0;
    constexpr int hop = HopOf<OP>::value;
    auto push = [&](int r, int pp) {
        st[sp] = contrib_vec<DT, OP>(__ldcs(reinterpret_cast<const uint4 *>(rank_ptr(a.bufs, pp, r)) + v), a.inv_p);
        sz[sp] = 1;
        sp++;
        while (sp >= 2 && sz[sp - 1] == sz[sp - 2]) {
            st[sp - 2] = hop_vec<DT, hop>(st[sp - 2], st[sp - 1]);
            sz[sp - 2] *= 2;
            sp--;
        }
    };
    if constexpr (P > 0) {
#pragma unroll
        for (int r = 0; r < P; r++) push(r, P);
    } else {
        for (int r = 0; r < p; r++) push(r, p);
    }
    while (sp > 1) {
        st[sp - 2] = hop_vec<DT, hop>(st[sp - 2], st[sp - 1]);
        sp--;
    }
    return st[0];
}

template <int DT, int OP, int P>
__device__ __forceinline__ uint32_t tree_fold_element(const FusedArgs &a, int p, long long i) {
    constexpr int kMaxDepth = 12;
    uint32_t st[kMaxDepth];
    int sz[kMaxDepth];
    int sp = 0;
    constexpr int hop = HopOf<OP>::value;
    for (int r = 0; r < p; r++) {
        st[sp] = contrib_word<DT, OP>(load_elem<DT>(rank_ptr(a.bufs, p, r), i), a.inv_p);
        sz[sp] = 1;
        sp++;
        while (sp >= 2 && sz[sp - 1] == sz[sp - 2]) {
            st[sp - 2] = hop_word<DT, hop>(st[sp - 2], st[sp - 1]);
            sz[sp - 2] *= 2;
            sp--;
        }
    }
    while (sp > 1) {
        st[sp - 2] = hop_word<DT, hop>(st[sp - 2], st[sp - 1]);
        sp--;
    }
    return st[0];
}

template <int DT, int OP, int P, bool VEC>
__global__ void __launch_bounds__(kFusedThreads) fused_tree_order_kernel(const __grid_constant__ FusedArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    const int p = P > 0 ? P : a.p;
    const long long n = a.n;
    const long long base = a.n_total / p, extra = a.n_total % p;
    const long long g0 = a.first;
    constexpr int VE = VEC ? 16 / ElemInfo<DT>::bytes : 1;
    const long long nvec = (n + VE - 1) / VE;
    const long long nfull = n / VE;
    for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < nvec;
         v += (long long)gridDim.x * blockDim.x) {
        const long long e0 = v * VE;
        const int ca = chunk_of(g0 + e0, base, extra);
        const int cb = chunk_of(g0 + (e0 + VE - 1 < n ? e0 + VE - 1 : n - 1), base, extra);
        if (VEC && v < nfull && (a.phase == PHASE_ALL || ca == cb)) {
            uint4 acc = tree_fold_vector<DT, OP, P>(a, p, v);
            if constexpr (OP == OP_AVG) acc = scale_vec<DT>(acc, a.inv_p);
            if (a.phase == PHASE_RS) {
                const int owner = (ca == 0) ? p - 1 : ca - 1;
                __stcs(reinterpret_cast<uint4 *>(rank_ptr(a.bufs, p, owner)) + v, acc);
            } else {
                for (int r = 0; r < p; r++) __stcs(reinterpret_cast<uint4 *>(rank_ptr(a.bufs, p, r)) + v, acc);
            }
            continue;
        }
        for (int l = 0; l < VE; l++) {
            const long long i = e0 + l;
            if (i >= n) break;
            uint32_t acc = tree_fold_element<DT, OP, P>(a, p, i);
            if constexpr (OP == OP_AVG) acc = scale_word<DT>(acc, a.inv_p);
            if (a.phase == PHASE_RS) {
                const int c = chunk_of(g0 + i, base, extra);
                store_elem<DT>(rank_ptr(a.bufs, p, (c == 0) ? p - 1 : c - 1), i, acc);
            } else {
                for (int r = 0; r < p; r++) store_elem<DT>(rank_ptr(a.bufs, p, r), i, acc);
            }
        }
    }
}

// ---------------------------------------------------------------- hierarchical order
//
// "Ring All-Reduce, in depth", "Hierarchy": p = m nodes of g ranks
// (rank = node * g + local); reduce-scatter inside the nodes on
// chunk_bounds(n, g), all-reduce of every 1/g shard across the nodes on
// chunk_bounds(shard, m), all-gather inside the nodes.  Element i of
// intra-node chunk c and shard sub-chunk s therefore becomes the fold over
// nodes s, s+1, ... (mod m) of node partials, each partial folding local
// ranks c, c+1, ... (mod g) of its node.  avg scales the final value once.

struct HierPos {
    int c;  // intra-node chunk
    int s;  // sub-chunk of that chunk across the nodes
};

__device__ __forceinline__ HierPos hier_pos(long long i, long long n, int g, int m) {
    const long long gb = n / g, ge = n % g;
    const int c = chunk_of(i, gb, ge);
    const long long c0 = chunk_start(c, gb, ge);
    const long long len = gb + (c < ge ? 1 : 0);
    return HierPos{c, chunk_of(i - c0, len / m, len % m)};
}

template <int DT, int OP>
__device__ __forceinline__ uint4 hier_fold_vector(const FusedArgs &a, int p, int g, HierPos hp, long long v) {
    constexpr int hop = HopOf<OP>::value;
    const int m = p / g;
    uint4 acc = make_uint4(0, 0, 0, 0);
    for (int t = 0; t < m; t++) {
        int node = hp.s + t;
        node -= node >= m ? m : 0;
        const int base = node * g;
        uint4 part = make_uint4(0, 0, 0, 0);
        for (int k0 = 0; k0 < g; k0 += 8) {
            uint4 x[8];
#pragma unroll
            for (int j = 0; j < 8; j++) {
                if (k0 + j < g) {
                    int l = hp.c + k0 + j;
                    l -= l >= g ? g : 0;
                    x[j] = contrib_vec<DT, OP>(__ldcs(reinterpret_cast<const uint4 *>(rank_ptr(a.bufs, p, base + l)) + v),
                                               a.inv_p);
                }
            }
#pragma unroll
            for (int j = 0; j < 8; j++)
                if (k0 + j < g) part = (k0 + j == 0) ? x[j] : hop_vec<DT, hop>(part, x[j]);
        }
        acc = t == 0 ? part : hop_vec<DT, hop>(acc, part);
    }
    if constexpr (OP == OP_AVG) acc = scale_vec<DT>(acc, a.inv_p);
    return acc;
}

template <int DT, int OP>
__device__ __forceinline__ uint32_t hier_fold_element(const FusedArgs &a, int p, int g, HierPos hp, long long i) {
    constexpr int hop = HopOf<OP>::value;
    const int m = p / g;
    uint32_t acc = 0;
    for (int t = 0; t < m; t++) {
        int node = hp.s + t;
        node -= node >= m ? m : 0;
        uint32_t part = 0;
        for (int k = 0; k < g; k++) {
            int l = hp.c + k;
            l -= l >= g ? g : 0;
            const uint32_t x = contrib_word<DT, OP>(load_elem<DT>(rank_ptr(a.bufs, p, node * g + l), i), a.inv_p);
            part = k == 0 ? x : hop_word<DT, hop>(part, x);
        }
        acc = t == 0 ? part : hop_word<DT, hop>(acc, part);
    }
    if constexpr (OP == OP_AVG) acc = scale_word<DT>(acc, a.inv_p);
    return acc;
}

template <int DT, int OP, bool VEC>
__global__ void __launch_bounds__(kFusedThreads) fused_hier_kernel(const __grid_constant__ FusedArgs a, int g) {
    pdl_wait();
    pdl_launch_dependents();
    const int p = a.p;
    const int m = p / g;
    const long long n = a.n;
    const long long nt = a.n_total, g0 = a.first;
    constexpr int VE = VEC ? 16 / ElemInfo<DT>::bytes : 1;
    const long long nvec = (n + VE - 1) / VE;
    const long long nfull = n / VE;
    for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < nvec;
         v += (long long)gridDim.x * blockDim.x) {
        const long long e0 = v * VE;
        if (VEC && v < nfull) {
            const HierPos a0 = hier_pos(g0 + e0, nt, g, m), a1 = hier_pos(g0 + e0 + VE - 1, nt, g, m);
            if (a0.c == a1.c && a0.s == a1.s) {
                const uint4 acc = hier_fold_vector<DT, OP>(a, p, g, a0, v);
                for (int r = 0; r < p; r++) __stcs(reinterpret_cast<uint4 *>(rank_ptr(a.bufs, p, r)) + v, acc);
                continue;
            }
        }
        for (int l = 0; l < VE; l++) {
            const long long i = e0 + l;
            if (i >= n) break;
            const uint32_t acc = hier_fold_element<DT, OP>(a, p, g, hier_pos(g0 + i, nt, g, m), i);
            for (int r = 0; r < p; r++) store_elem<DT>(rank_ptr(a.bufs, p, r), i, acc);
        }
    }
}

// The same order with all P ranks' vectors in flight at once (P a
// compile-time rank count): each thread keeps the rank order of the fold for
// its current (intra-node chunk, sub-chunk) segment and rebuilds it only when
// its vectors move into another segment, so a vector costs P loads, the fold
// and P stores.  Vectors across a segment boundary fold element by element.
template <int DT, int OP, int P, bool VEC>
__global__ void __launch_bounds__(kFusedThreads) fused_hier_kernel_p(const __grid_constant__ FusedArgs a, int g) {
    pdl_wait();
    pdl_launch_dependents();
    constexpr int hop = HopOf<OP>::value;
    constexpr int VE = VEC ? 16 / ElemInfo<DT>::bytes : 1;
    const int m = P / g;
    const long long n = a.n;
    const long long nt = a.n_total, g0 = a.first;
    const long long nvec = (n + VE - 1) / VE;
    const long long nfull = n / VE;
    long long seg_lo = 1, seg_hi = 0;  // current segment, global indices [seg_lo, seg_hi); none yet
    int ord[P];                        // its ranks in fold order
    for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < nvec;
         v += (long long)gridDim.x * blockDim.x) {
        const long long e0 = v * VE;
        const long long ge0 = g0 + e0;
        if (ge0 < seg_lo || ge0 >= seg_hi) {
            const HierPos hp = hier_pos(ge0, nt, g, m);
            const long long gb = nt / g, ge = nt % g;
            const long long c0 = chunk_start(hp.c, gb, ge);
            const long long len = gb + (hp.c < ge ? 1 : 0);
            seg_lo = c0 + chunk_start(hp.s, len / m, len % m);
            seg_hi = c0 + chunk_start(hp.s + 1, len / m, len % m);
            int t = 0, kk = 0;
#pragma unroll
            for (int k = 0; k < P; k++) {
                int node = hp.s + t;
                node -= node >= m ? m : 0;
                int l = hp.c + kk;
                l -= l >= g ? g : 0;
                ord[k] = node * g + l;
                if (++kk == g) {
                    kk = 0;
                    t++;
                }
            }
        }
        if (VEC && v < nfull && ge0 + VE <= seg_hi) {
            uint4 x[P];
#pragma unroll
            for (int k = 0; k < P; k++)
                x[k] = contrib_vec<DT, OP>(__ldcs(reinterpret_cast<const uint4 *>(rank_ptr(a.bufs, P, ord[k])) + v),
                                           a.inv_p);
            // node partials over g local ranks, then over the nodes in turn
            uint4 acc = x[0], part = x[0];
            int kk = 1;
#pragma unroll
            for (int k = 1; k < P; k++) {
                if (kk == g) {
                    acc = k == g ? part : hop_vec<DT, hop>(acc, part);
                    part = x[k];
                    kk = 1;
                } else {
                    part = hop_vec<DT, hop>(part, x[k]);
                    kk++;
                }
            }
            acc = g == P ? part : hop_vec<DT, hop>(acc, part);
            if constexpr (OP == OP_AVG) acc = scale_vec<DT>(acc, a.inv_p);
#pragma unroll
            for (int r = 0; r < P; r++) __stcs(reinterpret_cast<uint4 *>(rank_ptr(a.bufs, P, r)) + v, acc);
            continue;
        }
        for (int l = 0; l < VE; l++) {
            const long long i = e0 + l;
            if (i >= n) break;
            const uint32_t acc = hier_fold_element<DT, OP>(a, P, g, hier_pos(g0 + i, nt, g, m), i);
            for (int r = 0; r < P; r++) store_elem<DT>(rank_ptr(a.bufs, P, r), i, acc);
        }
    }
}

// ---------------------------------------------------------------- dispatch

template <typename K>
static int blocks_per_sm_of(K kernel, int threads) {
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, threads, 0) != cudaSuccess) return 1;
    return nb > 0 ? nb : 1;
}

static int sm_count_cached() {
    const int v = current_device_sm_count();
    return v > 0 ? v : 1;
}

template <typename K, typename... Extra>
static cudaError_t launch_persistent(K kernel, const FusedArgs &a, long long work_items, int threads,
                                     cudaStream_t stream, Extra... extra) {
    const int sms = sm_count_cached();
    const long long want = (work_items + threads - 1) / threads;
    long long grid = (long long)sms * blocks_per_sm_of(kernel, threads);
    if (grid > want) grid = want;
    if (grid < 1) grid = 1;
    cudaError_t e = launch_pdl(kernel, dim3((unsigned)grid), dim3((unsigned)threads), 0, stream, a, extra...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Whether a chunk start inside the launch's index range is not 16-byte
// aligned (so that a vector lies across the boundary).
static bool has_unaligned_chunk_start(const FusedArgs &a, int ve) {
    const long long base = a.n_total / a.p, extra = a.n_total % a.p;
    for (int c = 1; c < a.p; c++) {
        const long long b = (long long)c * base + (c < extra ? c : extra) - a.first;  // chunk_start(c)
        if (b > 0 && b < a.n && b % ve != 0) return true;
    }
    return false;
}

template <int DT, int OP, int P>
static cudaError_t launch_fused_p(const FusedArgs &a, bool tree, bool vec16, int threads, cudaStream_t stream) {
    constexpr int VE = 16 / ElemInfo<DT>::bytes;
    constexpr int U = (P > 0 && P <= 8) ? 2 : 1;
    if (tree) {
        if (vec16)
            return launch_persistent(fused_tree_order_kernel<DT, OP, P, true>, a, (a.n + VE - 1) / VE, threads,
                                     stream);
        return launch_persistent(fused_tree_order_kernel<DT, OP, P, false>, a, a.n, threads, stream);
    }
    if (vec16) {
        // One vector per thread for a buffer that the one-vector kernel
        // covers in at most two waves of its co-resident grid.  The U-vector
        // kernel's registers cannot hold all of its p * U loads at once, so it
        // has about as many bytes in flight per thread as the one-vector
        // kernel, on half the threads: below a full grid the one-vector
        // kernel keeps twice the loads in flight (GB300, p = 8: 1-2 M
        // elements per rank 27-40% faster, 2.4 M fp32 10%).  From about two
        // waves on the two kernels are within a few percent either way, and
        // the U-vector kernel is ahead at 25 MB per rank (p = 8 fp32, 2%).
        const long long nvec = (a.n + VE - 1) / VE;
        if (U > 1 && nvec <= 2ll * sm_count_cached() *
                                 blocks_per_sm_of(fused_ring_order_kernel<DT, OP, P, 1, true>, threads) * threads)
            return launch_persistent(fused_ring_order_kernel<DT, OP, P, 1, true>, a, nvec, threads, stream, 0);
        // Beyond p = 8 a vector across a chunk boundary costs its thread p
        // dependent element folds per element (p = 64 x 250,000 bf16: 108 us
        // against 37 us with aligned chunk starts), so those vectors go to a
        // warp each in a pass of their own.
        const int straddle_pass = a.phase == PHASE_ALL && a.p > 8 && has_unaligned_chunk_start(a, VE) ? 1 : 0;
        cudaError_t e = launch_persistent(fused_ring_order_kernel<DT, OP, P, U, true>, a, (nvec + U - 1) / U,
                                          threads, stream, straddle_pass);
        if (e != cudaSuccess || !straddle_pass) return e;
        const unsigned blocks = (unsigned)(((long long)(a.p - 1) * 32 + kFusedThreads - 1) / kFusedThreads);
        e = launch_pdl(fused_straddle_kernel<DT, OP>, dim3(blocks), dim3(kFusedThreads), 0, stream, a);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    return launch_persistent(fused_ring_order_kernel<DT, OP, P, 1, false>, a, a.n, threads, stream, 0);
}

template <int DT, int OP>
static cudaError_t launch_fused_op(const FusedArgs &a, bool tree, bool vec16, int threads, cudaStream_t stream) {
    switch (a.p) {
    case 4: return launch_fused_p<DT, OP, 4>(a, tree, vec16, threads, stream);
    case 8: return launch_fused_p<DT, OP, 8>(a, tree, vec16, threads, stream);
    case 16: return launch_fused_p<DT, OP, 16>(a, tree, vec16, threads, stream);
    default: return launch_fused_p<DT, OP, 0>(a, tree, vec16, threads, stream);
    }
}

}  // namespace rar
