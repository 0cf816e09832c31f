// fused_stream.cu -- engine (a), rank-sequential streaming path.
//
// Same arithmetic as the other fused paths: element i of chunk c becomes
// x_c (+) x_(c+1) (+) ... (+) x_(c+p-1) in the ring's hop order ("Ring
// All-Reduce, in depth", "The schedule" and "Tracing four GPUs"), scaled by
// 1/p for avg, then copied to every rank (the all-gather).
//
// The access pattern follows the ring instead of reading all p ranks at
// once: a CTA takes a tile of `tile_bytes` per rank and walks the ranks in
// hop order, one contiguous tile at a time, keeping the running values in
// registers.  Each CTA therefore streams one long run at a time: the number
// of concurrent DRAM streams is set by the CTA count, not by p.  (With all p
// tiles in flight at once, throughput falls off beyond p = 16 on GB300.)
//
// A tile inside one chunk c needs ranks c, c+1, ..., c+p-1.  A tile that
// crosses chunk boundaries has segments c, c+1, ..., c+m-1; at global step j
// the CTA loads rank (c + j) and segment s takes its step j - s, which is
// exactly the rank it needs.  Such a tile costs p + m - 1 rank loads instead
// of p.  The few 16-byte vectors that themselves straddle a boundary are
// folded lane by lane from global memory instead, so no vector ever mixes
// two chunks' orders.
//
// Warp roles: a producer warp issues one cp.async.bulk load per step into a
// ring of shared-memory stages (full/empty mbarriers); eight consumer warps
// fold.  The result of a tile goes to a double-buffered shared-memory row,
// and its p cp.async.bulk stores are issued one per step of the next tile,
// interleaved with that tile's loads.
//
// Failure path.  A consumer warp's wait for a stage is bounded by the call's
// timeout; one that runs out records RAR_ETIMEOUT (with the rank whose tile
// never arrived) and raises a shared flag, and from then on no consumer
// releases a stage: a stage is handed back only after its load was seen
// complete, so the producer never reissues into a stage with a load still in
// flight.  The producer's wait for a free stage gives up on the same flag or
// timeout.  Before the producer -- and with it the CTA -- finishes, it waits
// for every bulk load it issued, whatever the call's timeout: an issued load
// always completes, so that wait ends by itself; it still has its own fixed
// limit (kStreamDrainLimitNs), far beyond any load's latency.  Bulk stores
// are waited for with cp.async.bulk.wait_group.  A host-requested fault
// (RAR_FAULT_MUTE) makes the producer stop issuing at the first load of the
// muted rank, so the consumers' bounded waits run out as for a dead rank.
#include "fused_impl.cuh"

namespace rar {

constexpr int kStreamConsumerWarps = 8;
constexpr int kStreamConsumerThreads = 32 * kStreamConsumerWarps;  // fold threads
constexpr int kStreamThreads = 32 + kStreamConsumerThreads;        // + one producer warp
constexpr int kStreamMaxStages = 8;
constexpr int kStreamMaxVecPerThread = 8;  // tile_bytes <= 256 * 16 * 8 = 32 KB

__device__ __forceinline__ uint32_t st_smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void st_mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void st_mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool st_mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ void st_mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Barrier 1 over the consumer warps only (the producer warp never joins it).
__device__ __forceinline__ void st_named_barrier_consumers() {
    asm volatile("bar.sync 1, %0;" ::"n"(kStreamConsumerThreads) : "memory");
}
__device__ __forceinline__ void st_bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void st_bulk_store(void *dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void st_bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void st_bulk_wait_reads_leave_1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void st_bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void st_fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void st_fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ unsigned long long st_global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for the phase of `bar` with this parity; false once `timeout_ns`
// passed (globaltimer, with an iteration cap) or `*stop` became nonzero.
__device__ __forceinline__ bool st_mbar_wait_bounded(uint32_t bar, uint32_t parity, unsigned long long timeout_ns,
                                                     const volatile int *stop) {
    if (st_mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = st_global_ns();
    const unsigned long long max_iters = timeout_ns / 16ull + (1ull << 20);
    for (unsigned long long it = 0; it < max_iters; it++) {
        if (st_mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 63 && (*stop || st_global_ns() - t0 > timeout_ns)) return false;
    }
    return false;
}

// The producer's wait for a bulk load it issued itself.  It does not take
// the call's timeout: the load completes by itself, and the CTA must not
// finish while it can still write shared memory.  The fixed limit only
// guards against a broken device.
constexpr unsigned long long kStreamDrainLimitNs = 10000000000ull;  // 10 s
__device__ __forceinline__ void st_mbar_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = st_global_ns();
    for (unsigned long long it = 0; it < (1ull << 36); it++) {
        if (st_mbar_try_wait(bar, parity)) return;
        if ((it & 255) == 255 && st_global_ns() - t0 > kStreamDrainLimitNs) return;
    }
}

// A vector across a chunk boundary (at most p - 1 in a buffer): each lane is
// folded in its own chunk's order from global memory, where this tile's
// inputs are still unchanged, and written into the result row.
template <int DT, int OP>
__device__ __noinline__ void stream_straddling_vector(const FusedArgs &a, int p, long long base, long long extra,
                                                      long long i0, unsigned char *out) {
    constexpr int EB = ElemInfo<DT>::bytes;
    constexpr int VE = 16 / EB;
    for (int l = 0; l < VE; l++) {
        const long long i = i0 + l;
        const int c = chunk_of(a.first + i, base, extra);
        uint32_t acc = contrib_word<DT, OP>(load_elem<DT>(rank_ptr(a.bufs, p, c), i), a.inv_p);
        for (int k = 1; k < p; k++) {
            int r = c + k;
            r -= (r >= p) ? p : 0;
            acc = hop_word<DT, HopOf<OP>::value>(acc, contrib_word<DT, OP>(load_elem<DT>(rank_ptr(a.bufs, p, r), i),
                                                                          a.inv_p));
        }
        if constexpr (OP == OP_AVG) acc = scale_word<DT>(acc, a.inv_p);
        if constexpr (EB == 4) reinterpret_cast<uint32_t *>(out)[l] = acc;
        else reinterpret_cast<uint16_t *>(out)[l] = (uint16_t)acc;
    }
}

template <int DT, int OP, int VPT>
__global__ void __launch_bounds__(kStreamThreads, 1)
    fused_stream_kernel(const __grid_constant__ FusedArgs a, int tile_bytes, int n_stages) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_fail;  // a consumer warp's wait ran out (then s_fail_* say where)
    __shared__ int s_fail_rank, s_fail_step;
    __shared__ long long s_fail_tile;
    constexpr int EB = ElemInfo<DT>::bytes;
    constexpr int VE = 16 / EB;
    constexpr int hop_op = HopOf<OP>::value;
    const int p = a.p;
    const int TB = tile_bytes;
    const int NS = n_stages;
    const long long n = a.n;
    const long long bulk_bytes = (n * EB) & ~15ll;
    const long long ntiles = (bulk_bytes + TB - 1) / TB;
    const long long base = a.n_total / p, extra = a.n_total % p;
    const long long g0 = a.first;  // global index of local element 0
    unsigned char *stage = smem;                               // NS * TB
    unsigned char *result = smem + (size_t)NS * TB;            // 2 * TB
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)(NS + 2) * TB);
    uint64_t *empty = full + kStreamMaxStages;
    const long long my_tiles = ntiles > blockIdx.x ? (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    pdl_wait();
    pdl_launch_dependents();

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; s++) {
            st_mbar_init(st_smem_addr(&full[s]), 1);
            st_mbar_init(st_smem_addr(&empty[s]), kStreamConsumerWarps);
        }
        st_fence_mbar_init();
        s_fail = 0;
    }
    __syncthreads();  // the last CTA-wide barrier: the warps split into roles below

    auto tile_off = [&](long long k) { return ((long long)blockIdx.x + k * gridDim.x) * TB; };
    auto tile_len = [&](long long k) {
        const long long off = tile_off(k);
        return (uint32_t)(bulk_bytes - off < TB ? bulk_bytes - off : TB);
    };
    auto tile_first_chunk = [&](long long k) { return chunk_of(g0 + tile_off(k) / EB, base, extra); };
    auto tile_segments = [&](long long k) {
        const long long e0 = g0 + tile_off(k) / EB;
        return chunk_of(e0 + tile_len(k) / EB - 1, base, extra) - chunk_of(e0, base, extra) + 1;
    };

    if (warp == 0) {
        // ---- producer: one bulk load per step, into the next free stage
        if (lane != 0) return;
        const int muted_rank = a.fault_mode == RAR_FAULT_MUTE ? a.fault_rank : -1;
        long long g = 0;  // loads issued
        bool ok = true;
        for (long long k = 0; k < my_tiles && ok; k++) {
            const long long off = tile_off(k);
            const uint32_t bytes = tile_len(k);
            const int c0 = tile_first_chunk(k);
            const int steps = p + tile_segments(k) - 1;
            for (int j = 0; j < steps; j++, g++) {
                const int s = (int)(g % NS);
                const long long use = g / NS;
                // a stage comes back only once all consumer warps saw its
                // previous load complete; give up when they stopped
                if (use > 0 &&
                    !st_mbar_wait_bounded(st_smem_addr(&empty[s]), (uint32_t)((use - 1) & 1), a.timeout_ns, &s_fail)) {
                    ok = false;
                    break;
                }
                const int rank = (c0 + j) % p;
                if (rank == muted_rank) {  // injected dead rank: its data never comes
                    ok = false;
                    break;
                }
                st_fence_proxy_async();
                const uint32_t bar = st_smem_addr(&full[s]);
                st_mbar_expect_tx(bar, bytes);
                st_bulk_load(st_smem_addr(stage + (size_t)s * TB), rank_ptr(a.bufs, p, rank) + off, bytes, bar);
            }
        }
        // Every load before the last NS was seen complete by the consumers
        // (its stage came back); the last NS may still be writing this CTA's
        // shared memory, so wait for each of them before finishing.
        for (long long h = g - NS > 0 ? g - NS : 0; h < g; h++)
            st_mbar_drain(st_smem_addr(&full[h % NS]), (uint32_t)((h / NS) & 1));
        return;
    }

    // ---- consumers: warps 1 .. kStreamConsumerWarps
    const int ct = threadIdx.x - 32;  // 0 .. 255
    long long g = 0;
    long long k = 0;
    bool failed = false;
    // Bulk stores of the previous tile's result row, issued by consumer 0 one
    // per step of the next tile so that they interleave with its loads.
    const unsigned char *pend_row = nullptr;
    long long pend_off = 0;
    uint32_t pend_bytes = 0;
    int pend_next = 0;  // next rank to store; p when none are pending
    int pend_count = 0;
    auto issue_pending_store = [&]() {
        if (pend_next < pend_count) {
            st_bulk_store(rank_ptr(a.bufs, p, pend_next) + pend_off, st_smem_addr(pend_row), pend_bytes);
            if (++pend_next == pend_count) st_bulk_commit();  // one group per tile
        }
    };
    for (; k < my_tiles; k++) {
        const long long off = tile_off(k);
        const uint32_t bytes = tile_len(k);
        const int nvec = (int)(bytes / 16);
        const long long e0 = off / EB;
        const int c0 = tile_first_chunk(k);
        const int m = tile_segments(k);
        const int steps = p + m - 1;
        uint4 acc[VPT];
        int seg[VPT];  // segment of each vector; -1 if it straddles a boundary
#pragma unroll
        for (int u = 0; u < VPT; u++) {
            const int v = ct + u * kStreamConsumerThreads;
            seg[u] = 0;
            if (m > 1 && v < nvec) {
                const long long i0 = e0 + (long long)v * VE;
                const int ca = chunk_of(g0 + i0, base, extra), cb = chunk_of(g0 + i0 + VE - 1, base, extra);
                seg[u] = ca == cb ? ca - c0 : -1;
            }
        }
        for (int j = 0; j < steps; j++, g++) {
            const int s = (int)(g % NS);
            if (!failed) {
                // warp-uniform: the warp goes on only if every lane saw the load
                bool ok = !*(volatile int *)&s_fail &&
                          st_mbar_wait_bounded(st_smem_addr(&full[s]), (uint32_t)((g / NS) & 1), a.timeout_ns, &s_fail);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) {
                    failed = true;
                    if (lane == 0 && atomicCAS(&s_fail, 0, 1) == 0) {  // the first to fail records where
                        s_fail_rank = (c0 + j) % p;
                        s_fail_step = j;
                        s_fail_tile = blockIdx.x + k * gridDim.x;
                    }
                }
            }
            if (!failed) {
                const unsigned char *st = stage + (size_t)s * TB;
#pragma unroll
                for (int u = 0; u < VPT; u++) {
                    const int v = ct + u * kStreamConsumerThreads;
                    if (v >= nvec || seg[u] < 0) continue;
                    const int kk = j - seg[u];
                    if (kk >= 0 && kk < p) {
                        const uint4 x = contrib_vec<DT, OP>(*reinterpret_cast<const uint4 *>(st + (size_t)v * 16),
                                                            a.inv_p);
                        acc[u] = kk == 0 ? x : hop_vec<DT, hop_op>(acc[u], x);
                    }
                }
            }
            __syncwarp();
            if (!failed) {
                // this warp is done with the stage, whose load it saw complete
                if (lane == 0) st_mbar_arrive(st_smem_addr(&empty[s]));
                if (ct == 0) issue_pending_store();
            }
        }

        // tile end: result row (double-buffered), then p bulk stores
        unsigned char *res = result + (size_t)(k & 1) * TB;
        if (ct == 0) st_bulk_wait_reads_leave_1();  // stores of tile k - 2 finished reading res
        st_named_barrier_consumers();
        if (*(volatile int *)&s_fail) {
            failed = true;
            break;  // uniform: every consumer reads s_fail after the same barrier
        }
#pragma unroll
        for (int u = 0; u < VPT; u++) {
            const int v = ct + u * kStreamConsumerThreads;
            if (v >= nvec) continue;
            if (seg[u] >= 0) {
                uint4 r = acc[u];
                if constexpr (OP == OP_AVG) r = scale_vec<DT>(r, a.inv_p);
                *reinterpret_cast<uint4 *>(res + (size_t)v * 16) = r;
            } else {
                stream_straddling_vector<DT, OP>(a, p, base, extra, e0 + (long long)v * VE, res + (size_t)v * 16);
            }
        }
        st_fence_proxy_async();
        st_named_barrier_consumers();
        if (ct == 0) {
            // every tile has at least p steps, so the previous tile's stores
            // have all been issued by now
            pend_row = res;
            pend_off = off;
            pend_bytes = bytes;
            pend_next = 0;
            pend_count = p;
        }
    }

    if (failed) {
        // (s_fail_* were written before the barrier that ended the tile)
        if (ct == 0) {
            a.status->code = RAR_ETIMEOUT;
            a.status->rank = -1;  // no rank group: a tile of the fused engine
            a.status->step = s_fail_step;
            a.status->slice = (int)s_fail_tile;
            a.status->waited_on = s_fail_rank;
            a.status->flag_seen = 0;
            a.status->flag_wanted = 0;
            __threadfence();
            atomicAdd(&a.status->seq, 1u);
            st_bulk_commit();  // stores issued but not yet committed join a group
            st_bulk_wait_all();
        }
        return;
    }
    if (ct == 0)
        while (pend_next < pend_count) issue_pending_store();
    if (blockIdx.x == gridDim.x - 1 && ct == 0) {
        for (long long i = bulk_bytes / EB; i < n; i++) fused_fold_element<DT, OP>(a, p, chunk_of(g0 + i, base, extra), i);
    }
    if (ct == 0) st_bulk_wait_all();
}

template <int DT, int OP, int VPT>
static cudaError_t launch_stream_v(const FusedArgs &a, int tile_bytes, int n_stages, cudaStream_t stream) {
    auto kernel = fused_stream_kernel<DT, OP, VPT>;
    const size_t smem = (size_t)(n_stages + 2) * tile_bytes + 2 * kStreamMaxStages * sizeof(uint64_t);
    // the kernel's dynamic shared memory limit, raised once per device to
    // the largest size asked for (setting it again is harmless)
    static std::atomic<int> configured_smem[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::atomic<int> &conf = configured_smem[dev >= 0 && dev < 64 ? dev : 0];
    if ((size_t)conf.load(std::memory_order_relaxed) < smem || dev < 0 || dev >= 64) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        conf.store((int)smem, std::memory_order_relaxed);
    }
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kStreamThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int sms = current_device_sm_count();
    if (sms < 1) return cudaErrorInvalidDevice;
    const long long bulk_bytes = (a.n * ElemInfo<DT>::bytes) & ~15ll;
    const long long ntiles = (bulk_bytes + tile_bytes - 1) / tile_bytes;
    long long grid = (long long)sms * per_sm;
    if (grid > ntiles) grid = ntiles;
    if (grid < 1) grid = 1;
    e = launch_pdl(kernel, dim3((unsigned)grid), dim3(kStreamThreads), smem, stream, a, tile_bytes, n_stages);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// 8 vectors per consumer thread: tiles of up to 32 KB per rank.
template <int DT, int OP>
static cudaError_t launch_stream_t(const FusedArgs &a, int tile_bytes, int n_stages, cudaStream_t stream) {
    return launch_stream_v<DT, OP, kStreamMaxVecPerThread>(a, tile_bytes, n_stages, stream);
}

cudaError_t launch_fused_stream(const FusedArgs &a, int dtype, int op, int tile_bytes, int n_stages,
                                cudaStream_t stream) {
    if (tile_bytes < 512 || tile_bytes > kStreamConsumerThreads * 16 * kStreamMaxVecPerThread || tile_bytes % 512)
        return cudaErrorInvalidValue;
    if (n_stages < 2 || n_stages > kStreamMaxStages || (size_t)(n_stages + 2) * tile_bytes > 227 * 1024)
        return cudaErrorInvalidValue;
    return dispatch_dtype_op<true>(dtype, op, cudaErrorInvalidValue, [&](auto dt, auto o) {
        return launch_stream_t<decltype(dt)::value, decltype(o)::value>(a, tile_bytes, n_stages, stream);
    });
}

}  // namespace rar
