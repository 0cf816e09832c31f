// fused_bulk.cu -- engine (a) with bulk-copy (TMA) staging in shared memory.
//
// Same arithmetic as the register path in fused_impl.cuh: every element of
// chunk c is x_c (+) x_(c+1) (+) ... (+) x_(c+p-1) in the ring's hop order
// ("Ring All-Reduce, in depth", "The schedule" and "Tracing four GPUs"),
// then the avg scaling, then the all-gather's copy to every rank.  Here the
// data moves by the bulk-copy engine instead of per-thread loads:
//   - the buffer is cut into tiles of `tile_bytes` per rank; a persistent CTA
//     owns tiles blockIdx.x, blockIdx.x + gridDim.x, ...;
//   - one thread issues, for a tile, p cp.async.bulk loads (one contiguous
//     tile_bytes run from each rank buffer) into one stage of a 3-stage
//     shared-memory ring, completing on that stage's mbarrier;
//   - all threads fold the tile out of shared memory into a result row (a
//     chunk boundary inside a tile only changes the row order per vector or
//     per element, so vector lanes never mix two chunks' orders);
//   - one thread issues p cp.async.bulk stores of the result row, one per
//     rank buffer.
// HBM traffic is the minimum 2 p n e; loads for later tiles are in flight
// while a tile is folded.
//
// Every mbarrier wait is bounded.  A wait that runs out records RAR_ETIMEOUT
// in the status word, then the issuing thread waits (bounded again) for the
// loads it still has in flight and for its stores, and the CTA returns.
#include "fused_impl.cuh"

namespace rar {

constexpr int kBulkThreads = 256;
constexpr int kBulkStages = 3;

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void bulk_store(void *dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_reads_leave_2() {
    asm volatile("cp.async.bulk.wait_group.read 2;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ unsigned long long bulk_global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for one mbarrier phase: true once complete, false if the
// time or iteration budget ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, unsigned long long timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = bulk_global_ns();
    const unsigned long long max_iters = timeout_ns / 16ull + (1ull << 20);
    for (unsigned long long it = 0; it < max_iters; it++) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255) == 0 && bulk_global_ns() - t0 > timeout_ns) return false;
    }
    return false;
}

template <int DT, int OP>
__device__ __forceinline__ uint32_t lane_hop(uint32_t acc, uint32_t own) {
    return hop_word<DT, OP == OP_AVG ? OP_SUM : OP>(acc, own);
}

template <int DT, int OP>
__global__ void __launch_bounds__(kBulkThreads) fused_bulk_kernel(const __grid_constant__ FusedArgs a, int tile_bytes) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_fail;
    constexpr int EB = ElemInfo<DT>::bytes;
    constexpr int VE = 16 / EB;
    constexpr int hop_op = OP == OP_AVG ? OP_SUM : OP;
    const int p = a.p;
    const int TB = tile_bytes;
    const long long n = a.n;
    const long long bulk_bytes = (n * EB) & ~15ll;  // the bulk copies' part; the rest is the tail
    const long long ntiles = (bulk_bytes + TB - 1) / TB;
    const long long base = n / p, extra = n % p;
    const size_t stage_bytes = (size_t)(p + 1) * TB;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kBulkStages * stage_bytes);
    const long long my_tiles = ntiles > blockIdx.x ? (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kBulkStages; s++) mbar_init(smem_addr(&bars[s]), 1);
        fence_mbar_init();
        s_fail = 0;
    }
    __syncthreads();

    auto tile_off = [&](long long k) { return ((long long)blockIdx.x + k * gridDim.x) * TB; };
    auto tile_len = [&](long long k) {
        const long long off = tile_off(k);
        return (uint32_t)(bulk_bytes - off < TB ? bulk_bytes - off : TB);
    };
    auto issue = [&](long long k) {  // thread 0: the p loads of this CTA's k-th tile
        const int s = (int)(k % kBulkStages);
        const long long off = tile_off(k);
        const uint32_t bytes = tile_len(k);
        unsigned char *st = smem + (size_t)s * stage_bytes;
        const uint32_t bar = smem_addr(&bars[s]);
        mbar_arrive_expect_tx(bar, bytes * (uint32_t)p);
        for (int r = 0; r < p; r++) bulk_load(smem_addr(st + (size_t)r * TB), rank_ptr(a.bufs, p, r) + off, bytes, bar);
    };

    long long issued = 0;
    if (threadIdx.x == 0)
        for (; issued < my_tiles && issued < kBulkStages - 1; issued++) issue(issued);

    long long k = 0;
    for (; k < my_tiles; k++) {
        const int s = (int)(k % kBulkStages);
        const uint32_t parity = (uint32_t)((k / kBulkStages) & 1);
        if (threadIdx.x == 0) {
            if (issued < my_tiles) {
                // the stage being refilled was read by the fold of tile k - 1
                fence_proxy_async_smem();
                issue(issued);
                issued++;
            }
            // the stores that read this stage's result row (tile k - 3) are done
            bulk_wait_reads_leave_2();
        }
        if (!mbar_wait_bounded(smem_addr(&bars[s]), parity, a.timeout_ns)) s_fail = 1;
        __syncthreads();
        if (s_fail) break;

        const unsigned char *st = smem + (size_t)s * stage_bytes;
        unsigned char *res = smem + (size_t)s * stage_bytes + (size_t)p * TB;
        const long long off = tile_off(k);
        const uint32_t bytes = tile_len(k);
        const int nvec = (int)(bytes / 16);
        const long long e0 = off / EB;
        const int cfirst = chunk_of(e0, base, extra);
        const int clast = chunk_of(e0 + bytes / EB - 1, base, extra);
        for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
            const long long i0 = e0 + (long long)v * VE;
            int c = cfirst;
            bool uniform = cfirst == clast;
            if (!uniform) {
                c = chunk_of(i0, base, extra);
                uniform = chunk_of(i0 + VE - 1, base, extra) == c;
            }
            if (uniform) {
                uint4 acc = *reinterpret_cast<const uint4 *>(st + (size_t)c * TB + (size_t)v * 16);
                int r = c;
#pragma unroll 4
                for (int kk = 1; kk < p; kk++) {
                    r = (r + 1 == p) ? 0 : r + 1;
                    acc = hop_vec<DT, hop_op>(acc, *reinterpret_cast<const uint4 *>(st + (size_t)r * TB + (size_t)v * 16));
                }
                if constexpr (OP == OP_AVG) acc = scale_vec<DT>(acc, a.inv_p);
                *reinterpret_cast<uint4 *>(res + (size_t)v * 16) = acc;
            } else {
                for (int l = 0; l < VE; l++) {
                    const int cl = chunk_of(i0 + l, base, extra);
                    const size_t lo = (size_t)v * 16 + (size_t)l * EB;
                    auto lane = [&](int row) -> uint32_t {
                        if constexpr (EB == 4) return *reinterpret_cast<const uint32_t *>(st + (size_t)row * TB + lo);
                        else return (uint32_t)*reinterpret_cast<const uint16_t *>(st + (size_t)row * TB + lo);
                    };
                    uint32_t acc = lane(cl);
                    int r = cl;
                    for (int kk = 1; kk < p; kk++) {
                        r = (r + 1 == p) ? 0 : r + 1;
                        acc = lane_hop<DT, OP>(acc, lane(r));
                    }
                    if constexpr (OP == OP_AVG) acc = scale_word<DT>(acc, a.inv_p);
                    if constexpr (EB == 4) *reinterpret_cast<uint32_t *>(res + lo) = acc;
                    else *reinterpret_cast<uint16_t *>(res + lo) = (uint16_t)acc;
                }
            }
        }
        fence_proxy_async_smem();  // result row visible to the bulk-copy engine
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int r = 0; r < p; r++) bulk_store(rank_ptr(a.bufs, p, r) + off, smem_addr(res), bytes);
            bulk_commit();
        }
    }

    if (s_fail) {
        if (threadIdx.x == 0) {
            unsigned prev = atomicMax(&a.status->epoch, a.epoch);
            if (prev < a.epoch) {
                a.status->code = RAR_ETIMEOUT;
                a.status->rank = -1;
                a.status->step = -1;
                a.status->slice = (int)(blockIdx.x + k * gridDim.x);
                a.status->waited_on = -1;
                a.status->flag_seen = 0;
                a.status->flag_wanted = 0;
                __threadfence();
            }
            // loads still in flight land in this CTA's shared memory: wait for
            // them (bounded) before the CTA gives its shared memory up
            for (long long j = k; j < issued; j++) {
                const int s = (int)(j % kBulkStages);
                mbar_wait_bounded(smem_addr(&bars[s]), (uint32_t)((j / kBulkStages) & 1), a.timeout_ns);
            }
            bulk_wait_all();
        }
        return;
    }

    // the ragged tail (< 16 bytes of each rank buffer): per element, global
    // memory, by one thread of the last CTA
    if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) {
        for (long long i = bulk_bytes / EB; i < n; i++) fused_fold_element<DT, OP>(a, p, chunk_of(i, base, extra), i);
    }
    if (threadIdx.x == 0) bulk_wait_all();  // stores finished reading shared memory
}

template <int DT, int OP>
static cudaError_t launch_bulk_t(const FusedArgs &a, int tile_bytes, int grid_cap, cudaStream_t stream, int *out_grid) {
    auto kernel = fused_bulk_kernel<DT, OP>;
    const size_t smem = (size_t)kBulkStages * (size_t)(a.p + 1) * tile_bytes + kBulkStages * sizeof(uint64_t);
    static int configured_smem[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if ((size_t)configured_smem[dev] < smem) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured_smem[dev] = (int)smem;
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kBulkThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long bulk_bytes = (a.n * ElemInfo<DT>::bytes) & ~15ll;
    const long long ntiles = (bulk_bytes + tile_bytes - 1) / tile_bytes;
    long long grid = (long long)sms * per_sm;
    if (grid_cap > 0 && grid > grid_cap) grid = grid_cap;
    if (grid > ntiles) grid = ntiles;
    if (grid < 1) grid = 1;
    if (out_grid) *out_grid = (int)grid;
    kernel<<<(unsigned)grid, kBulkThreads, smem, stream>>>(a, tile_bytes);
    return cudaGetLastError();
}

// Tile size per rank: the largest power of two in [512, 8192] bytes whose
// three stages of p + 1 rows fit in about 110 KB (two CTAs per SM), else in
// about 220 KB (one CTA per SM); 0 if even 512 does not fit.
int fused_bulk_tile_bytes(int p) {
    for (const long long budget : {110ll * 1024, 220ll * 1024}) {
        for (int tb = 8192; tb >= 512; tb /= 2) {
            if ((long long)kBulkStages * (p + 1) * tb + 64 <= budget && (long long)p * tb < (1ll << 20)) {
                if (budget == 110ll * 1024 && tb < 2048) break;
                return tb;
            }
        }
    }
    return 0;
}

cudaError_t launch_fused_bulk(const FusedArgs &a, int dtype, int op, int tile_bytes, int grid_cap, cudaStream_t stream) {
    int grid = 0;
    switch (dtype) {
    case DT_I32:
        if (op == OP_SUM) return launch_bulk_t<DT_I32, OP_SUM>(a, tile_bytes, grid_cap, stream, &grid);
        if (op == OP_MAX) return launch_bulk_t<DT_I32, OP_MAX>(a, tile_bytes, grid_cap, stream, &grid);
        break;
    case DT_F32:
        if (op == OP_SUM) return launch_bulk_t<DT_F32, OP_SUM>(a, tile_bytes, grid_cap, stream, &grid);
        if (op == OP_MAX) return launch_bulk_t<DT_F32, OP_MAX>(a, tile_bytes, grid_cap, stream, &grid);
        if (op == OP_AVG) return launch_bulk_t<DT_F32, OP_AVG>(a, tile_bytes, grid_cap, stream, &grid);
        break;
    case DT_BF16:
        if (op == OP_SUM) return launch_bulk_t<DT_BF16, OP_SUM>(a, tile_bytes, grid_cap, stream, &grid);
        if (op == OP_MAX) return launch_bulk_t<DT_BF16, OP_MAX>(a, tile_bytes, grid_cap, stream, &grid);
        if (op == OP_AVG) return launch_bulk_t<DT_BF16, OP_AVG>(a, tile_bytes, grid_cap, stream, &grid);
        break;
    case DT_F16:
        if (op == OP_SUM) return launch_bulk_t<DT_F16, OP_SUM>(a, tile_bytes, grid_cap, stream, &grid);
        if (op == OP_MAX) return launch_bulk_t<DT_F16, OP_MAX>(a, tile_bytes, grid_cap, stream, &grid);
        if (op == OP_AVG) return launch_bulk_t<DT_F16, OP_AVG>(a, tile_bytes, grid_cap, stream, &grid);
        break;
    }
    return cudaErrorInvalidValue;
}

}  // namespace rar
