// flag_sync.cuh -- progress words between CTA groups of one cooperative
// launch (the ring and tree executors): release/acquire at GPU scope,
// bounded waits, and the status word a wait that runs out fills in.
//
// A CTA publishes its progress after each slice with a release store of a
// 64-bit word (epoch << 32) | (items done), counting the items (slice block,
// step, slice) of its processing order; a waiter acquires it.  Epoch-tagged
// words need no reset between calls.
// Every wait is bounded by the call's timeout (globaltimer) and an
// iteration cap; the first CTA to give up records where, raises the abort
// word (which every other wait polls) and returns.  Nothing traps.
#pragma once

#include "elem_ops.cuh"

namespace rar {

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ int mod_p(int v, int p) {
    v %= p;
    return v < 0 ? v + p : v;
}

// Record a timeout and raise the abort word.  The first CTA of the launch
// to give up fills in the details; every give-up bumps the sequence number.
static __device__ void ring_give_up(const RingArgs &a, unsigned epoch, int rank, int step, long long slice, int nb,
                                    unsigned long long seen, unsigned long long wanted) {
    unsigned prev = atomicMax(&a.status->epoch, epoch);
    if (prev < epoch) {
        a.status->code = RAR_ETIMEOUT;
        a.status->rank = rank;
        a.status->step = step;
        a.status->slice = (int)slice;
        a.status->waited_on = nb;
        a.status->flag_seen = seen;
        a.status->flag_wanted = wanted;
        __threadfence();
    }
    atomicAdd(&a.status->seq, 1u);
    atomicMax(a.abort_word, epoch);
}

// Bounded acquire-wait for the neighbour's progress word.  Returns false if
// the wait ran out or another CTA aborted the launch.
static __device__ bool ring_wait(const RingArgs &a, unsigned epoch, const unsigned long long *flag,
                                 unsigned long long target, int rank, int step, long long slice, int nb) {
    unsigned long long v = ld_acquire_u64(flag);
    if (v >= target) return true;
    const unsigned long long t0 = global_ns();
    const unsigned long long max_iters = a.timeout_ns / 16ull + (1ull << 20);
    // spin on the word first (a hand-off usually lands within a few polls),
    // then back off; the abort word and the clock are read every 16th poll
    for (unsigned long long it = 0;; it++) {
        if (it >= 64) __nanosleep(64);
        v = ld_acquire_u64(flag);
        if (v >= target) return true;
        if ((it & 15) == 15) {
            if (ld_relaxed_u32(a.abort_word) == epoch) return false;
            if (it >= max_iters || global_ns() - t0 > a.timeout_ns) {
                ring_give_up(a, epoch, rank, step, slice, nb, v, target);
                return false;
            }
        }
    }
}

// The epoch of this launch: one more than the last finished launch's.  All
// CTAs read the same value (the word only changes once every CTA finished).
__device__ __forceinline__ unsigned launch_epoch_begin(const RingArgs &a) {
    __shared__ unsigned s_epoch;
    if (threadIdx.x == 0) s_epoch = ld_relaxed_u32(a.epoch_word) + 1u;
    __syncthreads();
    return s_epoch;
}

// Every CTA calls this once, on every exit path, with all its threads.  The
// last CTA to finish publishes the epoch for the next launch; on wrap-around
// it first clears every progress word and mailbox word.
__device__ __forceinline__ void launch_epoch_end(const RingArgs &a, unsigned epoch) {
    __shared__ int s_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(a.finish_count, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last) return;
    if (epoch == 0xFFFFFFFFu) {
        for (int i = threadIdx.x; i < a.flag_capacity; i += blockDim.x) a.flags[i] = 0ull;
        for (long long i = threadIdx.x; i < a.mailbox_words; i += blockDim.x) a.mailbox[i] = 0ull;
        // the abort word and the status's first-reporter epoch only grow
        // (atomicMax) within a count: a stale value would abort the launch
        // that reaches it again after the wrap, or hide its timeout details
        if (threadIdx.x == 0) {
            *a.abort_word = 0u;
            a.status->epoch = 0u;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        *a.finish_count = 0u;
        *a.epoch_word = epoch == 0xFFFFFFFFu ? 0u : epoch;
        __threadfence();
    }
}

// Drop dead data from L2 without writing it back (PTX discard.global.L2:
// the line then holds an indeterminate value until it is written again).
// For a slice that the CTA's vector loop has just read, thread t taking the
// vectors vlo + t + m T of [vlo, vhi): warp w read the 32 vectors
// [vlo + 32 w + m T, + 32) for every m, so after __syncwarp, which orders
// the warp's reads before it, the warp may drop any 128-byte line that lies
// wholly in one of its segments -- lane l takes line l % 4 of segment
// m = l / 4 (mod 8).  The caller publishes the slice after this (barrier and
// release store), so a write that waits on that publication is ordered
// after the discard.
__device__ __forceinline__ void discard_read_lines(const uint4 *s4, long long vlo, long long vhi, int T) {
    __syncwarp();
    const int lane = threadIdx.x & 31;
    const uintptr_t end = reinterpret_cast<uintptr_t>(s4 + vhi);
    for (long long s0 = vlo + 32ll * (threadIdx.x >> 5) + (long long)(lane >> 2) * T; s0 < vhi; s0 += 8ll * T) {
        const uintptr_t seg = reinterpret_cast<uintptr_t>(s4 + s0);
        const uintptr_t line = ((seg + 127) & ~(uintptr_t)127) + 128u * (unsigned)(lane & 3);
        const uintptr_t seg_end = seg + 512 < end ? seg + 512 : end;
        if (line + 128 <= seg_end) asm volatile("discard.global.L2 [%0], 128;" ::"l"(line) : "memory");
    }
}

// Step trace (RingArgs::trace): the first warp of a CTA adds the time it
// waited for the neighbour and the time it then spent on the slice to its
// rank's entry for the step.  t0: before the wait, t1: after it.
__device__ __forceinline__ void trace_add(const RingArgs &a, int rank, int step, unsigned long long t0,
                                          unsigned long long t1) {
    const unsigned long long t2 = global_ns();
    unsigned long long *e = a.trace + 2 * ((long long)rank * a.trace_steps + step);
    atomicAdd(e, t2 - t1);      // work
    atomicAdd(e + 1, t1 - t0);  // wait
}

// Injected straggler: pause about `ns` (bounded by the same clock).
static __device__ void ring_delay(unsigned ns) {
    const unsigned long long t0 = global_ns();
    for (int it = 0; it < (1 << 22) && global_ns() - t0 < ns; it++) __nanosleep(256);
}

}  // namespace rar
