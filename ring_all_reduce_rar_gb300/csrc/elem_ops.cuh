// elem_ops.cuh -- one hop of the reduction and the avg epilogue, on 32-bit
// words (one int32/float32 element, or two bfloat16/float16 elements).
//
// A hop combines the running value arriving from the left neighbour (acc)
// with the receiver's own element (own), rounded to the dtype ("Ring
// All-Reduce, in depth", "The schedule": the receiver adds the chunk into its
// own copy; "Derive the cost of a ring all-reduce", last probe: in the
// buffer's dtype).  max keeps acc unless own is strictly greater.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <type_traits>
#include <utility>

#include "rar_internal.h"

namespace rar {

template <int V>
using IntC = std::integral_constant<int, V>;

// Runtime (dtype, op) to a kernel instantiation: calls
// f(IntC<dtype>{}, IntC<op>{}) for every pair the library offers -- sum and
// max on every dtype, avg on the floating types, avg_prediv on the floating
// types where kPrediv -- and returns `none` for any other pair.
template <bool kPrediv, typename R, typename F>
R dispatch_dtype_op(int dtype, int op, R none, F &&f) {
    auto floating = [&](auto dt) -> R {
        if (op == OP_SUM) return f(dt, IntC<OP_SUM>{});
        if (op == OP_MAX) return f(dt, IntC<OP_MAX>{});
        if (op == OP_AVG) return f(dt, IntC<OP_AVG>{});
        if constexpr (kPrediv) {
            if (op == OP_AVG_PREDIV) return f(dt, IntC<OP_AVG_PREDIV>{});
        }
        return none;
    };
    switch (dtype) {
    case DT_I32:
        if (op == OP_SUM) return f(IntC<DT_I32>{}, IntC<OP_SUM>{});
        if (op == OP_MAX) return f(IntC<DT_I32>{}, IntC<OP_MAX>{});
        return none;
    case DT_F32: return floating(IntC<DT_F32>{});
    case DT_BF16: return floating(IntC<DT_BF16>{});
    case DT_F16: return floating(IntC<DT_F16>{});
    }
    return none;
}

template <int DT> struct ElemInfo;
template <> struct ElemInfo<DT_I32> { static constexpr int bytes = 4; };
template <> struct ElemInfo<DT_F32> { static constexpr int bytes = 4; };
template <> struct ElemInfo<DT_BF16> { static constexpr int bytes = 2; };
template <> struct ElemInfo<DT_F16> { static constexpr int bytes = 2; };

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h16) { return __uint_as_float(h16 << 16); }
__device__ __forceinline__ uint32_t float_to_bf16_bits(float f) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ float f16_bits_to_float(uint32_t h16) {
    return __half2float(__ushort_as_half((unsigned short)h16));
}
__device__ __forceinline__ uint32_t float_to_f16_bits(float f) {
    return (uint32_t)__half_as_ushort(__float2half_rn(f));
}

// max on one 16-bit lane (bits in the low half): keep acc unless own > acc.
template <int DT>
__device__ __forceinline__ uint32_t max_lane16(uint32_t acc, uint32_t own) {
    float a = DT == DT_BF16 ? bf16_bits_to_float(acc) : f16_bits_to_float(acc);
    float b = DT == DT_BF16 ? bf16_bits_to_float(own) : f16_bits_to_float(own);
    return (b > a) ? own : acc;
}

template <int DT, int OP>
__device__ __forceinline__ uint32_t hop_word(uint32_t acc, uint32_t own) {
    constexpr bool is_max = OP == OP_MAX;
    if constexpr (DT == DT_I32) {
        if constexpr (is_max) return ((int32_t)own > (int32_t)acc) ? own : acc;
        else return acc + own;  // wraps modulo 2^32
    } else if constexpr (DT == DT_F32) {
        float a = __uint_as_float(acc), b = __uint_as_float(own);
        if constexpr (is_max) return (b > a) ? own : acc;
        else return __float_as_uint(__fadd_rn(a, b));
    } else if constexpr (DT == DT_BF16) {
        if constexpr (is_max) {
            uint32_t lo = max_lane16<DT>(acc & 0xFFFFu, own & 0xFFFFu);
            uint32_t hi = max_lane16<DT>(acc >> 16, own >> 16);
            return lo | (hi << 16);
        } else {
            // correctly rounded bf16 addition on both lanes
            __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162 *>(&acc);
            __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162 *>(&own);
            __nv_bfloat162 r = __hadd2(a, b);
            return *reinterpret_cast<uint32_t *>(&r);
        }
    } else {
        if constexpr (is_max) {
            uint32_t lo = max_lane16<DT>(acc & 0xFFFFu, own & 0xFFFFu);
            uint32_t hi = max_lane16<DT>(acc >> 16, own >> 16);
            return lo | (hi << 16);
        } else {
            __half2 a = *reinterpret_cast<__half2 *>(&acc);
            __half2 b = *reinterpret_cast<__half2 *>(&own);
            __half2 r = __hadd2(a, b);
            return *reinterpret_cast<uint32_t *>(&r);
        }
    }
}

// avg epilogue: x * (1/p) in binary32, rounded once, then to the 16-bit type
// (both lanes of a word converted by one paired round-to-nearest).
template <int DT>
__device__ __forceinline__ uint32_t scale_word(uint32_t w, float inv_p) {
    if constexpr (DT == DT_F32) {
        return __float_as_uint(__fmul_rn(__uint_as_float(w), inv_p));
    } else if constexpr (DT == DT_BF16) {
        const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xFFFF0000u);
        __nv_bfloat162 r = __floats2bfloat162_rn(__fmul_rn(lo, inv_p), __fmul_rn(hi, inv_p));
        return *reinterpret_cast<uint32_t *>(&r);
    } else if constexpr (DT == DT_F16) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w));
        __half2 r = __floats2half2_rn(__fmul_rn(f.x, inv_p), __fmul_rn(f.y, inv_p));
        return *reinterpret_cast<uint32_t *>(&r);
    } else {
        return w;
    }
}

// A rank's contribution as it enters the fold: unchanged, or (pre-divided
// average) times 1/p rounded to the dtype.
template <int DT, int OP>
__device__ __forceinline__ uint32_t contrib_word(uint32_t w, float inv_p) {
    if constexpr (OP == OP_AVG_PREDIV) return scale_word<DT>(w, inv_p);
    else return w;
}

template <int DT, int OP>
__device__ __forceinline__ uint4 hop_vec(uint4 acc, uint4 own) {
    acc.x = hop_word<DT, OP>(acc.x, own.x);
    acc.y = hop_word<DT, OP>(acc.y, own.y);
    acc.z = hop_word<DT, OP>(acc.z, own.z);
    acc.w = hop_word<DT, OP>(acc.w, own.w);
    return acc;
}

template <int DT>
__device__ __forceinline__ uint4 scale_vec(uint4 v, float inv_p) {
    v.x = scale_word<DT>(v.x, inv_p);
    v.y = scale_word<DT>(v.y, inv_p);
    v.z = scale_word<DT>(v.z, inv_p);
    v.w = scale_word<DT>(v.w, inv_p);
    return v;
}

template <int DT, int OP>
__device__ __forceinline__ uint4 contrib_vec(uint4 v, float inv_p) {
    if constexpr (OP == OP_AVG_PREDIV) return scale_vec<DT>(v, inv_p);
    else return v;
}

// The op a hop applies: both averages add.
template <int OP>
struct HopOf { static constexpr int value = (OP == OP_AVG || OP == OP_AVG_PREDIV) ? OP_SUM : OP; };

// Single elements (16-bit types use the low half of the word).
template <int DT>
__device__ __forceinline__ uint32_t load_elem(const char *base, long long i) {
    if constexpr (ElemInfo<DT>::bytes == 4) return __ldcg(reinterpret_cast<const unsigned int *>(base) + i);
    else return (uint32_t)__ldcg(reinterpret_cast<const unsigned short *>(base) + i);
}
template <int DT>
__device__ __forceinline__ void store_elem(char *base, long long i, uint32_t w) {
    if constexpr (ElemInfo<DT>::bytes == 4) reinterpret_cast<unsigned int *>(base)[i] = w;
    else reinterpret_cast<unsigned short *>(base)[i] = (unsigned short)w;
}

// Programmatic dependent launch.  A fused kernel is launched with
// programmatic stream serialization, so it may be scheduled while the
// previous kernel of the stream finishes; pdl_wait() then blocks until that
// kernel has completed and its memory is visible (a no-op when the previous
// operation was not a kernel), and must come before any access to the rank
// buffers.  pdl_launch_dependents() lets the next such kernel be scheduled
// once every CTA of this grid has run it; all of this grid's CTAs are then
// resident, so the waiting CTAs of the next grid cannot hold them back.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch `kernel` with programmatic stream serialization (see pdl_wait).
template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ char *rank_ptr(const RankPtrs &b, int p, int r) {
    return static_cast<char *>(p <= kInlineP ? b.inl[r] : b.table[r]);
}

// chunk_bounds ("Ring All-Reduce, in depth", "An implementation"): the first
// `extra` = n mod p chunks hold base + 1 elements, the rest base.
__device__ __forceinline__ int chunk_of(long long i, long long base, long long extra) {
    long long big = extra * (base + 1);
    return (int)(i < big ? i / (base + 1) : extra + (i - big) / base);
}
__device__ __forceinline__ long long chunk_start(int c, long long base, long long extra) {
    return (long long)c * base + (c < extra ? c : extra);
}

}  // namespace rar
