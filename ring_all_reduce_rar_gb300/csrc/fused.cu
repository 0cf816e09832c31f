// fused.cu -- instantiation and dispatch of the fused engines (ring order
// and tree order) for every dtype and op.
#include "fused_impl.cuh"

namespace rar {

cudaError_t launch_fused(const FusedArgs &a, int dtype, int op, bool tree, bool vec16, int threads,
                         cudaStream_t stream) {
    return dispatch_dtype_op<true>(dtype, op, cudaErrorInvalidValue, [&](auto dt, auto o) {
        return launch_fused_op<decltype(dt)::value, decltype(o)::value>(a, tree, vec16, threads, stream);
    });
}

template <typename K>
static cudaError_t launch_hier_grid(K kernel, const FusedArgs &a, int g, long long work, int threads,
                                    cudaStream_t stream) {
    long long grid = (long long)sm_count_cached() * blocks_per_sm_of(kernel, threads);
    const long long want = (work + threads - 1) / threads;
    if (grid > want) grid = want;
    if (grid < 1) grid = 1;
    cudaError_t e = launch_pdl(kernel, dim3((unsigned)grid), dim3((unsigned)threads), 0, stream, a, g);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int DT, int OP, int P>
static cudaError_t launch_hier_p(const FusedArgs &a, int g, bool vec16, int threads, cudaStream_t stream) {
    constexpr int VE = 16 / ElemInfo<DT>::bytes;
    if constexpr (P > 0) {
        if (vec16) return launch_hier_grid(fused_hier_kernel_p<DT, OP, P, true>, a, g, (a.n + VE - 1) / VE, threads, stream);
        return launch_hier_grid(fused_hier_kernel_p<DT, OP, P, false>, a, g, a.n, threads, stream);
    } else {
        if (vec16) return launch_hier_grid(fused_hier_kernel<DT, OP, true>, a, g, (a.n + VE - 1) / VE, threads, stream);
        return launch_hier_grid(fused_hier_kernel<DT, OP, false>, a, g, a.n, threads, stream);
    }
}

template <int DT, int OP>
static cudaError_t launch_hier_t(const FusedArgs &a, int g, bool vec16, int threads, cudaStream_t stream) {
    switch (a.p) {
    case 4: return launch_hier_p<DT, OP, 4>(a, g, vec16, threads, stream);
    case 8: return launch_hier_p<DT, OP, 8>(a, g, vec16, threads, stream);
    case 16: return launch_hier_p<DT, OP, 16>(a, g, vec16, threads, stream);
    default: return launch_hier_p<DT, OP, 0>(a, g, vec16, threads, stream);
    }
}

cudaError_t launch_fused_hier(const FusedArgs &a, int dtype, int op, int g, bool vec16, int threads,
                              cudaStream_t stream) {
    return dispatch_dtype_op<true>(dtype, op, cudaErrorInvalidValue, [&](auto dt, auto o) {
        return launch_hier_t<decltype(dt)::value, decltype(o)::value>(a, g, vec16, threads, stream);
    });
}

}  // namespace rar
