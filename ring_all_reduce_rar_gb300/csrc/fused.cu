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

template <int DT, int OP>
static cudaError_t launch_hier_t(const FusedArgs &a, int g, bool vec16, int threads, cudaStream_t stream) {
    constexpr int VE = 16 / ElemInfo<DT>::bytes;
    const int sms = sm_count_cached();
    const long long work = vec16 ? (a.n + VE - 1) / VE : a.n;
    long long grid = (long long)sms * (vec16 ? blocks_per_sm_of(fused_hier_kernel<DT, OP, true>, threads)
                                            : blocks_per_sm_of(fused_hier_kernel<DT, OP, false>, threads));
    const long long want = (work + threads - 1) / threads;
    if (grid > want) grid = want;
    if (grid < 1) grid = 1;
    if (vec16) fused_hier_kernel<DT, OP, true><<<(unsigned)grid, threads, 0, stream>>>(a, g);
    else fused_hier_kernel<DT, OP, false><<<(unsigned)grid, threads, 0, stream>>>(a, g);
    return cudaGetLastError();
}

cudaError_t launch_fused_hier(const FusedArgs &a, int dtype, int op, int g, bool vec16, int threads,
                              cudaStream_t stream) {
    return dispatch_dtype_op<true>(dtype, op, cudaErrorInvalidValue, [&](auto dt, auto o) {
        return launch_hier_t<decltype(dt)::value, decltype(o)::value>(a, g, vec16, threads, stream);
    });
}

}  // namespace rar
