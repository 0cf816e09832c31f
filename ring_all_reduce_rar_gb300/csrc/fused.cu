// fused.cu -- instantiation and dispatch of the fused engines (ring order
// and tree order) for every dtype and op.
#include "fused_impl.cuh"

namespace rar {

cudaError_t launch_fused(const FusedArgs &a, int dtype, int op, bool tree, bool vec16, int threads,
                         cudaStream_t stream) {
    switch (dtype) {
    case DT_I32:
        if (op == OP_SUM) return launch_fused_op<DT_I32, OP_SUM>(a, tree, vec16, threads, stream);
        if (op == OP_MAX) return launch_fused_op<DT_I32, OP_MAX>(a, tree, vec16, threads, stream);
        break;
    case DT_F32:
        if (op == OP_SUM) return launch_fused_op<DT_F32, OP_SUM>(a, tree, vec16, threads, stream);
        if (op == OP_MAX) return launch_fused_op<DT_F32, OP_MAX>(a, tree, vec16, threads, stream);
        if (op == OP_AVG) return launch_fused_op<DT_F32, OP_AVG>(a, tree, vec16, threads, stream);
        if (op == OP_AVG_PREDIV) return launch_fused_op<DT_F32, OP_AVG_PREDIV>(a, tree, vec16, threads, stream);
        break;
    case DT_BF16:
        if (op == OP_SUM) return launch_fused_op<DT_BF16, OP_SUM>(a, tree, vec16, threads, stream);
        if (op == OP_MAX) return launch_fused_op<DT_BF16, OP_MAX>(a, tree, vec16, threads, stream);
        if (op == OP_AVG) return launch_fused_op<DT_BF16, OP_AVG>(a, tree, vec16, threads, stream);
        if (op == OP_AVG_PREDIV) return launch_fused_op<DT_BF16, OP_AVG_PREDIV>(a, tree, vec16, threads, stream);
        break;
    case DT_F16:
        if (op == OP_SUM) return launch_fused_op<DT_F16, OP_SUM>(a, tree, vec16, threads, stream);
        if (op == OP_MAX) return launch_fused_op<DT_F16, OP_MAX>(a, tree, vec16, threads, stream);
        if (op == OP_AVG) return launch_fused_op<DT_F16, OP_AVG>(a, tree, vec16, threads, stream);
        if (op == OP_AVG_PREDIV) return launch_fused_op<DT_F16, OP_AVG_PREDIV>(a, tree, vec16, threads, stream);
        break;
    }
    return cudaErrorInvalidValue;
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
    switch (dtype) {
    case DT_I32:
        if (op == OP_SUM) return launch_hier_t<DT_I32, OP_SUM>(a, g, vec16, threads, stream);
        if (op == OP_MAX) return launch_hier_t<DT_I32, OP_MAX>(a, g, vec16, threads, stream);
        break;
    case DT_F32:
        if (op == OP_SUM) return launch_hier_t<DT_F32, OP_SUM>(a, g, vec16, threads, stream);
        if (op == OP_MAX) return launch_hier_t<DT_F32, OP_MAX>(a, g, vec16, threads, stream);
        if (op == OP_AVG) return launch_hier_t<DT_F32, OP_AVG>(a, g, vec16, threads, stream);
        if (op == OP_AVG_PREDIV) return launch_hier_t<DT_F32, OP_AVG_PREDIV>(a, g, vec16, threads, stream);
        break;
    case DT_BF16:
        if (op == OP_SUM) return launch_hier_t<DT_BF16, OP_SUM>(a, g, vec16, threads, stream);
        if (op == OP_MAX) return launch_hier_t<DT_BF16, OP_MAX>(a, g, vec16, threads, stream);
        if (op == OP_AVG) return launch_hier_t<DT_BF16, OP_AVG>(a, g, vec16, threads, stream);
        if (op == OP_AVG_PREDIV) return launch_hier_t<DT_BF16, OP_AVG_PREDIV>(a, g, vec16, threads, stream);
        break;
    case DT_F16:
        if (op == OP_SUM) return launch_hier_t<DT_F16, OP_SUM>(a, g, vec16, threads, stream);
        if (op == OP_MAX) return launch_hier_t<DT_F16, OP_MAX>(a, g, vec16, threads, stream);
        if (op == OP_AVG) return launch_hier_t<DT_F16, OP_AVG>(a, g, vec16, threads, stream);
        if (op == OP_AVG_PREDIV) return launch_hier_t<DT_F16, OP_AVG_PREDIV>(a, g, vec16, threads, stream);
        break;
    }
    return cudaErrorInvalidValue;
}

}  // namespace rar
