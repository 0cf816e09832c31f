// tree_plan.h -- how the tree executor spreads its CTAs over the ranks
// (see tree.cu): which levels a rank takes part in and where its CTAs
// start.  Plain integer functions, used by the kernel and by the host; they
// also compile as ordinary C++ (the host test of the closed forms).
#pragma once

#ifndef __CUDACC__
#define RAR_HD inline
#else
#define RAR_HD __host__ __device__ inline
#endif

namespace rar {

// ceil(log2 p)
RAR_HD int tree_levels(int p) {
    int L = 0;
    while ((1 << L) < p) L++;
    return L;
}
// Reduce levels in which rank r is a parent: l < ctz(r) (all L for the
// root) with r + 2^l < p; they are 0 .. m - 1.
RAR_HD int tree_reduce_levels(int r, int p, int L) {
    int m = 0;
    while (m < L && (r == 0 || ((r >> m) & 1) == 0) && r + (1 << m) < p) m++;
    return m;
}
// w_r: the steps rank r takes part in (its reduce levels, plus one
// broadcast for every rank but the root).
RAR_HD int tree_weight(int r, int p, int L) {
    return tree_reduce_levels(r, p, L) + (r == 0 ? 0 : 1);
}
// First CTA of rank r: scale * (w_0 + ... + w_(r-1)), or r * channels when
// scale is 0.  The sum in closed form: the root's L, one broadcast for each
// of ranks 1 .. r - 1, and per level l the ranks q in [1, r - 1] with
// 2^(l+1) | q and q + 2^l < p.
RAR_HD long long tree_first_cta(int r, int p, int L, int scale, int channels) {
    if (scale <= 0) return (long long)r * channels;
    if (r == 0) return 0;
    long long s = L + (r - 1);
    for (int l = 0; l < L; l++) {
        const long long M = (long long)(r - 1 < p - (1 << l) - 1 ? r - 1 : p - (1 << l) - 1);
        if (M >= 1) s += M >> (l + 1);
    }
    return s * scale;
}

}  // namespace rar
