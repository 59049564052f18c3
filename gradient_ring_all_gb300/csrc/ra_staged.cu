// ra_staged.cu -- launches of the staged kernel, one ring iteration each.
#include <string.h>

#include "ra_kernels.cuh"

namespace ra {

template <class E, bool VEC>
static cudaError_t staged_launch_one(const StagedLaunch &L, int op, int t, cudaStream_t s) {
    StagedParams p;
    memset(&p, 0, sizeof(p));
    for (int k = 0; k < L.n; ++k) p.rows[k] = L.rows[k];
    p.msg = L.msg;
    p.n = L.n;
    p.t = t;
    p.op = op;
    p.mis = L.mis;
    p.nseg = L.nseg;
    p.ntiles = L.ntiles;
    for (int k = 0; k < L.nseg; ++k) p.seg[k] = L.seg[k];
    // one tile per block, as for the fused kernel
    const int64_t grid = L.ntiles < kMaxGrid ? L.ntiles : kMaxGrid;
    staged_step_kernel<E, VEC><<<(unsigned)grid, kThreadsPerBlock, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_staged_step(const StagedLaunch &L, int op, int t, cudaStream_t s) {
    if (L.nseg > RA_MAX_N) return cudaErrorInvalidValue;
    if (L.dtype == RA_F32)
        return L.vector ? staged_launch_one<F32, true>(L, op, t, s) : staged_launch_one<F32, false>(L, op, t, s);
    return L.vector ? staged_launch_one<BF16, true>(L, op, t, s) : staged_launch_one<BF16, false>(L, op, t, s);
}

}  // namespace ra
