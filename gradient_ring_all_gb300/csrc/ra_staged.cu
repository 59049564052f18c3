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
    p.msg_lo = L.msg_lo;
    p.msg_hi = L.msg_hi;
    p.err = L.err;
    p.p = L.p;
    p.n = L.n;
    p.t = t;
    p.op = op;
    p.mis = L.mis;
    p.nseg = L.nseg;
    p.ntiles = L.ntiles;
    for (int k = 0; k < L.nseg; ++k) p.seg[k] = L.seg[k];
    // one tile per block, as for the fused kernel
    const int64_t grid = L.ntiles < kMaxGrid ? L.ntiles : kMaxGrid;
    if (VEC && L.tile_vec == kStagedTileVecLarge)
        return launch_pdl(staged_step_kernel<E, VEC, kStagedTileVecLarge>, grid, kThreadsPerBlock, 0, s, p);
    return launch_pdl(staged_step_kernel<E, VEC, kStagedTileVecSmall>, grid, kThreadsPerBlock, 0, s, p);
}

cudaError_t launch_staged_step(const StagedLaunch &L, int op, int t, cudaStream_t s) {
    if (L.nseg > RA_MAX_N) return cudaErrorInvalidValue;
    if (L.dtype == RA_F32)
        return L.vector ? staged_launch_one<F32, true>(L, op, t, s) : staged_launch_one<F32, false>(L, op, t, s);
    return L.vector ? staged_launch_one<BF16, true>(L, op, t, s) : staged_launch_one<BF16, false>(L, op, t, s);
}

template <class E>
static cudaError_t gather_scalar_launch(const GatherLaunch &L, cudaStream_t s) {
    GatherParams p;
    memset(&p, 0, sizeof(p));
    for (int k = 0; k < L.n; ++k) {
        p.rows[k] = L.rows[k];
        p.src[k] = L.src[k];
    }
    p.n = L.n;
    p.nseg = L.nseg;
    p.mis = L.mis;
    p.skip_owner = L.skip_owner ? 1 : 0;
    p.err = L.err;
    p.p = L.p;
    p.ntiles = L.ntiles;
    for (int k = 0; k < L.nseg; ++k) p.seg[k] = L.seg[k];
    const int64_t grid = L.ntiles < kMaxGrid ? L.ntiles : kMaxGrid;
    return launch_pdl(all_gather_scalar_kernel<E>, grid, kThreadsPerBlock, 0, s, p);
}

template <class E>
static cudaError_t gather_tma_launch(const GatherLaunch &L, cudaStream_t s) {
    GatherParams p;
    memset(&p, 0, sizeof(p));
    for (int k = 0; k < L.n; ++k) {
        p.rows[k] = L.rows[k];
        p.src[k] = L.src[k];
    }
    p.n = L.n;
    p.nseg = L.nseg;
    p.mis = L.mis;
    p.skip_owner = L.skip_owner ? 1 : 0;
    p.err = L.err;
    p.p = L.p;
    p.ntiles = L.ntiles;
    for (int k = 0; k < L.nseg; ++k) p.seg[k] = L.seg[k];
    const size_t smem = (size_t)kGatherTileBytes + 16;
    if (smem > 48 * 1024) {
        static unsigned long long opted_in = 0;  // bit per device
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 64 && !(__atomic_load_n(&opted_in, __ATOMIC_ACQUIRE) & (1ull << dev))) {
            e = cudaFuncSetAttribute(all_gather_tma_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            __atomic_fetch_or(&opted_in, 1ull << dev, __ATOMIC_ACQ_REL);
        }
    }
    const int64_t grid = L.ntiles < kMaxGrid ? L.ntiles : kMaxGrid;
    return launch_pdl(all_gather_tma_kernel<E>, grid, 32, smem, s, p, kGatherTileBytes);
}

cudaError_t launch_all_gather(const GatherLaunch &L, cudaStream_t s) {
    if (L.nseg > RA_MAX_N) return cudaErrorInvalidValue;
    if (L.vector) return L.dtype == RA_F32 ? gather_tma_launch<F32>(L, s) : gather_tma_launch<BF16>(L, s);
    return L.dtype == RA_F32 ? gather_scalar_launch<F32>(L, s) : gather_scalar_launch<BF16>(L, s);
}

}  // namespace ra
