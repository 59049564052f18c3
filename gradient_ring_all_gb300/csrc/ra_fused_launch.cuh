// ra_fused_launch.cuh -- host-side launch of the fused kernel for one
// element type (included by ra_fused_f32.cu and ra_fused_bf16.cu so the two
// instantiation sets compile in parallel).
#pragma once

#include <string.h>

#include "ra_kernels.cuh"

namespace ra {

template <class E, int NT, int OUT, bool VEC, int MAXSEG>
static cudaError_t fused_launch_one(const FusedLaunch &L, int64_t ntiles, cudaStream_t s) {
    FusedParams<MAXSEG> p;
    memset(&p, 0, sizeof(p));
    for (int k = 0; k < L.n; ++k) {
        p.rows[k] = L.rows[k];
        p.aux[k] = L.aux[k];
    }
    p.w = L.w;
    p.lr = L.lr;
    p.n = L.n;
    p.nseg = L.nseg;
    p.mis = L.mis;
    p.ntiles = ntiles;
    for (int k = 0; k < L.nseg; ++k) p.seg[k] = L.seg[k];
    // One tile per block.  The block scheduler hands out blocks in index
    // order, so the tiles in flight form one contiguous address window that
    // slides through the arrays; that keeps DRAM pages open far better than
    // a persistent grid whose blocks drift apart (measured on GB300: 7.09 vs
    // 6.28 TB/s at N=8, P=300M f32).  The kernel's tile loop only matters
    // past 2^31-1 tiles.
    const int64_t grid = ntiles < kMaxGrid ? ntiles : kMaxGrid;
    fused_allreduce_kernel<E, NT, OUT, VEC, MAXSEG><<<(unsigned)grid, kThreadsPerBlock, 0, s>>>(p);
    return cudaGetLastError();
}

template <class E, int NT>
static cudaError_t fused_launch_nt(const FusedLaunch &L, int64_t ntiles, cudaStream_t s) {
    const bool big = L.nseg > kSegSmall;
    if (L.out != kOutAll && big) return cudaErrorInvalidValue;  // SGD / reduce-scatter use n segments
    if (L.out == kOutAllWire) {
        if constexpr (sizeof(typename E::T) == 2) {
            if (L.vector) return fused_launch_one<E, NT, kOutAllWire, true, kSegSmall>(L, ntiles, s);
            return fused_launch_one<E, 0, kOutAllWire, false, kSegSmall>(L, ntiles, s);
        } else {
            return cudaErrorInvalidValue;  // bf16 arrays only
        }
    }
    if (L.vector) {
        if (L.out == kOutAllSgd) return fused_launch_one<E, NT, kOutAllSgd, true, kSegSmall>(L, ntiles, s);
        if (L.out == kOutOne) return fused_launch_one<E, NT, kOutOne, true, kSegSmall>(L, ntiles, s);
        if (big) return fused_launch_one<E, NT, kOutAll, true, kSegLarge>(L, ntiles, s);
        return fused_launch_one<E, NT, kOutAll, true, kSegSmall>(L, ntiles, s);
    }
    // scalar path: generic worker count only
    if (L.out == kOutAllSgd) return fused_launch_one<E, 0, kOutAllSgd, false, kSegSmall>(L, ntiles, s);
    if (L.out == kOutOne) return fused_launch_one<E, 0, kOutOne, false, kSegSmall>(L, ntiles, s);
    if (big) return fused_launch_one<E, 0, kOutAll, false, kSegLarge>(L, ntiles, s);
    return fused_launch_one<E, 0, kOutAll, false, kSegSmall>(L, ntiles, s);
}

template <class E>
static cudaError_t fused_launch_dtype(const FusedLaunch &L, int64_t ntiles, cudaStream_t s) {
    switch (L.vector ? fused_compile_time_n(L.n) : 0) {
        case 2: return fused_launch_nt<E, 2>(L, ntiles, s);
        case 4: return fused_launch_nt<E, 4>(L, ntiles, s);
        case 8: return fused_launch_nt<E, 8>(L, ntiles, s);
        case 16: return fused_launch_nt<E, 16>(L, ntiles, s);
        case 32: return fused_launch_nt<E, 32>(L, ntiles, s);
        default: return fused_launch_nt<E, 0>(L, ntiles, s);
    }
}

}  // namespace ra
