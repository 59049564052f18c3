// ra_fused_launch.cuh -- host-side launch of the fused kernel for one
// element type (included by ra_fused_f32.cu and ra_fused_bf16.cu so the two
// instantiation sets compile in parallel).
#pragma once

#include <string.h>

#include "ra_kernels.cuh"

namespace ra {

template <class E, int OUT, int MAXSEG>
static void fill_params(FusedParams<MAXSEG> &p, const FusedLaunch &L, int64_t ntiles) {
    memset(&p, 0, sizeof(p));
    for (int k = 0; k < L.n; ++k) {
        p.rows[k] = L.rows[k];
        p.aux[k] = L.aux[k];
    }
    p.w = L.w;
    p.err = L.err;
    p.lr = L.lr;
    p.n = L.n;
    p.nseg = L.nseg;
    p.mis = L.mis;
    p.p = L.p;
    p.ntiles = ntiles;
    for (int k = 0; k < L.nseg; ++k) p.seg[k] = L.seg[k];
}

// large dynamic shared memory needs an opt-in per kernel and device
template <class K>
static cudaError_t opt_in_smem(K kern, unsigned long long *opted_in) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !(__atomic_load_n(opted_in, __ATOMIC_ACQUIRE) & (1ull << dev))) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynamicSmem);
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(opted_in, 1ull << dev, __ATOMIC_ACQ_REL);
    }
    return cudaSuccess;
}

// rows that disagree modulo 16 bytes: the TMA kernel with widened copies
template <class E, int OUT, int MAXSEG>
static cudaError_t fused_unaligned_launch_one(const FusedLaunch &L, int64_t ntiles, cudaStream_t s) {
    auto kern = fused_tma_unaligned_kernel<E, OUT, MAXSEG>;
    static unsigned long long opted_in = 0;  // bit per device
    cudaError_t e = opt_in_smem(kern, &opted_in);
    if (e != cudaSuccess) return e;
    TmaFusedParams<MAXSEG> tp;
    fill_params<E, OUT, MAXSEG>(tp.f, L, ntiles);
    tp.tile_bytes = L.tile_bytes;
    const size_t smem = unaligned_smem_bytes(L.n, L.tile_bytes, OUT, (int)sizeof(typename E::T));
    if (smem > (size_t)kMaxDynamicSmem) return cudaErrorInvalidValue;
    // One tile per block.  The block scheduler hands out blocks in index
    // order, so the tiles in flight form one contiguous address window that
    // slides through the arrays; that keeps DRAM pages open far better than
    // a persistent grid whose blocks drift apart (measured on GB300: 7.09 vs
    // 6.28 TB/s at N=8, P=300M f32).  The kernel's tile loop only matters
    // past 2^31-1 tiles.
    const int64_t grid = ntiles < kMaxGrid ? ntiles : kMaxGrid;
    return launch_pdl(kern, grid, kThreadsPerBlock, smem, s, tp);
}

template <class E>
static cudaError_t fused_unaligned_dispatch(const FusedLaunch &L, int64_t ntiles, cudaStream_t s) {
    const bool big = L.nseg > kSegSmall;
    if (L.out != kOutAll && big) return cudaErrorInvalidValue;
    switch (L.out) {
        case kOutAllSgd: return fused_unaligned_launch_one<E, kOutAllSgd, kSegSmall>(L, ntiles, s);
        case kOutOne: return fused_unaligned_launch_one<E, kOutOne, kSegSmall>(L, ntiles, s);
        case kOutAllWire:
            if constexpr (sizeof(typename E::T) == 2)
                return fused_unaligned_launch_one<E, kOutAllWire, kSegSmall>(L, ntiles, s);
            return cudaErrorInvalidValue;
        default:
            if (big) return fused_unaligned_launch_one<E, kOutAll, kSegLarge>(L, ntiles, s);
            return fused_unaligned_launch_one<E, kOutAll, kSegSmall>(L, ntiles, s);
    }
}

template <class E, int NT, int OUT, int MAXSEG>
static cudaError_t fused_tma_launch_one(const FusedLaunch &L, int64_t ntiles, cudaStream_t s) {
    auto kern = fused_tma_kernel<E, NT, OUT, MAXSEG>;
    static unsigned long long opted_in = 0;  // bit per device
    cudaError_t e = opt_in_smem(kern, &opted_in);
    if (e != cudaSuccess) return e;
    TmaFusedParams<MAXSEG> tp;
    fill_params<E, OUT, MAXSEG>(tp.f, L, ntiles);
    tp.tile_bytes = L.tile_bytes;
    const int esz = (int)sizeof(typename E::T);
    const size_t smem = (size_t)L.n * L.tile_bytes + L.tile_bytes + (OUT == kOutAllSgd ? L.tile_bytes / esz * 4 : 0) + 16;
    if (smem > (size_t)kMaxDynamicSmem) return cudaErrorInvalidValue;
    // one tile per block (see fused_unaligned_launch_one)
    const int64_t grid = ntiles < kMaxGrid ? ntiles : kMaxGrid;
    return launch_pdl(kern, grid, kThreadsPerBlock, smem, s, tp);
}

// vector path: the TMA kernel, the fold unrolled for the common worker counts
template <class E, int NT>
static cudaError_t fused_tma_dispatch_nt(const FusedLaunch &L, int64_t ntiles, cudaStream_t s) {
    const bool big = L.nseg > kSegSmall;
    if (L.out != kOutAll && big) return cudaErrorInvalidValue;
    switch (L.out) {
        case kOutAllSgd: return fused_tma_launch_one<E, NT, kOutAllSgd, kSegSmall>(L, ntiles, s);
        case kOutOne: return fused_tma_launch_one<E, NT, kOutOne, kSegSmall>(L, ntiles, s);
        case kOutAllWire:
            if constexpr (sizeof(typename E::T) == 2)
                return fused_tma_launch_one<E, NT, kOutAllWire, kSegSmall>(L, ntiles, s);
            return cudaErrorInvalidValue;
        default:
            if (big) return fused_tma_launch_one<E, NT, kOutAll, kSegLarge>(L, ntiles, s);
            return fused_tma_launch_one<E, NT, kOutAll, kSegSmall>(L, ntiles, s);
    }
}

// Which worker counts get the unrolled fold was measured on GB300: binary32
// gains at n = 4 (7.05 vs 6.92 TB/s) and 8 (7.08 vs 6.94), and edges ahead at
// 32; bf16 keeps the runtime loop at 8 (7.06 vs 6.70 TB/s unrolled) and 16
// (7.05 vs 6.89), and is even at 2 and 4.
template <class E>
static cudaError_t fused_tma_dispatch(const FusedLaunch &L, int64_t ntiles, cudaStream_t s) {
    constexpr bool wide = sizeof(typename E::T) == 4;
    switch (L.n) {
        case 2: return fused_tma_dispatch_nt<E, 2>(L, ntiles, s);
        case 4: return fused_tma_dispatch_nt<E, 4>(L, ntiles, s);
        case 8:
            if constexpr (wide) return fused_tma_dispatch_nt<E, 8>(L, ntiles, s);
            return fused_tma_dispatch_nt<E, 0>(L, ntiles, s);
        case 16:
            if constexpr (wide) return fused_tma_dispatch_nt<E, 16>(L, ntiles, s);
            return fused_tma_dispatch_nt<E, 0>(L, ntiles, s);
        case 32:
            if constexpr (wide) return fused_tma_dispatch_nt<E, 32>(L, ntiles, s);
            return fused_tma_dispatch_nt<E, 0>(L, ntiles, s);
        default: return fused_tma_dispatch_nt<E, 0>(L, ntiles, s);
    }
}

template <class E>
static cudaError_t fused_launch_dtype(const FusedLaunch &L, int64_t ntiles, cudaStream_t s) {
    return L.vector ? fused_tma_dispatch<E>(L, ntiles, s) : fused_unaligned_dispatch<E>(L, ntiles, s);
}

}  // namespace ra
