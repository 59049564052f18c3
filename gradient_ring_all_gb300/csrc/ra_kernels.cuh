// ra_kernels.cuh -- device code of the ring all-reduce library (sm_103a).
//
// Work decomposition.  The host cuts every request into "segments": a
// contiguous element range of the workers' arrays in which every element
// belongs to the same ring chunk c (Gibiansky, "Scatter-Reduce": the array
// is split into N chunks, and the chunk decides where the scatter-reduce
// starts accumulating it).  A plain all-reduce has N segments, a bucketed
// one N per bucket.  Each segment is cut into tiles; every block takes one
// tile (a grid-stride loop covers grids past the launch limit), finds the
// tile's segment by binary search in the kernel-parameter table, and so
// knows c for the whole tile.  The few elements of a segment that do not
// fill a 16-byte vector (its ragged head and tail) are done with scalar
// accesses by the segment's first and last tiles.
//
// Kernels:
//   fused_tma_kernel     the one-pass all-reduce (and its SGD, reduce-scatter
//                        and bf16-wire variants): TMA bulk copies stage the N
//                        row tiles in shared memory, the fold runs in ring
//                        order from worker c in binary32, the mean is divided
//                        by N and bulk-stored to its destinations;
//   fused_tma_unaligned_kernel
//                        the same for rows that share no 16-byte vector
//                        boundary: each row's tile is copied widened to
//                        16-byte boundaries and read at its own offset;
//   staged_step_kernel   one iteration of the literal ring per launch;
//   all_gather_tma_kernel / all_gather_scalar_kernel
//                        the all-gather on its own (bulk copies through
//                        shared memory, or element by element).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ra_internal.h"

namespace ra {

// ---------------------------------------------------------------------------
// element types

struct F32 {
    using T = float;
    static constexpr int kVec = 4;  // elements per 16-byte vector
};
struct BF16 {
    using T = uint16_t;  // bf16 bit pattern
    static constexpr int kVec = 8;
};

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

// binary32 -> bf16, round to nearest even (hardware conversion)
__device__ __forceinline__ uint32_t f32_to_bf16_bits(float x) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return f32_to_bf16_bits(lo) | (f32_to_bf16_bits(hi) << 16);
}

// 16-byte vector load/store with the streaming (evict-first) hint.
__device__ __forceinline__ uint4 ld_vec(const void *p) { return __ldcs(reinterpret_cast<const uint4 *>(p)); }
__device__ __forceinline__ void st_vec(void *p, uint4 v) { __stcs(reinterpret_cast<uint4 *>(p), v); }

template <class E>
__device__ __forceinline__ void unpack(uint4 v, float (&x)[E::kVec]);
template <>
__device__ __forceinline__ void unpack<F32>(uint4 v, float (&x)[4]) {
    x[0] = __uint_as_float(v.x);
    x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z);
    x[3] = __uint_as_float(v.w);
}
template <>
__device__ __forceinline__ void unpack<BF16>(uint4 v, float (&x)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        x[2 * k] = bf16_bits_to_f32(w[k] & 0xffffu);
        x[2 * k + 1] = bf16_bits_to_f32(w[k] >> 16);
    }
}

// pack the binary32 mean into the stored vector; `back` receives the value
// the workers will hold (for the SGD update)
template <class E>
__device__ __forceinline__ uint4 pack(const float (&x)[E::kVec], float (&back)[E::kVec]);
template <>
__device__ __forceinline__ uint4 pack<F32>(const float (&x)[4], float (&back)[4]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) back[k] = x[k];
    return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]), __float_as_uint(x[3]));
}
template <>
__device__ __forceinline__ uint4 pack<BF16>(const float (&x)[8], float (&back)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        w[k] = pack_bf16x2(x[2 * k], x[2 * k + 1]);
        back[2 * k] = bf16_bits_to_f32(w[k] & 0xffffu);
        back[2 * k + 1] = bf16_bits_to_f32(w[k] >> 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <class E>
__device__ __forceinline__ float load_scalar(const void *row, int64_t i) {
    if constexpr (sizeof(typename E::T) == 4)
        return __ldcs(reinterpret_cast<const float *>(row) + i);
    else
        return bf16_bits_to_f32(__ldcs(reinterpret_cast<const unsigned short *>(row) + i));
}

// stores the mean, returns the value the workers hold
template <class E>
__device__ __forceinline__ float store_scalar_all(void *const *rows, int n, int64_t i, float avg) {
    if constexpr (sizeof(typename E::T) == 4) {
        for (int k = 0; k < n; ++k) __stcs(reinterpret_cast<float *>(rows[k]) + i, avg);
        return avg;
    } else {
        const unsigned short b = (unsigned short)f32_to_bf16_bits(avg);
        for (int k = 0; k < n; ++k) __stcs(reinterpret_cast<unsigned short *>(rows[k]) + i, b);
        return bf16_bits_to_f32(b);
    }
}

// Mean of a binary32 sum over n workers: one IEEE division, rounded to
// nearest even.  For n a power of two, x * (1/n) is the same correctly
// rounded value (1/n is exact, and both operations round the same real
// number x/n), so the cheaper multiplication is used there.
__device__ __forceinline__ float div_n(float x, int n) {
    return (n & (n - 1)) == 0 ? __fmul_rn(x, 1.0f / (float)n) : __fdiv_rn(x, (float)n);
}

// worker index (c + k) mod n for 0 <= c, k < n
__device__ __forceinline__ int ring_idx(int c, int k, int n) {
    int r = c + k;
    return r >= n ? r - n : r;
}

// ---------------------------------------------------------------------------
// segment table


// binary32 value of the nearest bf16 (ties to even)
__device__ __forceinline__ float round_bf16(float x) { return bf16_bits_to_f32(f32_to_bf16_bits(x)); }

// The bounds-checked build (compiled with RA_CHECKED=1 into a separate
// library for the tests): before each global access a kernel verifies that
// the range lies inside the caller's buffer it belongs to -- a row
// [rows[k], rows[k] + p), the weights [w, w + p), chunk c of a shard or of the
// all-gather's source, the staged workspace -- and the bulk copies of a tile
// also inside the tile's segment.  A violation sets bit 1 of the error word
// and the access is skipped, so nothing outside the buffers is touched.  The
// product build compiles every check away.
constexpr bool kChecked = RA_CHECKED != 0;
constexpr unsigned int kErrBounds = 2u;

__device__ __forceinline__ bool span_in(const void *a, int64_t bytes, const void *lo, int64_t len) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), b = reinterpret_cast<uintptr_t>(lo);
    return bytes >= 0 && len >= 0 && x >= b && x + (uintptr_t)bytes <= b + (uintptr_t)len;
}
// chunk c of a p-element array split for n workers (the first p mod n
// chunks hold one extra element)
__device__ __forceinline__ void chunk_span(int64_t p, int n, int c, int64_t *b, int64_t *e) {
    const int64_t q = p / n, r = p % n;
    *b = (int64_t)c * q + (c < r ? c : r);
    *e = *b + q + (c < r ? 1 : 0);
}

template <int MAXSEG>
struct FusedParams {
    void *rows[RA_MAX_N];  // worker arrays (device)
    void *aux[RA_MAX_N];   // kOutOne: element i of chunk c goes to aux[c] + i * element size
    float *w;              // SGD weights (device) or null
    unsigned int *err;     // the device's error word: bit 0 = a bounded wait gave up
    float lr;
    int n;                 // workers
    int nseg;
    int mis;               // rows' common misalignment, in elements (< kVec); vector mode only
    int64_t p;             // elements per row (the bounds the checked build verifies)
    int64_t ntiles;
    Seg seg[MAXSEG];
};

template <int MAXSEG>
__device__ __forceinline__ int find_seg(const Seg *seg, int nseg, int64_t tile) {
    // largest s with seg[s].tile0 <= tile
    int lo = 0, hi = nseg - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (seg[mid].tile0 <= tile)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// ---------------------------------------------------------------------------
// fused kernel

// one element through the scalar path: ring-order fold from worker c
template <class E, int OUT, int MAXSEG>
__device__ __forceinline__ void fused_scalar(const FusedParams<MAXSEG> &p, int c, int64_t i) {
    if constexpr (kChecked) {
        bool ok = i >= 0 && i < p.p;
        if constexpr (OUT == kOutOne) {
            int64_t b, e;
            chunk_span(p.p, p.n, c, &b, &e);
            ok = ok && i >= b && i < e;
        }
        if (!ok) {
            atomicOr(p.err, kErrBounds);
            return;
        }
    }
    const int n = p.n;
    float acc = load_scalar<E>(p.rows[c], i);
    for (int k = 1; k < n; ++k) {
        acc = __fadd_rn(load_scalar<E>(p.rows[ring_idx(c, k, n)], i), acc);
        if constexpr (OUT == kOutAllWire) acc = round_bf16(acc);
    }
    const float avg = div_n(acc, n);
    if constexpr (OUT == kOutOne) {
        store_scalar_all<E>(&p.aux[c], 1, i, avg);
    } else {
        const float held = store_scalar_all<E>(p.rows, n, i, avg);
        if constexpr (OUT == kOutAllSgd) p.w[i] = __fsub_rn(p.w[i], __fmul_rn(p.lr, held));
    }
}

constexpr int kThreads = kThreadsPerBlock;

// ---------------------------------------------------------------------------
// TMA fused kernel (the vector path).  One block per tile; a tile is up to
// tile_bytes of one segment's 16-byte-aligned interior in every row.  Thread
// 0 starts n bulk copies (cp.async.bulk, global -> shared) that complete on
// one mbarrier; every thread folds its 16-byte vectors over the n staged rows
// in ring order straight from shared memory, writes the mean to a shared
// output tile, and thread 0 stores that tile to every destination with bulk
// copies (shared -> global).  The copy engine holds the bytes in flight, so
// the fold needs no per-n register arrays and one kernel serves every n.

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of an mbarrier, giving up after limit_ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = global_ns();
    for (;;) {
        uint32_t ok;
        asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                     : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
        if (ok) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

// Programmatic dependent launch.  The fused kernels are launched with
// programmatic stream serialisation, so the next kernel on the stream may be
// launched while this one drains its last wave.  Every block first allows
// that (the next grid starts only once all blocks of this one have started),
// then waits until the previous grid on the stream has completed and its
// writes are visible, before touching global memory.  Without the launch
// attribute both instructions do nothing.
#ifndef RA_PDL
#define RA_PDL 1
#endif
__device__ __forceinline__ void pdl_enter() {
#if RA_PDL
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}

// host side: launch with programmatic stream serialisation (every kernel of
// this library calls pdl_enter before its first global access)
template <class K, class... P>
static cudaError_t launch_pdl(K kern, int64_t grid, int block, size_t smem, cudaStream_t s, const P &...params) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = RA_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, params...);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: copies of one tile take microseconds

template <int MAXSEG>
struct TmaFusedParams {
    FusedParams<MAXSEG> f;  // rows, aux, w, err, lr, n, nseg, mis, p, ntiles, seg
    int tile_bytes;         // bytes per row per tile (multiple of 16)
};

// fold one 16-byte vector q over the n staged rows, ring order from row c
template <class E, int NT, int OUT>
__device__ __forceinline__ void tma_fold(const unsigned char *stage, int B, int n, int c, int q,
                                         float (&acc)[E::kVec]) {
    constexpr int V = E::kVec;
    float t[V];
    unpack<E>(reinterpret_cast<const uint4 *>(stage + (size_t)c * B)[q], acc);
    if constexpr (NT > 0) {
#pragma unroll
        for (int k = 1; k < NT; ++k) {
            const int r = ring_idx(c, k, NT);
            unpack<E>(reinterpret_cast<const uint4 *>(stage + (size_t)r * B)[q], t);
#pragma unroll
            for (int e = 0; e < V; ++e) {
                acc[e] = __fadd_rn(t[e], acc[e]);
                if constexpr (OUT == kOutAllWire) acc[e] = round_bf16(acc[e]);
            }
        }
    } else {
        int r = c;
        for (int k = 1; k < n; ++k) {
            r = r + 1 == n ? 0 : r + 1;
            unpack<E>(reinterpret_cast<const uint4 *>(stage + (size_t)r * B)[q], t);
#pragma unroll
            for (int e = 0; e < V; ++e) {
                acc[e] = __fadd_rn(t[e], acc[e]);
                if constexpr (OUT == kOutAllWire) acc[e] = round_bf16(acc[e]);
            }
        }
    }
}

template <class E, int NT, int OUT, int MAXSEG>
__global__ void __launch_bounds__(kThreads) fused_tma_kernel(const __grid_constant__ TmaFusedParams<MAXSEG> tp) {
    constexpr int V = E::kVec;
    constexpr int esz = (int)sizeof(typename E::T);
    const FusedParams<MAXSEG> &p = tp.f;
    const int n = NT > 0 ? NT : p.n;
    const int B = tp.tile_bytes;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *stage = smem;                      // n rows of B bytes
    unsigned char *outb = smem + (size_t)n * B;       // B bytes
    float *wt = reinterpret_cast<float *>(outb + B);  // SGD: the weights of the tile, (B / esz) * 4 bytes
    const int wbytes_max = OUT == kOutAllSgd ? (B / esz) * 4 : 0;
    uint64_t *bar = reinterpret_cast<uint64_t *>(outb + B + wbytes_max);
    pdl_enter();

    for (int64_t tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x) {
        const int s = find_seg<MAXSEG>(p.seg, p.nseg, tile);
        const Seg sg = p.seg[s];
        const int c = sg.c;
        const int64_t t_in_seg = tile - sg.tile0;
        int64_t ab, ae;
        vector_interior(sg.begin, sg.end, p.mis, V, &ab, &ae);
        const int64_t first = ab + t_in_seg * (B / esz);  // first element of this tile
        const int64_t left = (ae - first) * esz;
        const int bytes = left <= 0 ? 0 : (int)(left < B ? left : B);
        const int wbytes = OUT == kOutAllSgd ? (bytes / esz) * 4 : 0;

        if (bytes > 0) {
            if constexpr (kChecked) {
                // every copy of the tile inside its segment of its buffer
                if (threadIdx.x == 0) {
                    bool ok = sg.begin >= 0 && sg.end <= p.p && first >= sg.begin && first * esz + bytes <= sg.end * esz;
                    for (int k = 0; k < n; ++k)
                        ok = ok && span_in(reinterpret_cast<const char *>(p.rows[k]) + first * esz, bytes, p.rows[k],
                                           p.p * esz);
                    if constexpr (OUT == kOutAllSgd) ok = ok && span_in(p.w + first, wbytes, p.w, p.p * 4);
                    if constexpr (OUT == kOutOne) {
                        int64_t b, e;
                        chunk_span(p.p, p.n, c, &b, &e);
                        ok = ok && span_in(reinterpret_cast<const char *>(p.aux[c]) + first * esz, bytes,
                                           reinterpret_cast<const char *>(p.aux[c]) + b * esz, (e - b) * esz);
                    }
                    if (!ok) atomicOr(p.err, kErrBounds);
                    reinterpret_cast<int *>(bar + 1)[0] = ok ? 0 : 1;  // the spare half of the barrier's slot
                }
                __syncthreads();
                if (reinterpret_cast<volatile int *>(bar + 1)[0]) return;
            }
            if (threadIdx.x == 0) {
                asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(smem_addr(bar)));
                asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                             :: "r"(smem_addr(bar)), "r"((uint32_t)bytes * (uint32_t)n + (uint32_t)wbytes) : "memory");
                for (int k = 0; k < n; ++k)
                    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                                 :: "r"(smem_addr(stage + (size_t)k * B)),
                                    "l"(reinterpret_cast<const char *>(p.rows[k]) + first * esz), "r"(bytes),
                                    "r"(smem_addr(bar)) : "memory");
                if constexpr (OUT == kOutAllSgd)
                    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                                 :: "r"(smem_addr(wt)), "l"(p.w + first), "r"(wbytes), "r"(smem_addr(bar)) : "memory");
            }
            __syncthreads();
            const bool ok = mbar_wait_bounded(smem_addr(bar), 0, kWaitLimitNs);
            if (__syncthreads_or(!ok)) {
                // the copies never landed: record it, let them finish (bounded), leave
                if (threadIdx.x == 0) {
                    atomicOr(p.err, 1u);
                    mbar_wait_bounded(smem_addr(bar), 0, kWaitLimitNs);
                }
                __syncthreads();
                return;
            }
            const int nvec = bytes / 16;
            for (int q = threadIdx.x; q < nvec; q += kThreads) {
                float acc[V];
                tma_fold<E, NT, OUT>(stage, B, n, c, q, acc);
                float avg[V], held[V];
#pragma unroll
                for (int e = 0; e < V; ++e) avg[e] = div_n(acc[e], n);
                reinterpret_cast<uint4 *>(outb)[q] = pack<E>(avg, held);
                if constexpr (OUT == kOutAllSgd) {
#pragma unroll
                    for (int e = 0; e < V; e += 4) {
                        float4 *wp = reinterpret_cast<float4 *>(wt + q * V + e);
                        float4 wv = *wp;
                        wv.x = __fsub_rn(wv.x, __fmul_rn(p.lr, held[e + 0]));
                        wv.y = __fsub_rn(wv.y, __fmul_rn(p.lr, held[e + 1]));
                        wv.z = __fsub_rn(wv.z, __fmul_rn(p.lr, held[e + 2]));
                        wv.w = __fsub_rn(wv.w, __fmul_rn(p.lr, held[e + 3]));
                        *wp = wv;
                    }
                }
            }
            // generic-proxy writes of the output tile -> visible to the bulk copies
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncthreads();
            if (threadIdx.x == 0) {
                if constexpr (OUT == kOutOne) {
                    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                                 :: "l"(reinterpret_cast<char *>(p.aux[c]) + first * esz), "r"(smem_addr(outb)),
                                    "r"(bytes) : "memory");
                } else {
                    for (int k = 0; k < n; ++k)
                        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                                     :: "l"(reinterpret_cast<char *>(p.rows[k]) + first * esz), "r"(smem_addr(outb)),
                                        "r"(bytes) : "memory");
                    if constexpr (OUT == kOutAllSgd)
                        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                                     :: "l"(p.w + first), "r"(smem_addr(wt)), "r"(wbytes) : "memory");
                }
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                // the shared tile must stay valid until the copies have read it
                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                asm volatile("mbarrier.inval.shared::cta.b64 [%0];" :: "r"(smem_addr(bar)) : "memory");
            }
            __syncthreads();
        }
        // ragged head and tail of the segment: scalar path
        if (t_in_seg == 0 && threadIdx.x < ab - sg.begin) fused_scalar<E, OUT>(p, c, sg.begin + threadIdx.x);
        const bool last = (s + 1 < p.nseg ? p.seg[s + 1].tile0 : p.ntiles) == tile + 1;
        if (last && threadIdx.x < sg.end - ae) fused_scalar<E, OUT>(p, c, ae + threadIdx.x);
    }
}

// TMA kernel for rows that disagree modulo 16 bytes.  A bulk copy needs
// 16-byte-aligned global addresses, and here every row sits at its own byte
// offset d_k from that boundary.
//   load:  for each row thread 0 copies the tile widened to 16-byte
//          boundaries (first byte rounded down, end rounded up) into a slot
//          of B + 16 bytes; the row's elements start d_k bytes into the slot.
//   fold:  each thread takes J elements of the tile and walks the rows in
//          ring order through a table thread 0 writes per tile (where row
//          (c + t) mod n starts in shared memory), reading every row at its
//          own offset, so the per-row work is shared by J elements; every
//          pass but the tile's last runs without bounds checks.
//   store: the mean leaves by scalar stores, coalesced across the warp, as
//          soon as it is known.  (Writing it back into shared memory first
//          and storing whole 16-byte granules -- by bulk copies, from one
//          slot per distinct row offset, or by 16-byte thread stores --
//          measured slower on GB300: the block barrier they need holds the
//          staging longer.)
// The SGD weights are one more widened bulk copy in and, for their whole
// granules, a bulk copy out.  Tiles keep 16 bytes away from both ends of
// their segment (those elements take the scalar path), so the widened copies
// never leave the segment's own bytes.
template <class T>
__device__ __forceinline__ float ld_staged(const unsigned char *p) {
    if constexpr (sizeof(T) == 4) return *reinterpret_cast<const float *>(p);
    else return bf16_bits_to_f32(*reinterpret_cast<const unsigned short *>(p));
}
// element stores of the unaligned kernel: plain (write-back) stores; the
// streaming hint measured 0.1-0.3 % slower on these partial-sector writes
template <class T>
__device__ __forceinline__ void put_elem(void *p, T v) {
    if constexpr (sizeof(T) == 4) *reinterpret_cast<float *>(p) = v;
    else *reinterpret_cast<unsigned short *>(p) = v;
}

// Elements per thread per pass of the unaligned kernel, measured on GB300
// with packed rows: 2 for the all-reduce (bf16 N=16: 6.47 TB/s, against 5.82
// with 1 and 5.87 with 4; binary32 within 1 %), 4 for the reduce-scatter
// (7.35 against 7.11 TB/s with 2).
#ifndef RA_UNALIGNED_J
#define RA_UNALIGNED_J 0
#endif
template <int OUT>
constexpr int unaligned_per_thread() { return RA_UNALIGNED_J > 0 ? RA_UNALIGNED_J : (OUT == kOutOne ? 4 : 2); }

// One pass of the unaligned kernel over elements j0 + u * kThreads (u < J)
// of the staged tile.  ringoff[t] is where row (c + t) mod n's elements
// start in shared memory, so the fold is one loop in ring order; rowptr[k]
// is row k's first element of the tile in global memory.  In a FULL pass
// every element exists (no bounds checks); the tile's last pass checks
// each against ne.
template <class E, int OUT, int J, bool FULL, int MAXSEG>
__device__ __forceinline__ void unaligned_pass(const FusedParams<MAXSEG> &p, const unsigned char *smem,
                                               const int *ringoff, char *const *rowptr, const int *shift,
                                               unsigned char *wslot, int n, int c, int ne, int64_t first, int j0) {
    using T = typename E::T;
    constexpr int esz = (int)sizeof(T);
    constexpr int step = kThreads * esz;  // bytes between one thread's elements
    const int boff = j0 * esz;
    bool in[J];
#pragma unroll
    for (int u = 0; u < J; ++u) in[u] = FULL || j0 + u * kThreads < ne;
    float acc[J];
    {
        const unsigned char *b = smem + ringoff[0] + boff;
#pragma unroll
        for (int u = 0; u < J; ++u) acc[u] = in[u] ? ld_staged<T>(b + u * step) : 0.f;
    }
#pragma unroll 4
    for (int t = 1; t < n; ++t) {
        const unsigned char *b = smem + ringoff[t] + boff;
#pragma unroll
        for (int u = 0; u < J; ++u)
            if (in[u]) {
                acc[u] = __fadd_rn(ld_staged<T>(b + u * step), acc[u]);
                if constexpr (OUT == kOutAllWire) acc[u] = round_bf16(acc[u]);
            }
    }
    T v[J];
    float held[J];
#pragma unroll
    for (int u = 0; u < J; ++u) {
        const float avg = div_n(acc[u], n);
        if constexpr (esz == 4) {
            v[u] = avg;
            held[u] = avg;
        } else {
            v[u] = (T)f32_to_bf16_bits(avg);
            held[u] = bf16_bits_to_f32(v[u]);
        }
    }
    if constexpr (OUT == kOutOne) {
        char *bp = reinterpret_cast<char *>(p.aux[c]) + first * esz + boff;
#pragma unroll
        for (int u = 0; u < J; ++u)
            if (in[u]) put_elem<T>(bp + u * step, v[u]);
    } else {
        for (int k = 0; k < n; ++k) {
            char *bp = rowptr[k] + boff;
#pragma unroll
            for (int u = 0; u < J; ++u)
                if (in[u]) put_elem<T>(bp + u * step, v[u]);
        }
        if constexpr (OUT == kOutAllSgd) {
            // whole granules of the weights go back by bulk copy, the
            // partial ones at the tile's ends element by element
            const int d = shift[n], lo = (d + 15) & ~15, hi = (d + ne * 4) & ~15;
#pragma unroll
            for (int u = 0; u < J; ++u) {
                const int j = j0 + u * kThreads;
                if (in[u]) {
                    const int pos = d + j * 4;
                    float *wp = reinterpret_cast<float *>(wslot + pos);
                    const float nw = __fsub_rn(*wp, __fmul_rn(p.lr, held[u]));
                    if (pos >= lo && pos < hi) *wp = nw;
                    else __stcs(p.w + first + j, nw);
                }
            }
        }
    }
}

template <class E, int OUT, int MAXSEG>
__global__ void __launch_bounds__(kThreads) fused_tma_unaligned_kernel(const __grid_constant__ TmaFusedParams<MAXSEG> tp) {
    using T = typename E::T;
    constexpr int V = E::kVec;
    constexpr int esz = (int)sizeof(T);
    constexpr int J = unaligned_per_thread<OUT>();
    const FusedParams<MAXSEG> &p = tp.f;
    const int n = p.n;
    const int B = tp.tile_bytes;  // bytes of each row per tile
    const int slot = B + 16;      // room for the widening
    extern __shared__ __align__(128) unsigned char smem[];
    // n row slots | weight slot (SGD) | mbarrier | offsets
    unsigned char *wslot = smem + (size_t)n * slot;
    const int wslot_bytes = OUT == kOutAllSgd ? (B / esz) * 4 + 16 : 0;
    uint64_t *bar = reinterpret_cast<uint64_t *>(wslot + wslot_bytes);
    int *shift = reinterpret_cast<int *>(wslot + wslot_bytes + 16);  // d_k of row k; shift[n]: the weights'
    // per tile (set by thread 0, so that the fold and the stores do no
    // per-row address arithmetic): ringoff[t], where row (c + t) mod n's
    // elements start in shared memory, in the fold's ring order; rowptr[k],
    // row k's first element of the tile in global memory
    int *ringoff = shift + n + 1;
    char **rowptr = reinterpret_cast<char **>(
        (reinterpret_cast<uintptr_t>(ringoff + n) + 7) & ~static_cast<uintptr_t>(7));
    pdl_enter();

    for (int64_t tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x) {
        const int s = find_seg<MAXSEG>(p.seg, p.nseg, tile);
        const Seg sg = p.seg[s];
        const int c = sg.c;
        const int64_t t_in_seg = tile - sg.tile0;
        int64_t ab, ae;
        unaligned_interior(sg.begin, sg.end, V, &ab, &ae);
        const int64_t first = ab + t_in_seg * (B / esz);
        const int64_t left = (ae - first) * esz;
        const int bytes = left <= 0 ? 0 : (int)(left < B ? left : B);
        const int ne = bytes / esz;

        if (bytes > 0) {
            if constexpr (kChecked) {
                // every widened copy inside the tile's segment of its row (or of w),
                // the stores inside the segment, the reduce-scatter's inside chunk c
                if (threadIdx.x == 0) {
                    bool ok = sg.begin >= 0 && sg.end <= p.p && first >= sg.begin && first + ne <= sg.end;
                    for (int k = 0; k < n; ++k) {
                        const char *a = reinterpret_cast<const char *>(p.rows[k]) + first * esz;
                        const int d = (int)(reinterpret_cast<uintptr_t>(a) & 15);
                        ok = ok && span_in(a - d, (d + bytes + 15) & ~15,
                                           reinterpret_cast<const char *>(p.rows[k]) + sg.begin * esz,
                                           (sg.end - sg.begin) * esz);
                    }
                    if constexpr (OUT == kOutAllSgd) {
                        const char *a = reinterpret_cast<const char *>(p.w + first);
                        const int d = (int)(reinterpret_cast<uintptr_t>(a) & 15);
                        ok = ok && span_in(a - d, (d + ne * 4 + 15) & ~15, p.w + sg.begin, (sg.end - sg.begin) * 4);
                    }
                    if constexpr (OUT == kOutOne) {
                        int64_t b, e;
                        chunk_span(p.p, p.n, c, &b, &e);
                        ok = ok && first >= b && first + ne <= e;
                    }
                    if (!ok) atomicOr(p.err, kErrBounds);
                    reinterpret_cast<int *>(bar + 1)[0] = ok ? 0 : 1;  // the spare half of the barrier's slot
                }
                __syncthreads();
                if (reinterpret_cast<volatile int *>(bar + 1)[0]) return;
            }
            if (threadIdx.x == 0) {
                uint32_t total = 0;
                for (int k = 0; k < n; ++k) {
                    const int d = (int)((reinterpret_cast<uintptr_t>(p.rows[k]) + (uintptr_t)first * esz) & 15);
                    shift[k] = d;
                    ringoff[k >= c ? k - c : k + n - c] = k * slot + d;
                    rowptr[k] = reinterpret_cast<char *>(p.rows[k]) + first * esz;
                    total += (uint32_t)((d + bytes + 15) & ~15);
                }
                if constexpr (OUT == kOutAllSgd) {
                    shift[n] = (int)((reinterpret_cast<uintptr_t>(p.w + first)) & 15);
                    total += (uint32_t)((shift[n] + ne * 4 + 15) & ~15);
                }
                asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(smem_addr(bar)));
                asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(smem_addr(bar)), "r"(total)
                             : "memory");
                for (int k = 0; k < n; ++k) {
                    const int d = shift[k];
                    const char *src = reinterpret_cast<const char *>(p.rows[k]) + first * esz - d;
                    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                                 :: "r"(smem_addr(smem + (size_t)k * slot)), "l"(src), "r"((d + bytes + 15) & ~15),
                                    "r"(smem_addr(bar)) : "memory");
                }
                if constexpr (OUT == kOutAllSgd) {
                    const int d = shift[n];
                    const char *src = reinterpret_cast<const char *>(p.w + first) - d;
                    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                                 :: "r"(smem_addr(wslot)), "l"(src), "r"((d + ne * 4 + 15) & ~15), "r"(smem_addr(bar))
                                 : "memory");
                }
            }
            __syncthreads();
            const bool ok = mbar_wait_bounded(smem_addr(bar), 0, kWaitLimitNs);
            if (__syncthreads_or(!ok)) {
                // the copies never landed: record it, let them finish (bounded), leave
                if (threadIdx.x == 0) {
                    atomicOr(p.err, 1u);
                    mbar_wait_bounded(smem_addr(bar), 0, kWaitLimitNs);
                }
                __syncthreads();
                return;
            }
            // passes of J * kThreads elements; in all but the last every
            // thread has J of them
            const int full_end = ne - ne % (J * kThreads);
            for (int base = 0; base < full_end; base += J * kThreads)
                unaligned_pass<E, OUT, J, true>(p, smem, ringoff, rowptr, shift, wslot, n, c, ne, first,
                                                base + (int)threadIdx.x);
            if (full_end < ne)
                unaligned_pass<E, OUT, J, false>(p, smem, ringoff, rowptr, shift, wslot, n, c, ne, first,
                                                 full_end + (int)threadIdx.x);
            if constexpr (OUT == kOutAllSgd) {
                // generic-proxy writes of the new weights -> visible to the bulk copy
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                if constexpr (OUT == kOutAllSgd) {
                    const int d = shift[n], lo = (d + 15) & ~15, hi = (d + ne * 4) & ~15;
                    if (hi > lo)
                        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                                     :: "l"(reinterpret_cast<char *>(p.w + first) - d + lo), "r"(smem_addr(wslot + lo)),
                                        "r"(hi - lo) : "memory");
                    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                    // the staged weights must stay valid until the copy has read them
                    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                }
                asm volatile("mbarrier.inval.shared::cta.b64 [%0];" :: "r"(smem_addr(bar)) : "memory");
            }
            __syncthreads();
        }
        // the margins and anything shorter than them: scalar path
        if (t_in_seg == 0)
            for (int64_t i = sg.begin + threadIdx.x; i < ab; i += kThreads) fused_scalar<E, OUT>(p, c, i);
        const bool last = (s + 1 < p.nseg ? p.seg[s + 1].tile0 : p.ntiles) == tile + 1;
        if (last)
            for (int64_t i = (ae > ab ? ae : ab) + threadIdx.x; i < sg.end; i += kThreads) fused_scalar<E, OUT>(p, c, i);
    }
}

// ---------------------------------------------------------------------------
// staged kernel: one ring iteration per launch

struct StagedParams {
    void *rows[RA_MAX_N];
    float *msg;  // binary32 partial sums (bf16 only), element i at msg[i]
    const char *msg_lo, *msg_hi;  // the workspace holding them (checked build)
    unsigned int *err;            // the device's error word (checked build)
    int64_t p;                    // elements per row (checked build)
    int n;
    int t;       // iteration
    int op;      // StagedOp
    int mis;     // rows' (and msg's) common misalignment in elements (< kVec)
    int nseg;
    int64_t ntiles;
    Seg seg[RA_MAX_N];
};

// One element of one staged iteration.  Chunk c's partial sits at worker
// (c + t) mod n in scatter-reduce iteration t and moves to (c + t + 1) mod n;
// the complete chunk sits at worker (c - 1) mod n; in all-gather iteration t
// worker (c + t - 1) mod n sends it to worker (c + t) mod n.
__device__ __forceinline__ bool staged_in_bounds(const StagedParams &p, int64_t i, int count) {
    // elements [i, i + count) of the rows, and of the workspace when in use
    bool ok = i >= 0 && i + count <= p.p;
    if (p.msg) ok = ok && span_in(p.msg + i, (int64_t)count * 4, p.msg_lo, p.msg_hi - p.msg_lo);
    if (!ok) atomicOr(p.err, kErrBounds);
    return ok;
}

template <class E>
__device__ __forceinline__ void staged_scalar(const StagedParams &p, int c, int64_t i) {
    if constexpr (kChecked)
        if (!staged_in_bounds(p, i, 1)) return;
    const int n = p.n;
    switch (p.op) {
        case kOpScatter: {  // receiver's own value + received partial
            const int rcv = ring_idx(c, p.t + 1 >= n ? p.t + 1 - n : p.t + 1, n);
            if constexpr (sizeof(typename E::T) == 4) {
                const int snd = ring_idx(c, p.t, n);
                float *d = reinterpret_cast<float *>(p.rows[rcv]);
                d[i] = __fadd_rn(d[i], reinterpret_cast<const float *>(p.rows[snd])[i]);
            } else {
                const float own = load_scalar<E>(p.rows[rcv], i);
                const float in = p.t == 0 ? load_scalar<E>(p.rows[c], i) : p.msg[i];
                p.msg[i] = __fadd_rn(own, in);
            }
            break;
        }
        case kOpDivide: {
            const int own = c == 0 ? n - 1 : c - 1;
            if constexpr (sizeof(typename E::T) == 4) {
                float *d = reinterpret_cast<float *>(p.rows[own]);
                d[i] = __fdiv_rn(d[i], (float)n);
            } else {
                reinterpret_cast<unsigned short *>(p.rows[own])[i] =
                    (unsigned short)f32_to_bf16_bits(__fdiv_rn(p.msg[i], (float)n));
            }
            break;
        }
        default: {  // kOpGather: overwrite
            const int rcv = ring_idx(c, p.t, n);
            const int snd = rcv == 0 ? n - 1 : rcv - 1;
            using T = typename E::T;
            reinterpret_cast<T *>(p.rows[rcv])[i] = reinterpret_cast<const T *>(p.rows[snd])[i];
            break;
        }
    }
}

template <class E>
__device__ __forceinline__ void staged_vector(const StagedParams &p, int c, int64_t i) {
    const int n = p.n;
    constexpr int V = E::kVec;
    if constexpr (kChecked)
        if (!staged_in_bounds(p, i, V)) return;
    constexpr int esz = (int)sizeof(typename E::T);
    switch (p.op) {
        case kOpScatter: {
            const int rcv = ring_idx(c, p.t + 1 >= n ? p.t + 1 - n : p.t + 1, n);
            float own[V], in[V];
            unpack<E>(ld_vec(reinterpret_cast<const char *>(p.rows[rcv]) + i * esz), own);
            if constexpr (sizeof(typename E::T) == 4) {
                const int snd = ring_idx(c, p.t, n);
                unpack<E>(ld_vec(reinterpret_cast<const char *>(p.rows[snd]) + i * esz), in);
                float s[V], back[V];
#pragma unroll
                for (int e = 0; e < V; ++e) s[e] = __fadd_rn(own[e], in[e]);
                st_vec(reinterpret_cast<char *>(p.rows[rcv]) + i * esz, pack<E>(s, back));
            } else {
                if (p.t == 0) {
                    unpack<E>(ld_vec(reinterpret_cast<const char *>(p.rows[c]) + i * esz), in);
                } else {
#pragma unroll
                    for (int e = 0; e < V; e += 4) {
                        const float4 m = __ldcs(reinterpret_cast<const float4 *>(p.msg + i + e));
                        in[e] = m.x, in[e + 1] = m.y, in[e + 2] = m.z, in[e + 3] = m.w;
                    }
                }
#pragma unroll
                for (int e = 0; e < V; e += 4)
                    __stcs(reinterpret_cast<float4 *>(p.msg + i + e),
                           make_float4(__fadd_rn(own[e], in[e]), __fadd_rn(own[e + 1], in[e + 1]),
                                       __fadd_rn(own[e + 2], in[e + 2]), __fadd_rn(own[e + 3], in[e + 3])));
            }
            break;
        }
        case kOpDivide: {
            const int own = c == 0 ? n - 1 : c - 1;
            float s[V], q[V], back[V];
            if constexpr (sizeof(typename E::T) == 4) {
                unpack<E>(ld_vec(reinterpret_cast<const char *>(p.rows[own]) + i * esz), s);
            } else {
#pragma unroll
                for (int e = 0; e < V; e += 4) {
                    const float4 m = __ldcs(reinterpret_cast<const float4 *>(p.msg + i + e));
                    s[e] = m.x, s[e + 1] = m.y, s[e + 2] = m.z, s[e + 3] = m.w;
                }
            }
#pragma unroll
            for (int e = 0; e < V; ++e) q[e] = __fdiv_rn(s[e], (float)n);
            st_vec(reinterpret_cast<char *>(p.rows[own]) + i * esz, pack<E>(q, back));
            break;
        }
        default: {
            const int rcv = ring_idx(c, p.t, n);
            const int snd = rcv == 0 ? n - 1 : rcv - 1;
            st_vec(reinterpret_cast<char *>(p.rows[rcv]) + i * esz,
                   ld_vec(reinterpret_cast<const char *>(p.rows[snd]) + i * esz));
            break;
        }
    }
}

template <class E, bool VECTOR, int TV>
__global__ void __launch_bounds__(kThreads) staged_step_kernel(const __grid_constant__ StagedParams p) {
    constexpr int V = E::kVec;
    pdl_enter();
    for (int64_t tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x) {
        const int s = find_seg<RA_MAX_N>(p.seg, p.nseg, tile);
        const Seg sg = p.seg[s];
        const int64_t t_in_seg = tile - sg.tile0;
        if constexpr (VECTOR) {
            int64_t ab, ae;
            vector_interior(sg.begin, sg.end, p.mis, V, &ab, &ae);
            const int64_t i0 = ab + (t_in_seg * TV + threadIdx.x) * V;
#pragma unroll
            for (int j = 0; j < TV / kThreads; ++j) {
                const int64_t i = i0 + (int64_t)j * kThreads * V;
                if (i < ae) staged_vector<E>(p, sg.c, i);
            }
            if (t_in_seg == 0 && threadIdx.x < ab - sg.begin) staged_scalar<E>(p, sg.c, sg.begin + threadIdx.x);
            const bool last = (s + 1 < p.nseg ? p.seg[s + 1].tile0 : p.ntiles) == tile + 1;
            if (last && threadIdx.x < sg.end - ae) staged_scalar<E>(p, sg.c, ae + threadIdx.x);
        } else {
            const int64_t i0 = sg.begin + t_in_seg * (int64_t)kThreads * kScalarPerThread + threadIdx.x;
            for (int j = 0; j < kScalarPerThread; ++j) {
                const int64_t i = i0 + (int64_t)j * kThreads;
                if (i < sg.end) staged_scalar<E>(p, sg.c, i);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// all-gather kernel: chunk c travels from the worker that owns it, worker
// (c - 1) mod n (or from a separate shard buffer), to every worker (Gibiansky,
// "Allgather": the received chunk overwrites the receiver's copy).

struct GatherParams {
    void *rows[RA_MAX_N];
    void *src[RA_MAX_N];  // element i of chunk c is read at src[c] + i * element size
    int n;
    int nseg;
    int mis;
    int skip_owner;       // 1: the source is the owner's own array, which is not rewritten
    unsigned int *err;    // the device's error word: bit 0 = a bounded wait gave up
    int64_t p;            // elements per row (checked build)
    int64_t ntiles;
    Seg seg[RA_MAX_N];
};

template <class E>
__device__ __forceinline__ void gather_scalar(const GatherParams &p, int c, int64_t i) {
    using T = typename E::T;
    if constexpr (kChecked) {
        int64_t b, e;
        chunk_span(p.p, p.n, c, &b, &e);
        if (!(i >= b && i < e && i < p.p)) {
            atomicOr(p.err, kErrBounds);
            return;
        }
    }
    const T v = reinterpret_cast<const T *>(p.src[c])[i];
    const int owner = c == 0 ? p.n - 1 : c - 1;
    for (int k = 0; k < p.n; ++k)
        if (!(p.skip_owner && k == owner)) reinterpret_cast<T *>(p.rows[k])[i] = v;
}

// scalar all-gather, for rows (or shards) that share no 16-byte boundary
template <class E>
__global__ void __launch_bounds__(kThreads) all_gather_scalar_kernel(const __grid_constant__ GatherParams p) {
    pdl_enter();
    for (int64_t tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x) {
        const int s = find_seg<RA_MAX_N>(p.seg, p.nseg, tile);
        const Seg sg = p.seg[s];
        const int64_t i0 = sg.begin + (tile - sg.tile0) * (int64_t)kThreads * kScalarPerThread + threadIdx.x;
        for (int j = 0; j < kScalarPerThread; ++j) {
            const int64_t i = i0 + (int64_t)j * kThreads;
            if (i < sg.end) gather_scalar<E>(p, sg.c, i);
        }
    }
}

// TMA all-gather: thread 0 of a one-warp block bulk-copies the owner's tile
// of chunk c into shared memory and bulk-stores it to every destination row;
// no arithmetic, so the copy engine does all the work.  The other lanes only
// take the scalar head and tail.
template <class E>
__global__ void __launch_bounds__(32) all_gather_tma_kernel(const __grid_constant__ GatherParams p, int tile_bytes) {
    constexpr int V = E::kVec;
    constexpr int esz = (int)sizeof(typename E::T);
    const int B = tile_bytes;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + B);
    pdl_enter();
    for (int64_t tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x) {
        const int s = find_seg<RA_MAX_N>(p.seg, p.nseg, tile);
        const Seg sg = p.seg[s];
        const int c = sg.c;
        const int owner = c == 0 ? p.n - 1 : c - 1;
        const int64_t t_in_seg = tile - sg.tile0;
        int64_t ab, ae;
        vector_interior(sg.begin, sg.end, p.mis, V, &ab, &ae);
        const int64_t first = ab + t_in_seg * (B / esz);
        const int64_t left = (ae - first) * esz;
        const int bytes = left <= 0 ? 0 : (int)(left < B ? left : B);
        int fail = 0;
        if constexpr (kChecked) {
            // the owner's chunk c in the source, every destination row
            if (bytes > 0 && threadIdx.x == 0) {
                int64_t b, e;
                chunk_span(p.p, p.n, c, &b, &e);
                bool ok = span_in(reinterpret_cast<const char *>(p.src[c]) + first * esz, bytes,
                                  reinterpret_cast<const char *>(p.src[c]) + b * esz, (e - b) * esz);
                for (int k = 0; k < p.n; ++k)
                    ok = ok && span_in(reinterpret_cast<const char *>(p.rows[k]) + first * esz, bytes, p.rows[k],
                                       p.p * esz);
                if (!ok) {
                    atomicOr(p.err, kErrBounds);
                    fail = 2;
                }
            }
            if (__shfl_sync(0xffffffffu, fail, 0)) return;
        }
        if (bytes > 0 && threadIdx.x == 0) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(smem_addr(bar)));
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                         :: "r"(smem_addr(bar)), "r"((uint32_t)bytes) : "memory");
            asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                         :: "r"(smem_addr(smem)), "l"(reinterpret_cast<const char *>(p.src[c]) + first * esz),
                            "r"(bytes), "r"(smem_addr(bar)) : "memory");
            fail = mbar_wait_bounded(smem_addr(bar), 0, kWaitLimitNs) ? 0 : 1;
        }
        // the whole warp leaves together if the copy never landed
        if (__shfl_sync(0xffffffffu, fail, 0)) {
            if (threadIdx.x == 0) {
                atomicOr(p.err, 1u);
                mbar_wait_bounded(smem_addr(bar), 0, kWaitLimitNs);
            }
            return;
        }
        if (bytes > 0 && threadIdx.x == 0) {
            for (int k = 0; k < p.n; ++k)
                if (!(p.skip_owner && k == owner))
                    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                                 :: "l"(reinterpret_cast<char *>(p.rows[k]) + first * esz), "r"(smem_addr(smem)),
                                    "r"(bytes) : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            asm volatile("mbarrier.inval.shared::cta.b64 [%0];" :: "r"(smem_addr(bar)) : "memory");
        }
        if (t_in_seg == 0 && threadIdx.x < ab - sg.begin) gather_scalar<E>(p, c, sg.begin + threadIdx.x);
        const bool last = (s + 1 < p.nseg ? p.seg[s + 1].tile0 : p.ntiles) == tile + 1;
        if (last && threadIdx.x < sg.end - ae) gather_scalar<E>(p, c, ae + threadIdx.x);
        __syncwarp();
    }
}

}  // namespace ra
