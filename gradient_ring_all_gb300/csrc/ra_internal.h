// ra_internal.h -- types shared by the library's host and device code.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/ring_allreduce.h"

namespace ra {

// A contiguous element range in which every element belongs to ring chunk c
// (so its scatter-reduce fold starts at worker c).  tile0 is the index of
// the segment's first tile in the launch.
struct Seg {
    int64_t begin;
    int64_t end;
    int64_t tile0;
    int32_t c;
    int32_t pad;
};
static_assert(sizeof(Seg) == 32, "Seg layout");

// RA_CHECKED=1 builds the bounds-checked library (see ra_kernels.cuh)
#ifndef RA_CHECKED
#define RA_CHECKED 0
#endif

constexpr int kThreadsPerBlock = 256;
constexpr int64_t kMaxGrid = 0x7fffffff;  // largest gridDim.x
constexpr int kScalarPerThread = 4;  // elements per thread per tile, scalar staged and gather paths
// 16-byte vectors per tile of the staged kernel: 1024 (4 per thread) when a
// launch still fills a wave of blocks with them, else 512.  Measured on
// GB300 (staged ring, GB/s over its schedule's bytes): 512 / 1024 / 2048 /
// 4096 gave 6921 / 7019 / 6984 / 6901 at n=8 binary32, 6947 / 7001 / 6949 /
// 6879 at n=16 bf16 and 6720 / 6876 / 6294 / 5592 at n=32; but the 1M-element
// ring (256 blocks of 1024) slowed to 38 us, against 28 with 512 and 29 with
// 256 vectors per tile.  The tile size is a template parameter: with a
// runtime loop bound the large cases lost 2-3 %.  Loading all of a
// thread's vectors before any store (the rows may alias, so the compiler
// keeps them in order) was slower: 6520 at n=8, 5576 at n=16 bf16.
constexpr int kStagedTileVecLarge = 1024, kStagedTileVecSmall = 512;
constexpr int64_t kStagedWaveBlocks = 152 * 8;  // SMs x resident blocks of 256 threads
inline int staged_tile_vec(int64_t vectors) {
    return vectors / kStagedTileVecLarge >= kStagedWaveBlocks ? kStagedTileVecLarge : kStagedTileVecSmall;
}

// The 16-byte-vector interior [ab, ae) of the element range [b, e) when the
// rows' addresses are `mis` elements past a 16-byte boundary (V elements per
// vector): ab is the first index >= b with (index + mis) % V == 0, ae the
// last such index <= e; [b, ab) and [ae, e) are the scalar head and tail.
__host__ __device__ inline void vector_interior(int64_t b, int64_t e, int mis, int V, int64_t *ab, int64_t *ae) {
    int64_t r = (b + mis) % V;
    int64_t up = r == 0 ? b : b + (V - r);
    if (up > e) up = e;
    int64_t down = e - (e + mis) % V;
    if (down < up) down = up;
    *ab = up;
    *ae = down;
}

// kernel-parameter segment tables: a small one for plain calls and a large
// one for bucketed calls (kernel parameters are limited to 32 KiB)
constexpr int kSegSmall = RA_MAX_N;
constexpr int kSegLarge = 896;

enum StagedOp { kOpScatter = 0, kOpDivide = 1, kOpGather = 2 };

// Where the fused kernel puts the mean: every worker's array (all-reduce),
// the same plus the SGD step, or one destination per chunk (reduce-scatter:
// the worker that owns the chunk, or a separate shard buffer).
// kOutAllWire: the all-reduce of bf16 arrays with every partial sum rounded
// to bf16, as a ring that keeps its arrays in bf16 would store them.
enum FusedOut { kOutAll = 0, kOutAllSgd = 1, kOutOne = 2, kOutAllWire = 3 };

struct FusedLaunch {
    void *rows[RA_MAX_N];
    void *aux[RA_MAX_N];  // reduce-scatter: destination base per chunk
    int out;              // FusedOut
    int n;
    int dtype;
    float *w;  // SGD weights
    float lr;
    bool vector;
    int mis;
    const Seg *seg;  // host table, tile0 filled by the launcher
    int nseg;
    int tile_bytes;  // bytes of each row per tile (fused_tile_bytes)
    unsigned int *err;  // the device's error word (device_error_word)
    int64_t p;          // elements per row: the rows are [rows[k], rows[k] + p)
};

// Tile size of the fused kernels: bytes of each row one block stages in
// shared memory.  The n staged rows take about a budget per block --
// RA_TMA_STAGE_BYTES for the vector path (RA_TMA_STAGE_BYTES_NPOT when n is
// not a power of two), more for the unaligned kernel,
// which holds its tile longer, and 64 KB for the reduce-scatter, which writes
// one row per tile instead of n -- with the tile a multiple of 16 bytes
// between 2 KB and 16 KB, and at most RA_TMA_MAX_STAGE_BYTES staged per
// block (so that several blocks share an SM even at n = 64).
// Measured on GB300, all-reduce at 9.6 GB per call:
//  - 16 KB budget against 64 KB: equal at n=8 (7.10 TB/s), +0.4 % at n=4,
//    -0.2 % for bf16 at n=16, +4 % on rows in host memory;
//  - tiles sized to the budget, not rounded down to a power of two: n=3
//    6.86 (was 6.32), n=5 6.98 (5.75), n=7 6.88 (6.54) TB/s in binary32;
//  - 1 KB minimum instead of 2 KB: n=32 6.01 against 6.97 TB/s;
//  - 64 KB cap per block: n=64 6.88 against 5.07 TB/s (one 128 KB block per
//    SM); a 96 KB cap gave 6.87 (binary32) and 6.66 (bf16, against 6.79).
#ifndef RA_TMA_STAGE_BYTES
#define RA_TMA_STAGE_BYTES 16384
#endif
// worker counts that are not powers of two stage more per block: n=3/5/7
// binary32 7.12/7.14/7.12 TB/s at 24 KB against 6.90/7.01/6.91 at 16 KB,
// while n=8 lost 0.2 % at 24 KB (from n=12 on the 2 KB minimum decides)
#ifndef RA_TMA_STAGE_BYTES_NPOT
#define RA_TMA_STAGE_BYTES_NPOT 24576
#endif
constexpr int64_t kTmaStageBytesOneOut = 65536;
#ifndef RA_UNALIGNED_STAGE_BYTES
#define RA_UNALIGNED_STAGE_BYTES 32768
#endif
#ifndef RA_TMA_MIN_TILE_BYTES
#define RA_TMA_MIN_TILE_BYTES 2048
#endif
#ifndef RA_TMA_MAX_STAGE_BYTES
#define RA_TMA_MAX_STAGE_BYTES 65536
#endif
inline int fused_tile_bytes(int n, bool one_destination, bool vector) {
    const bool pow2 = (n & (n - 1)) == 0;
    const int64_t budget = one_destination ? kTmaStageBytesOneOut
                           : !vector       ? RA_UNALIGNED_STAGE_BYTES
                           : pow2          ? RA_TMA_STAGE_BYTES
                                           : RA_TMA_STAGE_BYTES_NPOT;
    int64_t b = (budget / n) & ~(int64_t)15;
    if (b < RA_TMA_MIN_TILE_BYTES) b = RA_TMA_MIN_TILE_BYTES;
    if (b > 16384) b = 16384;
    if (b * n > RA_TMA_MAX_STAGE_BYTES) b = (RA_TMA_MAX_STAGE_BYTES / n) & ~(int64_t)15;
    return (int)b;
}
constexpr int kMaxDynamicSmem = 227 * 1024;

int64_t fused_tma_assign_tiles(Seg *seg, int nseg, int dtype, int mis, int tile_bytes);

// Rows that disagree modulo 16 bytes: the bulk-copied part of a segment
// keeps one 16-byte vector of elements away from each end, so the copies,
// widened to 16-byte boundaries, stay inside the segment.  The margins (and
// segments too short to have an interior) are done element by element.
__host__ __device__ inline void unaligned_interior(int64_t b, int64_t e, int V, int64_t *ab, int64_t *ae) {
    *ab = b + V;
    *ae = e - V;
    if (*ae < *ab) *ab = *ae = b;
}
// shared memory of the unaligned kernel: a slot of B + 16 bytes per row
// (room for the widening), a weight slot for SGD, the mbarrier, the per-row
// byte offsets and staging offsets, and (8-byte aligned) the rows' tile
// pointers
inline size_t unaligned_smem_bytes(int n, int tile_bytes, int out, int esz) {
    return (size_t)n * ((size_t)tile_bytes + 16) + (out == kOutAllSgd ? (size_t)(tile_bytes / esz) * 4 + 16 : 0) + 16 +
           (size_t)(2 * n + 1) * sizeof(int) + 8 + (size_t)n * sizeof(char *);
}
int64_t fused_unaligned_assign_tiles(Seg *seg, int nseg, int dtype, int tile_bytes);

// The current device's error word: one unsigned int in device memory that
// every kernel with a bounded wait ORs bit 0 into when the wait gives up.
// It is a file-scope __device__ variable of ra_api.cu; its address is looked
// up once per device (cudaGetSymbolAddress) and passed to the kernels in
// their parameters, so all translation units report to the same word.
cudaError_t device_error_word(unsigned int **out);
cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, unsigned int *err, cudaStream_t s);

// fill seg[].tile0 and return the tile count of the staged kernel
int64_t staged_assign_tiles(Seg *seg, int nseg, int dtype, bool vector, int mis, int tile_vec);

cudaError_t launch_fused_f32(const FusedLaunch &L, int64_t ntiles, cudaStream_t s);
cudaError_t launch_fused_bf16(const FusedLaunch &L, int64_t ntiles, cudaStream_t s);


struct StagedLaunch {
    void *rows[RA_MAX_N];
    float *msg;
    const char *msg_lo, *msg_hi;  // the caller's workspace
    unsigned int *err;            // the device's error word
    int64_t p;                    // elements per row
    int n;
    int dtype;
    bool vector;
    int mis;
    const Seg *seg;
    int nseg;
    int64_t ntiles;
    int tile_vec;  // vector mode: 16-byte vectors per tile (staged_tile_vec)
};
cudaError_t launch_staged_step(const StagedLaunch &L, int op, int t, cudaStream_t s);

struct GatherLaunch {
    void *rows[RA_MAX_N];
    void *src[RA_MAX_N];  // source base per chunk
    int n;
    int dtype;
    bool vector;
    int mis;
    bool skip_owner;
    const Seg *seg;
    int nseg;
    int64_t ntiles;  // scalar kernel: staged-size tiles; vector: kGatherTileBytes tiles
    unsigned int *err;  // the device's error word (device_error_word)
    int64_t p;          // elements per row
};
cudaError_t launch_all_gather(const GatherLaunch &L, cudaStream_t s);

// bytes of the owner's chunk one block of the TMA all-gather stages at a
// time: one block per SM at this size (measured on GB300, N=8 f32: 16 KB
// 6.78, 32 KB 6.85, 64 KB 6.88-6.89, 96 KB 6.91, 128 KB 7.02, 192 KB 7.01-
// 7.02 TB/s; bf16 N=16 and f32 N=4 gain the same 1.7 % from 64 to 128 KB)
#ifndef RA_GATHER_TILE_BYTES
#define RA_GATHER_TILE_BYTES 131072
#endif
constexpr int kGatherTileBytes = RA_GATHER_TILE_BYTES;

// set the value ra_last_cuda_error() reports on this thread
void record_cuda_error(cudaError_t e);

// argument checks shared by the calls that take n worker arrays of p elements
ra_status check_rows(void *const *bufs, int n, int64_t p, int dtype);

}  // namespace ra
