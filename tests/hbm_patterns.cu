// hbm_patterns.cu -- HBM throughput of bare data movement with the same TMA
// bulk copies the library's fused kernel uses, no arithmetic: read only,
// write only, a 1:1 copy, and the all-reduce's in-place pattern (one block
// per tile, a tile = B bytes of each of 8 rows, loaded to shared memory and
// stored back), plus two ways of grouping a block's writes in time and
// smaller blocks (more blocks, more bytes in flight per SM).  Test
// infrastructure: the ceiling the fused all-reduce is compared against.
//
//   hbm_patterns P REPS  -> one JSON line, GB/s of each pattern
//
// Every mbarrier wait is bounded (2 s) and recorded on expiry; every block
// touches only its own tile of each row, inside the buffers.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>

__device__ unsigned int g_wait_expired;

__device__ __forceinline__ uint32_t saddr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ bool wait_bounded(uint32_t bar) {
    const uint64_t t0 = now_ns();
    for (;;) {
        uint32_t ok;
        asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0; selp.u32 %0, 1, 0, p; }"
                     : "=r"(ok) : "r"(bar) : "memory");
        if (ok) return true;
        if (now_ns() - t0 > 2000000000ull) return false;
    }
}
__device__ __forceinline__ void init_bar(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(saddr(bar)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(saddr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void load(void *dst, const char *src, int bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(saddr(dst)), "l"(src), "r"(bytes), "r"(saddr(bar)) : "memory");
}
__device__ __forceinline__ void store(char *dst, const void *src, int bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" :: "l"(dst), "r"(saddr(src)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void store_done() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

enum { kRead = 0, kWrite = 1, kCopy = 2, kInPlace = 3 };

// one tile (B bytes of each of `rows` rows) per block
template <int MODE>
__global__ void one_tile(char *a, char *b, int64_t row_bytes, int rows, int B) {
    extern __shared__ __align__(128) unsigned char sm[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + rows * B);
    const int64_t off = (int64_t)blockIdx.x * B;
    if (threadIdx.x == 0) {
        bool ok = true;
        if (MODE != kWrite) {
            init_bar(bar, (uint32_t)(rows * B));
            for (int k = 0; k < rows; ++k) load(sm + k * B, a + k * row_bytes + off, B, bar);
            if (!wait_bounded(saddr(bar))) {
                atomicOr(&g_wait_expired, 1u);
                wait_bounded(saddr(bar));
                ok = false;
            }
        }
        if (ok && MODE != kRead) {
            char *d = MODE == kCopy ? b : a;
            for (int k = 0; k < rows; ++k) store(d + k * row_bytes + off, sm + k * B, B);
            store_done();
        }
    }
    __syncthreads();
}

// two consecutive tiles per block, in place: GROUPED loads both, then stores
// both; otherwise stores the first as soon as it has landed
template <bool GROUPED>
__global__ void two_tiles(char *a, int64_t row_bytes, int rows, int B) {
    extern __shared__ __align__(128) unsigned char sm[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + 2 * rows * B);
    if (threadIdx.x == 0) {
        const int nbar = GROUPED ? 1 : 2;
        for (int h = 0; h < nbar; ++h) init_bar(bar + h, (uint32_t)(rows * B * (GROUPED ? 2 : 1)));
        for (int h = 0; h < 2; ++h)
            for (int k = 0; k < rows; ++k)
                load(sm + (h * rows + k) * B, a + k * row_bytes + (2 * (int64_t)blockIdx.x + h) * B, B,
                     bar + (GROUPED ? 0 : h));
        bool ok = true;
        for (int h = 0; h < nbar; ++h)
            if (!wait_bounded(saddr(bar + h))) {
                atomicOr(&g_wait_expired, 1u);
                wait_bounded(saddr(bar + h));
                ok = false;
            } else if (!GROUPED && ok) {
                for (int k = 0; k < rows; ++k)
                    store(a + k * row_bytes + (2 * (int64_t)blockIdx.x + h) * B, sm + (h * rows + k) * B, B);
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            }
        if (ok && GROUPED)
            for (int h = 0; h < 2; ++h)
                for (int k = 0; k < rows; ++k)
                    store(a + k * row_bytes + (2 * (int64_t)blockIdx.x + h) * B, sm + (h * rows + k) * B, B);
        if (ok) store_done();
    }
    __syncthreads();
}

static void check(cudaError_t e, const char *what) {
    if (e != cudaSuccess) {
        fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
        exit(1);
    }
}

template <class F>
static double gbs(F launch, int reps, double bytes) {
    launch();
    cudaEvent_t e0, e1;
    check(cudaEventCreate(&e0), "event");
    check(cudaEventCreate(&e1), "event");
    check(cudaEventRecord(e0), "record");
    for (int r = 0; r < reps; ++r) launch();
    check(cudaEventRecord(e1), "record");
    check(cudaEventSynchronize(e1), "sync");
    check(cudaGetLastError(), "launch");
    float ms = 0;
    check(cudaEventElapsedTime(&ms, e0, e1), "elapsed");
    return bytes * reps / (ms / 1e3) / 1e9;
}

int main(int argc, char **argv) {
    const int64_t P = argc > 1 ? atoll(argv[1]) : 300000000;  // fp32 elements per row
    const int reps = argc > 2 ? atoi(argv[2]) : 10;
    const int rows = 8, B = 2048;                      // the fused kernel's tile at N = 8
    const int64_t tiles = (P * 4) / (2 * B) * 2;       // per row, even
    const int64_t row_bytes = tiles * B;
    char *a = nullptr, *b = nullptr;
    check(cudaMalloc(&a, rows * row_bytes), "malloc");
    check(cudaMalloc(&b, rows * row_bytes), "malloc");
    check(cudaMemset(a, 0, rows * row_bytes), "memset");
    check(cudaMemset(b, 0, rows * row_bytes), "memset");
    const size_t s1 = (size_t)rows * B + 16, s2 = (size_t)2 * rows * B + 16;
    check(cudaFuncSetAttribute(one_tile<kRead>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1), "attr");
    check(cudaFuncSetAttribute(one_tile<kWrite>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1), "attr");
    check(cudaFuncSetAttribute(one_tile<kCopy>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1), "attr");
    check(cudaFuncSetAttribute(one_tile<kInPlace>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1), "attr");
    check(cudaFuncSetAttribute(two_tiles<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2), "attr");
    check(cudaFuncSetAttribute(two_tiles<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2), "attr");
    const double one = (double)rows * row_bytes;
    const unsigned g1 = (unsigned)tiles, g2 = (unsigned)(tiles / 2);
    double r[9];
    r[0] = gbs([&] { one_tile<kRead><<<g1, 256, s1>>>(a, b, row_bytes, rows, B); }, reps, one);
    r[1] = gbs([&] { one_tile<kWrite><<<g1, 256, s1>>>(a, b, row_bytes, rows, B); }, reps, one);
    r[2] = gbs([&] { one_tile<kCopy><<<g1, 256, s1>>>(a, b, row_bytes, rows, B); }, reps, 2 * one);
    r[3] = gbs([&] { one_tile<kInPlace><<<g1, 256, s1>>>(a, b, row_bytes, rows, B); }, reps, 2 * one);
    r[4] = gbs([&] { two_tiles<true><<<g2, 256, s2>>>(a, row_bytes, rows, B); }, reps, 2 * one);
    r[5] = gbs([&] { two_tiles<false><<<g2, 256, s2>>>(a, row_bytes, rows, B); }, reps, 2 * one);
    const int th[3] = {32, 64, 128};
    for (int i = 0; i < 3; ++i)
        r[6 + i] = gbs([&] { one_tile<kInPlace><<<g1, th[i], s1>>>(a, b, row_bytes, rows, B); }, reps, 2 * one);
    unsigned int expired = 0;
    check(cudaMemcpyFromSymbol(&expired, g_wait_expired, sizeof(expired)), "symbol");
    printf("{\"rows\": %d, \"row_bytes\": %lld, \"tile_bytes_per_row\": %d, \"reps\": %d, \"read_only\": %.1f, "
           "\"write_only\": %.1f, \"copy\": %.1f, \"in_place\": %.1f, \"in_place_two_tiles_grouped\": %.1f, "
           "\"in_place_two_tiles_pipelined\": %.1f, \"in_place_32_threads\": %.1f, \"in_place_64_threads\": %.1f, "
           "\"in_place_128_threads\": %.1f, \"waits_expired\": %u}\n",
           rows, (long long)row_bytes, B, reps, r[0], r[1], r[2], r[3], r[4], r[5], r[6], r[7], r[8], expired);
    cudaFree(a);
    cudaFree(b);
    return expired ? 2 : 0;
}
