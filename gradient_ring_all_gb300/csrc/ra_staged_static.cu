// ra_staged_static.cu -- ra_allreduce_avg_staged_static: the staged ring for
// callers that cannot allocate device memory.
//
// The staged bf16 ring keeps its binary32 partial sums in a scratch array of
// p elements.  ra_allreduce_avg_staged takes that array from the caller; this
// entry point instead uses a fixed array compiled into the library, so the
// caller passes only the workers' buffers.  The call itself allocates
// nothing: no cudaMalloc/cudaFree, no allocating library routine, no heap
// memory on the host (fixed-size tables on the stack).
//
// Set-up: the first call on a device (that passes the argument checks) runs,
// with that device current, cudaGetSymbolAddress on the array and caches the
// address per device.
// That first call should therefore come before any stream capture.
//
// Sharing: every call on a device uses the same array.  Scatter-reduce
// iteration 0 writes every partial sum before any later iteration reads one,
// so nothing has to be cleared between calls; but two calls whose work
// overlaps on the GPU (different streams, no ordering between them) race on
// the array and give wrong results.
#include <mutex>
#include <string.h>

#include "ra_kernels.cuh"

namespace ra {
namespace {

// binary32 partial sums; 4 extra elements leave room for the shift that
// lines the array up with the rows' 16-byte vectors
static __device__ __align__(256) float g_staged_scratch[RA_STAGED_STATIC_MAX_P + 4];

constexpr int kMaxDevices = 64;

struct DeviceSetup {
    bool done;
    float *scratch;  // device address of g_staged_scratch on this device
};

std::mutex g_setup_mu;
DeviceSetup g_setup[kMaxDevices];

// once per device, with that device current
cudaError_t setup_device(int dev, DeviceSetup *out) {
    std::lock_guard<std::mutex> lk(g_setup_mu);
    DeviceSetup &d = g_setup[dev];
    if (!d.done) {
        void *addr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&addr, g_staged_scratch);
        if (e != cudaSuccess) return e;
        d.scratch = static_cast<float *>(addr);
        d.done = true;
    }
    *out = d;
    return cudaSuccess;
}

// one tile per block, as for the other staged launches
template <class E, bool VEC>
cudaError_t launch_step(const StagedParams &p, int tile_vec, cudaStream_t s) {
    const int64_t grid = p.ntiles < kMaxGrid ? p.ntiles : kMaxGrid;
    if (VEC && tile_vec == kStagedTileVecLarge)
        return launch_pdl(staged_step_kernel<E, VEC, kStagedTileVecLarge>, grid, kThreadsPerBlock, 0, s, p);
    return launch_pdl(staged_step_kernel<E, VEC, kStagedTileVecSmall>, grid, kThreadsPerBlock, 0, s, p);
}

cudaError_t launch_step_any(const StagedParams &p, int dtype, bool vec, int tile_vec, cudaStream_t s) {
    if (dtype == RA_F32) return vec ? launch_step<F32, true>(p, tile_vec, s) : launch_step<F32, false>(p, tile_vec, s);
    return vec ? launch_step<BF16, true>(p, tile_vec, s) : launch_step<BF16, false>(p, tile_vec, s);
}

}  // namespace
}  // namespace ra

using namespace ra;

extern "C" ra_status ra_allreduce_avg_staged_static(void *const *bufs, int n, int64_t p, int dtype,
                                                    ra_traffic *per_worker, void *stream) {
    // argument checks, without heap memory
    if (n < 1 || n > RA_MAX_N || p < 0 || bufs == nullptr || (dtype != RA_F32 && dtype != RA_BF16))
        return RA_ERR_INVALID_ARG;
    const int esz = dtype == RA_F32 ? 4 : 2;
    if (p > INT64_MAX / 16) return RA_ERR_INVALID_ARG;
    if (p > 0) {
        for (int k = 0; k < n; ++k) {
            const uintptr_t a = reinterpret_cast<uintptr_t>(bufs[k]);
            if (a == 0 || a % esz != 0) return RA_ERR_INVALID_ARG;
        }
        for (int a = 0; a < n; ++a)
            for (int b = a + 1; b < n; ++b) {
                const uintptr_t x = reinterpret_cast<uintptr_t>(bufs[a]), y = reinterpret_cast<uintptr_t>(bufs[b]);
                if (x < y + (uintptr_t)p * esz && y < x + (uintptr_t)p * esz) return RA_ERR_OVERLAP;
            }
    }
    // the scratch holds the bf16 ring's partial sums: p is bounded by its size
    if (dtype == RA_BF16 && p > (int64_t)RA_STAGED_STATIC_MAX_P) return RA_ERR_UNSUPPORTED;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return RA_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return RA_ERR_UNSUPPORTED;
    DeviceSetup d;
    e = setup_device(dev, &d);
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return RA_ERR_CUDA;
    }

    // chunks of the ring: chunk c = [c*q + min(c, r), ...) (Gibiansky,
    // "Scatter-Reduce": N chunks, the first p mod n one element longer)
    const int64_t q = p / n, r = p % n;
    if (per_worker) {
        // in iteration t worker m sends chunk (m - t) mod N (scatter-reduce),
        // resp. (m + 1 - t) mod N (all-gather), to worker m + 1
        for (int m = 0; m < n; ++m) per_worker[m].sent = per_worker[m].received = 0;
        for (int phase = 0; phase < 2; ++phase)
            for (int t = 0; t < n - 1; ++t)
                for (int m = 0; m < n; ++m) {
                    const int c = (((phase == 0 ? m - t : m + 1 - t) % n) + n) % n;
                    const int64_t len = q + (c < r ? 1 : 0);
                    per_worker[m].sent += len;
                    per_worker[(m + 1) % n].received += len;
                }
    }
    if (n == 1 || p == 0) return RA_OK;

    StagedParams prm;
    memset(&prm, 0, sizeof(prm));
    for (int k = 0; k < n; ++k) prm.rows[k] = bufs[k];
    prm.n = n;
    const int V = 16 / esz;
    const int mis = (int)((reinterpret_cast<uintptr_t>(bufs[0]) / esz) % V);
    bool vec = true;
    for (int k = 1; k < n; ++k)
        if ((int)((reinterpret_cast<uintptr_t>(bufs[k]) / esz) % V) != mis) vec = false;
    prm.mis = vec ? mis : 0;
    // partial sums at scratch + shift, so that msg + i is 16-byte aligned
    // exactly when the rows' element i starts a vector
    prm.msg = dtype == RA_BF16 ? d.scratch + (vec ? mis % 4 : 0) : nullptr;
    prm.msg_lo = reinterpret_cast<const char *>(d.scratch);
    prm.msg_hi = reinterpret_cast<const char *>(d.scratch + RA_STAGED_STATIC_MAX_P + 4);
    prm.p = p;
    e = device_error_word(&prm.err);
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return RA_ERR_CUDA;
    }
    int nseg = 0;
    for (int c = 0; c < n; ++c) {
        const int64_t b = (int64_t)c * q + (c < r ? c : r), len = q + (c < r ? 1 : 0);
        if (len > 0) prm.seg[nseg++] = Seg{b, b + len, 0, c, 0};
    }
    prm.nseg = nseg;
    const int tile_vec = staged_tile_vec(p / V);
    prm.ntiles = staged_assign_tiles(prm.seg, nseg, dtype, vec, prm.mis, tile_vec);

    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int t = 0; t < n - 1 && e == cudaSuccess; ++t) {
        prm.op = kOpScatter;
        prm.t = t;
        e = launch_step_any(prm, dtype, vec, tile_vec, s);
    }
    if (e == cudaSuccess) {
        prm.op = kOpDivide;
        prm.t = 0;
        e = launch_step_any(prm, dtype, vec, tile_vec, s);
    }
    for (int t = 0; t < n - 1 && e == cudaSuccess; ++t) {
        prm.op = kOpGather;
        prm.t = t;
        e = launch_step_any(prm, dtype, vec, tile_vec, s);
    }
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return RA_ERR_CUDA;
    }
    return RA_OK;
}
