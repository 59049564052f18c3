// ra_api.cu -- the C ABI (include/ring_allreduce.h): argument checks, the
// cutting of a request into ring-chunk segments, and kernel dispatch.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <utility>
#include <vector>

#include "ra_internal.h"

namespace ra {

// The error word every bounded wait reports to (one per device, since a
// __device__ variable exists once in each device's copy of the module).
static __device__ unsigned int g_device_error_word = 0;

namespace {
constexpr int kMaxDevices = 64;
std::atomic<unsigned int *> g_error_word_addr[kMaxDevices];
std::mutex g_error_word_mu;
}  // namespace

cudaError_t device_error_word(unsigned int **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    unsigned int *a = g_error_word_addr[dev].load(std::memory_order_acquire);
    if (a == nullptr) {
        std::lock_guard<std::mutex> lk(g_error_word_mu);
        a = g_error_word_addr[dev].load(std::memory_order_acquire);
        if (a == nullptr) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_device_error_word);
            if (e != cudaSuccess) return e;
            a = static_cast<unsigned int *>(p);
            g_error_word_addr[dev].store(a, std::memory_order_release);
        }
    }
    *out = a;
    return cudaSuccess;
}

namespace {

thread_local int g_last_cuda_error = 0;

ra_status cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return RA_ERR_CUDA;
}

int elem_size(int dtype) { return dtype == RA_F32 ? 4 : (dtype == RA_BF16 ? 2 : 0); }

int vec_elems(int dtype) { return 16 / elem_size(dtype); }

// chunk c of a p-element array split for n workers (Gibiansky,
// "Scatter-Reduce": the array is cut into N chunks; the first p mod n
// chunks take one extra element)
void chunk_of(int64_t p, int n, int c, int64_t *b, int64_t *e) {
    const int64_t q = p / n, r = p % n;
    *b = (int64_t)c * q + std::min<int64_t>(c, r);
    *e = *b + q + (c < r ? 1 : 0);
}

// byte ranges must be pairwise disjoint
bool ranges_disjoint(std::vector<std::pair<uintptr_t, uintptr_t>> r) {
    std::sort(r.begin(), r.end());
    for (size_t k = 1; k < r.size(); ++k)
        if (r[k].first < r[k - 1].second) return false;
    return true;
}

// 16-byte vector path: all rows sit the same number of elements past a
// 16-byte boundary (*mis), so one element index starts a vector in all of
// them.
bool common_misalignment(void *const *bufs, int n, int dtype, int *mis) {
    const int esz = elem_size(dtype), V = vec_elems(dtype);
    const int m0 = (int)((reinterpret_cast<uintptr_t>(bufs[0]) / esz) % V);
    for (int k = 1; k < n; ++k)
        if ((int)((reinterpret_cast<uintptr_t>(bufs[k]) / esz) % V) != m0) return false;
    *mis = m0;
    return true;
}

// segments of one ring over [off, off + count): chunk c of that ring
void ring_segments(int64_t off, int64_t count, int n, std::vector<Seg> *out) {
    for (int c = 0; c < n; ++c) {
        int64_t b, e;
        chunk_of(count, n, c, &b, &e);
        if (e > b) out->push_back(Seg{off + b, off + e, 0, c, 0});
    }
}

ra_status run_fused(void *const *bufs, int n, int64_t p, int dtype, float *w, float lr, const Seg *segs, int nseg,
                    bool vector, int mis, cudaStream_t s, void *const *aux = nullptr, bool bf16_wire = false) {
    FusedLaunch L;
    L.p = p;
    for (int k = 0; k < n; ++k) {
        L.rows[k] = bufs[k];
        L.aux[k] = aux ? aux[k] : nullptr;
    }
    L.out = bf16_wire ? kOutAllWire : (aux ? kOutOne : (w ? kOutAllSgd : kOutAll));
    L.n = n;
    L.dtype = dtype;
    L.w = w;
    L.lr = lr;
    L.vector = vector;
    L.mis = mis;
    std::vector<Seg> tab(segs, segs + nseg);
    L.tile_bytes = fused_tile_bytes(n, L.out == kOutOne, vector);
    const int64_t ntiles = vector ? fused_tma_assign_tiles(tab.data(), nseg, dtype, mis, L.tile_bytes)
                                  : fused_unaligned_assign_tiles(tab.data(), nseg, dtype, L.tile_bytes);
    L.seg = tab.data();
    L.nseg = nseg;
    if (ntiles == 0) return RA_OK;
    cudaError_t e = device_error_word(&L.err);
    if (e != cudaSuccess) return cuda_fail(e);
    e = dtype == RA_F32 ? launch_fused_f32(L, ntiles, s) : launch_fused_bf16(L, ntiles, s);
    return e == cudaSuccess ? RA_OK : cuda_fail(e);
}

// Per-chunk base addresses for the shard calls: element i of chunk c lives at
// base[c] + i * esz -- the owning worker's own array, or its shard buffer
// shifted back by the chunk's first index.  Checks the shards (non-null,
// aligned, disjoint from each other and from the rows) and whether the
// vector path still applies.
ra_status shard_bases(void *const *bufs, int n, int64_t p, int dtype, void *const *shards, void **base,
                      bool *vector, int mis) {
    const int esz = elem_size(dtype), V = vec_elems(dtype);
    std::vector<std::pair<uintptr_t, uintptr_t>> r;
    if (shards) {
        for (int k = 0; k < n; ++k) {
            const uintptr_t a = reinterpret_cast<uintptr_t>(bufs[k]);
            r.emplace_back(a, a + (uintptr_t)p * esz);
        }
    }
    for (int c = 0; c < n; ++c) {
        const int owner = (c + n - 1) % n;
        int64_t b, e;
        chunk_of(p, n, c, &b, &e);
        if (!shards) {
            base[c] = bufs[owner];
            continue;
        }
        const uintptr_t a = reinterpret_cast<uintptr_t>(shards[owner]);
        if (e > b) {
            if (a == 0 || a % esz != 0) return RA_ERR_INVALID_ARG;
            r.emplace_back(a, a + (uintptr_t)(e - b) * esz);
        }
        const uintptr_t shifted = a - (uintptr_t)b * esz;  // never dereferenced below index b
        base[c] = reinterpret_cast<void *>(shifted);
        if (e > b && (int)((shifted / esz) % V) != mis) *vector = false;
    }
    if (shards && !ranges_disjoint(std::move(r))) return RA_ERR_OVERLAP;
    return RA_OK;
}

}  // namespace

// Checks shared by every call that reads `bufs` of p elements.
ra_status check_rows(void *const *bufs, int n, int64_t p, int dtype) {
    if (n < 1 || n > RA_MAX_N || p < 0 || elem_size(dtype) == 0 || bufs == nullptr) return RA_ERR_INVALID_ARG;
    const int esz = elem_size(dtype);
    if (p > INT64_MAX / 16) return RA_ERR_INVALID_ARG;
    if (p == 0) return RA_OK;
    std::vector<std::pair<uintptr_t, uintptr_t>> r;
    for (int k = 0; k < n; ++k) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(bufs[k]);
        if (a == 0 || a % esz != 0) return RA_ERR_INVALID_ARG;
        r.emplace_back(a, a + (uintptr_t)p * esz);
    }
    return ranges_disjoint(std::move(r)) ? RA_OK : RA_ERR_OVERLAP;
}

void record_cuda_error(cudaError_t e) { g_last_cuda_error = (int)e; }

int64_t fused_unaligned_assign_tiles(Seg *seg, int nseg, int dtype, int tile_bytes) {
    const int V = vec_elems(dtype), esz = elem_size(dtype);
    int64_t t = 0;
    for (int k = 0; k < nseg; ++k) {
        seg[k].tile0 = t;
        int64_t ab, ae;
        unaligned_interior(seg[k].begin, seg[k].end, V, &ab, &ae);
        t += std::max<int64_t>(1, ((ae - ab) * esz + tile_bytes - 1) / tile_bytes);
    }
    return t;
}

int64_t fused_tma_assign_tiles(Seg *seg, int nseg, int dtype, int mis, int tile_bytes) {
    const int V = vec_elems(dtype), esz = elem_size(dtype);
    int64_t t = 0;
    for (int k = 0; k < nseg; ++k) {
        seg[k].tile0 = t;
        int64_t ab, ae;
        vector_interior(seg[k].begin, seg[k].end, mis, V, &ab, &ae);
        t += std::max<int64_t>(1, ((ae - ab) * esz + tile_bytes - 1) / tile_bytes);
    }
    return t;
}

int64_t staged_assign_tiles(Seg *seg, int nseg, int dtype, bool vector, int mis, int tile_vec) {
    const int V = vec_elems(dtype);
    const int64_t ts = (int64_t)kThreadsPerBlock * kScalarPerThread;
    int64_t t = 0;
    for (int k = 0; k < nseg; ++k) {
        seg[k].tile0 = t;
        int64_t tiles;
        if (vector) {
            int64_t ab, ae;
            vector_interior(seg[k].begin, seg[k].end, mis, V, &ab, &ae);
            tiles = std::max<int64_t>(1, ((ae - ab) / V + tile_vec - 1) / tile_vec);
        } else {
            tiles = std::max<int64_t>(1, (seg[k].end - seg[k].begin + ts - 1) / ts);
        }
        t += tiles;
    }
    return t;
}

}  // namespace ra

using namespace ra;

extern "C" {

ra_status ra_allreduce_avg(void *const *bufs, int n, int64_t p, int dtype, void *stream) {
    ra_status st = check_rows(bufs, n, p, dtype);
    if (st != RA_OK || n == 1 || p == 0) return st;
    std::vector<Seg> segs;
    ring_segments(0, p, n, &segs);
    int mis = 0;
    const bool vector = common_misalignment(bufs, n, dtype, &mis);
    return run_fused(bufs, n, p, dtype, nullptr, 0.f, segs.data(), (int)segs.size(), vector, mis,
                     static_cast<cudaStream_t>(stream));
}

ra_status ra_allreduce_sgd(void *const *bufs, int n, int64_t p, int dtype, float *w, float lr, void *stream) {
    ra_status st = check_rows(bufs, n, p, dtype);
    if (st != RA_OK) return st;
    if (p == 0) return RA_OK;
    const uintptr_t wa = reinterpret_cast<uintptr_t>(w);
    if (wa == 0 || wa % 4 != 0) return RA_ERR_INVALID_ARG;
    std::vector<std::pair<uintptr_t, uintptr_t>> r;
    const int esz = elem_size(dtype);
    for (int k = 0; k < n; ++k) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(bufs[k]);
        r.emplace_back(a, a + (uintptr_t)p * esz);
    }
    r.emplace_back(wa, wa + (uintptr_t)p * 4);
    if (!ranges_disjoint(std::move(r))) return RA_ERR_OVERLAP;
    std::vector<Seg> segs;
    ring_segments(0, p, n, &segs);
    int mis = 0;
    bool vector = common_misalignment(bufs, n, dtype, &mis);
    // the weights are read as float4 at the rows' vector boundaries
    if (vector && (int)((wa / 4) % 4) != mis % 4) vector = false;
    return run_fused(bufs, n, p, dtype, w, lr, segs.data(), (int)segs.size(), vector, mis,
                     static_cast<cudaStream_t>(stream));
}

size_t ra_staged_workspace_bytes(int n, int64_t p, int dtype) {
    (void)n;
    if (dtype != RA_BF16 || p <= 0) return 0;
    return (size_t)p * 4 + 64;
}

ra_status ra_allreduce_avg_staged(void *const *bufs, int n, int64_t p, int dtype, void *ws, size_t ws_bytes,
                                  ra_traffic *per_worker, void *stream) {
    ra_status st = check_rows(bufs, n, p, dtype);
    if (st != RA_OK) return st;
    const size_t need = ra_staged_workspace_bytes(n, p, dtype);
    uintptr_t wsa = reinterpret_cast<uintptr_t>(ws);
    if (need > 0 && n > 1) {
        if (wsa == 0 || ws_bytes < need) return RA_ERR_INVALID_ARG;
        std::vector<std::pair<uintptr_t, uintptr_t>> r;
        const int esz = elem_size(dtype);
        for (int k = 0; k < n; ++k) {
            const uintptr_t a = reinterpret_cast<uintptr_t>(bufs[k]);
            r.emplace_back(a, a + (uintptr_t)p * esz);
        }
        r.emplace_back(wsa, wsa + ws_bytes);
        if (!ranges_disjoint(std::move(r))) return RA_ERR_OVERLAP;
    }
    // per-worker traffic: walk the schedule (Gibiansky, "Scatter-Reduce" and
    // "Allgather": in iteration t worker m sends chunk (m - t) mod N, resp.
    // (m + 1 - t) mod N, to worker m + 1)
    if (per_worker) {
        for (int m = 0; m < n; ++m) per_worker[m].sent = per_worker[m].received = 0;
        for (int phase = 0; phase < 2; ++phase)
            for (int t = 0; t < n - 1; ++t)
                for (int m = 0; m < n; ++m) {
                    const int c = (((phase == 0 ? m - t : m + 1 - t) % n) + n) % n;
                    int64_t b, e;
                    chunk_of(p, n, c, &b, &e);
                    per_worker[m].sent += e - b;
                    per_worker[(m + 1) % n].received += e - b;
                }
    }
    if (n == 1 || p == 0) return RA_OK;

    StagedLaunch L;
    for (int k = 0; k < n; ++k) L.rows[k] = bufs[k];
    L.n = n;
    L.dtype = dtype;
    int mis = 0;
    L.vector = common_misalignment(bufs, n, dtype, &mis);
    L.mis = mis;
    // binary32 partial sums for bf16, placed so that msg + i is 16-byte
    // aligned exactly when the rows' element i starts a vector
    L.msg = nullptr;
    L.msg_lo = L.msg_hi = nullptr;
    if (dtype == RA_BF16) {
        const uintptr_t base = (wsa + 15) & ~(uintptr_t)15;
        L.msg = reinterpret_cast<float *>(base + (uintptr_t)(L.vector ? 4 * (mis % 4) : 0));
        L.msg_lo = reinterpret_cast<const char *>(wsa);
        L.msg_hi = reinterpret_cast<const char *>(wsa + ws_bytes);
    }
    L.p = p;
    {
        cudaError_t e = device_error_word(&L.err);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    std::vector<Seg> segs;
    ring_segments(0, p, n, &segs);
    L.tile_vec = staged_tile_vec(p / vec_elems(dtype));
    L.ntiles = staged_assign_tiles(segs.data(), (int)segs.size(), dtype, L.vector, mis, L.tile_vec);
    L.seg = segs.data();
    L.nseg = (int)segs.size();
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int t = 0; t < n - 1; ++t) {
        cudaError_t e = launch_staged_step(L, kOpScatter, t, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    cudaError_t e = launch_staged_step(L, kOpDivide, 0, s);
    if (e != cudaSuccess) return cuda_fail(e);
    for (int t = 0; t < n - 1; ++t) {
        e = launch_staged_step(L, kOpGather, t, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return RA_OK;
}

ra_status ra_bucket_plan(const int64_t *numel, int ntensors, int elem_bytes, int64_t cap_bytes, ra_bucket *out,
                         int max_out, int *n_out) {
    if (ntensors < 0 || elem_bytes <= 0 || cap_bytes <= 0 || n_out == nullptr || (ntensors > 0 && !numel) ||
        max_out < 0 || (max_out > 0 && !out))
        return RA_ERR_INVALID_ARG;
    int64_t total = 0;
    for (int k = 0; k < ntensors; ++k) {
        if (numel[k] < 0 || numel[k] > INT64_MAX / 16 - total) return RA_ERR_INVALID_ARG;
        total += numel[k];
    }
    // walk from the output layer back to the input layer; close the open
    // bucket [lo, hi) once it holds at least cap_bytes
    int nb = 0;
    int64_t hi = total, lo = total;
    for (int k = ntensors - 1; k >= 0; --k) {
        lo -= numel[k];
        if ((hi - lo) * (int64_t)elem_bytes >= cap_bytes) {
            if (nb >= max_out) return RA_ERR_INVALID_ARG;
            out[nb++] = ra_bucket{lo, hi - lo};
            hi = lo;
        }
    }
    if (hi > 0) {
        if (nb >= max_out) return RA_ERR_INVALID_ARG;
        out[nb++] = ra_bucket{0, hi};
    }
    *n_out = nb;
    return RA_OK;
}

ra_status ra_allreduce_avg_buckets(void *const *bufs, int n, int dtype, const ra_bucket *b, int nb, void *stream) {
    if (nb < 0 || (nb > 0 && b == nullptr)) return RA_ERR_INVALID_ARG;
    int64_t extent = 0;
    std::vector<std::pair<int64_t, int64_t>> br;
    for (int k = 0; k < nb; ++k) {
        if (b[k].offset < 0 || b[k].count < 0 || b[k].offset > INT64_MAX / 16 - b[k].count)
            return RA_ERR_INVALID_ARG;
        extent = std::max(extent, b[k].offset + b[k].count);
        if (b[k].count > 0) br.emplace_back(b[k].offset, b[k].offset + b[k].count);
    }
    std::sort(br.begin(), br.end());
    for (size_t k = 1; k < br.size(); ++k)
        if (br[k].first < br[k - 1].second) return RA_ERR_OVERLAP;
    ra_status st = check_rows(bufs, n, extent, dtype);
    if (st != RA_OK || n == 1 || extent == 0) return st;
    std::vector<Seg> segs;
    for (int k = 0; k < nb; ++k) ring_segments(b[k].offset, b[k].count, n, &segs);
    int mis = 0;
    const bool vector = common_misalignment(bufs, n, dtype, &mis);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (size_t k0 = 0; k0 < segs.size(); k0 += kSegLarge) {
        const int cnt = (int)std::min<size_t>(kSegLarge, segs.size() - k0);
        st = run_fused(bufs, n, extent, dtype, nullptr, 0.f, segs.data() + k0, cnt, vector, mis, s);
        if (st != RA_OK) return st;
    }
    return RA_OK;
}

ra_status ra_allreduce_avg_host(void *const *host_bufs, void *const *dev_bufs, int n, int64_t p, int dtype, int mode,
                                void *stream) {
    if (n < 1 || n > RA_MAX_N || p < 0 || elem_size(dtype) == 0 || host_bufs == nullptr ||
        (mode != RA_HOST_AUTO && mode != RA_HOST_DIRECT && mode != RA_HOST_STAGED))
        return RA_ERR_INVALID_ARG;
    ra_status st = check_rows(host_bufs, n, p, dtype);
    if (st != RA_OK) return st;
    if (p == 0) return RA_OK;
    // Direct path: on GB300 the GPU reaches host memory over the coherent
    // NVLink-C2C link, so the fused kernel can read every worker's host
    // array and write the mean back in place, with no staging copies.  That
    // needs a device address for each host array: page-locked (pinned or
    // registered) memory has one; ordinary pageable memory is usable as is
    // when the device walks the host page tables.
    int dev = 0, pageable = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    void *direct[RA_MAX_N];
    bool all_direct = mode != RA_HOST_STAGED;
    for (int k = 0; k < n && all_direct; ++k) {
        cudaPointerAttributes a;
        e = cudaPointerGetAttributes(&a, host_bufs[k]);
        if (e != cudaSuccess) return cuda_fail(e);
        if (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr)
            direct[k] = a.devicePointer;
        else if (a.type == cudaMemoryTypeUnregistered && pageable)
            direct[k] = host_bufs[k];
        else
            all_direct = false;
    }
    if (all_direct) return ra_allreduce_avg(direct, n, p, dtype, stream);
    if (mode == RA_HOST_DIRECT) return RA_ERR_UNSUPPORTED;

    // Staging path: copy in, reduce on the device, copy the mean back.
    if (dev_bufs == nullptr) return RA_ERR_UNSUPPORTED;
    st = check_rows(dev_bufs, n, p, dtype);
    if (st != RA_OK) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t bytes = (size_t)p * elem_size(dtype);
    for (int k = 0; k < n; ++k) {
        e = cudaMemcpyAsync(dev_bufs[k], host_bufs[k], bytes, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (n > 1) {
        st = ra_allreduce_avg(dev_bufs, n, p, dtype, stream);
        if (st != RA_OK) return st;
    }
    for (int k = 0; k < n; ++k) {
        e = cudaMemcpyAsync(host_bufs[k], dev_bufs[k], bytes, cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return RA_OK;
}

ra_status ra_reduce_scatter_avg(void *const *bufs, int n, int64_t p, int dtype, void *const *shards, void *stream) {
    ra_status st = check_rows(bufs, n, p, dtype);
    if (st != RA_OK || p == 0 || (n == 1 && shards == nullptr)) return st;
    int mis = 0;
    bool vector = common_misalignment(bufs, n, dtype, &mis);
    void *base[RA_MAX_N];
    st = shard_bases(bufs, n, p, dtype, shards, base, &vector, mis);
    if (st != RA_OK) return st;
    std::vector<Seg> segs;
    ring_segments(0, p, n, &segs);
    return run_fused(bufs, n, p, dtype, nullptr, 0.f, segs.data(), (int)segs.size(), vector, mis,
                     static_cast<cudaStream_t>(stream), base);
}

ra_status ra_all_gather(void *const *bufs, int n, int64_t p, int dtype, void *const *shards, void *stream) {
    ra_status st = check_rows(bufs, n, p, dtype);
    if (st != RA_OK || p == 0 || (n == 1 && shards == nullptr)) return st;
    GatherLaunch L;
    for (int k = 0; k < n; ++k) L.rows[k] = bufs[k];
    L.n = n;
    L.dtype = dtype;
    int mis = 0;
    L.vector = common_misalignment(bufs, n, dtype, &mis);
    L.mis = mis;
    L.skip_owner = shards == nullptr;
    L.p = p;
    st = shard_bases(bufs, n, p, dtype, shards, L.src, &L.vector, mis);
    if (st != RA_OK) return st;
    std::vector<Seg> segs;
    ring_segments(0, p, n, &segs);
    L.ntiles = L.vector ? fused_tma_assign_tiles(segs.data(), (int)segs.size(), dtype, mis, kGatherTileBytes)
                        : staged_assign_tiles(segs.data(), (int)segs.size(), dtype, false, mis, 0);
    L.seg = segs.data();
    L.nseg = (int)segs.size();
    cudaError_t e = device_error_word(&L.err);
    if (e != cudaSuccess) return cuda_fail(e);
    e = launch_all_gather(L, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? RA_OK : cuda_fail(e);
}

ra_status ra_allreduce_avg_bf16_wire(void *const *bufs, int n, int64_t p, void *stream) {
    ra_status st = check_rows(bufs, n, p, RA_BF16);
    if (st != RA_OK || n == 1 || p == 0) return st;
    std::vector<Seg> segs;
    ring_segments(0, p, n, &segs);
    int mis = 0;
    const bool vector = common_misalignment(bufs, n, RA_BF16, &mis);
    return run_fused(bufs, n, p, RA_BF16, nullptr, 0.f, segs.data(), (int)segs.size(), vector, mis,
                     static_cast<cudaStream_t>(stream), nullptr, true);
}

ra_status ra_allreduce_avg_single_reducer(void *const *bufs, int n, int64_t p, int dtype, ra_traffic *per_worker,
                                          void *stream) {
    ra_status st = check_rows(bufs, n, p, dtype);
    if (st != RA_OK) return st;
    // Gibiansky, "The Communication Problem": the reducer (worker 0) receives
    // every other worker's array and sends the mean back to each of them
    if (per_worker) {
        for (int m = 0; m < n; ++m) per_worker[m].sent = per_worker[m].received = m == 0 ? (int64_t)(n - 1) * p : p;
    }
    if (n == 1 || p == 0) return RA_OK;
    // one segment: every element's sum starts at worker 0 and takes the
    // workers in order
    const Seg seg{0, p, 0, 0, 0};
    int mis = 0;
    const bool vector = common_misalignment(bufs, n, dtype, &mis);
    return run_fused(bufs, n, p, dtype, nullptr, 0.f, &seg, 1, vector, mis, static_cast<cudaStream_t>(stream));
}

ra_status ra_check_device_errors(void) {
    unsigned int flags = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&flags, g_device_error_word, sizeof(flags));
    if (e == cudaSuccess && flags) e = cudaMemcpyToSymbol(g_device_error_word, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e);
    return (flags & 2u) ? RA_ERR_BOUNDS : (flags ? RA_ERR_TIMEOUT : RA_OK);
}

ra_status ra_selftest_bounds_check(void *const *bufs, int n, int64_t p, int dtype, void *stream) {
    ra_status st = check_rows(bufs, n, p, dtype);
    if (st != RA_OK) return st;
    if (n < 2 || p < 2) return RA_ERR_INVALID_ARG;
    if (!RA_CHECKED) return RA_ERR_UNSUPPORTED;
    // the ring's segments over all p elements, the kernel's bound one short
    std::vector<Seg> segs;
    ring_segments(0, p, n, &segs);
    int mis = 0;
    const bool vector = common_misalignment(bufs, n, dtype, &mis);
    return run_fused(bufs, n, p - 1, dtype, nullptr, 0.f, segs.data(), (int)segs.size(), vector, mis,
                     static_cast<cudaStream_t>(stream));
}

ra_status ra_selftest_wait_timeout(int timeout_us, void *stream) {
    if (timeout_us < 1 || timeout_us > 10000000) return RA_ERR_INVALID_ARG;
    unsigned int *err = nullptr;
    cudaError_t e = device_error_word(&err);
    if (e == cudaSuccess)
        e = launch_wait_timeout_selftest((uint64_t)timeout_us * 1000ull, err, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? RA_OK : cuda_fail(e);
}

void ra_chunk_range(int64_t p, int n, int c, int64_t *begin, int64_t *end) {
    if (n < 1 || c < 0 || c >= n || p < 0) {
        if (begin) *begin = 0;
        if (end) *end = 0;
        return;
    }
    int64_t b, e;
    chunk_of(p, n, c, &b, &e);
    if (begin) *begin = b;
    if (end) *end = e;
}

const char *ra_status_str(int status) {
    switch (status) {
        case RA_OK: return "RA_OK";
        case RA_ERR_INVALID_ARG: return "RA_ERR_INVALID_ARG";
        case RA_ERR_UNSUPPORTED: return "RA_ERR_UNSUPPORTED";
        case RA_ERR_OVERLAP: return "RA_ERR_OVERLAP";
        case RA_ERR_CUDA: return "RA_ERR_CUDA";
        case RA_ERR_TIMEOUT: return "RA_ERR_TIMEOUT";
        case RA_ERR_BOUNDS: return "RA_ERR_BOUNDS";
        default: return "RA_UNKNOWN_STATUS";
    }
}

int ra_last_cuda_error(void) { return g_last_cuda_error; }

}  // extern "C"
