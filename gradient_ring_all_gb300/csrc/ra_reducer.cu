// ra_reducer.cu -- per-bucket all-reduce that overlaps the backward pass.
//
// Gibiansky, "Applying the Allreduce to Deep Learning": backpropagation
// produces the output layer's gradients first, and the all-reduce can run on
// a subset of the parameters, so the all-reduce of the last layers starts
// while earlier layers are still being computed.  The reducer holds the
// reverse-order bucket plan of a model's layer tensors; the training loop
// marks each tensor's gradient ready on its compute stream, and as soon as
// every tensor of a bucket is ready the bucket's ring all-reduce is queued on
// the reducer's own stream behind an event recorded on the compute stream.
// ra_reducer_finish makes the compute stream wait for all of them.
#include <string.h>

#include <new>
#include <vector>

#include "ra_internal.h"

struct ra_reducer {
    int device;
    int n;
    int dtype;
    void *bufs[RA_MAX_N];
    std::vector<ra_bucket> buckets;      // closing order: output side first
    std::vector<int> tensor_bucket;      // bucket of each tensor (-1: empty tensor)
    std::vector<int> bucket_tensors;     // non-empty tensors per bucket
    std::vector<int> bucket_ready;       // tensors marked this step
    std::vector<char> bucket_launched;
    std::vector<char> marked;
    cudaStream_t side;
    std::vector<cudaEvent_t> ready;      // per bucket
    cudaEvent_t done;
};

namespace {

ra_status fail(cudaError_t e) {
    ra::record_cuda_error(e);
    return RA_ERR_CUDA;
}

ra_status same_device(const ra_reducer *r) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(e);
    return dev == r->device ? RA_OK : RA_ERR_INVALID_ARG;
}

ra_status launch_bucket(ra_reducer *r, int b) {
    r->bucket_launched[b] = 1;
    return ra_allreduce_avg_buckets(r->bufs, r->n, r->dtype, &r->buckets[b], 1, r->side);
}

void release(ra_reducer *r) {
    for (cudaEvent_t ev : r->ready)
        if (ev) cudaEventDestroy(ev);
    if (r->done) cudaEventDestroy(r->done);
    if (r->side) cudaStreamDestroy(r->side);
    delete r;
}

}  // namespace

extern "C" {

ra_status ra_reducer_create(void *const *bufs, int n, int dtype, const int64_t *numel, int ntensors,
                            int64_t cap_bytes, ra_reducer **out) {
    if (out == nullptr || ntensors < 0 || (ntensors > 0 && numel == nullptr) || cap_bytes <= 0)
        return RA_ERR_INVALID_ARG;
    *out = nullptr;
    if (dtype != RA_F32 && dtype != RA_BF16) return RA_ERR_INVALID_ARG;
    int64_t total = 0;
    for (int k = 0; k < ntensors; ++k) {
        if (numel[k] < 0 || numel[k] > INT64_MAX / 16 - total) return RA_ERR_INVALID_ARG;
        total += numel[k];
    }
    ra_status st = ra::check_rows(bufs, n, total, dtype);
    if (st != RA_OK) return st;

    ra_reducer *r = new (std::nothrow) ra_reducer();
    if (!r) return RA_ERR_INVALID_ARG;
    r->n = n;
    r->dtype = dtype;
    for (int k = 0; k < n; ++k) r->bufs[k] = bufs[k];
    r->buckets.resize((size_t)ntensors + 1);
    int nb = 0;
    st = ra_bucket_plan(numel, ntensors, dtype == RA_F32 ? 4 : 2, cap_bytes, r->buckets.data(), ntensors + 1, &nb);
    if (st != RA_OK) {
        release(r);
        return st;
    }
    r->buckets.resize((size_t)nb);
    // tensors to buckets: bucket b covers whole tensors [offset, offset + count)
    r->tensor_bucket.assign((size_t)ntensors, -1);
    r->bucket_tensors.assign((size_t)nb, 0);
    int64_t off = 0;
    for (int t = 0; t < ntensors; ++t) {
        if (numel[t] > 0)
            for (int b = 0; b < nb; ++b)
                if (off >= r->buckets[b].offset && off < r->buckets[b].offset + r->buckets[b].count) {
                    r->tensor_bucket[t] = b;
                    ++r->bucket_tensors[b];
                    break;
                }
        off += numel[t];
    }
    r->bucket_ready.assign((size_t)nb, 0);
    r->bucket_launched.assign((size_t)nb, 0);
    r->marked.assign((size_t)ntensors, 0);
    r->ready.assign((size_t)nb, nullptr);

    cudaError_t e = cudaGetDevice(&r->device);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&r->side, cudaStreamNonBlocking);
    for (int b = 0; b < nb && e == cudaSuccess; ++b) e = cudaEventCreateWithFlags(&r->ready[b], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r->done, cudaEventDisableTiming);
    if (e != cudaSuccess) {
        release(r);
        return fail(e);
    }
    *out = r;
    return RA_OK;
}

ra_status ra_reducer_buckets(const ra_reducer *r, ra_bucket *out, int max_out, int *n_out) {
    if (!r || !n_out || max_out < 0 || (max_out > 0 && !out)) return RA_ERR_INVALID_ARG;
    const int nb = (int)r->buckets.size();
    if (max_out < nb) return RA_ERR_INVALID_ARG;
    for (int b = 0; b < nb; ++b) out[b] = r->buckets[b];
    *n_out = nb;
    return RA_OK;
}

ra_status ra_reducer_mark_ready(ra_reducer *r, int tensor, void *stream) {
    if (!r || tensor < 0 || tensor >= (int)r->marked.size() || r->marked[tensor]) return RA_ERR_INVALID_ARG;
    ra_status st = same_device(r);
    if (st != RA_OK) return st;
    r->marked[tensor] = 1;
    const int b = r->tensor_bucket[tensor];
    if (b < 0) return RA_OK;  // an empty tensor has nothing to reduce
    if (++r->bucket_ready[b] < r->bucket_tensors[b]) return RA_OK;
    // the bucket's last gradient is queued on `stream`: its ring may start
    // once that work has run
    cudaError_t e = cudaEventRecord(r->ready[b], static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = cudaStreamWaitEvent(r->side, r->ready[b], 0);
    if (e != cudaSuccess) return fail(e);
    return launch_bucket(r, b);
}

ra_status ra_reducer_finish(ra_reducer *r, void *stream) {
    if (!r) return RA_ERR_INVALID_ARG;
    ra_status st = same_device(r);
    if (st != RA_OK) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    // buckets with tensors never marked are reduced now, after the work
    // already queued on `stream`
    bool pending = false;
    for (size_t b = 0; b < r->buckets.size(); ++b) pending |= !r->bucket_launched[b];
    if (pending) {
        cudaError_t e = cudaEventRecord(r->done, s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(r->side, r->done, 0);
        if (e != cudaSuccess) return fail(e);
        for (size_t b = 0; b < r->buckets.size(); ++b)
            if (!r->bucket_launched[b] && (st = launch_bucket(r, (int)b)) != RA_OK) return st;
    }
    cudaError_t e = cudaEventRecord(r->done, r->side);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, r->done, 0);
    if (e != cudaSuccess) return fail(e);
    // ready for the next step
    for (size_t b = 0; b < r->buckets.size(); ++b) r->bucket_ready[b] = 0, r->bucket_launched[b] = 0;
    for (size_t t = 0; t < r->marked.size(); ++t) r->marked[t] = 0;
    return RA_OK;
}

ra_status ra_reducer_destroy(ra_reducer *r) {
    if (!r) return RA_OK;
    // the side stream may still hold queued all-reduces: let them finish
    cudaError_t e = cudaStreamSynchronize(r->side);
    release(r);
    return e == cudaSuccess ? RA_OK : fail(e);
}

}  // extern "C"
