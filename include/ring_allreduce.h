/*
 * ring_allreduce.h -- C ABI of the GB300 ring all-reduce library
 * (libgradient_ring_all.so).
 *
 * The library computes the data-parallel gradient all-reduce-average of the
 * ring algorithm for N logical workers whose gradient arrays all sit in the
 * HBM of one GPU.  The result is what the ring of
 *   Gibiansky, "Bringing HPC Techniques to Deep Learning" (Korean
 *   translation), sections "Ring Allreduce", "Scatter-Reduce", "Allgather"
 * leaves on every worker, divided by N so that every worker holds the mean
 * gradient ("The Communication Problem": the GPUs average their gradients;
 * "[PyTorch] GPU 분산 학습 1 - DP / DDP / FSDP 개념", section DDP: every GPU
 * ends with the identical gradient).
 *
 * Numerics (identical bits to a step-by-step simulation of the ring):
 *   - the array of P elements is split into N chunks; chunk c is
 *     [c*q + min(c,r), (c+1)*q + min(c+1,r)), q = P / N, r = P mod N;
 *   - element i of chunk c is summed in binary32 in ring order, a left fold
 *     that starts at worker c: ((g_c + g_{c+1}) + g_{c+2}) + ... + g_{c+N-1}
 *     (worker indices mod N) -- the order in which the scatter-reduce
 *     accumulates it;
 *   - the sum is divided by N with one IEEE binary32 division (round to
 *     nearest even);
 *   - bf16 gradients are widened exactly, summed in binary32 and the mean is
 *     rounded to bf16 (nearest even) once;
 *   - the SGD variant computes w - (lr * avg) with two roundings.
 *
 * Conventions shared by every call:
 *   - `dtype` is an int holding an ra_dtype value and `stream` a void *
 *     holding a cudaStream_t, so that this header needs no CUDA header and
 *     compiles as plain C; the values are those of the enum and the
 *     runtime's stream handle.
 *   - `bufs` is a HOST array of n DEVICE pointers, one per worker; each
 *     points at p elements of `dtype`, element-aligned.  The array itself
 *     is read during the call only.  The buffers must not overlap.
 *   - All device memory is owned by the caller and must stay valid until
 *     the work queued on `stream` has finished.  Calls are asynchronous on
 *     `stream` (a cudaStream_t; NULL = the legacy default stream): they only
 *     queue kernels and return.  One exception is the first launch of each
 *     kernel variant in a process, which loads its module; with CUDA's lazy
 *     module loading (the default) that load may synchronise the context,
 *     so warm a call up once (or set CUDA_MODULE_LOADING=EAGER) before
 *     relying on overlap.  The first launching call on a device also looks
 *     up the address of the device's error word (cudaGetSymbolAddress);
 *     like that first launch, it belongs before any stream capture.
 *   - Arguments are checked before anything is queued; a non-OK status
 *     means nothing was launched.  RA_ERR_CUDA reports a failed launch or
 *     device query; ra_last_cuda_error() returns its cudaError_t value.
 *   - n == 1 or p == 0: nothing to reduce, RA_OK without a launch (x / 1 is
 *     exact).  The SGD call still updates w when n == 1.
 *   - Pointers whose addresses agree modulo 16 bytes take the vector path
 *     (TMA bulk copies of whole 16-byte granules); any other element-aligned
 *     pointers take the unaligned path (bulk copies widened to 16-byte
 *     boundaries inside each row's own range) with the same results.
 *   - Kernels are launched with programmatic dependent launch: the next
 *     launch on the stream may start while the current one drains, and
 *     every kernel waits for the previous grid on the stream to finish
 *     before touching memory, so stream order holds as usual.
 *   - Every function is thread-safe; the library keeps no state besides
 *     the per-device addresses of its built-in scratch array and of its
 *     error word.
 */
#ifndef RING_ALLREDUCE_H
#define RING_ALLREDUCE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { RA_F32 = 0, RA_BF16 = 1 } ra_dtype;

typedef enum {
    RA_OK = 0,
    RA_ERR_INVALID_ARG = 1, /* null pointer, n out of range, p < 0, bad dtype, misaligned element */
    RA_ERR_UNSUPPORTED = 2, /* a valid request outside what the called function handles (see its notes) */
    RA_ERR_OVERLAP = 3,     /* two buffers (or w and a buffer) share bytes */
    RA_ERR_CUDA = 4,        /* a CUDA call failed; see ra_last_cuda_error() */
    RA_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up */
    RA_ERR_BOUNDS = 6       /* bounds-checked build only: a kernel found a range outside the caller's buffers */
} ra_status;

/* A contiguous element range [offset, offset + count) of every worker's array. */
typedef struct {
    int64_t offset;
    int64_t count;
} ra_bucket;

/* Elements one worker sent and received over a full ring all-reduce. */
typedef struct {
    int64_t sent;
    int64_t received;
} ra_traffic;

#define RA_MAX_N 64 /* most workers one call accepts */

/*
 * ra_allreduce_avg -- every worker's array becomes the element-wise mean of
 * all n arrays (scatter-reduce, divide by N, all-gather; Gibiansky,
 * "Scatter-Reduce" and "Allgather").  One fused pass: each element's n
 * values are read once and the mean is written to all n arrays.
 *   bufs   host array of n device pointers, p elements each, in place
 *   n      1 .. RA_MAX_N workers
 *   p      elements per worker (>= 0)
 *   dtype  RA_F32 or RA_BF16
 *   stream cudaStream_t to queue the kernel on
 */
ra_status ra_allreduce_avg(void *const *bufs, int n, int64_t p, int dtype, void *stream);

/*
 * ra_allreduce_sgd -- ra_allreduce_avg plus the synchronous SGD step
 * w <- w - lr * avg in the same pass (Gibiansky, "The Communication
 * Problem": the averaged gradient is applied to the weights; DDP: every
 * replica applies the same update, so one binary32 weight copy stands for
 * all of them).
 *   w      device pointer to p binary32 weights, updated in place; must
 *          not overlap any gradient buffer
 *   lr     learning rate
 * With RA_BF16 gradients the update uses the bf16-rounded mean.
 */
ra_status ra_allreduce_sgd(void *const *bufs, int n, int64_t p, int dtype, float *w, float lr, void *stream);

/*
 * ra_staged_workspace_bytes -- device workspace ra_allreduce_avg_staged
 * needs: 0 for RA_F32 (the partial sums live in the workers' own arrays),
 * p * 4 + 64 bytes for RA_BF16 (the binary32 partial sums "on the wire").
 */
size_t ra_staged_workspace_bytes(int n, int64_t p, int dtype);

/*
 * ra_allreduce_avg_staged -- the same result as ra_allreduce_avg, computed
 * the way the ring moves data: N-1 scatter-reduce iterations (in iteration
 * t every worker m adds the chunk (m-1-t) mod N it receives from worker
 * m-1), one division step by the worker holding each complete chunk, and
 * N-1 all-gather iterations (worker m overwrites chunk (m-t) mod N with its
 * left neighbour's copy); one kernel launch per iteration, 2(N-1)+1 in all
 * (Gibiansky, "Scatter-Reduce" and "Allgather", first-iteration tables).
 *   ws, ws_bytes  device workspace of at least
 *                 ra_staged_workspace_bytes(n, p, dtype) bytes (may be
 *                 NULL when that is 0); owned by the caller
 *   per_worker    optional HOST array of n ra_traffic entries; receives the
 *                 elements each worker sent and received (Gibiansky,
 *                 "Allreduce Communication Cost": 2(N-1)/N * P each when N
 *                 divides P)
 */
ra_status ra_allreduce_avg_staged(void *const *bufs, int n, int64_t p, int dtype, void *ws, size_t ws_bytes,
                                  ra_traffic *per_worker, void *stream);

/*
 * ra_bucket_plan -- groups layer tensors into buckets for per-subset
 * all-reduce, output layer first (Gibiansky, "Applying the Allreduce to
 * Deep Learning": the all-reduce can start on the output layer's
 * parameters while backpropagation is still computing earlier layers).
 * Rule: walk the tensors from the last to the first, add each to the open
 * bucket and close the bucket once it holds >= cap_bytes; what is left
 * forms the last bucket.  Buckets are contiguous element ranges of the
 * forward-ordered flat array, written to out[] in closing order.
 *   numel      host array of ntensors element counts (forward order)
 *   elem_bytes bytes per element (> 0); cap_bytes > 0
 *   out        host array of max_out entries; *n_out receives the count
 * RA_ERR_INVALID_ARG if max_out is too small or an argument is bad.
 */
ra_status ra_bucket_plan(const int64_t *numel, int ntensors, int elem_bytes, int64_t cap_bytes, ra_bucket *out,
                         int max_out, int *n_out);

/*
 * ra_allreduce_avg_buckets -- every bucket of every worker's array is
 * all-reduced-averaged as a ring of its own (its own P = count and its own
 * N chunks): the all-reduce run on a subset of the parameters at a time
 * (Gibiansky, "Applying the Allreduce to Deep Learning").  The (bucket, chunk) pieces go to the fused kernel in as few
 * launches as the kernel-parameter space allows (at most 896 pieces per
 * launch); the result does not depend on that split.
 *   bufs   host array of n device pointers; each buffer must hold every
 *          bucket, i.e. at least max(offset + count) elements
 *   b, nb  host array of nb buckets (offset >= 0, count >= 0); buckets
 *          must not overlap one another (RA_ERR_OVERLAP)
 */
ra_status ra_allreduce_avg_buckets(void *const *bufs, int n, int dtype, const ra_bucket *b, int nb, void *stream);

/*
 * ra_allreduce_avg_staged_static -- the same staged ring as
 * ra_allreduce_avg_staged, for callers that cannot allocate device memory:
 * the call takes no workspace and allocates nothing (no cudaMalloc/cudaFree,
 * no allocating library routine).  The pages have no counterpart; this is
 * an interface convenience of this library.
 *
 * Who needs it: code that runs inside a host framework which owns all device
 * memory through its own pool and does not let plug-ins call cudaMalloc;
 * latency-critical loops where cudaMalloc/cudaFree would synchronise the
 * device; and programs whose device-memory budget is fixed when they start.
 *
 * How: the bf16 ring's binary32 partial sums go to a scratch array compiled
 * into the library (RA_STAGED_STATIC_MAX_P binary32 elements, 16 MiB), which
 * every GPU that loads the library holds until the process exits.  RA_F32
 * needs no scratch (its partial sums live in the workers' own arrays).
 *   bufs, n, p, dtype, per_worker, stream  as for ra_allreduce_avg_staged
 * Returns RA_ERR_UNSUPPORTED, before doing anything, when dtype is RA_BF16
 * and p > RA_STAGED_STATIC_MAX_P.
 * The first call on a device (that passes the argument checks) looks up the
 * array's device address and caches it; make that first call before any
 * stream capture.  All calls on a device share the
 * array and it keeps the last call's contents; nothing in it needs clearing
 * (each call writes every partial sum before reading it), but calls whose
 * work overlaps on the GPU race on it: order them on one stream or with
 * events.
 */
#define RA_STAGED_STATIC_MAX_P 4194304
ra_status ra_allreduce_avg_staged_static(void *const *bufs, int n, int64_t p, int dtype, ra_traffic *per_worker,
                                         void *stream);

/*
 * ra_allreduce_avg_host -- ra_allreduce_avg for workers whose gradients
 * live in HOST memory: every host array ends holding the mean (the end-to-end
 * path of a data-parallel step whose gradients start and end on the host).
 * Two ways:
 *   - direct: the device addresses every host array -- page-locked memory
 *     (cudaHostAlloc / cudaHostRegister), or any host memory on a device
 *     that walks the host page tables (Grace-Blackwell's coherent
 *     NVLink-C2C) -- and the fused kernel reads the host arrays and writes
 *     the mean back to them directly; dev_bufs is not touched;
 *   - staged: each host array is copied to its device buffer in dev_bufs,
 *     reduced there, and the mean copied back.
 *   host_bufs  host array of n HOST pointers, p elements each, not
 *              overlapping
 *   dev_bufs   host array of n DEVICE pointers, p elements each (caller-owned
 *              staging), or NULL
 *   mode       RA_HOST_AUTO: direct when possible, else staged;
 *              RA_HOST_DIRECT: direct or RA_ERR_UNSUPPORTED;
 *              RA_HOST_STAGED: staged (RA_ERR_UNSUPPORTED if dev_bufs is NULL)
 * All work is queued on `stream`; the host arrays must not be read before
 * the stream has finished.
 */
enum { RA_HOST_AUTO = 0, RA_HOST_DIRECT = 1, RA_HOST_STAGED = 2 };
ra_status ra_allreduce_avg_host(void *const *host_bufs, void *const *dev_bufs, int n, int64_t p, int dtype, int mode,
                                void *stream);

/*
 * ra_reduce_scatter_avg -- the scatter-reduce half of the ring on its own,
 * with the owner's division: afterwards the worker that holds the complete
 * chunk c, worker (c - 1) mod n, has the mean of chunk c (Gibiansky,
 * "Scatter-Reduce": each GPU ends with one chunk of the final result;
 * "[PyTorch] GPU 분산 학습 1 - DP / DDP / FSDP 개념", FSDP: the gradients are
 * reduce-scattered so each GPU keeps the part it updates).  Same summation
 * order and rounding as ra_allreduce_avg.  One fused pass: N*P reads, P
 * writes.
 *   shards  NULL: the mean of chunk c is written into bufs[(c-1) mod n] at
 *           chunk c's elements; every other element keeps its input.
 *           Otherwise a host array of n DEVICE pointers: shards[m] receives
 *           the mean of chunk (m+1) mod n (ra_chunk_range gives its length);
 *           bufs are not written.  Shards must not overlap each other or
 *           the worker arrays.
 */
ra_status ra_reduce_scatter_avg(void *const *bufs, int n, int64_t p, int dtype, void *const *shards, void *stream);

/*
 * ra_all_gather -- the all-gather half of the ring on its own: chunk c,
 * held by worker (c - 1) mod n, is copied to every worker (Gibiansky,
 * "Allgather": received chunks overwrite; FSDP: the parameter shards are
 * all-gathered before a layer runs).  P reads, (N-1)*P writes in place.
 *   shards  NULL: the source of chunk c is bufs[(c-1) mod n] at chunk c's
 *           elements, and the other n-1 workers' chunk c is overwritten.
 *           Otherwise a host array of n DEVICE pointers: shards[m] holds
 *           chunk (m+1) mod n, which is written to every worker's array.
 */
ra_status ra_all_gather(void *const *bufs, int n, int64_t p, int dtype, void *const *shards, void *stream);

/*
 * ra_allreduce_avg_bf16_wire -- the ring over bf16 arrays as a ring that
 * keeps every array in bf16 computes it: each receiver adds its own value
 * and the received partial in binary32 and stores the sum back in bf16
 * (nearest even), so every partial sum is rounded; the owner divides its
 * bf16 sum by N in binary32 and rounds the mean to bf16 (Gibiansky,
 * "Scatter-Reduce" with bf16 buffers).  Less accurate than ra_allreduce_avg
 * with RA_BF16, whose partials stay binary32; offered to reproduce such
 * rings bit for bit.  One fused pass, same traffic as ra_allreduce_avg.
 */
ra_status ra_allreduce_avg_bf16_wire(void *const *bufs, int n, int64_t p, void *stream);

/*
 * ra_allreduce_avg_single_reducer -- the averaging scheme the ring replaces
 * (Gibiansky, "The Communication Problem"): every worker sends its gradient
 * to one reducer, worker 0, which adds them in worker order
 * ((g_0 + g_1) + g_2) + ... + g_{N-1} in binary32, divides by N, and sends
 * the mean back to every worker.  Computed in one fused pass here; the
 * result differs from the ring's only in summation order.
 *   per_worker  optional HOST array of n ra_traffic entries: the elements
 *               each worker sends and receives in that scheme -- (N-1)*P
 *               each way for the reducer, P each way for every other worker
 *               (the reducer's load grows with N, the ring's does not)
 */
ra_status ra_allreduce_avg_single_reducer(void *const *bufs, int n, int64_t p, int dtype, ra_traffic *per_worker,
                                          void *stream);

/*
 * ra_reducer -- per-bucket all-reduce overlapped with the backward pass
 * (Gibiansky, "Applying the Allreduce to Deep Learning": backpropagation
 * yields the output layer's gradients first and the all-reduce can run on a
 * subset of the parameters, so communication starts while earlier layers
 * are still computing).
 *
 * The reducer holds the ra_bucket_plan of a model's layer tensors (forward
 * order, packed back to back in every worker's flat gradient array) and a
 * stream of its own.  Each step the training loop calls
 * ra_reducer_mark_ready(tensor, stream) once per tensor, when the work that
 * completes that tensor's gradient (on every worker) has been queued on
 * `stream`; as soon as all tensors of a bucket are marked, the bucket's ring
 * all-reduce (the same bits as ra_allreduce_avg_buckets) is queued on the
 * reducer's stream behind an event recorded on `stream`.
 * ra_reducer_finish(stream) queues the buckets whose tensors were not all
 * marked, makes `stream` wait for every bucket, and resets the marks for
 * the next step.  A reducer belongs to the device current at creation and
 * to one host thread at a time; it allocates host memory, one stream and
 * nb + 1 events, but no device memory.
 *   ra_reducer_create   bufs: n device pointers, each holding sum(numel)
 *                       elements of dtype; numel: host array of ntensors
 *                       element counts; cap_bytes: bucket size (> 0)
 *   ra_reducer_buckets  copies the plan (closing order) into out[max_out]
 *   ra_reducer_destroy  waits for the reducer's stream, then frees it
 * RA_ERR_INVALID_ARG for a tensor marked twice in one step or a call from
 * another device.
 */
typedef struct ra_reducer ra_reducer;
ra_status ra_reducer_create(void *const *bufs, int n, int dtype, const int64_t *numel, int ntensors,
                            int64_t cap_bytes, ra_reducer **out);
ra_status ra_reducer_buckets(const ra_reducer *r, ra_bucket *out, int max_out, int *n_out);
ra_status ra_reducer_mark_ready(ra_reducer *r, int tensor, void *stream);
ra_status ra_reducer_finish(ra_reducer *r, void *stream);
ra_status ra_reducer_destroy(ra_reducer *r);

/*
 * ra_check_device_errors -- whether a kernel of this library on the current
 * device gave up a bounded wait since the last check.  The TMA kernels
 * (fused all-reduce in all its variants, all-gather) wait for their bulk
 * copies (global -> shared memory) on an mbarrier; each wait is limited to
 * 2 s (the copies of one tile take microseconds), after which the kernel
 * records the failure in the device's error word, skips its stores and
 * returns, so the context stays usable.  Returns RA_ERR_TIMEOUT if such a
 * record exists (the results of the calls in flight at the time are then
 * invalid), RA_ERR_BOUNDS if the bounds-checked build recorded an access
 * outside the caller's buffers (see ra_selftest_bounds_check; it takes
 * precedence), RA_OK otherwise, and clears the record.  Reads device memory
 * synchronously: call it after the streams in question have finished.
 */
ra_status ra_check_device_errors(void);

/*
 * ra_selftest_bounds_check -- the bounds-checked build (libgradient_ring_all_
 * checked.so, built for the tests) verifies inside every kernel that each
 * global range it reads or writes lies in the caller's buffers, skips the
 * access otherwise, and records RA_ERR_BOUNDS for ra_check_device_errors().
 * This call exercises that check: it runs the fused all-reduce over the p
 * elements of `bufs` (arguments as ra_allreduce_avg) while telling the
 * kernel that the rows hold only p - 1 elements, so the tile holding the
 * last element must be reported and skipped.  No memory outside the rows
 * is touched; the rows' contents afterwards are unspecified.  Needs p >= 2
 * and n >= 2.  The product build returns RA_ERR_UNSUPPORTED.
 */
ra_status ra_selftest_bounds_check(void *const *bufs, int n, int64_t p, int dtype, void *stream);

/*
 * ra_selftest_wait_timeout -- exercises that timeout path on purpose: queues
 * on `stream` a one-block kernel whose mbarrier expects 16 bytes that no copy
 * delivers; its bounded wait gives up after timeout_us (1 .. 10^7) and
 * records the failure, so ra_check_device_errors() then returns
 * RA_ERR_TIMEOUT.  Nothing hangs and no memory is touched.
 */
ra_status ra_selftest_wait_timeout(int timeout_us, void *stream);

/* ra_chunk_range -- [begin, end) of chunk c of a p-element array split for
 * n workers.  Gibiansky, "Scatter-Reduce", divides the array into N chunks
 * but leaves open how the split goes when N does not divide P; this
 * library's reading, used by every call, gives the first p mod n chunks one
 * extra element: chunk c = [c*q + min(c,r), (c+1)*q + min(c+1,r)) with
 * q = p / n, r = p mod n.  0 <= c < n; nothing is checked. */
void ra_chunk_range(int64_t p, int n, int c, int64_t *begin, int64_t *end);

/* ra_status_str -- a static, human-readable name for a status. */
const char *ra_status_str(int status);

/* ra_last_cuda_error -- the cudaError_t behind this thread's most recent
 * RA_ERR_CUDA (0 if none). */
int ra_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* RING_ALLREDUCE_H */
