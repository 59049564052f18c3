/*
 * ring_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU simulation of the ring all-reduce used for
 * data-parallel gradient averaging.  Only the tests, the smoke check and the
 * CPU leg of the benchmark (its timed CPU baseline, and its check of the
 * GPU's result against host copies of the same inputs) may load this file's
 * library; the product path (the CUDA library) never calls it and shares no
 * code with it.
 *
 * Sources (page title, section):
 *   [G]  "Andrew Gibiansky: Bringing HPC Techniques to Deep Learning"
 *        (Korean translation), sections "The Communication Problem",
 *        "Ring Allreduce", "Scatter-Reduce", "Allgather",
 *        "Allreduce Communication Cost", "Applying the Allreduce to Deep Learning".
 *   [M]  "[AI System] Training With Multiple GPUs", "Comparison With
 *        Centralized Training" (gradient averaging = full-batch gradient).
 *   [D]  "[PyTorch] GPU 분산 학습 1 - DP / DDP / FSDP 개념", section DDP
 *        (every GPU ends with the same gradient and updates its own weights).
 *
 * Readings of points the pages leave open:
 *   - uneven split: chunk c = [c*q + min(c,r), (c+1)*q + min(c+1,r)),
 *     q = P / N, r = P mod N (the first r chunks hold one extra element);
 *   - the receiving worker adds the received partial to its own value
 *     (own + received; IEEE addition is commutative, so only the
 *     association -- a left fold that starts at worker c for chunk c -- matters);
 *   - averaging is one IEEE binary32 division by N, done by the worker that
 *     holds the complete chunk after the scatter-reduce, before the all-gather;
 *   - bf16 gradients: partial sums travel in binary32 and the mean is rounded
 *     to bf16 (round to nearest, ties to even) once;
 *   - SGD: w <- w - (lr * avg) with two roundings (compile with
 *     -ffp-contract=off so no fused multiply-add is formed).
 *
 * Pins: tests/test_oracle_*.py check every function here against the pages'
 * worked tables, exact rational arithmetic, closed forms and invariants.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* chunks and the neighbour map ([G] "Scatter-Reduce": split into N chunks;
 * [G] "Ring Allreduce": send right, receive left).                     */

static int mod_n(int64_t a, int n) {
    int64_t m = a % n;
    return (int)(m < 0 ? m + n : m);
}

void oracle_chunk_range(int64_t p, int n, int c, int64_t *begin, int64_t *end) {
    int64_t q = p / n, r = p % n;
    int64_t b = (int64_t)c * q + (c < r ? c : r);
    *begin = b;
    *end = b + q + (c < r ? 1 : 0);
}

/* Scatter-reduce: GPU n first sends chunk n and receives chunk n-1, then
 * works backwards, each iteration sending the chunk it received in the
 * previous one ([G] "Scatter-Reduce", first-iteration table).            */
int oracle_scatter_send_chunk(int n_workers, int n, int t) { return mod_n((int64_t)n - t, n_workers); }
int oracle_scatter_recv_chunk(int n_workers, int n, int t) { return mod_n((int64_t)n - 1 - t, n_workers); }
/* All-gather: GPU n first sends chunk n+1 and receives chunk n, then always
 * forwards what it has just received ([G] "Allgather", first-iteration table). */
int oracle_gather_send_chunk(int n_workers, int n, int t) { return mod_n((int64_t)n + 1 - t, n_workers); }
int oracle_gather_recv_chunk(int n_workers, int n, int t) { return mod_n((int64_t)n - t, n_workers); }

/* ------------------------------------------------------------------ */
/* bf16 helpers (IEEE-754 binary32 upper half; round to nearest even).   */

static float bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

uint16_t oracle_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) /* NaN: keep it quiet */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lower = u & 0xffffu;
    uint32_t upper = u >> 16;
    /* round half to even on the 16 discarded bits */
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;
    return (uint16_t)upper;
}

/* ------------------------------------------------------------------ */
/* The literal ring, binary32 working rows.
 *
 * rows[n][0..p) is worker n's array, modified in place.  The run is split so
 * that a test can stop it part-way and look at the intermediate state:
 *   n_scatter  scatter-reduce iterations to run (N-1 for the full method),
 *   do_avg     1: after them, the worker that holds a complete chunk divides
 *              it by N (only meaningful after all N-1 iterations),
 *   bf16_out   1: the divided chunk is rounded to bf16 (and kept as the
 *              binary32 value of that bf16) -- the bf16-gradient reading,
 *   n_gather   all-gather iterations to run (N-1 for the full method).
 * sent / received (may be NULL) accumulate per-worker element counts.
 * Returns 0, or -1 on bad arguments / out of memory.
 *
 * Every iteration is simulated as the pages describe it: all workers first
 * put the chunk they send on the wire (a message buffer), then every worker
 * takes the chunk from its left neighbour and accumulates (scatter-reduce)
 * or overwrites (all-gather).                                             */
int oracle_ring_run_f32(float *const *rows, int n_workers, int64_t p, int n_scatter, int do_avg,
                        int bf16_out, int n_gather, int64_t *sent, int64_t *received) {
    int N = n_workers;
    if (N < 1 || p < 0 || n_scatter < 0 || n_gather < 0 || n_scatter > N - 1 || n_gather > N - 1)
        return -1;
    float *wire = (float *)malloc((size_t)(p > 0 ? p : 1) * sizeof(float));
    if (!wire)
        return -1;

    /* scatter-reduce ([G] "Scatter-Reduce") */
    for (int t = 0; t < n_scatter; ++t) {
        for (int n = 0; n < N; ++n) { /* sends: worker n -> worker n+1 */
            int c = oracle_scatter_send_chunk(N, n, t);
            int64_t b, e;
            oracle_chunk_range(p, N, c, &b, &e);
            for (int64_t i = b; i < e; ++i)
                wire[i] = rows[n][i];
            if (sent)
                sent[n] += e - b;
        }
        for (int m = 0; m < N; ++m) { /* receives: worker m <- worker m-1, accumulate */
            int c = oracle_scatter_recv_chunk(N, m, t);
            int left = mod_n((int64_t)m - 1, N);
            if (oracle_scatter_send_chunk(N, left, t) != c) {
                free(wire);
                return -1; /* the schedule must match sender to receiver */
            }
            int64_t b, e;
            oracle_chunk_range(p, N, c, &b, &e);
            for (int64_t i = b; i < e; ++i)
                rows[m][i] = rows[m][i] + wire[i];
            if (received)
                received[m] += e - b;
        }
    }

    /* average: after the scatter-reduce worker n holds the complete chunk
     * n+1 ([G] "Allgather": the all-gather starts by sending chunk n+1);
     * divide by N to turn the sum into the mean ([G] "The Communication
     * Problem": the GPUs average their gradients).                        */
    if (do_avg) {
        float fn = (float)N;
        for (int n = 0; n < N; ++n) {
            int c = mod_n((int64_t)n + 1, N);
            int64_t b, e;
            oracle_chunk_range(p, N, c, &b, &e);
            for (int64_t i = b; i < e; ++i) {
                float avg = rows[n][i] / fn;
                rows[n][i] = bf16_out ? bf16_to_f32(oracle_f32_to_bf16(avg)) : avg;
            }
        }
    }

    /* all-gather ([G] "Allgather"): same pattern, overwrite instead of add */
    for (int t = 0; t < n_gather; ++t) {
        for (int n = 0; n < N; ++n) {
            int c = oracle_gather_send_chunk(N, n, t);
            int64_t b, e;
            oracle_chunk_range(p, N, c, &b, &e);
            for (int64_t i = b; i < e; ++i)
                wire[i] = rows[n][i];
            if (sent)
                sent[n] += e - b;
        }
        for (int m = 0; m < N; ++m) {
            int c = oracle_gather_recv_chunk(N, m, t);
            int left = mod_n((int64_t)m - 1, N);
            if (oracle_gather_send_chunk(N, left, t) != c) {
                free(wire);
                return -1;
            }
            int64_t b, e;
            oracle_chunk_range(p, N, c, &b, &e);
            for (int64_t i = b; i < e; ++i)
                rows[m][i] = wire[i];
            if (received)
                received[m] += e - b;
        }
    }
    free(wire);
    return 0;
}

/* The full method on binary32 gradients: every worker ends with the mean. */
int oracle_ring_allreduce_avg_f32(float *const *rows, int n_workers, int64_t p, int64_t *sent,
                                  int64_t *received) {
    return oracle_ring_run_f32(rows, n_workers, p, n_workers - 1, 1, 0, n_workers - 1, sent, received);
}

/* The full method on bf16 gradients: rows are widened exactly to binary32,
 * the ring runs with binary32 partials, the mean is rounded to bf16 once and
 * written back to every worker.                                          */
int oracle_ring_allreduce_avg_bf16(uint16_t *const *rows, int n_workers, int64_t p, int64_t *sent,
                                   int64_t *received) {
    int N = n_workers;
    if (N < 1 || p < 0)
        return -1;
    float **work = (float **)calloc((size_t)N, sizeof(float *));
    if (!work)
        return -1;
    int rc = 0;
    for (int n = 0; n < N && rc == 0; ++n) {
        work[n] = (float *)malloc((size_t)(p > 0 ? p : 1) * sizeof(float));
        if (!work[n])
            rc = -1;
        else
            for (int64_t i = 0; i < p; ++i)
                work[n][i] = bf16_to_f32(rows[n][i]);
    }
    if (rc == 0)
        rc = oracle_ring_run_f32(work, N, p, N - 1, 1, 1, N - 1, sent, received);
    if (rc == 0)
        for (int n = 0; n < N; ++n)
            for (int64_t i = 0; i < p; ++i)
                rows[n][i] = oracle_f32_to_bf16(work[n][i]); /* exact: already bf16 values */
    for (int n = 0; n < N; ++n)
        free(work[n]);
    free(work);
    return rc;
}

/* Synchronous SGD step after the all-reduce ([G] "The Communication Problem":
 * the averaged gradient is applied to the weights; [D] DDP: every replica
 * applies the same gradient).  One binary32 weight copy w[p] stands for the N
 * identical replicas.  avg is worker 0's row after the all-reduce.         */
void oracle_sgd_update_f32(float *w, const float *avg, int64_t p, float lr) {
    for (int64_t i = 0; i < p; ++i) {
        float step = lr * avg[i];
        w[i] = w[i] - step;
    }
}

void oracle_sgd_update_bf16avg(float *w, const uint16_t *avg, int64_t p, float lr) {
    for (int64_t i = 0; i < p; ++i) {
        float step = lr * bf16_to_f32(avg[i]);
        w[i] = w[i] - step;
    }
}

/* One element of the ring, for checking a few sampled outputs of a run too
 * large to simulate whole.  vals[n] is worker n's input at element i of a
 * ring over p elements.  The partial for chunk c starts at worker c and each
 * scatter-reduce iteration t adds it to the value of receiver c+1+t, exactly
 * as oracle_ring_run_f32 does for every element.                         */
float oracle_ring_avg_point_f32(const float *vals, int n_workers, int64_t p, int64_t i) {
    int N = n_workers;
    int c = 0;
    for (int k = 0; k < N; ++k) {
        int64_t b, e;
        oracle_chunk_range(p, N, k, &b, &e);
        if (i >= b && i < e) {
            c = k;
            break;
        }
    }
    float partial = vals[c];
    for (int t = 0; t < N - 1; ++t) {
        int receiver = mod_n((int64_t)c + 1 + t, N);
        partial = vals[receiver] + partial;
    }
    return partial / (float)N;
}

/* The ring's result over the element range [begin, end) of a p-element ring,
 * for comparing every output of a run too large to simulate whole at once.
 * rows[k] points at worker k's element `begin` (the caller holds only that
 * slice of each row); out receives end - begin results.  Every element gets
 * what the scatter-reduce makes of it: the partial for chunk c starts as
 * worker c's value, iteration t adds it to the value of receiver c+1+t, and
 * the owner divides once by N ([G] "Scatter-Reduce"; the average as in
 * oracle_ring_run_f32).  Elements do not interact, so a slice holds exactly
 * the values the full run gives there.  The loops take one chunk at a time
 * and, inside it, one ring iteration at a time over all its elements; each
 * element still sees the same additions in the same order.
 * Returns 0, or -1 on bad arguments.                                      */
int oracle_ring_avg_range_f32(const float *const *rows, int n_workers, int64_t p, int64_t begin, int64_t end,
                              float *out) {
    int N = n_workers;
    if (N < 1 || p < 0 || begin < 0 || end < begin || end > p)
        return -1;
    float fn = (float)N;
    for (int c = 0; c < N; ++c) {
        int64_t b, e;
        oracle_chunk_range(p, N, c, &b, &e);
        if (b < begin)
            b = begin;
        if (e > end)
            e = end;
        if (b >= e)
            continue;
        for (int64_t i = b; i < e; ++i)
            out[i - begin] = rows[c][i - begin];
        for (int t = 0; t < N - 1; ++t) {
            const float *recv = rows[mod_n((int64_t)c + 1 + t, N)];
            for (int64_t i = b; i < e; ++i)
                out[i - begin] = recv[i - begin] + out[i - begin];
        }
        for (int64_t i = b; i < e; ++i)
            out[i - begin] = out[i - begin] / fn;
    }
    return 0;
}

/* The same for bf16 rows: widened exactly, binary32 partials, the mean
 * rounded to bf16 once (the bf16 reading above).                        */
int oracle_ring_avg_range_bf16(const uint16_t *const *rows, int n_workers, int64_t p, int64_t begin, int64_t end,
                               uint16_t *out) {
    int N = n_workers;
    if (N < 1 || p < 0 || begin < 0 || end < begin || end > p)
        return -1;
    float *acc = (float *)malloc((size_t)(end > begin ? end - begin : 1) * sizeof(float));
    if (!acc)
        return -1;
    float fn = (float)N;
    for (int c = 0; c < N; ++c) {
        int64_t b, e;
        oracle_chunk_range(p, N, c, &b, &e);
        if (b < begin)
            b = begin;
        if (e > end)
            e = end;
        if (b >= e)
            continue;
        for (int64_t i = b; i < e; ++i)
            acc[i - begin] = bf16_to_f32(rows[c][i - begin]);
        for (int t = 0; t < N - 1; ++t) {
            const uint16_t *recv = rows[mod_n((int64_t)c + 1 + t, N)];
            for (int64_t i = b; i < e; ++i)
                acc[i - begin] = bf16_to_f32(recv[i - begin]) + acc[i - begin];
        }
        for (int64_t i = b; i < e; ++i)
            out[i - begin] = oracle_f32_to_bf16(acc[i - begin] / fn);
    }
    free(acc);
    return 0;
}

/* The plain definition the ring reaches up to rounding order: the binary64
 * mean of the N inputs, summed in worker order.                          */
void oracle_mean_f64(const float *const *rows, int n_workers, int64_t p, double *out) {
    for (int64_t i = 0; i < p; ++i) {
        double s = 0.0;
        for (int n = 0; n < n_workers; ++n)
            s += (double)rows[n][i];
        out[i] = s / (double)n_workers;
    }
}

/* ------------------------------------------------------------------ */
/* Buckets ([G] "Applying the Allreduce to Deep Learning": the all-reduce
 * can run on a subset of the parameters, output layer first, while the
 * backward pass is still computing the rest).
 *
 * Reading: walk the tensors from the last (output) to the first; add each
 * to the open bucket; close the bucket once its size in bytes reaches
 * cap_bytes; whatever remains at the end forms the last bucket.  A bucket
 * is a contiguous element range [off, off+cnt) of the forward-ordered flat
 * buffer and is reduced as a ring of its own.  Buckets are emitted in the
 * order they are closed (output side first).  Returns the bucket count, or
 * -1 if max_out is too small or an argument is bad.                     */
int oracle_bucket_plan(const int64_t *numel, int ntensors, int64_t elem_bytes, int64_t cap_bytes,
                       int64_t *off, int64_t *cnt, int max_out) {
    if (ntensors < 0 || elem_bytes <= 0 || cap_bytes <= 0)
        return -1;
    int64_t total = 0;
    for (int k = 0; k < ntensors; ++k) {
        if (numel[k] < 0)
            return -1;
        total += numel[k];
    }
    int nb = 0;
    int64_t end = total;  /* the open bucket covers [start, end) */
    int64_t start = total;
    for (int k = ntensors - 1; k >= 0; --k) {
        start -= numel[k];
        if ((end - start) * elem_bytes >= cap_bytes) {
            if (nb >= max_out)
                return -1;
            off[nb] = start;
            cnt[nb] = end - start;
            ++nb;
            end = start;
        }
    }
    if (end > 0) {
        if (nb >= max_out)
            return -1;
        off[nb] = 0;
        cnt[nb] = end;
        ++nb;
    }
    return nb;
}

/* Per-worker traffic of the full ring (both phases), by walking the same
 * schedule as oracle_ring_run_f32 without touching data ([G] "Allreduce
 * Communication Cost": N-1 sends and N-1 receives per phase, one chunk each). */
void oracle_ring_traffic(int n_workers, int64_t p, int64_t *sent, int64_t *received) {
    int N = n_workers;
    for (int n = 0; n < N; ++n)
        sent[n] = received[n] = 0;
    for (int phase = 0; phase < 2; ++phase)
        for (int t = 0; t < N - 1; ++t)
            for (int n = 0; n < N; ++n) {
                int c = phase == 0 ? oracle_scatter_send_chunk(N, n, t) : oracle_gather_send_chunk(N, n, t);
                int64_t b, e;
                oracle_chunk_range(p, N, c, &b, &e);
                sent[n] += e - b;
                received[mod_n((int64_t)n + 1, N)] += e - b;
            }
}

/* bf16 point evaluation: inputs are bf16 bit patterns, widened exactly; the
 * binary32 ring result is rounded to bf16 once (the bf16 reading above). */
uint16_t oracle_ring_avg_point_bf16(const uint16_t *vals, int n_workers, int64_t p, int64_t i) {
    float wide[1024];
    if (n_workers < 1 || n_workers > 1024)
        return 0;
    for (int n = 0; n < n_workers; ++n)
        wide[n] = bf16_to_f32(vals[n]);
    return oracle_f32_to_bf16(oracle_ring_avg_point_f32(wide, n_workers, p, i));
}

/* ------------------------------------------------------------------ */
/* The two phases on their own ([D] FSDP: gradients are reduce-scattered so
 * that each GPU keeps the part it owns; parameters are all-gathered before
 * use; [G] Scatter-Reduce / Allgather).                                 */

/* Reduce-scatter-average of bf16 rows: the scatter-reduce with binary32
 * partials and the owner's division, as in the full method; afterwards
 * worker n's chunk n+1 holds the bf16 mean and every other chunk keeps the
 * worker's input (only the owned chunks are results).                   */
int oracle_reduce_scatter_avg_bf16(uint16_t *const *rows, int n_workers, int64_t p) {
    int N = n_workers;
    if (N < 1 || p < 0)
        return -1;
    float **work = (float **)calloc((size_t)N, sizeof(float *));
    if (!work)
        return -1;
    int rc = 0;
    for (int n = 0; n < N && rc == 0; ++n) {
        work[n] = (float *)malloc((size_t)(p > 0 ? p : 1) * sizeof(float));
        if (!work[n])
            rc = -1;
        else
            for (int64_t i = 0; i < p; ++i)
                work[n][i] = bf16_to_f32(rows[n][i]);
    }
    if (rc == 0)
        rc = oracle_ring_run_f32(work, N, p, N - 1, 1, 1, 0, 0, 0);
    if (rc == 0)
        for (int n = 0; n < N; ++n) {
            int64_t b, e;
            oracle_chunk_range(p, N, mod_n((int64_t)n + 1, N), &b, &e);
            for (int64_t i = b; i < e; ++i)
                rows[n][i] = oracle_f32_to_bf16(work[n][i]); /* exact: bf16 values */
        }
    for (int n = 0; n < N; ++n)
        free(work[n]);
    free(work);
    return rc;
}

/* All-gather of any element type, literally: N-1 iterations in which worker
 * n sends chunk (n+1-t) mod N to worker n+1, which overwrites its copy.
 * Starting from worker (c-1) mod N holding chunk c, every worker ends with
 * every chunk.                                                           */
int oracle_all_gather(void *const *rows, int n_workers, int64_t p, int elem_bytes) {
    int N = n_workers;
    if (N < 1 || p < 0 || elem_bytes < 1)
        return -1;
    unsigned char *wire = (unsigned char *)malloc((size_t)(p > 0 ? p : 1) * (size_t)elem_bytes);
    if (!wire)
        return -1;
    for (int t = 0; t < N - 1; ++t) {
        for (int n = 0; n < N; ++n) {
            int64_t b, e;
            oracle_chunk_range(p, N, oracle_gather_send_chunk(N, n, t), &b, &e);
            memcpy(wire + b * elem_bytes, (unsigned char *)rows[n] + b * elem_bytes, (size_t)(e - b) * elem_bytes);
        }
        for (int m = 0; m < N; ++m) {
            int64_t b, e;
            oracle_chunk_range(p, N, oracle_gather_recv_chunk(N, m, t), &b, &e);
            memcpy((unsigned char *)rows[m] + b * elem_bytes, wire + b * elem_bytes, (size_t)(e - b) * elem_bytes);
        }
    }
    free(wire);
    return 0;
}

/* ------------------------------------------------------------------ */
/* bf16 on the wire: the literal ring over bf16 arrays.  A receiver widens
 * its own value and the received partial to binary32, adds them, and stores
 * the sum back into its bf16 array (rounded to nearest even), so every
 * partial sum is a bf16 number; the owner divides its bf16 sum by N in
 * binary32 and rounds the mean to bf16.  ([G] Scatter-Reduce with the
 * arrays kept in bf16.)                                                  */
int oracle_ring_allreduce_avg_bf16_wire(uint16_t *const *rows, int n_workers, int64_t p) {
    int N = n_workers;
    if (N < 1 || p < 0)
        return -1;
    uint16_t *wire = (uint16_t *)malloc((size_t)(p > 0 ? p : 1) * sizeof(uint16_t));
    if (!wire)
        return -1;
    for (int t = 0; t < N - 1; ++t) {
        for (int n = 0; n < N; ++n) {
            int64_t b, e;
            oracle_chunk_range(p, N, oracle_scatter_send_chunk(N, n, t), &b, &e);
            for (int64_t i = b; i < e; ++i)
                wire[i] = rows[n][i];
        }
        for (int m = 0; m < N; ++m) {
            int64_t b, e;
            oracle_chunk_range(p, N, oracle_scatter_recv_chunk(N, m, t), &b, &e);
            for (int64_t i = b; i < e; ++i) {
                float sum = bf16_to_f32(rows[m][i]) + bf16_to_f32(wire[i]);
                rows[m][i] = oracle_f32_to_bf16(sum);
            }
        }
    }
    float fn = (float)N;
    for (int n = 0; n < N; ++n) {
        int64_t b, e;
        oracle_chunk_range(p, N, mod_n((int64_t)n + 1, N), &b, &e);
        for (int64_t i = b; i < e; ++i)
            rows[n][i] = oracle_f32_to_bf16(bf16_to_f32(rows[n][i]) / fn);
    }
    free(wire);
    return oracle_all_gather((void *const *)rows, N, p, 2);
}

/* ------------------------------------------------------------------ */
/* The single reducer ([G] The Communication Problem: every GPU sends its
 * gradient to one GPU, which averages them and sends the average back to
 * all).  Reading: worker 0 is the reducer; it receives the other workers'
 * arrays in worker order 1, 2, ..., N-1 and adds each to its running sum
 * (own + received), divides by N, and sends the mean to every other worker.
 * Binary32 rows; sent / received count elements per worker.              */
int oracle_single_reducer_avg_f32(float *const *rows, int n_workers, int64_t p, int64_t *sent, int64_t *received) {
    int N = n_workers;
    if (N < 1 || p < 0)
        return -1;
    for (int m = 1; m < N; ++m) {
        for (int64_t i = 0; i < p; ++i)
            rows[0][i] = rows[0][i] + rows[m][i];
        if (sent)
            sent[m] += p;
        if (received)
            received[0] += p;
    }
    float fn = (float)N;
    for (int64_t i = 0; i < p; ++i)
        rows[0][i] = rows[0][i] / fn;
    for (int m = 1; m < N; ++m) {
        memcpy(rows[m], rows[0], (size_t)p * sizeof(float));
        if (sent)
            sent[0] += p;
        if (received)
            received[m] += p;
    }
    return 0;
}

/* The same with bf16 arrays: widened exactly, binary32 running sum, the
 * mean rounded to bf16 once.                                             */
int oracle_single_reducer_avg_bf16(uint16_t *const *rows, int n_workers, int64_t p, int64_t *sent,
                                   int64_t *received) {
    int N = n_workers;
    if (N < 1 || p < 0)
        return -1;
    float *acc = (float *)malloc((size_t)(p > 0 ? p : 1) * sizeof(float));
    if (!acc)
        return -1;
    for (int64_t i = 0; i < p; ++i)
        acc[i] = bf16_to_f32(rows[0][i]);
    for (int m = 1; m < N; ++m) {
        for (int64_t i = 0; i < p; ++i)
            acc[i] = acc[i] + bf16_to_f32(rows[m][i]);
        if (sent)
            sent[m] += p;
        if (received)
            received[0] += p;
    }
    float fn = (float)N;
    for (int64_t i = 0; i < p; ++i)
        rows[0][i] = oracle_f32_to_bf16(acc[i] / fn);
    for (int m = 1; m < N; ++m) {
        memcpy(rows[m], rows[0], (size_t)p * sizeof(uint16_t));
        if (sent)
            sent[0] += p;
        if (received)
            received[m] += p;
    }
    free(acc);
    return 0;
}
