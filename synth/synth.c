/*
 * synth.c -- seeded synthetic gradient generator (shared by the tests, the
 * oracle side and the benchmark; contains none of the all-reduce arithmetic).
 *
 * Every value depends only on (seed, stream, index), so any element can be
 * regenerated on its own and the bulk fill can be split over threads freely.
 *
 * Generator: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014), accessed by counter: the
 * k-th output of the stream with key K is mix(K + (k+1)*GAMMA).
 * Normal deviates: the Box-Muller transform (G. Box, M. Muller, 1958).
 * Student-t with nu=3: Z / sqrt((Z1^2 + Z2^2 + Z3^2) / 3) from four
 * independent standard normals (the textbook definition of Student's t).
 *
 * Streams: stream s of seed S uses the key mix(S ^ mix(s + STREAM_SALT)).
 * Worker n's gradient row is stream n.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9e3779b97f4a7c15ULL
#define STREAM_SALT 0x632be59bd9b4e019ULL

static uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}

static uint64_t stream_key(uint64_t seed, uint64_t stream) { return mix64(seed ^ mix64(stream + STREAM_SALT)); }

static uint64_t draw(uint64_t key, uint64_t k) { return mix64(key + (k + 1) * GAMMA); }

/* standard normals 2*pair and 2*pair+1 of the stream (one Box-Muller pair) */
static void normal_pair(uint64_t key, uint64_t pair, double *z0, double *z1) {
    double u1 = ((double)(draw(key, 2 * pair) >> 11) + 1.0) * 0x1.0p-53; /* (0, 1] */
    double u2 = (double)(draw(key, 2 * pair + 1) >> 11) * 0x1.0p-53;     /* [0, 1) */
    double r = sqrt(-2.0 * log(u1));
    double a = 6.283185307179586476925286766559 * u2;
    *z0 = r * cos(a);
    *z1 = r * sin(a);
}

static double normal_at(uint64_t key, uint64_t j) {
    double z0, z1;
    normal_pair(key, j >> 1, &z0, &z1);
    return (j & 1) ? z1 : z0;
}

/* Student-t value i uses standard normals 4i .. 4i+3 (pairs 2i and 2i+1) */
static double student_t3_at(uint64_t key, uint64_t i) {
    double z, a, b, c;
    normal_pair(key, 2 * i, &z, &a);
    normal_pair(key, 2 * i + 1, &b, &c);
    return z / sqrt((a * a + b * b + c * c) / 3.0);
}

static uint16_t to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t hi = u >> 16, lo = u & 0xffffu;
    if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u)))
        hi += 1u;
    return (uint16_t)hi;
}

/* ------------------------------------------------------------------ */

typedef struct {
    int kind; /* 0: normal -> f32, 1: student-t3 -> bf16 bits, 2: student-t3 -> f32 */
    uint64_t key;
    double scale;
    int64_t start, count;
    void *out;
} job_t;

static void run_job(const job_t *j) {
    if (j->kind == 0) {
        float *o = (float *)j->out;
        int64_t k = 0;
        if (j->count > 0 && (j->start & 1)) { /* odd start: second half of a pair */
            o[0] = (float)(j->scale * normal_at(j->key, (uint64_t)j->start));
            k = 1;
        }
        for (; k + 1 < j->count; k += 2) {
            double z0, z1;
            normal_pair(j->key, (uint64_t)(j->start + k) >> 1, &z0, &z1);
            o[k] = (float)(j->scale * z0);
            o[k + 1] = (float)(j->scale * z1);
        }
        if (k < j->count)
            o[k] = (float)(j->scale * normal_at(j->key, (uint64_t)(j->start + k)));
    } else if (j->kind == 1) {
        uint16_t *o = (uint16_t *)j->out;
        for (int64_t k = 0; k < j->count; ++k)
            o[k] = to_bf16_rne((float)(j->scale * student_t3_at(j->key, (uint64_t)(j->start + k))));
    } else {
        float *o = (float *)j->out;
        for (int64_t k = 0; k < j->count; ++k)
            o[k] = (float)(j->scale * student_t3_at(j->key, (uint64_t)(j->start + k)));
    }
}

static void *thread_main(void *arg) {
    run_job((const job_t *)arg);
    return 0;
}

static void fill(int kind, uint64_t seed, uint64_t stream, double scale, int64_t start, int64_t count,
                 void *out, int nthreads) {
    size_t esz = kind == 1 ? 2 : 4;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    if (count < (int64_t)nthreads * 65536)
        nthreads = 1;
    job_t jobs[256];
    pthread_t th[256];
    int64_t per = (count + nthreads - 1) / nthreads;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        int64_t b = (int64_t)t * per, e = b + per < count ? b + per : count;
        if (b >= e)
            break;
        jobs[t].kind = kind;
        jobs[t].key = stream_key(seed, stream);
        jobs[t].scale = scale;
        jobs[t].start = start + b;
        jobs[t].count = e - b;
        jobs[t].out = (char *)out + (size_t)b * esz;
        if (nthreads == 1) {
            run_job(&jobs[t]);
        } else if (pthread_create(&th[t], 0, thread_main, &jobs[t]) == 0) {
            ++started;
            continue;
        } else {
            run_job(&jobs[t]);
        }
    }
    for (int t = 0; t < started; ++t)
        pthread_join(th[t], 0);
}

/* out[k] = float(sigma * Z_{start+k}) for stream (seed, stream) */
void synth_normal_f32(uint64_t seed, uint64_t stream, double sigma, int64_t start, int64_t count, float *out,
                      int nthreads) {
    fill(0, seed, stream, sigma, start, count, out, nthreads);
}

/* out[k] = bf16_rne(float(scale * T3_{start+k})) */
void synth_student_t3_bf16(uint64_t seed, uint64_t stream, double scale, int64_t start, int64_t count,
                           uint16_t *out, int nthreads) {
    fill(1, seed, stream, scale, start, count, out, nthreads);
}

void synth_student_t3_f32(uint64_t seed, uint64_t stream, double scale, int64_t start, int64_t count,
                          float *out, int nthreads) {
    fill(2, seed, stream, scale, start, count, out, nthreads);
}

/* the same values at arbitrary indices */
void synth_normal_f32_at(uint64_t seed, uint64_t stream, double sigma, const int64_t *idx, int64_t n, float *out) {
    uint64_t key = stream_key(seed, stream);
    for (int64_t k = 0; k < n; ++k)
        out[k] = (float)(sigma * normal_at(key, (uint64_t)idx[k]));
}

void synth_student_t3_bf16_at(uint64_t seed, uint64_t stream, double scale, const int64_t *idx, int64_t n,
                              uint16_t *out) {
    uint64_t key = stream_key(seed, stream);
    for (int64_t k = 0; k < n; ++k)
        out[k] = to_bf16_rne((float)(scale * student_t3_at(key, (uint64_t)idx[k])));
}

/* raw 64-bit draws (for the generator's own tests) */
void synth_raw_u64(uint64_t seed, uint64_t stream, int64_t start, int64_t count, uint64_t *out) {
    uint64_t key = stream_key(seed, stream);
    for (int64_t k = 0; k < count; ++k)
        out[k] = draw(key, (uint64_t)(start + k));
}

/* the plain SplitMix64 sequence of a raw key (for checking the generator
 * against the published reference outputs) */
void synth_splitmix64(uint64_t key, int64_t start, int64_t count, uint64_t *out) {
    for (int64_t k = 0; k < count; ++k)
        out[k] = draw(key, (uint64_t)(start + k));
}
