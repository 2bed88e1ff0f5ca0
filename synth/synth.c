/*
 * Seeded synthetic inputs shared by the oracle and the CUDA path.
 *
 * This file holds no attention arithmetic: it only turns (seed, stream id,
 * element index) into numbers. Every draw is counter based, so element i of a
 * stream can be produced by any thread in any order and the result does not
 * depend on the thread count.
 *
 *   splitmix64 finaliser (Steele, Lea, Flood, "Fast splittable pseudorandom
 *   number generators", OOPSLA 2014) applied to key + (i + 1) * golden gamma,
 *   uniform in [0, 1) from the top 53 bits, standard normal by the Box-Muller
 *   transform (Box and Muller, 1958) on two uniforms of the same counter pair,
 *   and bf16 by round-to-nearest-even of the fp32 value.
 *
 * Built as a small shared library and called through ctypes.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Stream key: one independent counter sequence per (seed, stream id). */
static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(mix64(seed + GOLDEN_GAMMA) ^ (stream * 0xD1B54A32D192ED03ULL + 0x632BE59BD9B4E019ULL));
}

static inline uint64_t draw_u64(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN_GAMMA); }

/* Uniform in [0, 1) with 53 random bits. */
static inline double draw_unit(uint64_t key, uint64_t i) {
    return (double)(draw_u64(key, i) >> 11) * (1.0 / 9007199254740992.0);
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t b;
    memcpy(&b, &f, 4);
    if ((b & 0x7f800000u) == 0x7f800000u) return (uint16_t)((b >> 16) | ((b & 0xffffu) ? 0x40u : 0u));
    uint32_t lsb = (b >> 16) & 1u;
    b += 0x7fffu + lsb;
    return (uint16_t)(b >> 16);
}

/* Standard normal number i of a stream: Box-Muller on uniforms (2i, 2i+1). */
static inline double draw_normal(uint64_t key, uint64_t i) {
    double u1 = 1.0 - draw_unit(key, 2 * i); /* (0, 1] so the log is finite */
    double u2 = draw_unit(key, 2 * i + 1);
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

typedef struct {
    uint64_t key, okey, lo, hi;
    double outlier_frac, outlier_scale;
    uint16_t* out;
} normal_job;

static void* normal_worker(void* arg) {
    normal_job* j = (normal_job*)arg;
    for (uint64_t i = j->lo; i < j->hi; ++i) {
        double x = draw_normal(j->key, i);
        if (j->outlier_frac > 0.0 && draw_unit(j->okey, i) < j->outlier_frac) x *= j->outlier_scale;
        j->out[i] = f32_to_bf16_rne((float)x);
    }
    return NULL;
}

/*
 * n bf16 values ~ N(0,1) (as raw bits). With outlier_frac > 0 each element is,
 * independently with that probability (decided by stream id + 0x5151 of the same
 * seed), multiplied by outlier_scale before the single rounding to bf16.
 */
int synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t n, double outlier_frac, double outlier_scale,
                      uint16_t* out, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    uint64_t key = stream_key(seed, stream);
    uint64_t okey = stream_key(seed, stream + 0x5151);
    if (n < 65536 || nthreads == 1) {
        normal_job j = {key, okey, 0, n, outlier_frac, outlier_scale, out};
        normal_worker(&j);
        return 0;
    }
    pthread_t th[256];
    normal_job jobs[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = (normal_job){key, okey, n * (uint64_t)t / (uint64_t)nthreads,
                               n * (uint64_t)(t + 1) / (uint64_t)nthreads, outlier_frac, outlier_scale, out};
        if (pthread_create(&th[t], NULL, normal_worker, &jobs[t]) != 0) {
            normal_worker(&jobs[t]);
            th[t] = 0;
        }
    }
    for (int t = 0; t < nthreads; ++t)
        if (th[t]) pthread_join(th[t], NULL);
    return 0;
}

/* n integers uniform in [lo, hi] inclusive. */
int synth_uniform_int(uint64_t seed, uint64_t stream, uint64_t n, int64_t lo, int64_t hi, int64_t* out) {
    if (hi < lo) return -1;
    uint64_t key = stream_key(seed, stream);
    double span = (double)(hi - lo + 1);
    for (uint64_t i = 0; i < n; ++i) {
        int64_t v = lo + (int64_t)floor(draw_unit(key, i) * span);
        if (v > hi) v = hi;
        out[i] = v;
    }
    return 0;
}

/* A permutation of 0..n-1 by Fisher-Yates, swap index for step i drawn from counter i. */
int synth_permutation(uint64_t seed, uint64_t stream, int64_t n, int64_t* out) {
    uint64_t key = stream_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) out[i] = i;
    for (int64_t i = n - 1; i > 0; --i) {
        int64_t j = (int64_t)floor(draw_unit(key, (uint64_t)i) * (double)(i + 1));
        if (j > i) j = i;
        int64_t t = out[i];
        out[i] = out[j];
        out[j] = t;
    }
    return 0;
}

/* Exposed so tests can check the raw generator against its published definition. */
uint64_t synth_mix64(uint64_t z) { return mix64(z); }
double synth_unit(uint64_t seed, uint64_t stream, uint64_t i) { return draw_unit(stream_key(seed, stream), i); }
