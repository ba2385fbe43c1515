/*
 * Seeded synthetic inputs: weights, prompt ids and batch prompt lengths.
 *
 * This module holds none of the decode step's arithmetic. It only draws
 * numbers. Both the oracle (tests, CPU baseline) and the CUDA library are fed
 * from it, so the two sides read identical bytes.
 *
 * Generator (defined here, the same on every host):
 *   mix64(z)            SplitMix64 output function (Steele, Lea & Flood,
 *                       "Fast splittable pseudorandom number generators",
 *                       OOPSLA 2014): xor-shift 30/27/31 with the two
 *                       published multipliers.
 *   key(seed, stream)   = mix64(mix64(seed + G) ^ (stream * S))
 *   word(seed, stream, k) = mix64(key + (k + 1) * G),  G = 0x9E3779B97F4A7C15
 *   uniform(...)        = ((word >> 11) + 0.5) * 2^-53, strictly inside (0, 1)
 *   normal(seed, k)     Box-Muller (Box & Muller 1958) in double on the pair
 *                       j = k / 2: u1 = uniform(seed, W, 2j), u2 = uniform(seed,
 *                       W, 2j + 1), r = sqrt(-2 ln u1); even k takes
 *                       r cos(2 pi u2), odd k takes r sin(2 pi u2).
 *
 * Being counter-based, any slice of a 27 GB blob can be drawn independently,
 * in parallel, and reproducibly.
 *
 * Build: gcc -O2 -fPIC -shared -pthread synth.c -o libsynth.so -lm
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>

#define SYNTH_GAMMA 0x9E3779B97F4A7C15ULL
#define SYNTH_STREAM_MUL 0xD1B54A32D192ED03ULL

uint64_t synth_mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static uint64_t synth_key(uint64_t seed, uint64_t stream) {
    return synth_mix64(synth_mix64(seed + SYNTH_GAMMA) ^ (stream * SYNTH_STREAM_MUL));
}

uint64_t synth_word(uint64_t seed, uint64_t stream, uint64_t k) {
    return synth_mix64(synth_key(seed, stream) + (k + 1ULL) * SYNTH_GAMMA);
}

static double word_to_unit(uint64_t w) {
    return ((double)(w >> 11) + 0.5) * (1.0 / 9007199254740992.0); /* 2^-53 */
}

double synth_uniform(uint64_t seed, uint64_t stream, uint64_t k) {
    return word_to_unit(synth_word(seed, stream, k));
}

static double normal_with_key(uint64_t key, uint64_t k) {
    const uint64_t j = k >> 1;
    const double u1 = word_to_unit(synth_mix64(key + (2 * j + 1ULL) * SYNTH_GAMMA));
    const double u2 = word_to_unit(synth_mix64(key + (2 * j + 2ULL) * SYNTH_GAMMA));
    const double r = sqrt(-2.0 * log(u1));
    const double a = 6.283185307179586476925286766559 * u2;
    return (k & 1) ? r * sin(a) : r * cos(a);
}

double synth_normal(uint64_t seed, uint64_t stream, uint64_t k) {
    return normal_with_key(synth_key(seed, stream), k);
}

/* out[i] = (float)(scale * normal(seed, stream, k0 + i)), i in [0, n).
 * Each worker walks whole Box-Muller pairs, so one log/sqrt serves two values;
 * the result is the same as calling synth_normal element by element. */
typedef struct {
    uint64_t key, k0;
    size_t begin, end;
    double scale;
    float* out;
    int spawned;
    pthread_t tid;
} fill_job;

static void* fill_worker(void* arg) {
    fill_job* j = (fill_job*)arg;
    size_t i = j->begin;
    while (i < j->end) {
        const uint64_t k = j->k0 + i;
        const uint64_t p = k >> 1;
        const double u1 = word_to_unit(synth_mix64(j->key + (2 * p + 1ULL) * SYNTH_GAMMA));
        const double u2 = word_to_unit(synth_mix64(j->key + (2 * p + 2ULL) * SYNTH_GAMMA));
        const double r = sqrt(-2.0 * log(u1));
        const double a = 6.283185307179586476925286766559 * u2;
        if ((k & 1) == 0) {
            j->out[i++] = (float)(j->scale * (r * cos(a)));
            if (i >= j->end) break;
        }
        j->out[i++] = (float)(j->scale * (r * sin(a)));
    }
    return NULL;
}

int synth_fill_normal(uint64_t seed, uint64_t stream, uint64_t k0, size_t n, double scale,
                      float* out, int n_threads) {
    enum { MAX_THREADS = 256 };
    if (n_threads < 1) n_threads = 1;
    if (n_threads > MAX_THREADS) n_threads = MAX_THREADS;
    if ((size_t)n_threads > n / 65536 + 1) n_threads = (int)(n / 65536 + 1);
    const uint64_t key = synth_key(seed, stream);
    fill_job jobs[MAX_THREADS];
    const size_t per = (n + (size_t)n_threads - 1) / (size_t)n_threads;
    int used = 0;
    for (int t = 0; t < n_threads; ++t) {
        const size_t b = (size_t)t * per;
        if (b >= n) break;
        const size_t e = (b + per > n) ? n : b + per;
        jobs[t] = (fill_job){key, k0, b, e, scale, out, 0, 0};
        used = t + 1;
    }
    for (int t = 0; t + 1 < used; ++t)
        jobs[t].spawned = pthread_create(&jobs[t].tid, NULL, fill_worker, &jobs[t]) == 0;
    if (used > 0) fill_worker(&jobs[used - 1]);
    for (int t = 0; t + 1 < used; ++t) {
        if (jobs[t].spawned)
            pthread_join(jobs[t].tid, NULL);
        else
            fill_worker(&jobs[t]);
    }
    return 0;
}

/* out[i] = lo + floor(uniform(seed, stream, k0 + i) * (hi - lo)), i in [0, n). */
int synth_fill_ids(uint64_t seed, uint64_t stream, uint64_t k0, size_t n, int32_t lo, int32_t hi,
                   int32_t* out) {
    if (hi <= lo) return -1;
    const double span = (double)(hi - lo);
    for (size_t i = 0; i < n; ++i) {
        int32_t v = lo + (int32_t)floor(synth_uniform(seed, stream, k0 + i) * span);
        if (v >= hi) v = hi - 1;
        out[i] = v;
    }
    return 0;
}
