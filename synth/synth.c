/*
 * Seeded synthetic inputs for split-KV decode attention.
 *
 * This file holds no attention arithmetic. It turns (seed, stream, index)
 * into numbers, and nothing else, so that the float64 oracle and the CUDA
 * path can be fed the identical bytes.
 *
 * Generator (counter based, so any element can be produced on its own):
 *   mix64(z)       the SplitMix64 output function (Steele, Lea, Flood,
 *                  "Fast splittable pseudorandom number generators",
 *                  OOPSLA 2014): z ^= z>>30; z *= 0xBF58476D1CE4E5B9;
 *                  z ^= z>>27; z *= 0x94D049BB133111EB; z ^= z>>31.
 *   key(seed, s)   mix64(seed ^ (s * 0xD1B54A32D192ED03))
 *   word(key, j)   mix64(key + (j + 1) * 0x9E3779B97F4A7C15)
 *   unit(w)        ((w >> 11) + 1) * 2^-53, in (0, 1]
 *   normal(i)      Box-Muller on the pair (unit(word(2i)), unit(word(2i+1))):
 *                  sqrt(-2 ln u1) * cos(2 pi u2), computed in double, then
 *                  rounded once, to nearest-even, to binary16 or bfloat16.
 *   uniform_int(i) lo + word(i) mod (hi - lo + 1).
 *
 * The rounding helpers below are written from the IEEE 754 binary16 and the
 * bfloat16 (IEEE binary32 with the low 16 bits dropped) encodings.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <pthread.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL
#define STREAM_MUL 0xD1B54A32D192ED03ULL

static inline uint64_t mix64(uint64_t z) {
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ULL;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBULL;
    z ^= z >> 31;
    return z;
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(seed ^ (stream * STREAM_MUL));
}

static inline uint64_t word_at(uint64_t key, uint64_t j) {
    return mix64(key + (j + 1) * GOLDEN);
}

static inline double unit_open0(uint64_t w) {
    return (double)((w >> 11) + 1) * (1.0 / 9007199254740992.0);
}

static inline double normal_at(uint64_t key, uint64_t i) {
    const double two_pi = 6.283185307179586476925286766559;
    double u1 = unit_open0(word_at(key, 2 * i));
    double u2 = unit_open0(word_at(key, 2 * i + 1));
    return sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
}

/* double -> binary16, round to nearest, ties to even (one rounding). */
uint16_t synth_double_to_f16(double x) {
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (isnan(x)) return (uint16_t)(sign | 0x7e00u);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u); /* max finite 65504; midpoint 65520 ties to inf */
    if (a < 6.103515625e-05) {                            /* below 2^-14: subnormal grid of 2^-24 */
        double q = rint(ldexp(a, 24));                    /* q <= 1024; 1024 is the smallest normal */
        return (uint16_t)(sign | (uint16_t)q);
    }
    int e;
    frexp(a, &e);                       /* a = f * 2^e, f in [0.5, 1) */
    double r = rint(ldexp(a, 11 - e));  /* significand on [1024, 2048] */
    int E = e - 1;
    if (r == 2048.0) { r = 1024.0; E += 1; }
    if (E > 15) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)((int)r - 1024));
}

/* double -> bfloat16, round to nearest, ties to even (one rounding). */
uint16_t synth_double_to_bf16(double x) {
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (isnan(x)) return (uint16_t)(sign | 0x7fc0u);
    const double min_normal = ldexp(1.0, -126);
    if (a < min_normal) {                               /* subnormal grid of 2^-133 */
        double q = rint(ldexp(a, 133));                 /* q <= 128; 128 is the smallest normal */
        return (uint16_t)(sign | (uint16_t)q);
    }
    int e;
    frexp(a, &e);
    double r = rint(ldexp(a, 8 - e));   /* significand on [128, 256] */
    int E = e - 1;
    if (r == 256.0) { r = 128.0; E += 1; }
    if (E > 127) return (uint16_t)(sign | 0x7f80u);
    return (uint16_t)(sign | (uint16_t)((E + 127) << 7) | (uint16_t)((int)r - 128));
}

typedef struct {
    uint64_t key;
    uint64_t first;
    uint64_t count;
    int kind;        /* 0 = f16, 1 = bf16, 2 = f64 */
    double mean;
    double std;
    void* out;
} fill_job;

static void* fill_worker(void* arg) {
    fill_job* jb = (fill_job*)arg;
    for (uint64_t t = 0; t < jb->count; ++t) {
        uint64_t i = jb->first + t;
        double z = jb->mean + jb->std * normal_at(jb->key, i);
        if (jb->kind == 0) ((uint16_t*)jb->out)[t] = synth_double_to_f16(z);
        else if (jb->kind == 1) ((uint16_t*)jb->out)[t] = synth_double_to_bf16(z);
        else ((double*)jb->out)[t] = z;
    }
    return NULL;
}

/*
 * Fill out[0..n) with N(mean, std^2) elements first..first+n-1 of stream
 * (seed, stream). kind: 0 binary16 bits, 1 bfloat16 bits, 2 double.
 * Uses up to nthreads POSIX threads; the result does not depend on it.
 * Returns 0, or -1 on a bad argument.
 */
int synth_normal(uint64_t seed, uint64_t stream, uint64_t first, uint64_t n, int kind,
                 double mean, double std, void* out, int nthreads) {
    if (kind < 0 || kind > 2 || (n > 0 && out == NULL)) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((uint64_t)nthreads > n / 65536 + 1) nthreads = (int)(n / 65536 + 1);
    uint64_t key = stream_key(seed, stream);
    size_t esz = kind == 2 ? 8 : 2;
    fill_job jobs[256];
    pthread_t th[256];
    uint64_t per = (n + (uint64_t)nthreads - 1) / (uint64_t)nthreads;
    int launched = 0;
    for (int t = 0; t < nthreads; ++t) {
        uint64_t lo = (uint64_t)t * per;
        if (lo >= n) break;
        uint64_t hi = lo + per < n ? lo + per : n;
        jobs[t].key = key;
        jobs[t].first = first + lo;
        jobs[t].count = hi - lo;
        jobs[t].kind = kind;
        jobs[t].mean = mean;
        jobs[t].std = std;
        jobs[t].out = (char*)out + lo * esz;
        launched = t + 1;
    }
    if (launched <= 1) {
        if (launched == 1) fill_worker(&jobs[0]);
        return 0;
    }
    int spawned = 0;
    for (int t = 1; t < launched; ++t) {
        if (pthread_create(&th[t], NULL, fill_worker, &jobs[t]) != 0) break;
        spawned = t;
    }
    fill_worker(&jobs[0]);
    for (int t = spawned + 1; t < launched; ++t) fill_worker(&jobs[t]);
    for (int t = 1; t <= spawned; ++t) pthread_join(th[t], NULL);
    return 0;
}

/* out[t] = lo + word(first + t) mod (hi - lo + 1), for t in [0, n). Requires lo <= hi. */
int synth_uniform_int(uint64_t seed, uint64_t stream, uint64_t first, uint64_t n,
                      int64_t lo, int64_t hi, int64_t* out) {
    if (hi < lo || (n > 0 && out == NULL)) return -1;
    uint64_t key = stream_key(seed, stream);
    uint64_t span = (uint64_t)(hi - lo) + 1u;
    for (uint64_t t = 0; t < n; ++t) {
        uint64_t w = word_at(key, first + t);
        out[t] = lo + (int64_t)(span == 0 ? w : w % span);
    }
    return 0;
}
