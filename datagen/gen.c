/*
 * Seeded synthetic-input generator shared by the fp64 oracle and the CUDA
 * path.  It holds none of the operators' arithmetic: only random draws and
 * the rounding of those draws into the storage types.
 *
 * Streams.  Every tensor has its own stream, keyed by its name:
 *     key = master_seed XOR fnv1a64(name)
 * and draw i of that stream is SplitMix64's output for counter i+1:
 *     z = key + (i + 1) * 0x9E3779B97F4A7C15
 *     z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
 *     z = (z ^ (z >> 27)) * 0x94D049BB133111EB
 *     out = z ^ (z >> 31)
 * (SplitMix64 as published by Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014.)  Because a draw depends only
 * on (key, i), a tensor can be filled in any order and by any number of
 * threads with identical results.
 *
 * Normals.  Element pair (2j, 2j+1) uses draws 2j and 2j+1 in the Box-Muller
 * transform, computed in double precision:
 *     u1 = ((d0 >> 11) + 1) * 2^-53        in (0, 1]
 *     u2 =  (d1 >> 11)      * 2^-53        in [0, 1)
 *     r  = sqrt(-2 ln u1)
 *     n0 = r cos(2 pi u2),  n1 = r sin(2 pi u2)
 * then value = mean + std * n.  The double is rounded to the storage type:
 * to float by C's round-to-nearest-even conversion; to bfloat16 by rounding
 * that float to nearest-even on its upper 16 bits.
 *
 * Labels.  Uniform in [0, V) by Lemire's multiply-shift of a 64-bit draw
 * (Lemire, "Fast random integer generation in an interval", 2019).  Ignored
 * rows: exactly n_ignore distinct rows chosen by a partial Fisher-Yates
 * shuffle of the row indices driven by a second stream keyed by
 * name + ":ignore"; their labels are then overwritten with ignore_index.
 *
 * Plain C11, no architecture-specific code; builds with gcc on x86_64 and
 * aarch64 and gives identical results on both.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GEN_GAMMA 0x9E3779B97F4A7C15ULL

uint64_t gen_fnv1a64(const char* s) {
    uint64_t h = 0xCBF29CE484222325ULL;
    for (const unsigned char* p = (const unsigned char*)s; *p; ++p) {
        h ^= (uint64_t)(*p);
        h *= 0x100000001B3ULL;
    }
    return h;
}

uint64_t gen_stream_key(uint64_t seed, const char* name) { return seed ^ gen_fnv1a64(name); }

static inline uint64_t splitmix_at(uint64_t key, uint64_t i) {
    uint64_t z = key + (i + 1ULL) * GEN_GAMMA;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t gen_draw(uint64_t key, uint64_t i) { return splitmix_at(key, i); }

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u) {          /* inf / nan: keep, quiet nan */
        uint16_t h = (uint16_t)(u >> 16);
        if (u & 0x007FFFFFu) h |= 0x0040u;
        return h;
    }
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

uint16_t gen_f32_to_bf16(float f) { return f32_to_bf16_rne(f); }

/* dtype codes: 0 = float64, 1 = float32, 2 = bfloat16 (uint16 bits) */
static void normal_range(uint64_t key, double mean, double stdv, int dtype, void* out,
                         uint64_t begin, uint64_t end) {
    const double two_pi = 6.283185307179586476925286766559;
    const double inv53 = 1.0 / 9007199254740992.0;
    uint64_t j0 = begin / 2, j1 = (end + 1) / 2;
    for (uint64_t j = j0; j < j1; ++j) {
        uint64_t d0 = splitmix_at(key, 2 * j), d1 = splitmix_at(key, 2 * j + 1);
        double u1 = (double)((d0 >> 11) + 1ULL) * inv53;
        double u2 = (double)(d1 >> 11) * inv53;
        double r = sqrt(-2.0 * log(u1));
        double a = two_pi * u2;
        double v[2] = {mean + stdv * (r * cos(a)), mean + stdv * (r * sin(a))};
        for (int t = 0; t < 2; ++t) {
            uint64_t e = 2 * j + (uint64_t)t;
            if (e < begin || e >= end) continue;
            if (dtype == 0) ((double*)out)[e] = v[t];
            else if (dtype == 1) ((float*)out)[e] = (float)v[t];
            else ((uint16_t*)out)[e] = f32_to_bf16_rne((float)v[t]);
        }
    }
}

typedef struct {
    uint64_t key;
    double mean, stdv;
    int dtype;
    void* out;
    uint64_t begin, end;
} normal_job;

static void* normal_worker(void* p) {
    normal_job* j = (normal_job*)p;
    normal_range(j->key, j->mean, j->stdv, j->dtype, j->out, j->begin, j->end);
    return NULL;
}

/* Fill out[0..n) with mean + std * N(0,1) draws of stream (seed, name).
 * threads <= 1 runs inline.  Returns 0, or -1 on a bad argument. */
int gen_normal(uint64_t seed, const char* name, double mean, double stdv, int dtype, void* out,
               uint64_t n, int threads) {
    if (!name || (!out && n) || dtype < 0 || dtype > 2) return -1;
    uint64_t key = gen_stream_key(seed, name);
    if (threads <= 1 || n < (1u << 20)) {
        normal_range(key, mean, stdv, dtype, out, 0, n);
        return 0;
    }
    if (threads > 256) threads = 256;
    pthread_t tid[256];
    normal_job jobs[256];
    /* split on even boundaries so each Box-Muller pair stays in one job */
    uint64_t per = ((n / (uint64_t)threads) + 1) & ~1ULL;
    int started = 0;
    for (int t = 0; t < threads; ++t) {
        uint64_t b = (uint64_t)t * per, e = b + per;
        if (b >= n) break;
        if (e > n) e = n;
        jobs[t] = (normal_job){key, mean, stdv, dtype, out, b, e};
        if (pthread_create(&tid[t], NULL, normal_worker, &jobs[t]) != 0) {
            normal_worker(&jobs[t]);
            tid[t] = 0;
        }
        started = t + 1;
    }
    for (int t = 0; t < started; ++t)
        if (tid[t]) pthread_join(tid[t], NULL);
    return 0;
}

static inline uint64_t lemire(uint64_t d, uint64_t range) {
    return (uint64_t)(((unsigned __int128)d * (unsigned __int128)range) >> 64);
}

/* Labels uniform in [0, V), then exactly n_ignore distinct rows (partial
 * Fisher-Yates over row indices, stream name + ":ignore") set to
 * ignore_index.  Returns 0, or -1 on a bad argument. */
int gen_labels(uint64_t seed, const char* name, int64_t* out, int64_t T, int64_t V,
               int64_t n_ignore, int64_t ignore_index) {
    if (!name || (!out && T) || T < 0 || V <= 0 || n_ignore < 0 || n_ignore > T) return -1;
    uint64_t key = gen_stream_key(seed, name);
    for (int64_t t = 0; t < T; ++t) out[t] = (int64_t)lemire(splitmix_at(key, (uint64_t)t), (uint64_t)V);
    if (n_ignore == 0) return 0;
    size_t nlen = strlen(name);
    char* iname = (char*)malloc(nlen + 8);
    if (!iname) return -1;
    memcpy(iname, name, nlen);
    memcpy(iname + nlen, ":ignore", 8);
    uint64_t ikey = gen_stream_key(seed, iname);
    free(iname);
    int64_t* perm = (int64_t*)malloc(sizeof(int64_t) * (size_t)T);
    if (!perm) return -1;
    for (int64_t t = 0; t < T; ++t) perm[t] = t;
    for (int64_t i = 0; i < n_ignore; ++i) {
        int64_t j = i + (int64_t)lemire(splitmix_at(ikey, (uint64_t)i), (uint64_t)(T - i));
        int64_t tmp = perm[i];
        perm[i] = perm[j];
        perm[j] = tmp;
        out[perm[i]] = ignore_index;
    }
    free(perm);
    return 0;
}

/* Positions [B, S]: uniform in [0, max_pos) by the same multiply-shift. */
int gen_positions(uint64_t seed, const char* name, int32_t* out, int64_t n, int64_t max_pos) {
    if (!name || (!out && n) || n < 0 || max_pos <= 0 || max_pos > 2147483647LL) return -1;
    uint64_t key = gen_stream_key(seed, name);
    for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)lemire(splitmix_at(key, (uint64_t)i), (uint64_t)max_pos);
    return 0;
}
