/*
 * Seeded synthetic KV records for the host pool (input generation only).
 *
 * Every record is a pure function of (seed, stream, position): element pair
 * j of record `pos` in stream `s` (s = request * n_layers + layer) takes the
 * 64-bit word
 *
 *     h = splitmix64(key(seed, s) + pos * (W / 4) + j),
 *     key(seed, s) = splitmix64(splitmix64(seed) ^ (s + 1) * 0x9E3779B97F4A7C15)
 *
 * where splitmix64 is Steele, Lea and Flood's finaliser ("Fast splittable
 * pseudorandom number generators", OOPSLA 2014):
 *     z += 0x9E3779B97F4A7C15; z = (z ^ z>>30) * 0xBF58476D1CE4E5B9;
 *     z = (z ^ z>>27) * 0x94D049BB133111EB; return z ^ z>>31.
 * The two 24-bit fields u1 = h>>40 and u2 = (h>>16) & 0xFFFFFF give the pair:
 *   format 0 (fp16 U(-1,1)):  x = (u + 0.5) / 2^23 - 1 for u = u1, u2,
 *                             rounded to fp16 (nearest, ties to even);
 *   format 1 (bf16 N(0,1)):   Box-Muller on a = (u1 + 0.5) / 2^24,
 *                             b = (u2 + 0.5) / 2^24:
 *                             r = sqrt(-2 ln a), (r cos 2 pi b, r sin 2 pi b),
 *                             computed in float and rounded to bf16 (nearest,
 *                             ties to even).
 * Elements are little-endian 16-bit values, pair j at bytes [4j, 4j + 4).
 *
 * This file draws inputs only; it holds nothing of the resolve method.
 */
#define _GNU_SOURCE
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t splitmix64(uint64_t z) {
    z += 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return splitmix64(splitmix64(seed) ^ ((stream + 1) * 0x9E3779B97F4A7C15ull));
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))  /* NaN */
        return (uint16_t)((u >> 16) | 0x40);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

static inline uint16_t f32_to_f16_rne(float f) {
    _Float16 h = (_Float16)f;  /* C rounding mode: to nearest, ties to even */
    uint16_t u;
    memcpy(&u, &h, 2);
    return u;
}

static inline void make_pair(uint64_t h, int fmt, uint16_t *e) {
    uint32_t u1 = (uint32_t)(h >> 40);
    uint32_t u2 = (uint32_t)((h >> 16) & 0xFFFFFFu);
    if (fmt == 0) {
        float x0 = ((float)u1 + 0.5f) * (1.0f / 8388608.0f) - 1.0f;
        float x1 = ((float)u2 + 0.5f) * (1.0f / 8388608.0f) - 1.0f;
        e[0] = f32_to_f16_rne(x0);
        e[1] = f32_to_f16_rne(x1);
    } else {
        float a = ((float)u1 + 0.5f) * (1.0f / 16777216.0f);
        float b = ((float)u2 + 0.5f) * (1.0f / 16777216.0f);
        float r = sqrtf(-2.0f * logf(a));
        float th = 6.28318530717958647692f * b, sn, cs;
        sincosf(th, &sn, &cs);
        e[0] = f32_to_bf16_rne(r * cs);
        e[1] = f32_to_bf16_rne(r * sn);
    }
}

static void gen_one(uint8_t *dst, int64_t pos, int32_t W, int fmt, uint64_t key) {
    int64_t npair = W / 4;
    uint64_t base = key + (uint64_t)pos * (uint64_t)npair;
    uint16_t *e = (uint16_t *)dst;
    for (int64_t j = 0; j < npair; ++j)
        make_pair(splitmix64(base + (uint64_t)j), fmt, e + 2 * j);
}

/* Records for an explicit list of positions: dst[i] = record(positions[i]). */
void wl_gen_records(uint8_t *dst, const int32_t *positions, int64_t n, int32_t W,
                    int fmt, uint64_t seed, uint64_t stream) {
    uint64_t key = stream_key(seed, stream);
    for (int64_t i = 0; i < n; ++i)
        gen_one(dst + i * (int64_t)W, positions[i], W, fmt, key);
}

typedef struct {
    uint8_t *dst;
    int64_t pos0, n;
    int32_t W;
    int fmt;
    uint64_t key;
} fill_job;

static void *fill_worker(void *arg) {
    fill_job *j = (fill_job *)arg;
    for (int64_t i = 0; i < j->n; ++i)
        gen_one(j->dst + i * (int64_t)j->W, j->pos0 + i, j->W, j->fmt, j->key);
    return 0;
}

/* Records for the contiguous positions [pos0, pos0 + n) of one stream,
 * written to dst[0..n) and split over n_threads threads. Returns 0 on success. */
int wl_fill_records(uint8_t *dst, int64_t pos0, int64_t n, int32_t W, int fmt,
                    uint64_t seed, uint64_t stream, int n_threads) {
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    uint64_t key = stream_key(seed, stream);
    pthread_t th[256];
    fill_job jobs[256];
    int64_t per = (n + n_threads - 1) / n_threads;
    int started = 0;
    for (int t = 0; t < n_threads; ++t) {
        int64_t a = t * per, b = a + per;
        if (b > n) b = n;
        if (a >= b) break;
        jobs[t] = (fill_job){dst + a * (int64_t)W, pos0 + a, b - a, W, fmt, key};
        if (pthread_create(&th[started], 0, fill_worker, &jobs[t]) == 0)
            ++started;
        else
            fill_worker(&jobs[t]);  /* no thread: do this share inline */
    }
    for (int t = 0; t < started; ++t) pthread_join(th[t], 0);
    return 0;
}
