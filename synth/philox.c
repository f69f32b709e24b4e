/*
 * Seeded synthetic inputs: Philox4x32-10 counters + Box-Muller normals.
 *
 * This module produces the random inputs (Q, K, V, dO, ...) that both the
 * CUDA path and the float64 oracle consume.  It contains none of the
 * attention arithmetic; it only turns (seed, stream, element index) into a
 * reproducible N(0,1) sample.
 *
 * Generator: Philox4x32 with 10 rounds, as defined in Salmon, Moraes, Dror,
 * Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11), section 4:
 *   round:  (hi0,lo0) = mulhilo(0xD2511F53, c0); (hi1,lo1) = mulhilo(0xCD9E8D57, c2)
 *           c <- (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0)
 *   key bump between rounds: k0 += 0x9E3779B9, k1 += 0xBB67AE85.
 * Counter for element e: (e/4 low 32 bits, e/4 high 32 bits, stream, 0);
 * key = (seed low 32 bits, seed high 32 bits).
 *
 * Normals: the four 32-bit words x0..x3 become uniforms u = (x + 0.5) * 2^-32
 * in (0,1); Box-Muller in float64 turns (u0,u1) and (u2,u3) into two pairs
 * r*cos(2 pi u'), r*sin(2 pi u') with r = sqrt(-2 ln u).  Element e takes
 * output word e % 4 of block e / 4.  The float64 value is rounded to float32
 * (round to nearest) and, for bf16 output, float32 -> bf16 round to nearest
 * even (inputs are finite, so no NaN handling is needed).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

static void philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; ++r) {
        uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Raw generator, exported so that the known-answer vectors of the published
 * definition can be checked. */
void synth_philox4x32_10(const uint32_t* ctr, const uint32_t* key, uint32_t* out) {
    philox4x32_10(ctr, key, out);
}

static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static void normals_of_block(uint64_t seed, uint32_t stream, uint64_t block, double z[4]) {
    uint32_t ctr[4] = {(uint32_t)block, (uint32_t)(block >> 32), stream, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t x[4];
    philox4x32_10(ctr, key, x);
    const double two32inv = 1.0 / 4294967296.0;
    const double two_pi = 6.283185307179586476925286766559;
    double u0 = ((double)x[0] + 0.5) * two32inv;
    double u1 = ((double)x[1] + 0.5) * two32inv;
    double u2 = ((double)x[2] + 0.5) * two32inv;
    double u3 = ((double)x[3] + 0.5) * two32inv;
    double r0 = sqrt(-2.0 * log(u0));
    double r1 = sqrt(-2.0 * log(u2));
    z[0] = r0 * cos(two_pi * u1);
    z[1] = r0 * sin(two_pi * u1);
    z[2] = r1 * cos(two_pi * u3);
    z[3] = r1 * sin(two_pi * u3);
}

typedef struct {
    uint64_t seed;
    uint32_t stream;
    uint64_t offset;
    uint64_t begin, end; /* element range relative to offset */
    int out_dtype;       /* 0 = float32, 1 = bf16 (uint16 bits) */
    double scale;
    void* out;
} job_t;

static void* run_job(void* arg) {
    job_t* j = (job_t*)arg;
    uint64_t e = j->begin;
    double z[4];
    uint64_t cached = ~(uint64_t)0;
    for (; e < j->end; ++e) {
        uint64_t g = j->offset + e;
        uint64_t blk = g >> 2;
        if (blk != cached) {
            normals_of_block(j->seed, j->stream, blk, z);
            cached = blk;
        }
        float f = (float)(z[g & 3] * j->scale);
        if (j->out_dtype == 0)
            ((float*)j->out)[e] = f;
        else
            ((uint16_t*)j->out)[e] = f32_to_bf16_rne(f);
    }
    return 0;
}

/* Fill out[0..n) with samples for global elements offset..offset+n of the
 * (seed, stream) sequence, each multiplied by `scale` (in float64) before
 * rounding.  Returns 0 on success, 1 on a bad dtype code. */
int synth_normal(uint64_t seed, uint32_t stream, uint64_t offset, uint64_t n,
                 int out_dtype, double scale, void* out, int nthreads) {
    if (out_dtype != 0 && out_dtype != 1) return 1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((uint64_t)nthreads > n / 65536 + 1) nthreads = (int)(n / 65536 + 1);
    pthread_t th[256];
    int created[256];
    job_t jobs[256];
    uint64_t per = (n + (uint64_t)nthreads - 1) / (uint64_t)nthreads;
    for (int t = 0; t < nthreads; ++t) {
        uint64_t b = per * (uint64_t)t, en = b + per;
        if (b > n) b = n;
        if (en > n) en = n;
        jobs[t].seed = seed;
        jobs[t].stream = stream;
        jobs[t].offset = offset;
        jobs[t].begin = b;
        jobs[t].end = en;
        jobs[t].out_dtype = out_dtype;
        jobs[t].scale = scale;
        jobs[t].out = out;
        created[t] = 0;
    }
    for (int t = 1; t < nthreads; ++t)
        created[t] = pthread_create(&th[t], 0, run_job, &jobs[t]) == 0;
    run_job(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) {
        if (created[t])
            pthread_join(th[t], 0);
        else
            run_job(&jobs[t]);
    }
    return 0;
}
