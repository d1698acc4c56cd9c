/*
 * Seeded synthetic input generators, shared by the tests, the smoke check and
 * the benchmark for both the CUDA path and the oracle. It holds none of the
 * reduction or data-movement arithmetic: it only turns (seed, element index)
 * into input values.
 *
 * Stream: SplitMix64 (G. L. Steele, D. Lea, C. H. Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014). Its k-th output (k = 0, 1, ..)
 * for a start state `seed` is mix(seed + (k+1) * 0x9E3779B97F4A7C15), so any
 * element can be computed on its own and large fills split across threads.
 *
 * Kinds (element i of a fill that starts at counter `start`; k = start + i):
 *   RAW64    z_k
 *   UNIF_F32 lo + (hi - lo) * u, u = (z_k >> 40) * 2^-24, binary32, unfused
 *   NORM_F32 Box-Muller in binary64 on draws 2k and 2k+1:
 *            u1 = ((z >> 11) + 1) * 2^-53 in (0, 1], u2 = (z' >> 11) * 2^-53,
 *            sqrt(-2 ln u1) * cos(2 pi u2), then rounded to binary32
 *   UNIF_I32 lo + ((z_k >> 11) mod (hi - lo + 1)), inclusive range
 *   BITS16   z_k >> 48
 * Compiled with -ffp-contract=off so the binary32 formula is two roundings.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

enum { RAW64 = 0, UNIF_F32 = 1, NORM_F32 = 2, UNIF_I32 = 3, BITS16 = 4 };

static const uint64_t GAMMA = 0x9E3779B97F4A7C15ull;

static uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static uint64_t draw(uint64_t seed, uint64_t k) { return mix64(seed + (k + 1u) * GAMMA); }

typedef struct {
    int kind;
    uint64_t seed, start;
    int64_t lo_i, hi_i;
    double lo, hi;
    void* out;
    int64_t begin, end;
} job_t;

static void run(const job_t* j)
{
    const double two_pi = 6.283185307179586476925286766559;
    for (int64_t i = j->begin; i < j->end; ++i) {
        uint64_t k = j->start + (uint64_t)i;
        switch (j->kind) {
        case RAW64:
            ((uint64_t*)j->out)[i] = draw(j->seed, k);
            break;
        case UNIF_F32: {
            float u = (float)(draw(j->seed, k) >> 40) * (1.0f / 16777216.0f);
            float span = (float)j->hi - (float)j->lo;
            float t = span * u;
            ((float*)j->out)[i] = (float)j->lo + t;
            break;
        }
        case NORM_F32: {
            double u1 = (double)((draw(j->seed, 2u * k) >> 11) + 1u) * (1.0 / 9007199254740992.0);
            double u2 = (double)(draw(j->seed, 2u * k + 1u) >> 11) * (1.0 / 9007199254740992.0);
            ((float*)j->out)[i] = (float)(sqrt(-2.0 * log(u1)) * cos(two_pi * u2));
            break;
        }
        case UNIF_I32: {
            uint64_t span = (uint64_t)(j->hi_i - j->lo_i) + 1u;
            ((int32_t*)j->out)[i] = (int32_t)(j->lo_i + (int64_t)((draw(j->seed, k) >> 11) % span));
            break;
        }
        case BITS16:
            ((uint16_t*)j->out)[i] = (uint16_t)(draw(j->seed, k) >> 48);
            break;
        }
    }
}

static void* thread_main(void* p)
{
    run((const job_t*)p);
    return 0;
}

/* Fill out[0..n) with elements start..start+n-1 of stream `seed`. Returns 0,
 * or -1 on an unknown kind or a bad range. */
int synth_fill(int kind, uint64_t seed, uint64_t start, int64_t n,
               double lo, double hi, int64_t lo_i, int64_t hi_i, void* out, int nthreads)
{
    if (kind < RAW64 || kind > BITS16 || n < 0) return -1;
    if (kind == UNIF_I32 && hi_i < lo_i) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 64) nthreads = 64;
    if (n < (int64_t)1 << 20) nthreads = 1;
    job_t jobs[64];
    pthread_t tid[64];
    for (int t = 0; t < nthreads; ++t) {
        job_t j = {kind, seed, start, lo_i, hi_i, lo, hi, out,
                   n * t / nthreads, n * (t + 1) / nthreads};
        jobs[t] = j;
    }
    for (int t = 1; t < nthreads; ++t)
        if (pthread_create(&tid[t], 0, thread_main, &jobs[t]) != 0) {
            run(&jobs[t]);
            tid[t] = 0;
        }
    run(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (tid[t]) pthread_join(tid[t], 0);
    return 0;
}
