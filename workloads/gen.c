/*
 * Seeded synthetic inputs for the fused LM-head loss workloads.
 *
 * This module holds no loss arithmetic.  It only draws random numbers and
 * shapes them into logits, targets, masks, margins and segments.  Both the
 * CUDA path (through device copies of these host arrays) and the oracle read
 * the very same bits.
 *
 * Randomness: Philox4x32-10, the counter-based generator of Salmon, Moraes,
 * Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11):
 * ten rounds of two 32x32->64 multiplies with the published multipliers and
 * Weyl key increments.  Every output is a pure function of
 * (seed, stream, config, index), so any row can be regenerated on its own.
 * Normals come from the Box-Muller transform in double precision.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

typedef struct { uint32_t v[4]; } gen_u4;

gen_u4 gen_philox4x32_10(gen_u4 ctr, uint32_t k0, uint32_t k1)
{
    for (int round = 0; round < 10; ++round) {
        uint64_t p0 = (uint64_t)PHILOX_M0 * ctr.v[0];
        uint64_t p1 = (uint64_t)PHILOX_M1 * ctr.v[2];
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        gen_u4 nx;
        nx.v[0] = hi1 ^ ctr.v[1] ^ k0;
        nx.v[1] = lo1;
        nx.v[2] = hi0 ^ ctr.v[3] ^ k1;
        nx.v[3] = lo0;
        ctr = nx;
        k0 += PHILOX_W0;
        k1 += PHILOX_W1;
    }
    return ctr;
}

/* Exported for the known-answer test. */
void gen_philox_kat(const uint32_t ctr_in[4], const uint32_t key[2], uint32_t out[4])
{
    gen_u4 c;
    memcpy(c.v, ctr_in, sizeof c.v);
    gen_u4 r = gen_philox4x32_10(c, key[0], key[1]);
    memcpy(out, r.v, sizeof r.v);
}

/* Counter layout: (index lo, index hi, row lo, row hi ^ (config << 24)). */
static gen_u4 gen_draw(uint32_t seed, uint32_t cfg, uint32_t stream, int64_t row, int64_t idx)
{
    gen_u4 c;
    c.v[0] = (uint32_t)((uint64_t)idx & 0xffffffffu);
    c.v[1] = (uint32_t)((uint64_t)idx >> 32);
    c.v[2] = (uint32_t)((uint64_t)row & 0xffffffffu);
    c.v[3] = (uint32_t)((uint64_t)row >> 32) ^ (cfg << 24);
    return gen_philox4x32_10(c, seed, stream);
}

/* Uniform double in (0, 1) from 53 bits. */
static double gen_unit(uint32_t hi, uint32_t lo)
{
    uint64_t b = (((uint64_t)hi << 32) | lo) >> 11;
    return ((double)b + 0.5) * (1.0 / 9007199254740992.0);
}

static void gen_box_muller(gen_u4 x, double* n0, double* n1)
{
    double u1 = gen_unit(x.v[0], x.v[1]);
    double u2 = gen_unit(x.v[2], x.v[3]);
    double r = sqrt(-2.0 * log(u1));
    double th = 6.283185307179586 * u2;
    *n0 = r * cos(th);
    *n1 = r * sin(th);
}

/* Round-to-nearest-even of an fp32 value to bf16 bits (inputs are finite). */
static uint16_t gen_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u) return (uint16_t)((u >> 16) | ((u & 0xffffu) ? 0x40u : 0u));
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float gen_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

enum { GEN_BF16 = 0, GEN_FP32 = 1 };

static void gen_store(int dtype, void* out, int64_t idx, double x)
{
    if (dtype == GEN_BF16) ((uint16_t*)out)[idx] = gen_bf16_rne((float)x);
    else ((float*)out)[idx] = (float)x;
}

static double gen_load(int dtype, const void* in, int64_t idx)
{
    if (dtype == GEN_BF16) return (double)gen_bf16_to_f32(((const uint16_t*)in)[idx]);
    return (double)((const float*)in)[idx];
}

static int gen_nthreads(int n)
{
#ifdef _OPENMP
    return n > 0 ? n : omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* Rows [row0, row0 + nrows) of an N(mean, sigma^2) matrix, columns [0, V),
 * written to out[(r - row0) * ld + j] as bf16 bits or fp32. */
void gen_normal_rows(uint32_t seed, uint32_t cfg, uint32_t stream, int64_t row0, int64_t nrows,
                     int64_t V, int64_t ld, double mean, double sigma, int dtype, void* out, int nthreads)
{
#pragma omp parallel for schedule(static) num_threads(gen_nthreads(nthreads))
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t row = row0 + i;
        for (int64_t k = 0; 2 * k < V; ++k) {
            double a, b;
            gen_box_muller(gen_draw(seed, cfg, stream, row, k), &a, &b);
            gen_store(dtype, out, i * ld + 2 * k, mean + sigma * a);
            if (2 * k + 1 < V) gen_store(dtype, out, i * ld + 2 * k + 1, mean + sigma * b);
        }
    }
}

/* out = round(base + N(0, sigma^2)) element-wise over the same rows/columns. */
void gen_add_normal_rows(uint32_t seed, uint32_t cfg, uint32_t stream, int64_t row0, int64_t nrows,
                         int64_t V, int64_t ld, double sigma, int dtype, const void* base, void* out,
                         int nthreads)
{
#pragma omp parallel for schedule(static) num_threads(gen_nthreads(nthreads))
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t row = row0 + i;
        for (int64_t k = 0; 2 * k < V; ++k) {
            double a, b;
            gen_box_muller(gen_draw(seed, cfg, stream, row, k), &a, &b);
            int64_t j = i * ld + 2 * k;
            gen_store(dtype, out, j, gen_load(dtype, base, j) + sigma * a);
            if (2 * k + 1 < V) gen_store(dtype, out, j + 1, gen_load(dtype, base, j + 1) + sigma * b);
        }
    }
}

/* 1-D draws indexed by i0 + i. */
void gen_normal_1d(uint32_t seed, uint32_t cfg, uint32_t stream, int64_t i0, int64_t n,
                   double mean, double sigma, double* out)
{
    for (int64_t i = 0; i < n; ++i) {
        double a, b;
        gen_box_muller(gen_draw(seed, cfg, stream, -1, i0 + i), &a, &b);
        out[i] = mean + sigma * a;
    }
}

void gen_uniform_1d(uint32_t seed, uint32_t cfg, uint32_t stream, int64_t i0, int64_t n,
                    double lo, double hi, double* out)
{
    for (int64_t i = 0; i < n; ++i) {
        gen_u4 x = gen_draw(seed, cfg, stream, -1, i0 + i);
        out[i] = lo + (hi - lo) * gen_unit(x.v[0], x.v[1]);
    }
}

/* Integers in [0, range) by 64-bit multiply-shift of a 32-bit draw
 * (bias below range / 2^32). */
void gen_randint_1d(uint32_t seed, uint32_t cfg, uint32_t stream, int64_t i0, int64_t n,
                    int64_t range, int64_t* out)
{
    for (int64_t i = 0; i < n; ++i) {
        gen_u4 x = gen_draw(seed, cfg, stream, -1, i0 + i);
        out[i] = (int64_t)(((uint64_t)x.v[0] * (uint64_t)range) >> 32);
    }
}

/* Fisher-Yates shuffle of 0..n-1; swap position i draws from index i. */
void gen_permutation(uint32_t seed, uint32_t cfg, uint32_t stream, int64_t n, int64_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = i;
    for (int64_t i = n - 1; i > 0; --i) {
        gen_u4 x = gen_draw(seed, cfg, stream, -2, i);
        int64_t j = (int64_t)(((uint64_t)x.v[0] * (uint64_t)(i + 1)) >> 32);
        int64_t t = out[i];
        out[i] = out[j];
        out[j] = t;
    }
}

/* Plant a target margin: for each row i with a finite margin[i],
 * z_t := round(max_{j != t} z_j + margin[i]).  Rows with NaN margin are left alone. */
void gen_plant_rows(int dtype, int64_t nrows, int64_t V, int64_t ld, void* logits,
                    const int64_t* targets, const double* margin, int nthreads)
{
#pragma omp parallel for schedule(static) num_threads(gen_nthreads(nthreads))
    for (int64_t i = 0; i < nrows; ++i) {
        if (isnan(margin[i])) continue;
        int64_t t = targets[i];
        if (t < 0 || t >= V) continue;
        double m = -INFINITY;
        for (int64_t j = 0; j < V; ++j) {
            if (j == t) continue;
            double z = gen_load(dtype, logits, i * ld + j);
            if (z > m) m = z;
        }
        gen_store(dtype, logits, i * ld + t, m + margin[i]);
    }
}
