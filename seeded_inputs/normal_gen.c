/*
 * Seeded synthetic inputs for the attention forward path.
 *
 * Both the CUDA path's tests and the CPU oracle draw their Q/K/V from here, so
 * this file holds no attention arithmetic at all: it only produces iid N(0,1)
 * samples and rounds them to a 16-bit storage type.
 *
 *   uniform bits : the splitmix64 sequence (Steele, Lea and Flood, "Fast
 *                  splittable pseudorandom number generators", OOPSLA 2014;
 *                  the constants are those of Vigna's public-domain
 *                  splitmix64.c).  Output i of the stream started at `seed`
 *                  is mix(seed + (i + 1) * GOLDEN_GAMMA), so any sub-range of
 *                  the stream can be produced independently (counter based).
 *   normals      : Box-Muller (Box and Muller 1958).  Normal 2p uses
 *                  uniforms 2p and 2p+1 through the cosine branch, normal
 *                  2p+1 the same pair through the sine branch.
 *   rounding     : float64 -> IEEE binary16 or bfloat16, round to nearest,
 *                  ties to even, subnormals kept, overflow to infinity.
 *
 * Element g of the stream is normal number g.  A caller that wants "Q, then
 * K, then V from one stream" passes offsets 0, nQ and nQ + nK.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

#define GOLDEN_GAMMA 0x9e3779b97f4a7c15ULL

static uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}

uint64_t si_splitmix64_at(uint64_t seed, uint64_t i) { return mix64(seed + (i + 1) * GOLDEN_GAMMA); }

/* 53 random bits -> a double in [0, 1). */
static double unit_interval(uint64_t bits) { return (double)(bits >> 11) * 0x1.0p-53; }

/* Normal number g of the stream started at `seed`. */
double si_normal_at(uint64_t seed, uint64_t g) {
    uint64_t p = g >> 1;
    double u1 = 1.0 - unit_interval(si_splitmix64_at(seed, 2 * p)); /* (0, 1]: log() stays finite */
    double u2 = unit_interval(si_splitmix64_at(seed, 2 * p + 1));
    double r = sqrt(-2.0 * log(u1));
    double t = 2.0 * M_PI * u2;
    return (g & 1) ? r * sin(t) : r * cos(t);
}

/* Round a double to a storage format with `sig` significant bits (implicit bit
 * included), exponent bias `bias` and `ebits` exponent bits; ties to even. */
static uint16_t round_to_small_float(double x, int sig, int ebits, int bias) {
    const int mant_bits = sig - 1;
    const uint16_t sign = signbit(x) ? (uint16_t)(1u << 15) : 0;
    const uint16_t exp_all_ones = (uint16_t)(((1u << ebits) - 1) << mant_bits);
    if (isnan(x)) return (uint16_t)(exp_all_ones | (1u << (mant_bits - 1)));
    double a = fabs(x);
    if (isinf(a)) return sign | exp_all_ones;
    const int emin = 1 - bias;                 /* exponent of the smallest normal */
    if (a < ldexp(1.0, emin)) {                /* subnormal range: a = m * 2^(emin - mant_bits) */
        double m = nearbyint(ldexp(a, mant_bits - emin));
        return sign | (uint16_t)m;             /* m == 2^mant_bits is the smallest normal: still right */
    }
    int e;
    double f = frexp(a, &e);                   /* a = f * 2^e, f in [0.5, 1) */
    double m = nearbyint(ldexp(f, sig));       /* sig significant bits, in [2^(sig-1), 2^sig] */
    if (m == ldexp(1.0, sig)) { m = ldexp(1.0, sig - 1); e += 1; }
    int biased = e - 1 + bias;
    if (biased >= (1 << ebits) - 1) return sign | exp_all_ones;
    return sign | (uint16_t)((unsigned)biased << mant_bits) | (uint16_t)((uint64_t)m - (1ull << mant_bits));
}

uint16_t si_round_f16(double x) { return round_to_small_float(x, 11, 5, 15); }
uint16_t si_round_bf16(double x) { return round_to_small_float(x, 8, 8, 127); }

typedef struct {
    uint64_t seed, offset;
    int64_t begin, end;
    int dtype; /* 0: fp16, 1: bf16, 2: keep float64 */
    void* out;
} gen_job;

static void* gen_worker(void* arg) {
    gen_job* j = (gen_job*)arg;
    for (int64_t i = j->begin; i < j->end; ++i) {
        double z = si_normal_at(j->seed, j->offset + (uint64_t)i);
        if (j->dtype == 2) ((double*)j->out)[i] = z;
        else ((uint16_t*)j->out)[i] = j->dtype == 0 ? si_round_f16(z) : si_round_bf16(z);
    }
    return NULL;
}

/* Fill out[0..n) with normals offset..offset+n-1 of the stream `seed`.
 * dtype 0/1 write uint16 bit patterns (fp16/bf16), dtype 2 writes float64.
 * Returns 0 on success, -1 on bad arguments. */
int si_fill_normal(uint64_t seed, uint64_t offset, int64_t n, int dtype, void* out, int nthreads) {
    if (n < 0 || dtype < 0 || dtype > 2 || (n > 0 && out == NULL)) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (n < 65536) nthreads = 1;
    gen_job jobs[256];
    pthread_t tid[256];
    int created[256] = {0};
    int64_t chunk = (n + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        int64_t b = (int64_t)t * chunk, e = b + chunk < n ? b + chunk : n;
        if (b >= e) break;
        jobs[t] = (gen_job){seed, offset, b, e, dtype, out};
        if (nthreads > 1 && pthread_create(&tid[t], NULL, gen_worker, &jobs[t]) == 0) created[t] = 1;
        else gen_worker(&jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t)
        if (created[t]) pthread_join(tid[t], NULL);
    return 0;
}
