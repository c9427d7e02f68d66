/*
 * Seeded synthetic inputs for the MaxSim operator: token embeddings, lengths,
 * masks, per-token INT8 quantisation and upstream gradients.
 *
 * This module holds input preparation only. It computes no part of the
 * operator itself (no dot products, maxima, scores or gradients), so both the
 * CUDA path and the CPU oracle can consume its bytes without sharing any of
 * the method's arithmetic.
 *
 * Random numbers: PCG32 (M. E. O'Neill, "PCG: A Family of Simple Fast
 * Space-Efficient Statistically Good Algorithms for Random Number Generation",
 * 2014; the pcg32_random_r / pcg32_srandom_r definitions). Every row (or
 * element) draws from its own stream, selected by (seed, tensor id, index), so
 * any subset of rows can be regenerated independently and the generation is
 * parallel without changing a single byte.
 *
 * Normal deviates: Box-Muller transform on two uniforms in (0,1).
 * Token rows are l2-normalised in double and rounded once to the storage type
 * (binary16 or bfloat16, round-to-nearest-even written from the IEEE formats).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    uint64_t state;
    uint64_t inc;
} pcg32_t;

static uint32_t pcg32_next(pcg32_t *r) {
    uint64_t old = r->state;
    r->state = old * 6364136223846793005ULL + r->inc;
    uint32_t xorshifted = (uint32_t)(((old >> 18u) ^ old) >> 27u);
    uint32_t rot = (uint32_t)(old >> 59u);
    return (xorshifted >> rot) | (xorshifted << ((-rot) & 31u));
}

static void pcg32_seed(pcg32_t *r, uint64_t initstate, uint64_t initseq) {
    r->state = 0u;
    r->inc = (initseq << 1u) | 1u;
    pcg32_next(r);
    r->state += initstate;
    pcg32_next(r);
}

/* SplitMix64 finaliser, used only to spread (seed, tensor id) into a state. */
static uint64_t mix64(uint64_t z) {
    z += 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static void stream_for(pcg32_t *r, uint64_t seed, uint64_t tensor_id, uint64_t index) {
    pcg32_seed(r, mix64(seed * 0x100000001B3ULL + tensor_id), index);
}

/* Uniform double in the open interval (0,1) with 53 random bits. */
static double uniform01(pcg32_t *r) {
    uint64_t hi = pcg32_next(r) >> 5;   /* 27 bits */
    uint64_t lo = pcg32_next(r) >> 6;   /* 26 bits */
    uint64_t m = (hi << 26) | lo;       /* 53 bits */
    return ((double)m + 0.5) * (1.0 / 9007199254740992.0);
}

/* Uniform integer in [0, n) by rejection (no modulo bias). */
static uint32_t uniform_below(pcg32_t *r, uint32_t n) {
    if (n <= 1) return 0;
    uint32_t threshold = (uint32_t)(-n) % n;
    for (;;) {
        uint32_t x = pcg32_next(r);
        if (x >= threshold) return x % n;
    }
}

static void normal_pair(pcg32_t *r, double *z0, double *z1) {
    const double two_pi = 6.283185307179586476925286766559;
    double u1 = uniform01(r), u2 = uniform01(r);
    double rad = sqrt(-2.0 * log(u1));
    *z0 = rad * cos(two_pi * u2);
    *z1 = rad * sin(two_pi * u2);
}

/* ---- IEEE rounding from double, round-to-nearest-even ------------------- */

/* binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static uint16_t double_to_f16(double x) {
    uint64_t b;
    memcpy(&b, &x, 8);
    uint16_t sign = (uint16_t)((b >> 48) & 0x8000u);
    int e = (int)((b >> 52) & 0x7FF);
    uint64_t frac = b & 0xFFFFFFFFFFFFFULL;
    if (e == 0x7FF) return (uint16_t)(sign | 0x7C00u | (frac ? 0x200u : 0u));
    if (e == 0 && frac == 0) return sign;
    /* value = 1.frac * 2^(e-1023) (subnormal doubles underflow to 0 below) */
    int exp = e - 1023;
    uint64_t mant = frac | (1ULL << 52); /* 53 significant bits */
    if (e == 0) return sign;             /* double subnormal: far below f16 range */
    int shift;                           /* bits to drop from the 53-bit significand */
    uint32_t hexp;
    if (exp >= -14) {
        hexp = (uint32_t)(exp + 15);
        shift = 42;                      /* keep 11 bits (implicit + 10) */
    } else {
        hexp = 0;                        /* subnormal: value = m * 2^-24 */
        shift = 42 + (-14 - exp);
        if (shift > 63) return sign;     /* rounds to zero */
    }
    uint64_t kept = mant >> shift;
    uint64_t rem = mant & ((1ULL << shift) - 1);
    uint64_t half = 1ULL << (shift - 1);
    if (rem > half || (rem == half && (kept & 1))) kept++;
    if (hexp == 0) {
        /* kept <= 2^10; kept == 2^10 is the smallest normal, encoded naturally */
        return (uint16_t)(sign | (uint16_t)kept);
    }
    if (kept == (1ULL << 11)) { kept >>= 1; hexp++; }
    if (hexp >= 31) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (hexp << 10) | (uint16_t)(kept & 0x3FFu));
}

/* bfloat16: the upper 16 bits of binary32 (8 exponent bits, 7 fraction bits).
 * Rounded once from double: handled as a float with a 7-bit fraction. */
static uint16_t double_to_bf16(double x) {
    uint64_t b;
    memcpy(&b, &x, 8);
    uint16_t sign = (uint16_t)((b >> 48) & 0x8000u);
    int e = (int)((b >> 52) & 0x7FF);
    uint64_t frac = b & 0xFFFFFFFFFFFFFULL;
    if (e == 0x7FF) return (uint16_t)(sign | 0x7F80u | (frac ? 0x40u : 0u));
    if (e == 0) return sign;
    int exp = e - 1023;
    uint64_t mant = frac | (1ULL << 52);
    int shift;
    uint32_t bexp;
    if (exp >= -126) {
        bexp = (uint32_t)(exp + 127);
        shift = 45;                      /* keep 8 bits (implicit + 7) */
    } else {
        bexp = 0;
        shift = 45 + (-126 - exp);
        if (shift > 63) return sign;
    }
    uint64_t kept = mant >> shift;
    uint64_t rem = mant & ((1ULL << shift) - 1);
    uint64_t half = 1ULL << (shift - 1);
    if (rem > half || (rem == half && (kept & 1))) kept++;
    if (bexp == 0) return (uint16_t)(sign | (uint16_t)kept);
    if (kept == (1ULL << 8)) { kept >>= 1; bexp++; }
    if (bexp >= 255) return (uint16_t)(sign | 0x7F80u);
    return (uint16_t)(sign | (bexp << 7) | (uint16_t)(kept & 0x7Fu));
}

/* ---- exported generators -------------------------------------------------- */

static void gaussian_row(uint64_t seed, uint64_t tensor_id, int64_t row, int64_t dim,
                         int normalize, double *buf) {
    pcg32_t r;
    stream_for(&r, seed, tensor_id, (uint64_t)row);
    for (int64_t k = 0; k < dim; k += 2) {
        double z0, z1;
        normal_pair(&r, &z0, &z1);
        buf[k] = z0;
        if (k + 1 < dim) buf[k + 1] = z1;
    }
    if (normalize) {
        double ss = 0.0;
        for (int64_t k = 0; k < dim; ++k) ss += buf[k] * buf[k];
        double inv = 1.0 / sqrt(ss);
        for (int64_t k = 0; k < dim; ++k) buf[k] *= inv;
    }
}

/* out_dtype: 0 = binary16, 1 = bfloat16, 2 = float64, 3 = float32.
 * Rows [row0, row0 + nrows) of a [*, dim] tensor; row r uses stream r. */
int dg_gaussian_rows(uint64_t seed, uint64_t tensor_id, int64_t row0, int64_t nrows,
                     int64_t dim, int normalize, int out_dtype, void *out) {
    if (dim <= 0 || dim > 4096 || nrows < 0) return 1;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < nrows; ++i) {
        double b[4096];
        gaussian_row(seed, tensor_id, row0 + i, dim, normalize, b);
        for (int64_t k = 0; k < dim; ++k) {
            int64_t o = i * dim + k;
            switch (out_dtype) {
            case 0: ((uint16_t *)out)[o] = double_to_f16(b[k]); break;
            case 1: ((uint16_t *)out)[o] = double_to_bf16(b[k]); break;
            case 2: ((double *)out)[o] = b[k]; break;
            default: ((float *)out)[o] = (float)b[k]; break;
            }
        }
    }
    return 0;
}

/* Per-token symmetric INT8 quantisation of l2-normalised Gaussian rows:
 * scale = max_k |x_k| / 127 (stored as float32), q = clamp(rint(x / scale)).
 * rint is round-half-to-even under the default rounding mode. */
int dg_int8_rows(uint64_t seed, uint64_t tensor_id, int64_t row0, int64_t nrows, int64_t dim,
                 int8_t *q_out, float *scale_out) {
    if (dim <= 0 || dim > 1024 || nrows < 0) return 1;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < nrows; ++i) {
        double b[1024];
        gaussian_row(seed, tensor_id, row0 + i, dim, 1, b);
        double amax = 0.0;
        for (int64_t k = 0; k < dim; ++k) {
            double a = fabs(b[k]);
            if (a > amax) amax = a;
        }
        float s = (float)(amax / 127.0);
        if (!(s > 0.0f)) s = 1.0f; /* all-zero row cannot come from a normalised draw */
        scale_out[i] = s;
        for (int64_t k = 0; k < dim; ++k) {
            double v = nearbyint(b[k] / (double)s);
            if (v > 127.0) v = 127.0;
            if (v < -127.0) v = -127.0;
            q_out[i * dim + k] = (int8_t)v;
        }
    }
    return 0;
}

/* n integers uniform in [lo, hi] (inclusive); element e uses stream e. */
int dg_uniform_int(uint64_t seed, uint64_t tensor_id, int64_t n, int32_t lo, int32_t hi,
                   int32_t *out) {
    if (hi < lo || n < 0) return 1;
    uint32_t span = (uint32_t)((int64_t)hi - (int64_t)lo + 1);
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < n; ++e) {
        pcg32_t r;
        stream_for(&r, seed, tensor_id, (uint64_t)e);
        out[e] = lo + (int32_t)uniform_below(&r, span);
    }
    return 0;
}

/* n float32 standard normal values (for upstream gradients); element pairs
 * (2p, 2p+1) share stream p. */
int dg_normal_f32(uint64_t seed, uint64_t tensor_id, int64_t n, float *out) {
    if (n < 0) return 1;
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < (n + 1) / 2; ++p) {
        pcg32_t r;
        stream_for(&r, seed, tensor_id, (uint64_t)p);
        double z0, z1;
        normal_pair(&r, &z0, &z1);
        out[2 * p] = (float)z0;
        if (2 * p + 1 < n) out[2 * p + 1] = (float)z1;
    }
    return 0;
}

/* Mask that keeps the first L - k tokens of each of n items, k ~ U{0..kmax}
 * (clamped to L); item e uses stream e. mask is [n, L] bytes, 1 = active. */
int dg_mask_drop_tail(uint64_t seed, uint64_t tensor_id, int64_t n, int64_t L, int32_t kmax,
                      uint8_t *mask) {
    if (n < 0 || L < 0 || kmax < 0) return 1;
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < n; ++e) {
        pcg32_t r;
        stream_for(&r, seed, tensor_id, (uint64_t)e);
        int64_t k = (int64_t)uniform_below(&r, (uint32_t)kmax + 1u);
        if (k > L) k = L;
        for (int64_t t = 0; t < L; ++t) mask[e * L + t] = (uint8_t)(t < L - k ? 1 : 0);
    }
    return 0;
}

/* Mask that hides a uniformly random subset of k ~ U{0..kmax} positions
 * (clamped to L) of each of n items, chosen by a partial Fisher-Yates shuffle
 * on the item's stream. mask is [n, L] bytes, 1 = active. */
int dg_mask_random_subset(uint64_t seed, uint64_t tensor_id, int64_t n, int64_t L,
                          int32_t kmax, uint8_t *mask) {
    if (n < 0 || L < 0 || L > (1 << 24) || kmax < 0) return 1;
#pragma omp parallel
    {
        int32_t perm[4096];
#pragma omp for schedule(static)
        for (int64_t e = 0; e < n; ++e) {
            pcg32_t r;
            stream_for(&r, seed, tensor_id, (uint64_t)e);
            int64_t k = (int64_t)uniform_below(&r, (uint32_t)kmax + 1u);
            if (k > L) k = L;
            uint8_t *m = mask + e * L;
            for (int64_t t = 0; t < L; ++t) m[t] = 1;
            if (L <= 4096) {
                for (int64_t t = 0; t < L; ++t) perm[t] = (int32_t)t;
                for (int64_t a = 0; a < k; ++a) {
                    int64_t b = a + (int64_t)uniform_below(&r, (uint32_t)(L - a));
                    int32_t tmp = perm[a];
                    perm[a] = perm[b];
                    perm[b] = tmp;
                    m[perm[a]] = 0;
                }
            } else {
                /* long items: rejection sampling of distinct positions */
                int64_t hidden = 0;
                while (hidden < k) {
                    int64_t t = (int64_t)uniform_below(&r, (uint32_t)L);
                    if (m[t]) { m[t] = 0; ++hidden; }
                }
            }
        }
    }
    return 0;
}

int dg_version(void) { return 1; }
