/*
 * Seeded synthetic inputs shared by the CPU oracle, the tests and the bench.
 *
 * This file holds no arithmetic of the method under test: it only draws
 * seeded pseudo-random tensors and packs them into the storage formats the
 * method consumes (fp32, bf16, MXFP4).  Both sides of every parity test take
 * their inputs from here.
 *
 * Generator.  Element i of tensor (seed, id) is derived from two SplitMix64
 * outputs (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014: the increment 0x9E3779B97F4A7C15 and the
 * variant-13 finaliser of Stafford's Mix13), written here from that
 * published definition:
 *     key  = splitmix64(seed ^ splitmix64(id))
 *     h1   = splitmix64(key + 2p),   h2 = splitmix64(key + 2p + 1),
 * where p = floor(i / 2) is the element's pair.  Their top 53 bits give two
 * uniforms, u1 = ((h1 >> 11) + 1) * 2^-53 in (0, 1] and u2 = (h2 >> 11) *
 * 2^-53 in [0, 1), and the Box-Muller transform (Box and Muller, "A note on
 * the generation of random normal deviates", Ann. Math. Stat. 1958) gives
 * two independent standard normal draws
 *     z = sqrt(-2 ln u1) * cos(2 pi u2)  (element 2p),
 *     z = sqrt(-2 ln u1) * sin(2 pi u2)  (element 2p + 1),
 * so v = fp32(z * sigma) is N(0, sigma^2) with untruncated tails (|z| <=
 * 8.6 at u1 = 2^-53).  ln and cos are computed here in double precision with
 * a fixed sequence of IEEE operations (no libm transcendental, built with
 * -ffp-contract=off; sqrt is IEEE-exact), so every machine draws the same
 * bits:
 *   ln u = e ln2 + 2 atanh(f),  u = m 2^e with m in [sqrt(1/2), sqrt(2)),
 *          f = (m - 1)/(m + 1), atanh by its odd series to f^25
 *          (|f| <= 0.1716: remainder below 1e-21);
 *   cos and sin of 2 pi t by the half-, quarter- and eighth-turn symmetries
 *          down to an angle x in [0, pi/4], then the Taylor series of cos x
 *          (to x^18) and sin x (to x^19), remainder below 1e-19.
 *
 * bf16 storage rounds v to nearest-even on its fp32 bits.
 *
 * MXFP4 (OCP Microscaling spec v1.0): E2M1 elements, one E8M0 scale per 32
 * consecutive elements along K.  The quantiser takes the block amax, sets
 * the shared exponent e = floor(log2(amax)) - 2 (the spec's suggested
 * scale: E2M1's largest normal exponent is 2), and rounds v / 2^e to the
 * nearest E2M1 value with ties to the even code, saturating at +-6.
 * Packed layout: byte k/2 of a row holds element k in its low nibble when
 * k is even and in its high nibble when k is odd.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>
#include <stdlib.h>

static inline uint64_t splitmix64(uint64_t z) {
    z += 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline uint64_t tensor_key(uint64_t seed, uint64_t id) {
    return splitmix64(seed ^ splitmix64(id));
}

/* ln u for u in (0, 1] (see the header: fixed operation order).  u is a
 * normal double (u >= 2^-53), so its exponent and mantissa come from its bits:
 * u = m 2^e, m in [1, 2), then m is halved when above sqrt(2). */
static inline double ln_fixed(double u) {
    uint64_t b;
    memcpy(&b, &u, 8);
    int e = (int)((b >> 52) & 0x7FF) - 1023;
    b = (b & 0x000FFFFFFFFFFFFFull) | 0x3FF0000000000000ull;
    double m;
    memcpy(&m, &b, 8);                           /* [1, 2) */
    if (m > 1.41421356237309504880) {
        m *= 0.5;                                /* exact */
        e += 1;
    }
    const double f = (m - 1.0) / (m + 1.0);
    const double f2 = f * f;
    /* atanh(f) / f = sum f^(2q) / (2q + 1), q = 0..12, in Horner form */
    double p = 1.0 / 25.0;
    p = p * f2 + 1.0 / 23.0;
    p = p * f2 + 1.0 / 21.0;
    p = p * f2 + 1.0 / 19.0;
    p = p * f2 + 1.0 / 17.0;
    p = p * f2 + 1.0 / 15.0;
    p = p * f2 + 1.0 / 13.0;
    p = p * f2 + 1.0 / 11.0;
    p = p * f2 + 1.0 / 9.0;
    p = p * f2 + 1.0 / 7.0;
    p = p * f2 + 1.0 / 5.0;
    p = p * f2 + 1.0 / 3.0;
    p = p * f2 + 1.0;
    const double ln_m = 2.0 * f * p;
    /* ln 2 split so that e * LN2_HI is exact for |e| < 2^11 */
    const double LN2_HI = 6.93147180369123816490e-01, LN2_LO = 1.90821492927058770002e-10;
    return ((double)e * LN2_HI + (double)e * LN2_LO) + ln_m;
}

/* cos x and sin x for x in [0, pi/4]: Taylor series to x^18 and x^19 in
 * Horner form (coefficients 1/((2q-1) 2q) and 1/(2q (2q+1)) folded at
 * compile time). */
static inline void cos_sin_series(double x, double* c, double* s) {
    const double x2 = x * x;
    double pc = 1.0 - x2 * (1.0 / (17.0 * 18.0));
    pc = 1.0 - x2 * (1.0 / (15.0 * 16.0)) * pc;
    pc = 1.0 - x2 * (1.0 / (13.0 * 14.0)) * pc;
    pc = 1.0 - x2 * (1.0 / (11.0 * 12.0)) * pc;
    pc = 1.0 - x2 * (1.0 / (9.0 * 10.0)) * pc;
    pc = 1.0 - x2 * (1.0 / (7.0 * 8.0)) * pc;
    pc = 1.0 - x2 * (1.0 / (5.0 * 6.0)) * pc;
    pc = 1.0 - x2 * (1.0 / (3.0 * 4.0)) * pc;
    pc = 1.0 - x2 * (1.0 / (1.0 * 2.0)) * pc;
    double ps = 1.0 - x2 * (1.0 / (18.0 * 19.0));
    ps = 1.0 - x2 * (1.0 / (16.0 * 17.0)) * ps;
    ps = 1.0 - x2 * (1.0 / (14.0 * 15.0)) * ps;
    ps = 1.0 - x2 * (1.0 / (12.0 * 13.0)) * ps;
    ps = 1.0 - x2 * (1.0 / (10.0 * 11.0)) * ps;
    ps = 1.0 - x2 * (1.0 / (8.0 * 9.0)) * ps;
    ps = 1.0 - x2 * (1.0 / (6.0 * 7.0)) * ps;
    ps = 1.0 - x2 * (1.0 / (4.0 * 5.0)) * ps;
    ps = 1.0 - x2 * (1.0 / (2.0 * 3.0)) * ps;
    *c = pc;
    *s = x * ps;
}

/* (cos 2 pi t, sin 2 pi t) for t in [0, 1): the octant symmetries reduce the
 * angle to [0, pi/4]; every reduction step is exact (t has 53 bits). */
static inline void cos_sin_turns(double t, double* c, double* s) {
    const double TWO_PI = 6.28318530717958647692;
    double sgn_s = 1.0;
    if (t >= 0.5) {                              /* angle - pi: both change sign... */
        t = 1.0 - t;                             /* ...or mirror: cos even, sin odd */
        sgn_s = -1.0;
    }
    double sgn_c = 1.0;
    if (t > 0.25) {                              /* pi - angle */
        t = 0.5 - t;
        sgn_c = -1.0;
    }
    double cc, ss;
    if (t > 0.125) {                             /* pi/2 - angle: cos <-> sin */
        cos_sin_series(TWO_PI * (0.25 - t), &ss, &cc);
    } else {
        cos_sin_series(TWO_PI * t, &cc, &ss);
    }
    *c = sgn_c * cc;
    *s = sgn_s * ss;
}

/* Box-Muller pair p of stream `key`: two independent standard normals. */
static inline void normal_pair(uint64_t key, uint64_t p, double* z0, double* z1) {
    const uint64_t h1 = splitmix64(key + 2u * p);
    const uint64_t h2 = splitmix64(key + 2u * p + 1u);
    const double u1 = (double)((h1 >> 11) + 1u) * 0x1.0p-53;
    const double u2 = (double)(h2 >> 11) * 0x1.0p-53;
    const double rad = sqrt(-2.0 * ln_fixed(u1));
    double c, s;
    cos_sin_turns(u2, &c, &s);
    *z0 = rad * c;
    *z1 = rad * s;
}

/* Elements [offset, offset + count) of stream `key` as fp32 values z * sigma:
 * element i is the cosine (i even) or sine (i odd) member of pair i / 2. */
static void draw_range(uint64_t key, int64_t offset, int64_t count, double sigma, float* out) {
#pragma omp parallel for schedule(static)
    for (int64_t q = (offset >> 1); q <= ((offset + count - 1) >> 1); ++q) {
        double z[2];
        normal_pair(key, (uint64_t)q, &z[0], &z[1]);
        for (int h = 0; h < 2; ++h) {
            const int64_t i = 2 * q + h;
            if (i >= offset && i < offset + count) out[i - offset] = (float)(z[h] * sigma);
        }
    }
}

static inline uint16_t f32_to_bf16_rne(float v) {
    uint32_t u;
    memcpy(&u, &v, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* out[j] = value of element (offset + j) of tensor (seed, id), j < count. */
void qbgen_normal_f32(uint64_t seed, uint64_t id, int64_t offset, int64_t count,
                      float sigma, float* out) {
    if (count <= 0) return;
    draw_range(tensor_key(seed, id), offset, count, (double)sigma, out);
}

void qbgen_normal_bf16(uint64_t seed, uint64_t id, int64_t offset, int64_t count,
                       float sigma, uint16_t* out) {
    if (count <= 0) return;
    /* fp32 values in chunks, then bf16 rounding of their bits */
    const int64_t CH = 1 << 20;
    float* buf = (float*)malloc((size_t)(count < CH ? count : CH) * sizeof(float));
    for (int64_t a = 0; a < count; a += CH) {
        const int64_t c = count - a < CH ? count - a : CH;
        draw_range(tensor_key(seed, id), offset + a, c, (double)sigma, buf);
#pragma omp parallel for schedule(static)
        for (int64_t j = 0; j < c; ++j) out[a + j] = f32_to_bf16_rne(buf[j]);
    }
    free(buf);
}

/* E2M1 magnitudes by code 0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
static int e2m1_code(float q) {
    float a = fabsf(q);
    int code;
    /* round to nearest; ties go to the even code */
    if (a <= 0.25f) code = 0;
    else if (a < 0.75f) code = 1;
    else if (a <= 1.25f) code = 2;
    else if (a < 1.75f) code = 3;
    else if (a <= 2.5f) code = 4;
    else if (a < 3.5f) code = 5;
    else if (a <= 5.0f) code = 6;
    else code = 7;
    if (q < 0.0f && code != 0) code |= 8;
    return code;
}

/*
 * Quantise rows x K bf16 values (given as uint16 bits) to MXFP4.
 * packed: [rows, K/2] bytes; scales: [rows, K/32] E8M0 bytes.  K % 32 == 0.
 */
void qbgen_quantize_mxfp4(const uint16_t* src, int64_t rows, int64_t K,
                          uint8_t* packed, uint8_t* scales) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* row = src + r * K;
        for (int64_t b0 = 0; b0 < K; b0 += 32) {
            float v[32];
            float amax = 0.0f;
            for (int t = 0; t < 32; ++t) {
                uint32_t u = (uint32_t)row[b0 + t] << 16;
                memcpy(&v[t], &u, 4);
                float a = fabsf(v[t]);
                if (a > amax) amax = a;
            }
            int e = 0;
            if (amax > 0.0f) {
                int ex;
                frexpf(amax, &ex);          /* amax = f * 2^ex, f in [0.5, 1) */
                e = (ex - 1) - 2;           /* floor(log2 amax) - 2 */
            }
            if (e < -127) e = -127;
            if (e > 127) e = 127;
            scales[r * (K / 32) + b0 / 32] = (uint8_t)(e + 127);
            const float inv = ldexpf(1.0f, -e);   /* exact power of two */
            for (int t = 0; t < 32; t += 2) {
                int lo = e2m1_code(v[t] * inv);
                int hi = e2m1_code(v[t + 1] * inv);
                packed[r * (K / 2) + (b0 + t) / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
}
