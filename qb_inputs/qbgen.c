/*
 * Seeded synthetic inputs shared by the CPU oracle, the tests and the bench.
 *
 * This file holds no arithmetic of the method under test: it only draws
 * seeded pseudo-random tensors and packs them into the storage formats the
 * method consumes (fp32, bf16, MXFP4).  Both sides of every parity test take
 * their inputs from here.
 *
 * Generator.  Element i of tensor (seed, id) is derived from one SplitMix64
 * output (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014: the increment 0x9E3779B97F4A7C15 and the
 * variant-13 finaliser of Stafford's Mix13), written here from that
 * published definition:
 *     key  = splitmix64(seed ^ splitmix64(id))
 *     h    = splitmix64(key + i)
 * The 64-bit word h is split into four 16-bit fields a0..a3; each field
 * maps to the odd integer 2a+1-65536 (uniform and symmetric on
 * [-65535, 65535]) and the four are summed, an Irwin-Hall(4) draw with
 * mean 0 and variance 4*65536^2/3 (to within 1e-9 relative).  The value is
 *     v = fp32( fp32(S) * c ),   c = fp32(sigma * sqrt(3) / 131072),
 * so v has mean 0 and standard deviation sigma, with tails cut at
 * +-2*sqrt(3)*sigma (= 3.46 sigma).  S is an integer below 2^19, so fp32(S)
 * is exact and v is one IEEE multiply: identical on every machine.
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

static inline uint64_t splitmix64(uint64_t z) {
    z += 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline uint64_t tensor_key(uint64_t seed, uint64_t id) {
    return splitmix64(seed ^ splitmix64(id));
}

static inline float draw(uint64_t key, uint64_t i, float c) {
    uint64_t h = splitmix64(key + i);
    int32_t s = 0;
    for (int f = 0; f < 4; ++f) {
        int32_t a = (int32_t)((h >> (16 * f)) & 0xFFFFu);
        s += 2 * a + 1 - 65536;
    }
    return (float)s * c;   /* (float)s is exact: |s| < 2^19 */
}

static inline float scale_of(float sigma) {
    return (float)((double)sigma * sqrt(3.0) / 131072.0);
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
    const uint64_t key = tensor_key(seed, id);
    const float c = scale_of(sigma);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < count; ++j) out[j] = draw(key, (uint64_t)(offset + j), c);
}

void qbgen_normal_bf16(uint64_t seed, uint64_t id, int64_t offset, int64_t count,
                       float sigma, uint16_t* out) {
    const uint64_t key = tensor_key(seed, id);
    const float c = scale_of(sigma);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < count; ++j)
        out[j] = f32_to_bf16_rne(draw(key, (uint64_t)(offset + j), c));
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
