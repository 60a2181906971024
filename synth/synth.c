/*
 * Seeded synthetic inputs: SplitMix64 in counter form (Steele, Lea, Flood,
 * OOPSLA 2014), z_i = mix(seed + i * 0x9E3779B97F4A7C15) for counters i >= 1,
 * turned into float32 draws or int16 values.  Rounding to bf16 happens in the
 * Python module.  Holds none of the GEMM or copy arithmetic.
 */
#include <math.h>
#include <stdint.h>

static inline uint64_t mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline uint64_t draw(uint64_t seed, int64_t counter) {
    return mix(seed + (uint64_t)counter * 0x9E3779B97F4A7C15ull);
}

void synth_splitmix64(uint64_t seed, int64_t offset, int64_t n, uint64_t *out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = draw(seed, offset + i + 1);
}

/* u = ((z >> 40) - 2^23) / 2^23, exact in float32 */
void synth_uniform_pm1_f32(uint64_t seed, int64_t n, float *out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        int64_t v = (int64_t)(draw(seed, i + 1) >> 40) - (1ll << 23);
        out[i] = (float)v * 0x1p-23f;
    }
}

/* Box-Muller, cosine branch, on counters 2i+1 and 2i+2; result scaled, then rounded to float32 */
void synth_normal_f32(uint64_t seed, int64_t n, double scale, float *out) {
    const double two_pi = 6.283185307179586476925286766559;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double u1 = ((double)(draw(seed, 2 * i + 1) >> 11) + 1.0) * 0x1p-53;
        double u2 = (double)(draw(seed, 2 * i + 2) >> 11) * 0x1p-53;
        out[i] = (float)(sqrt(-2.0 * log(u1)) * cos(two_pi * u2) * scale);
    }
}

/* lo + (z mod (hi - lo + 1)) */
void synth_int_uniform_f32(uint64_t seed, int64_t n, int32_t lo, int32_t hi, float *out) {
    const uint64_t span = (uint64_t)((int64_t)hi - lo + 1);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (float)((int64_t)(draw(seed, i + 1) % span) + lo);
}

/* low 16 bits of z */
void synth_int16(uint64_t seed, int64_t n, int16_t *out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (int16_t)(uint16_t)(draw(seed, i + 1) & 0xFFFFu);
}
