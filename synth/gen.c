/*
 * Fast host generator for the seeded synthetic inputs.  Same definition as
 * the numpy version in synth/__init__.py (which the tests compare it with):
 * counter-based SplitMix64, x_i = mix(seed + (i + 1) * 0x9E3779B97F4A7C15),
 * with Vigna's splitmix64.c finaliser.  Holds no merge arithmetic.
 */
#include <stdint.h>

static inline uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* out[t] = top 32 bits of draw (start + t), t in [0, count). */
void synth_top32(uint64_t seed, int64_t start, int64_t count, uint32_t *out)
{
    for (int64_t t = 0; t < count; ++t) {
        uint64_t x = mix64(seed + (uint64_t)(start + t + 1) * 0x9E3779B97F4A7C15ULL);
        out[t] = (uint32_t)(x >> 32);
    }
}

/* out[t] = ((top 32 bits) * bound) >> 32, i.e. uniform in [0, bound). */
void synth_below(uint64_t seed, int64_t start, int64_t count, uint64_t bound,
                 uint32_t *out)
{
    for (int64_t t = 0; t < count; ++t) {
        uint64_t x = mix64(seed + (uint64_t)(start + t + 1) * 0x9E3779B97F4A7C15ULL);
        out[t] = (uint32_t)(((x >> 32) * bound) >> 32);
    }
}
