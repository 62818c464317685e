/*
 * Seeded synthetic inputs shared by the CUDA path and the CPU oracle.
 *
 * This file holds only input generation: counter-based random words
 * (SplitMix64 finaliser applied to a Weyl sequence, Steele, Lea & Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014), uniform
 * doubles, Box-Muller normals and round-to-nearest-even conversion of the
 * generated values to bfloat16 storage.  None of the model arithmetic of the
 * verify pass lives here.
 *
 * Every value is a pure function of (seed, stream, index), so any slice of a
 * tensor can be regenerated independently and in parallel, and the result
 * does not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SV_GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t sv_fmix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Key of one (seed, stream) pair: two finaliser rounds keep nearby seeds and
 * nearby stream ids far apart. */
uint64_t sv_key(uint64_t seed, uint64_t stream) {
    return sv_fmix(sv_fmix(seed + SV_GOLDEN) ^ (stream * 0xD1B54A32D192ED03ULL));
}

/* Word i of a stream: the finaliser of the (i+1)-th Weyl step. */
uint64_t sv_word(uint64_t key, uint64_t i) { return sv_fmix(key + (i + 1) * SV_GOLDEN); }

/* Uniform double in the open interval (0, 1) from the top 53 bits. */
static inline double sv_unit(uint64_t w) { return ((double)(w >> 11) + 0.5) * (1.0 / 9007199254740992.0); }

double sv_uniform(uint64_t seed, uint64_t stream, uint64_t i) { return sv_unit(sv_word(sv_key(seed, stream), i)); }

/* float -> bfloat16 bits, round to nearest even (inputs here are finite). */
static inline uint16_t sv_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* out[i] = bf16(float(std * N_i)), N_i standard normal.  Normals come in
 * Box-Muller pairs: pair j uses words 2j and 2j+1 of the stream; element 2j
 * takes the cosine branch and 2j+1 the sine branch.  `first` is the index of
 * out[0] within the stream, so a tensor can be generated in pieces. */
void sv_normal_bf16(uint16_t* out, int64_t count, uint64_t seed, uint64_t stream, int64_t first, double stdev) {
    const uint64_t key = sv_key(seed, stream);
    const double two_pi = 6.283185307179586476925286766559;
    const int64_t p0 = first >> 1, p1 = (first + count + 1) >> 1;
#pragma omp parallel for schedule(static)
    for (int64_t pair = p0; pair < p1; ++pair) {
        const double u1 = sv_unit(sv_word(key, (uint64_t)(2 * pair)));
        const double u2 = sv_unit(sv_word(key, (uint64_t)(2 * pair + 1)));
        const double r = sqrt(-2.0 * log(u1));
        const int64_t i0 = 2 * pair - first, i1 = i0 + 1;
        if (i0 >= 0 && i0 < count) out[i0] = sv_bf16((float)(stdev * (r * cos(two_pi * u2))));
        if (i1 >= 0 && i1 < count) out[i1] = sv_bf16((float)(stdev * (r * sin(two_pi * u2))));
    }
}

/* Same normals as float32 (used for synthetic KV in fp32 form if needed). */
void sv_normal_f32(float* out, int64_t count, uint64_t seed, uint64_t stream, int64_t first, double stdev) {
    const uint64_t key = sv_key(seed, stream);
    const double two_pi = 6.283185307179586476925286766559;
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < count; ++k) {
        const int64_t idx = first + k;
        const int64_t pair = idx >> 1;
        const double u1 = sv_unit(sv_word(key, (uint64_t)(2 * pair)));
        const double u2 = sv_unit(sv_word(key, (uint64_t)(2 * pair + 1)));
        const double r = sqrt(-2.0 * log(u1));
        const double z = (idx & 1) ? r * sin(two_pi * u2) : r * cos(two_pi * u2);
        out[k] = (float)(stdev * z);
    }
}

/* Fill with one constant stored as bf16 (RMSNorm gains are 1). */
void sv_const_bf16(uint16_t* out, int64_t count, float value) {
    const uint16_t b = sv_bf16(value);
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < count; ++k) out[k] = b;
}

/* Uniform integers in [lo, hi): floor(u * (hi - lo)) + lo, word i -> out[i]. */
void sv_uniform_int(int32_t* out, int64_t count, uint64_t seed, uint64_t stream, int32_t lo, int32_t hi) {
    const uint64_t key = sv_key(seed, stream);
    const double span = (double)hi - (double)lo;
    for (int64_t k = 0; k < count; ++k) {
        int64_t v = (int64_t)floor(sv_unit(sv_word(key, (uint64_t)k)) * span) + lo;
        if (v >= hi) v = hi - 1;
        out[k] = (int32_t)v;
    }
}

/* Uniform doubles in (0,1), word i -> out[i]. */
void sv_uniform_f64(double* out, int64_t count, uint64_t seed, uint64_t stream) {
    const uint64_t key = sv_key(seed, stream);
    for (int64_t k = 0; k < count; ++k) out[k] = sv_unit(sv_word(key, (uint64_t)k));
}
