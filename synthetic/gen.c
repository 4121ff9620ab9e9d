/*
 * Seeded synthetic inputs for the layerwise weight-streaming DiT forward.
 *
 * This file holds no arithmetic of the method itself. It only draws the
 * random numbers that stand in for checkpoint weights, latent tokens and
 * conditioning vectors, so that the CPU oracle and the CUDA path can be fed
 * the very same bits.
 *
 * Generator (counter-based, so any element can be drawn independently and
 * the fill parallelises):
 *   splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
 *   generators", OOPSLA 2014): the k-th output of a stream started at state
 *   s is mix(s + (k+1) * 0x9E3779B97F4A7C15).
 *   Each tensor gets its own stream state  s = mix(seed ^ mix(tensor_id + GAMMA)).
 *   Standard normals come in pairs by the Box-Muller transform (Box & Muller,
 *   1958): with u1 = (hi53(x_{2j}) + 0.5) / 2^53 in (0,1) and
 *   u2 = hi53(x_{2j+1}) / 2^53, element 2j = r cos(2 pi u2) and element
 *   2j+1 = r sin(2 pi u2), r = sqrt(-2 ln u1), all in double.
 *   A value drawn as N(0, std) is  (float)(std * z)  (round to nearest even).
 *   A bf16 weight is that float rounded to bf16 with round-to-nearest-even.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SYN_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t syn_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t syn_state(uint64_t seed, uint64_t tensor_id) {
    return syn_mix(seed ^ syn_mix(tensor_id + SYN_GAMMA));
}

/* k-th raw 64-bit output of the stream that starts at state s. */
static inline uint64_t syn_raw(uint64_t s, uint64_t k) {
    return syn_mix(s + (k + 1) * SYN_GAMMA);
}

static inline void syn_normal_pair(uint64_t s, uint64_t j, double* z0, double* z1) {
    const double two53 = 9007199254740992.0;
    double u1 = ((double)(syn_raw(s, 2 * j) >> 11) + 0.5) / two53;
    double u2 = (double)(syn_raw(s, 2 * j + 1) >> 11) / two53;
    double r = sqrt(-2.0 * log(u1));
    double t = 6.283185307179586476925286766559 * u2;
    *z0 = r * cos(t);
    *z1 = r * sin(t);
}

static inline uint16_t syn_f32_to_bf16_rne(float f) {
    uint32_t b;
    memcpy(&b, &f, 4);
    uint32_t bias = 0x7FFFu + ((b >> 16) & 1u);
    return (uint16_t)((b + bias) >> 16);
}

/* The raw splitmix64 outputs 0..n-1 of the stream for (seed, tensor_id). */
void syn_raw_u64(uint64_t seed, uint64_t tensor_id, int64_t n, uint64_t* out) {
    uint64_t s = syn_state(seed, tensor_id);
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < n; ++k) out[k] = syn_raw(s, (uint64_t)k);
}

/* n values ~ N(0, std) as float. */
void syn_normal_f32(uint64_t seed, uint64_t tensor_id, int64_t n, double std, float* out) {
    uint64_t s = syn_state(seed, tensor_id);
    int64_t pairs = (n + 1) / 2;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < pairs; ++j) {
        double z0, z1;
        syn_normal_pair(s, (uint64_t)j, &z0, &z1);
        out[2 * j] = (float)(std * z0);
        if (2 * j + 1 < n) out[2 * j + 1] = (float)(std * z1);
    }
}

/* n values ~ N(0, std), each rounded float -> bf16 (RNE); raw bf16 bits. */
void syn_normal_bf16(uint64_t seed, uint64_t tensor_id, int64_t n, double std, uint16_t* out) {
    uint64_t s = syn_state(seed, tensor_id);
    int64_t pairs = (n + 1) / 2;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < pairs; ++j) {
        double z0, z1;
        syn_normal_pair(s, (uint64_t)j, &z0, &z1);
        out[2 * j] = syn_f32_to_bf16_rne((float)(std * z0));
        if (2 * j + 1 < n) out[2 * j + 1] = syn_f32_to_bf16_rne((float)(std * z1));
    }
}

int syn_max_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
