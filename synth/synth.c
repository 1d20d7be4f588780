/*
 * Seeded synthetic input generator shared by the oracle side and the GPU side.
 *
 * It holds none of the MoE layer's arithmetic: it only turns (seed, stream,
 * element index) into numbers.  Every value is a pure function of its index
 * (counter-based), so any slice of a tensor can be produced on its own and
 * large tensors are generated in parallel with identical bits.
 *
 * Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014; the finaliser constants are Vigna's
 * published mix13 variant).  Output number n (n = 1, 2, ...) of a SplitMix64
 * stream whose state starts at s is mix64(s + n * 0x9E3779B97F4A7C15).
 *
 * Normals: Box-Muller (Box and Muller, 1958), cosine branch only, in double:
 *   u1 = ((b1 >> 11) + 1) * 2^-53  in (0, 1]
 *   u2 =  (b2 >> 11)      * 2^-53  in [0, 1)
 *   z  = sqrt(-2 ln u1) * cos(2 pi u2)
 * with b1, b2 the stream outputs 2i+1 and 2i+2 for element i.
 *
 * bf16 values: mean + std * z is rounded to float32 (round to nearest even,
 * by the C conversion), then float32 -> bf16 by round to nearest even on the
 * bit pattern.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

uint64_t synth_mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* State that starts the SplitMix64 stream `stream` of seed `seed`. */
uint64_t synth_stream_key(uint64_t seed, uint64_t stream) {
    return synth_mix64(seed * 0xD1B54A32D192ED03ULL + synth_mix64(stream + 0x632BE59BD9B4E019ULL));
}

/* Output number n (n >= 1) of the stream that starts at state `key`. */
static inline uint64_t nth(uint64_t key, uint64_t n) { return synth_mix64(key + n * GOLDEN); }

uint16_t synth_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0x7FC0; /* NaN */
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static inline double box_muller(uint64_t key, uint64_t i) {
    const double two53 = 1.0 / 9007199254740992.0; /* 2^-53 */
    uint64_t b1 = nth(key, 2 * i + 1), b2 = nth(key, 2 * i + 2);
    double u1 = ((double)(b1 >> 11) + 1.0) * two53;
    double u2 = (double)(b2 >> 11) * two53;
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

/* out[i] = bf16(mean + std * N_{start+i}) for i in [0, n). */
void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t start, uint64_t n,
                       double mean, double std, uint16_t* out) {
    uint64_t key = synth_stream_key(seed, stream);
    int64_t nn = (int64_t)n;
#pragma omp parallel for schedule(static, 1 << 16)
    for (int64_t i = 0; i < nn; ++i) {
        double v = mean + std * box_muller(key, start + (uint64_t)i);
        out[i] = synth_f32_to_bf16((float)v);
    }
}

/* out[i] = mean + std * N_{start+i} in double (no rounding). */
void synth_normal_f64(uint64_t seed, uint64_t stream, uint64_t start, uint64_t n,
                      double mean, double std, double* out) {
    uint64_t key = synth_stream_key(seed, stream);
    int64_t nn = (int64_t)n;
#pragma omp parallel for schedule(static, 1 << 16)
    for (int64_t i = 0; i < nn; ++i) out[i] = mean + std * box_muller(key, start + (uint64_t)i);
}

/* out[i] = raw 64-bit output number start+i+1 of the stream. */
void synth_u64(uint64_t seed, uint64_t stream, uint64_t start, uint64_t n, uint64_t* out) {
    uint64_t key = synth_stream_key(seed, stream);
    for (uint64_t i = 0; i < n; ++i) out[i] = nth(key, start + i + 1);
}

/* Raw SplitMix64 from an explicit initial state (for checking the definition). */
void synth_splitmix64_raw(uint64_t state, uint64_t n, uint64_t* out) {
    for (uint64_t i = 0; i < n; ++i) out[i] = nth(state, i + 1);
}
