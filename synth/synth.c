/*
 * synth.c -- seeded synthetic inputs, shared by the tests, the bench and the
 * oracle driver.  It holds none of the attention arithmetic: it only turns a
 * (seed, stream, element index) triple into a normally distributed value and
 * rounds that value to bf16.
 *
 * Generator (counter-based, so every element is independent of thread count):
 *   SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
 *   generators", OOPSLA 2014): from a state x, the n-th output (n >= 1) is
 *   mix(x + n * 0x9E3779B97F4A7C15) with
 *     mix(z): z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9;
 *             z = (z ^ (z >> 27)) * 0x94D049BB133111EB;
 *             return z ^ (z >> 31);
 *   The state of stream s under seed S is x = mix(S * 0x9E3779B97F4A7C15 + s + 1).
 *   Uniform: u = ((z >> 11) + 0.5) * 2^-53, in the open interval (0, 1).
 *   Normal (Box & Muller 1958): element 2p and 2p+1 take u1 = uniform of
 *   output 2p+1 and u2 = uniform of output 2p+2; r = sqrt(-2 ln u1),
 *   t = 2 pi u2; element 2p = r cos t, element 2p+1 = r sin t.
 *   Value = mean + sigma * normal, rounded to binary32 (C cast, round to
 *   nearest even), then to bf16 by round-to-nearest-even on the 16 low bits.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SM64_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t synth_stream_state(uint64_t seed, uint64_t stream) {
  return sm64_mix(seed * SM64_GAMMA + stream + 1ULL);
}

/* n-th output (n >= 1) of SplitMix64 started at state x. */
uint64_t synth_splitmix64_at(uint64_t x, uint64_t n) { return sm64_mix(x + n * SM64_GAMMA); }

static inline double unit_open(uint64_t z) {
  return ((double)(z >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t w;
  memcpy(&w, &f, sizeof w);
  if ((w & 0x7F800000u) == 0x7F800000u) /* inf / nan: keep class */
    return (uint16_t)((w >> 16) | ((w & 0xFFFFu) ? 0x40u : 0u));
  uint32_t lsb = (w >> 16) & 1u;
  w += 0x7FFFu + lsb;
  return (uint16_t)(w >> 16);
}

static const double TWO_PI = 6.283185307179586476925286766559;

/* Fill out[0..count) with bf16 bits of mean + sigma * N(0,1), element index
 * offset by first (so that a slice of a big tensor can be made alone). */
void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t first, uint64_t count,
                       double mean, double sigma, uint16_t* out) {
  const uint64_t x = synth_stream_state(seed, stream);
  long long n = (long long)count;
#pragma omp parallel for schedule(static)
  for (long long t = 0; t < n; ++t) {
    uint64_t e = first + (uint64_t)t;
    uint64_t p = e >> 1;
    double u1 = unit_open(sm64_mix(x + (2 * p + 1) * SM64_GAMMA));
    double u2 = unit_open(sm64_mix(x + (2 * p + 2) * SM64_GAMMA));
    double r = sqrt(-2.0 * log(u1));
    double z = (e & 1) ? r * sin(TWO_PI * u2) : r * cos(TWO_PI * u2);
    out[t] = f32_to_bf16_rne((float)(mean + sigma * z));
  }
}

/* Same values as binary32 (the bf16 bits widened), for callers that want them. */
void synth_bf16_to_f32(const uint16_t* in, uint64_t count, float* out) {
  long long n = (long long)count;
#pragma omp parallel for schedule(static)
  for (long long t = 0; t < n; ++t) {
    uint32_t w = ((uint32_t)in[t]) << 16;
    memcpy(&out[t], &w, sizeof w);
  }
}
