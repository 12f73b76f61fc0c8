/*
 * synth.c — seeded synthetic inputs shared by the tests, the benchmark and
 * the oracle checks.  It holds none of the quantized-matmul arithmetic: only
 * a counter-based uniform generator (splitmix64, Steele/Lea/Flood 2014:
 * state += 0x9E3779B97F4A7C15, then the two xor-shift-multiply rounds and a
 * final xor-shift) turned into normal deviates by the Box-Muller transform
 * (Box & Muller 1958), computed in fp64 and rounded to fp32.
 *
 * Element i of a stream with seed s uses the splitmix64 outputs at counters
 * 2i and 2i+1, so any element can be regenerated on its own and the result
 * does not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>

static uint64_t splitmix64_at(uint64_t seed, uint64_t i) {
  uint64_t z = seed + (i + 1u) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t synth_splitmix64(uint64_t seed, uint64_t i) { return splitmix64_at(seed, i); }

/* out[i] = mean + sigma * N(0,1) deviate number (offset + i) of stream seed. */
void synth_normal_f32(uint64_t seed, int64_t offset, int64_t n, double mean, double sigma,
                      float* out) {
  const double two_pi = 6.283185307179586476925286766559;
  int64_t i;
#pragma omp parallel for schedule(static)
  for (i = 0; i < n; ++i) {
    uint64_t c = (uint64_t)(offset + i);
    uint64_t a = splitmix64_at(seed, 2u * c);
    uint64_t b = splitmix64_at(seed, 2u * c + 1u);
    double u1 = (double)((a >> 11) + 1u) * 0x1.0p-53; /* (0, 1] */
    double u2 = (double)(b >> 11) * 0x1.0p-53;        /* [0, 1) */
    double r = sqrt(-2.0 * log(u1));
    out[i] = (float)(mean + sigma * r * cos(two_pi * u2));
  }
}

/* out[i] = uniform double in [0,1) number (offset + i) of stream seed. */
void synth_uniform_f64(uint64_t seed, int64_t offset, int64_t n, double* out) {
  int64_t i;
#pragma omp parallel for schedule(static)
  for (i = 0; i < n; ++i)
    out[i] = (double)(splitmix64_at(seed, (uint64_t)(offset + i)) >> 11) * 0x1.0p-53;
}
