/*
 * Seeded synthetic-input generator shared by the tests, the bench and the
 * oracle harness.  It holds no arithmetic of the DiT itself: it only turns a
 * (seed, tensor name) pair into reproducible numbers.
 *
 * The scheme follows the shared-PRNG idea described on the page
 * "feat(minimax-h3): port the MiniMax-H3 omni-modal video+audio DiT",
 * section "How this is gated (no weight bytes checked in)": both sides rebuild
 * weights from an FNV-1a-keyed splitmix64 stream, so no weight bytes are
 * stored.  Here the stream is counter based (value i is a pure function of the
 * key and i) so that generation can be split across threads.
 *
 *   key    = FNV-1a 64 of the string "seed=<k>/<name>"
 *   z(c)   = splitmix64 finaliser of (key + c * 0x9E3779B97F4A7C15), c = 1, 2, ...
 *   u1     = ((z(2j+1) >> 11) + 1) * 2^-53          in (0, 1]
 *   u2     =  (z(2j+2) >> 11)      * 2^-53          in [0, 1)
 *   n0, n1 = sqrt(-2 ln u1) * (cos, sin)(2 pi u2)   (Box-Muller, double)
 *   value  = (float)(n * std), optionally rounded to bf16 (round to nearest even)
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static const uint64_t kGolden = 0x9E3779B97F4A7C15ull;

uint64_t synth_fnv1a64(const char* s) {
  uint64_t h = 0xcbf29ce484222325ull;
  for (const unsigned char* p = (const unsigned char*)s; *p; ++p) {
    h ^= (uint64_t)(*p);
    h *= 0x100000001b3ull;
  }
  return h;
}

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static inline uint64_t draw(uint64_t key, uint64_t c) { return mix64(key + c * kGolden); }

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u) return (uint16_t)(u >> 16); /* inf / nan: keep */
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

static inline float bf16_to_f32(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* n values of N(0, std^2).  out_f32 gets the fp32 values (bf16-rounded if
 * out_bf16 != NULL, so both arrays then hold the same numbers). */
void synth_normal(uint64_t key, uint64_t n, double stddev, float* out_f32, uint16_t* out_bf16) {
  const double two_pi = 6.283185307179586476925286766559;
  const double inv53 = 1.0 / 9007199254740992.0;
  int64_t npairs = (int64_t)((n + 1) / 2);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < npairs; ++j) {
    uint64_t a = draw(key, 2 * (uint64_t)j + 1);
    uint64_t b = draw(key, 2 * (uint64_t)j + 2);
    double u1 = (double)((a >> 11) + 1) * inv53;
    double u2 = (double)(b >> 11) * inv53;
    double r = sqrt(-2.0 * log(u1));
    double v[2] = {r * cos(two_pi * u2), r * sin(two_pi * u2)};
    for (int q = 0; q < 2; ++q) {
      uint64_t i = 2 * (uint64_t)j + (uint64_t)q;
      if (i >= n) break;
      float f = (float)(v[q] * stddev);
      if (out_bf16) {
        uint16_t bb = f32_to_bf16_rne(f);
        out_bf16[i] = bb;
        f = bf16_to_f32(bb);
      }
      if (out_f32) out_f32[i] = f;
    }
  }
}

/* n values uniform in [lo, hi), as double. */
void synth_uniform(uint64_t key, uint64_t n, double lo, double hi, double* out) {
  const double inv53 = 1.0 / 9007199254740992.0;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) {
    double u = (double)(draw(key, (uint64_t)i + 1) >> 11) * inv53;
    out[i] = lo + (hi - lo) * u;
  }
}
