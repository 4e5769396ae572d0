/*
 * Seeded synthetic inputs for the S2-Pro Dual-AR frame decode.
 *
 * This module holds no arithmetic of the method itself: it only turns
 * (seed, stream, index) into numbers.  Both the CPU oracle and the CUDA path
 * are fed from it, so the two see the same bytes.
 *
 * Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014) used counter-style: the 64-bit output for
 * element i of stream s under seed k is mix(key(k, s) + (i+1)·γ), with
 * γ = 0x9E3779B97F4A7C15 and mix the SplitMix64 finaliser.  Every element is
 * a pure function of its index, so generation parallelises without changing
 * a single value.
 *
 *   uniform01(b)   = ((b >> 11) + 0.5) · 2^-53        in (0, 1), never 0 or 1
 *   normal(2j), normal(2j+1) = r·cos(t), r·sin(t) with r = sqrt(-2 ln u(2j)),
 *                  t = 2π u(2j+1)                       (Box–Muller, double)
 *   exponential(i) = -ln u(i)                          (inverse CDF, double)
 *   integer(i)     = lo + (b mod (hi - lo + 1))
 *
 * bf16 outputs are the fp32 value rounded to nearest-even on its top 16 bits; fp16 outputs are
 * the double rounded to nearest-even binary16 (subnormals kept, overflow to infinity).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define SM64_GAMMA 0x9E3779B97F4A7C15ull

static inline uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return sm64_mix(sm64_mix(seed + SM64_GAMMA) ^ (stream * 0xD1B54A32D192ED03ull + 0x632BE59BD9B4E019ull));
}

static inline uint64_t draw_bits(uint64_t key, uint64_t i) {
  return sm64_mix(key + (i + 1) * SM64_GAMMA);
}

static inline double u01(uint64_t b) {
  return ((double)(b >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u) return (uint16_t)(u >> 16);  /* inf/nan: never produced here */
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

/* Box–Muller pair j: (r cos t, r sin t) with r = sqrt(-2 ln u(2j)), t = 2π u(2j+1);
 * element 2j takes the cosine branch and element 2j+1 the sine branch. */
static inline void normal_pair(uint64_t key, uint64_t j, double* z0, double* z1) {
  double a = u01(draw_bits(key, 2 * j));
  double b = u01(draw_bits(key, 2 * j + 1));
  double r = sqrt(-2.0 * log(a)), t = 6.283185307179586476925286766559 * b;
  *z0 = r * cos(t);
  *z1 = r * sin(t);
}

/* n values of mean + std·N(0,1) as fp32. */
void synth_normal_f32(uint64_t seed, uint64_t stream, int64_t n, double mean, double std, float* out) {
  uint64_t key = stream_key(seed, stream);
  int64_t pairs = (n + 1) / 2;
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < pairs; ++j) {
    double z0, z1;
    normal_pair(key, (uint64_t)j, &z0, &z1);
    out[2 * j] = (float)(mean + std * z0);
    if (2 * j + 1 < n) out[2 * j + 1] = (float)(mean + std * z1);
  }
}

/* n values of mean + std·N(0,1), rounded fp64 -> fp32 -> bf16 (raw 16-bit patterns). */
void synth_normal_bf16(uint64_t seed, uint64_t stream, int64_t n, double mean, double std, uint16_t* out) {
  uint64_t key = stream_key(seed, stream);
  int64_t pairs = (n + 1) / 2;
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < pairs; ++j) {
    double z0, z1;
    normal_pair(key, (uint64_t)j, &z0, &z1);
    out[2 * j] = f32_to_bf16_rne((float)(mean + std * z0));
    if (2 * j + 1 < n) out[2 * j + 1] = f32_to_bf16_rne((float)(mean + std * z1));
  }
}

/* double -> IEEE binary16 bits, round to nearest even.  Scaling by a power of two is exact, so
 * rint() (default rounding mode: nearest even) does the only rounding. */
static inline uint16_t f64_to_f16_rne(double x) {
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  double a = fabs(x);
  if (a == 0.0) return sign;
  int e2;
  (void)frexp(a, &e2);               /* a = m * 2^e2, m in [0.5, 1) */
  int e = e2 - 1;                    /* a in [2^e, 2^(e+1)) */
  if (e < -14) {                     /* subnormal range: steps of 2^-24 */
    double q = rint(ldexp(a, 24));   /* q = 1024 lands on the smallest normal, bits 0x0400 */
    return (uint16_t)(sign | (uint16_t)q);
  }
  double q = rint(ldexp(a, 10 - e)); /* in [1024, 2048] */
  if (q >= 2048.0) {
    q = 1024.0;
    e += 1;
  }
  if (e > 15) return (uint16_t)(sign | 0x7c00u);
  return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(q - 1024.0));
}

/* n values of mean + std·N(0,1), rounded fp64 -> fp16 (raw 16-bit patterns). */
void synth_normal_f16(uint64_t seed, uint64_t stream, int64_t n, double mean, double std, uint16_t* out) {
  uint64_t key = stream_key(seed, stream);
  int64_t pairs = (n + 1) / 2;
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < pairs; ++j) {
    double z0, z1;
    normal_pair(key, (uint64_t)j, &z0, &z1);
    out[2 * j] = f64_to_f16_rne(mean + std * z0);
    if (2 * j + 1 < n) out[2 * j + 1] = f64_to_f16_rne(mean + std * z1);
  }
}

/* n standard exponential variates -ln(u), u uniform in (0,1), as fp32. */
void synth_exponential_f32(uint64_t seed, uint64_t stream, int64_t n, float* out) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = (float)(-log(u01(draw_bits(key, (uint64_t)i))));
}

/* n uniform doubles in (0,1). */
void synth_uniform_f64(uint64_t seed, uint64_t stream, int64_t n, double* out) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = u01(draw_bits(key, (uint64_t)i));
}

/* n integers uniform in [lo, hi] (inclusive). */
void synth_uniform_int(uint64_t seed, uint64_t stream, int64_t n, int32_t lo, int32_t hi, int32_t* out) {
  uint64_t key = stream_key(seed, stream);
  uint64_t span = (uint64_t)((int64_t)hi - (int64_t)lo + 1);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)((int64_t)lo + (int64_t)(draw_bits(key, (uint64_t)i) % span));
}
