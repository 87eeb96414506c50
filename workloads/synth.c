/*
 * Seeded synthetic input generator for the paged-attention workloads.
 *
 * This file only draws numbers. It holds none of the attention arithmetic; the
 * oracle and the CUDA path both receive what it produces and nothing else of it.
 *
 * Random stream: the SplitMix64 output function (Steele, Lea and Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014) applied to a Weyl
 * sequence. Value i of stream s under seed k is
 *     mix64(key(k, s) + (i + 1) * GOLDEN)
 * so any slice of a stream can be produced independently (counter based), which is
 * what lets the large page pools be filled in parallel with identical results.
 *
 * Normal deviates use the Box-Muller transform (two deviates per pair of uniforms).
 * The logarithm, cosine and sine are evaluated here from their series with plain
 * IEEE additions and multiplications so that x86_64 and aarch64 hosts produce the
 * same bits (this file is compiled with -ffp-contract=off and calls no libm
 * transcendental).
 */
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(mix64(seed + GOLDEN) ^ (stream * 0xD1B54A32D192ED03ULL + 0x2545F4914F6CDD1DULL));
}

static inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN); }

/* uniform double in [0, 1) from the top 53 bits */
static inline double unit53(uint64_t x) { return (double)(x >> 11) * (1.0 / 9007199254740992.0); }

/* natural log for x in (0, 1]: x = m * 2^e with m in [sqrt(1/2), sqrt(2)),
 * ln m = 2 atanh(z) = 2 (z + z^3/3 + z^5/5 + ...), z = (m - 1) / (m + 1), |z| <= 0.1716;
 * twelve terms leave a remainder below 1e-18. */
static double series_log(double x) {
  uint64_t bits;
  memcpy(&bits, &x, 8);
  int e = (int)((bits >> 52) & 0x7FF) - 1023;
  bits = (bits & 0x000FFFFFFFFFFFFFULL) | 0x3FF0000000000000ULL; /* m in [1, 2) */
  double m;
  memcpy(&m, &bits, 8);
  if (m > 1.4142135623730951) { m *= 0.5; e += 1; }
  double z = (m - 1.0) / (m + 1.0);
  double z2 = z * z;
  double s = 1.0 / 23.0;
  s = s * z2 + 1.0 / 21.0;
  s = s * z2 + 1.0 / 19.0;
  s = s * z2 + 1.0 / 17.0;
  s = s * z2 + 1.0 / 15.0;
  s = s * z2 + 1.0 / 13.0;
  s = s * z2 + 1.0 / 11.0;
  s = s * z2 + 1.0 / 9.0;
  s = s * z2 + 1.0 / 7.0;
  s = s * z2 + 1.0 / 5.0;
  s = s * z2 + 1.0 / 3.0;
  s = s * z2 + 1.0;
  return 2.0 * z * s + (double)e * 0.6931471805599453;
}

/* (cos 2 pi u, sin 2 pi u) for u in [0, 1). With v = 4u, r = floor(v + 1/2) and
 * t = (v - r) pi/2 in [-pi/4, pi/4] (v - r is exact), the angle is r pi/2 + t, so the
 * pair is a signed permutation of (cos t, sin t) chosen by r mod 4. Taylor series to
 * t^18 / t^17 (remainders below 1e-18). */
static void series_cos_sin_2pi(double u, double* cos_out, double* sin_out) {
  double v = 4.0 * u;
  double r = __builtin_floor(v + 0.5);
  double t = (v - r) * 1.5707963267948966;
  double t2 = t * t;
  double c = -1.0 / 6402373705728000.0;           /* -1/18! */
  c = c * t2 + 1.0 / 20922789888000.0;             /* 1/16! */
  c = c * t2 - 1.0 / 87178291200.0;                /* 1/14! */
  c = c * t2 + 1.0 / 479001600.0;                  /* 1/12! */
  c = c * t2 - 1.0 / 3628800.0;                    /* 1/10! */
  c = c * t2 + 1.0 / 40320.0;
  c = c * t2 - 1.0 / 720.0;
  c = c * t2 + 1.0 / 24.0;
  c = c * t2 - 0.5;
  c = c * t2 + 1.0;
  double s = 1.0 / 355687428096000.0;              /* 1/17! */
  s = s * t2 - 1.0 / 1307674368000.0;              /* 1/15! */
  s = s * t2 + 1.0 / 6227020800.0;                 /* 1/13! */
  s = s * t2 - 1.0 / 39916800.0;                   /* 1/11! */
  s = s * t2 + 1.0 / 362880.0;
  s = s * t2 - 1.0 / 5040.0;
  s = s * t2 + 1.0 / 120.0;
  s = s * t2 - 1.0 / 6.0;
  s = s * t2 + 1.0;
  s = s * t;
  int q = ((int)r) & 3;
  *cos_out = (q == 0) ? c : (q == 1) ? -s : (q == 2) ? -c : s;
  *sin_out = (q == 0) ? s : (q == 1) ? c : (q == 2) ? -s : -c;
}

/* Box-Muller: pair k of a stream uses uniforms 2k and 2k+1 and yields two independent
 * standard normal deviates, the cosine one first. */
static void normal_pair(uint64_t key, uint64_t k, double* z0, double* z1) {
  double u1 = 1.0 - unit53(draw(key, 2 * k));     /* (0, 1] */
  double u2 = unit53(draw(key, 2 * k + 1));       /* [0, 1) */
  double r2 = -2.0 * series_log(u1);
  double r = r2 > 0.0 ? __builtin_sqrt(r2) : 0.0; /* IEEE sqrt: correctly rounded */
  double c, s;
  series_cos_sin_2pi(u2, &c, &s);
  *z0 = r * c;
  *z1 = r * s;
}

/* deviate i of a normal stream: element 2k is the cosine deviate of pair k, 2k+1 the sine */
static double std_normal(uint64_t key, uint64_t i) {
  double z0, z1;
  normal_pair(key, i >> 1, &z0, &z1);
  return (i & 1) ? z1 : z0;
}

/* float32 -> bfloat16 bits, round to nearest even (NaN kept quiet) */
static uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* float32 -> IEEE binary16 bits, round to nearest even, with subnormals and overflow */
static uint16_t f32_to_f16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  uint32_t a = u & 0x7FFFFFFFu;
  if (a >= 0x7F800000u) return sign | (a > 0x7F800000u ? 0x7E00u : 0x7C00u);
  if (a >= 0x477FF000u) return sign | 0x7C00u; /* rounds to >= 65520: overflow to inf */
  if (a < 0x33000000u) return sign;            /* at most half the smallest subnormal */
  int e = (int)(a >> 23) - 127;
  uint32_t mant = (a & 0x7FFFFFu) | 0x800000u; /* 24-bit significand */
  int shift = e >= -14 ? 13 : 13 + (-14 - e);  /* bits dropped from the significand */
  uint32_t kept = mant >> shift;
  uint32_t rem = mant & ((1u << shift) - 1u);
  uint32_t half = 1u << (shift - 1);
  if (rem > half || (rem == half && (kept & 1u))) kept += 1u;
  if (e >= -14) /* a carry out of the significand moves into the exponent field */
    return sign | (uint16_t)(((uint32_t)(e + 15) << 10) + (kept - 0x400u));
  return sign | (uint16_t)kept;
}

static inline uint16_t to_bits(double x, int dtype) {
  float f = (float)x;
  return dtype == 1 ? f32_to_bf16(f) : f32_to_f16(f);
}

/* ---- exported ---------------------------------------------------------------- */

void synth_u64(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, uint64_t* out) {
  uint64_t key = stream_key(seed, stream);
  for (int64_t i = 0; i < n; ++i) out[i] = draw(key, offset + (uint64_t)i);
}

void synth_uniform(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double* out) {
  uint64_t key = stream_key(seed, stream);
  for (int64_t i = 0; i < n; ++i) out[i] = unit53(draw(key, offset + (uint64_t)i));
}

/* n standard normal deviates (elements offset .. offset+n-1 of the stream) rounded to
 * fp16 (dtype 0) or bf16 (dtype 1) */
void synth_normal_bits(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, int dtype,
                       uint16_t* out) {
  uint64_t key = stream_key(seed, stream);
  if (n <= 0) return;
  int64_t head = (offset & 1) ? 1 : 0; /* a leading sine deviate */
  if (head) out[0] = to_bits(std_normal(key, offset), dtype);
  int64_t pairs = (n - head) / 2;
  uint64_t k0 = (offset + (uint64_t)head) >> 1;
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < pairs; ++k) {
    double z0, z1;
    normal_pair(key, k0 + (uint64_t)k, &z0, &z1);
    out[head + 2 * k] = to_bits(z0, dtype);
    out[head + 2 * k + 1] = to_bits(z1, dtype);
  }
  if (head + 2 * pairs < n) out[n - 1] = to_bits(std_normal(key, offset + (uint64_t)(n - 1)), dtype);
}

/* n deviates uniform in [lo, hi) rounded to fp16 / bf16 */
void synth_uniform_bits(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double lo,
                        double hi, int dtype, uint16_t* out) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i)
    out[i] = to_bits(lo + (hi - lo) * unit53(draw(key, offset + (uint64_t)i)), dtype);
}

/* the deviates themselves in double, for checking the generator's distribution */
void synth_normal_f64(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double* out) {
  uint64_t key = stream_key(seed, stream);
  for (int64_t i = 0; i < n; ++i) out[i] = std_normal(key, offset + (uint64_t)i);
}
