/*
 * Seeded synthetic inputs for the sharded MLA decode workloads.
 *
 * This file generates input bytes only.  It holds no attention arithmetic:
 * no dot products, no softmax, no merge, and no fp8 *decoding*.  Both the
 * fp64 oracle and the CUDA path consume the bytes written here.
 *
 * Generator: a counter-based stream.  Value pair j of stream (seed, id) is
 * derived from splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014; finaliser constants as published by
 * S. Vigna) applied to key + 2j and key + 2j + 1, then turned into two
 * standard normals with the Box-Muller transform (Box and Muller, 1958).
 * Because every value is a pure function of (seed, id, index), the output
 * does not depend on the number of OpenMP threads.
 *
 * bf16 values: the normal is drawn in double, rounded to float (RNE), then
 * rounded to bf16 (RNE).  fp8 rows: one fp32 scale per row equal to
 * max|x| / 448 (1 when the row is all zero); codes are OCP e4m3 ("fn") of
 * x / scale, rounded to nearest even and saturated at +-448.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + GOLDEN;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t id) {
  return splitmix64(splitmix64(seed) ^ (id * GOLDEN));
}

/* Two standard normals from counter pair j. */
static inline void normal_pair(uint64_t key, uint64_t j, double* z0, double* z1) {
  uint64_t a = splitmix64(key + 2 * j);
  uint64_t b = splitmix64(key + 2 * j + 1);
  double u1 = ((double)((a >> 11) + 1)) * 0x1.0p-53; /* (0, 1] */
  double u2 = ((double)(b >> 11)) * 0x1.0p-53;       /* [0, 1) */
  double r = sqrt(-2.0 * log(u1));
  double th = 6.283185307179586476925286766559 * u2;
  *z0 = r * cos(th);
  *z1 = r * sin(th);
}

static inline double normal_at(uint64_t key, uint64_t k) {
  double z0, z1;
  normal_pair(key, k >> 1, &z0, &z1);
  return (k & 1) ? z1 : z0;
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x7FFFFFu)) return 0x7FC0;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* OCP e4m3 encoder: round to nearest even, saturate to +-448, NaN -> 0x7F. */
static uint8_t e4m3_encode(float v) {
  if (isnan(v)) return 0x7F;
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs((double)v);
  if (a == 0.0) return sign;
  if (a >= 448.0) return sign | 0x7E;
  int e2;
  frexp(a, &e2);          /* a = f * 2^e2, f in [0.5, 1) */
  int E = e2 - 1;         /* floor(log2 a) */
  if (E < -6) E = -6;     /* subnormal spacing 2^-9 below 2^-6 */
  double quantum = ldexp(1.0, E - 3);
  double r = nearbyint(a / quantum); /* exact division by a power of two; RNE */
  double val = r * quantum;
  if (val >= 448.0) return sign | 0x7E;
  if (val == 0.0) return sign;
  if (val < 0x1.0p-6) return sign | (uint8_t)r; /* exponent field 0 */
  int e3;
  double f = frexp(val, &e3);            /* val = f * 2^e3 */
  int exp_field = (e3 - 1) + 7;
  int mant = (int)(f * 16.0) - 8;        /* f*16 in [8, 16) */
  return sign | (uint8_t)((exp_field << 3) | mant);
}

/* n bf16 values ~ N(0, sigma^2) from stream (seed, id), indices offset..offset+n-1. */
void gen_normal_bf16(uint64_t seed, uint64_t id, uint64_t offset, size_t n,
                     double sigma, uint16_t* out) {
  uint64_t key = stream_key(seed, id);
#pragma omp parallel for schedule(static)
  for (long long c = 0; c < (long long)((n + 4095) / 4096); ++c) {
    size_t lo = (size_t)c * 4096, hi = lo + 4096 < n ? lo + 4096 : n;
    for (size_t k = lo; k < hi; ++k)
      out[k] = f32_to_bf16_rne((float)(sigma * normal_at(key, offset + k)));
  }
}

/* n fp32 values ~ N(0, sigma^2). */
void gen_normal_f32(uint64_t seed, uint64_t id, uint64_t offset, size_t n,
                    double sigma, float* out) {
  uint64_t key = stream_key(seed, id);
#pragma omp parallel for schedule(static)
  for (long long c = 0; c < (long long)((n + 4095) / 4096); ++c) {
    size_t lo = (size_t)c * 4096, hi = lo + 4096 < n ? lo + 4096 : n;
    for (size_t k = lo; k < hi; ++k)
      out[k] = (float)(sigma * normal_at(key, offset + k));
  }
}

/* Rows of `width` values ~ N(0, sigma^2), quantised per row to e4m3 codes
 * plus one fp32 scale (max|x|/448, or 1 for an all-zero row). */
void gen_normal_fp8_rows(uint64_t seed, uint64_t id, uint64_t row0, size_t nrows,
                         int width, double sigma, uint8_t* codes, float* scales) {
  uint64_t key = stream_key(seed, id);
#pragma omp parallel for schedule(static)
  for (long long r = 0; r < (long long)nrows; ++r) {
    float x[1024];
    int w = width > 1024 ? 1024 : width;
    float amax = 0.0f;
    uint64_t base = (row0 + (uint64_t)r) * (uint64_t)width;
    for (int d = 0; d < w; ++d) {
      x[d] = (float)(sigma * normal_at(key, base + (uint64_t)d));
      float ax = fabsf(x[d]);
      if (ax > amax) amax = ax;
    }
    float s = amax > 0.0f ? amax / 448.0f : 1.0f;
    scales[r] = s;
    for (int d = 0; d < w; ++d) codes[(size_t)r * width + d] = e4m3_encode(x[d] / s);
  }
}

/* Quantise given fp32 rows (same rule as above). */
void quantize_fp8_rows(const float* x, size_t nrows, int width, uint8_t* codes,
                       float* scales) {
#pragma omp parallel for schedule(static)
  for (long long r = 0; r < (long long)nrows; ++r) {
    const float* xr = x + (size_t)r * width;
    float amax = 0.0f;
    for (int d = 0; d < width; ++d) {
      float ax = fabsf(xr[d]);
      if (ax > amax) amax = ax;
    }
    float s = amax > 0.0f ? amax / 448.0f : 1.0f;
    scales[r] = s;
    for (int d = 0; d < width; ++d) codes[(size_t)r * width + d] = e4m3_encode(xr[d] / s);
  }
}

/* Encode single floats (exposed so tests can pin the encoder). */
void encode_e4m3(const float* x, size_t n, uint8_t* out) {
  for (size_t k = 0; k < n; ++k) out[k] = e4m3_encode(x[k]);
}

/* n raw 64-bit counter outputs of stream (seed, id). */
void gen_u64(uint64_t seed, uint64_t id, size_t n, uint64_t* out) {
  uint64_t key = stream_key(seed, id);
  for (size_t k = 0; k < n; ++k) out[k] = splitmix64(key + k);
}

/* Uniform random permutation of 0..n-1 (Fisher-Yates driven by the stream;
 * bounded integers by Lemire's multiply-shift, bias below 2^-32). */
void gen_permutation(uint64_t seed, uint64_t id, size_t n, int32_t* out) {
  uint64_t key = stream_key(seed, id);
  for (size_t i = 0; i < n; ++i) out[i] = (int32_t)i;
  for (size_t i = n; i > 1; --i) {
    uint64_t r = splitmix64(key + (uint64_t)i) >> 32;
    size_t j = (size_t)((r * (uint64_t)i) >> 32);
    int32_t t = out[i - 1];
    out[i - 1] = out[j];
    out[j] = t;
  }
}

/* Fill every row of a bf16 page pool whose (page,row) flag is set with a
 * 16-bit pattern (used to poison unused cache rows with NaN / huge values). */
void fill_rows_u16(uint16_t* pool, const uint8_t* row_flag, size_t nrows, int width,
                   uint16_t pattern) {
#pragma omp parallel for schedule(static)
  for (long long r = 0; r < (long long)nrows; ++r)
    if (row_flag[r])
      for (int d = 0; d < width; ++d) pool[(size_t)r * width + d] = pattern;
}

void fill_rows_u8(uint8_t* pool, const uint8_t* row_flag, size_t nrows, int width,
                  uint8_t pattern) {
#pragma omp parallel for schedule(static)
  for (long long r = 0; r < (long long)nrows; ++r)
    if (row_flag[r])
      for (int d = 0; d < width; ++d) pool[(size_t)r * width + d] = pattern;
}
