/*
 * Seeded synthetic inputs for the two-tier sparse-attention step.
 *
 * This file holds no arithmetic of the attention method. It only turns
 * (seed, tensor tag, element index) into numbers with the distributions the
 * workloads call for: N(0,1)/sqrt(d) values stored as bf16, as MXFP8 (e4m3
 * codes plus one UE8M0 scale per 32 elements) or as MXFP4 (e2m1 codes, two a
 * byte, plus one UE8M0 scale per 32 elements), and U(0,1) head weights.
 * Both the CUDA path and the CPU oracle are fed the bytes this file writes.
 *
 * Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014), used counter-style: the draw for counter c
 * of a stream is the SplitMix64 output mix(key + (c + 1) * GAMMA), so every
 * element can be produced independently and in parallel. Normals come from
 * the Box-Muller transform in double precision on the host.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Key of the stream (seed, tag). */
static inline uint64_t stream_key(uint64_t seed, uint64_t tag) {
  return mix64(seed * GAMMA + mix64(tag + GAMMA));
}

static inline uint64_t draw(uint64_t key, uint64_t c) { return mix64(key + (c + 1) * GAMMA); }

/* Uniform in (0, 1] with 53 random bits. */
static inline double unit53(uint64_t z) { return (double)((z >> 11) + 1) * 0x1.0p-53; }

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* e4m3 (bias 7, no infinities, max 448) code nearest to y, ties to even,
 * saturating at +-448. */
static uint8_t e4m3_code(double y) {
  uint8_t s = (y < 0) ? 0x80 : 0x00;
  double a = fabs(y);
  if (a >= 448.0) return s | 0x7E;
  if (a < 0x1.0p-6) {
    double m = nearbyint(a * 0x1.0p9); /* 0..8; 8 is the smallest normal */
    return s | (uint8_t)m;
  }
  int e;
  double fr = frexp(a, &e); /* a = fr * 2^e, fr in [0.5, 1) */
  int E = e - 1;            /* a in [2^E, 2^(E+1)) */
  double m = nearbyint((a / ldexp(1.0, E) - 1.0) * 8.0);
  (void)fr;
  if (m >= 8.0) {
    m = 0.0;
    E += 1;
  }
  if (E > 8 || (E == 8 && m > 6.0)) return s | 0x7E;
  return s | (uint8_t)(((E + 7) << 3) | (int)m);
}

/* e2m1 (1 sign, 2 exponent bits with bias 1, 1 mantissa bit; magnitudes 0,
 * 0.5, 1, 1.5, 2, 3, 4, 6) code nearest to y, ties to the even mantissa,
 * saturating at +-6. */
static uint8_t e2m1_code(double y) {
  uint8_t s = (y < 0) ? 0x8 : 0x0;
  double a = fabs(y);
  if (a >= 6.0) return s | 0x7;
  if (a < 1.0) return s | (uint8_t)nearbyint(a * 2.0); /* 0, 1, or 2 (= 1.0) */
  int e;
  frexp(a, &e);
  int E = e - 1; /* a in [2^E, 2^(E+1)), E in 0..2 */
  double m = nearbyint((a / ldexp(1.0, E) - 1.0) * 2.0);
  if (m >= 2.0) {
    m = 0.0;
    E += 1;
  }
  if (E > 2) return s | 0x7;
  return s | (uint8_t)(((E + 1) << 1) | (int)m);
}

/* Both normals of pair j: element 2j takes the cosine, 2j + 1 the sine. */
static inline void normal_pair(uint64_t key, uint64_t j, double* z0, double* z1) {
  double u1 = unit53(draw(key, 2 * j));
  double u2 = unit53(draw(key, 2 * j + 1));
  double r = sqrt(-2.0 * log(u1));
  double th = 6.283185307179586476925286766559 * u2;
  *z0 = r * cos(th);
  *z1 = r * sin(th);
}

/* Calls put(i, N(offset + i)) for i in [0, n), one Box-Muller pair at a time. */
#define FOR_EACH_NORMAL(key, offset, n, PUT)                                   \
  do {                                                                         \
    int64_t first_pair = (offset) >> 1;                                        \
    int64_t last_pair = ((offset) + (n) - 1) >> 1;                             \
    _Pragma("omp parallel for schedule(static)")                               \
    for (int64_t p = first_pair; p <= last_pair; ++p) {                        \
      double z[2];                                                             \
      normal_pair(key, (uint64_t)p, &z[0], &z[1]);                             \
      for (int t = 0; t < 2; ++t) {                                            \
        int64_t i = 2 * p + t - (offset);                                      \
        if (i >= 0 && i < (n)) PUT(i, z[t]);                                   \
      }                                                                        \
    }                                                                          \
  } while (0)

/* out[i] = bf16(float(scale * N(offset + i))) for i in [0, n). */
void synth_normal_bf16(uint64_t seed, uint64_t tag, int64_t offset, int64_t n, double scale,
                       uint16_t* out) {
  if (n <= 0) return;
  uint64_t key = stream_key(seed, tag);
#define PUT_BF16(i, z) out[i] = f32_to_bf16_rne((float)(scale * (z)))
  FOR_EACH_NORMAL(key, offset, n, PUT_BF16);
#undef PUT_BF16
}

/* out[i] = fp32(float(scale * N(offset + i))). */
void synth_normal_f32(uint64_t seed, uint64_t tag, int64_t offset, int64_t n, double scale,
                      float* out) {
  if (n <= 0) return;
  uint64_t key = stream_key(seed, tag);
#define PUT_F32(i, z) out[i] = (float)(scale * (z))
  FOR_EACH_NORMAL(key, offset, n, PUT_F32);
#undef PUT_F32
}

/* out[i] = e4m3 code of fp32(scale * N(offset + i)) / kv_scale (an fp8 cache
 * with one scale; kv_scale a power of two, so the division is exact). */
void synth_normal_e4m3(uint64_t seed, uint64_t tag, int64_t offset, int64_t n, double scale,
                       double kv_scale, uint8_t* out) {
  if (n <= 0) return;
  uint64_t key = stream_key(seed, tag);
#define PUT_E4M3(i, z) out[i] = e4m3_code((double)(float)(scale * (z)) / kv_scale)
  FOR_EACH_NORMAL(key, offset, n, PUT_E4M3);
#undef PUT_E4M3
}

/* out[i] = k * 2^-24 with k the top 24 bits of draw(offset + i): U[0,1), exact in fp32. */
void synth_uniform_f32(uint64_t seed, uint64_t tag, int64_t offset, int64_t n, float* out) {
  uint64_t key = stream_key(seed, tag);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    out[i] = (float)(draw(key, (uint64_t)(offset + i)) >> 40) * 0x1.0p-24f;
  }
}

/*
 * Rows of `dim` (a multiple of 32) values scale * N(row * dim + j), taken to
 * fp32 and stored as MXFP8: per group of 32, X = floor(log2(amax)) - 8 clamped
 * to [-127, 127] (X = 0 for an all-zero group), scale byte X + 127, codes =
 * e4m3(v / 2^X). codes is [rows, dim], scales is [rows, dim / 32].
 */
void synth_normal_mxfp8(uint64_t seed, uint64_t tag, int64_t row_offset, int64_t rows, int dim,
                        double scale, uint8_t* codes, uint8_t* scales) {
  uint64_t key = stream_key(seed, tag);
  int groups = dim / 32;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int g = 0; g < groups; ++g) {
      float v[32];
      float amax = 0.0f;
      for (int j = 0; j < 32; j += 2) {
        uint64_t c = (uint64_t)((row_offset + r) * dim + g * 32 + j); /* even */
        double z0, z1;
        normal_pair(key, c >> 1, &z0, &z1);
        v[j] = (float)(scale * z0);
        v[j + 1] = (float)(scale * z1);
      }
      for (int j = 0; j < 32; ++j) {
        float a = fabsf(v[j]);
        if (a > amax) amax = a;
      }
      int X = 0;
      if (amax > 0.0f) {
        int e;
        frexpf(amax, &e);
        X = (e - 1) - 8;
        if (X < -127) X = -127;
        if (X > 127) X = 127;
      }
      scales[r * groups + g] = (uint8_t)(X + 127);
      for (int j = 0; j < 32; ++j) {
        codes[r * dim + g * 32 + j] = e4m3_code(ldexp((double)v[j], -X));
      }
    }
  }
}

/*
 * As synth_normal_mxfp8, stored as MXFP4: per group of 32, X = floor(log2(amax))
 * - 2 clamped to [-127, 127] (X = 0 for an all-zero group), scale byte X + 127,
 * codes = e2m1(v / 2^X), two a byte (element 2i in the low nibble). packed is
 * [rows, dim / 2], scales is [rows, dim / 32].
 */
void synth_normal_mxfp4(uint64_t seed, uint64_t tag, int64_t row_offset, int64_t rows, int dim,
                        double scale, uint8_t* packed, uint8_t* scales) {
  uint64_t key = stream_key(seed, tag);
  int groups = dim / 32;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int g = 0; g < groups; ++g) {
      float v[32];
      float amax = 0.0f;
      for (int j = 0; j < 32; j += 2) {
        uint64_t c = (uint64_t)((row_offset + r) * dim + g * 32 + j); /* even */
        double z0, z1;
        normal_pair(key, c >> 1, &z0, &z1);
        v[j] = (float)(scale * z0);
        v[j + 1] = (float)(scale * z1);
      }
      for (int j = 0; j < 32; ++j) {
        float a = fabsf(v[j]);
        if (a > amax) amax = a;
      }
      int X = 0;
      if (amax > 0.0f) {
        int e;
        frexpf(amax, &e);
        X = (e - 1) - 2;
        if (X < -127) X = -127;
        if (X > 127) X = 127;
      }
      scales[r * groups + g] = (uint8_t)(X + 127);
      for (int j = 0; j < 32; j += 2) {
        uint8_t lo = e2m1_code(ldexp((double)v[j], -X));
        uint8_t hi = e2m1_code(ldexp((double)v[j + 1], -X));
        packed[r * (dim / 2) + g * 16 + j / 2] = (uint8_t)(lo | (hi << 4));
      }
    }
  }
}

int synth_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}
