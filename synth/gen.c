/*
 * Seeded synthetic inputs for the stage forward: weights, norm gains, token ids.
 *
 * This file holds input generation only.  It contains none of the stage's
 * arithmetic: no dequantisation, no matmul, no attention.  Both the CPU oracle
 * and the CUDA path receive the arrays written here.
 *
 * Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014), used counter-style: draw c of stream k is
 * the SplitMix64 finaliser applied to k + (c + 1) * 0x9E3779B97F4A7C15, which is
 * exactly the c-th output of a SplitMix64 generator seeded with k.  Any element
 * of any tensor can therefore be regenerated on its own.
 *
 * Normals: Box-Muller (Box and Muller, 1958) in double precision.  Element
 * pair p of a stream uses draws 2p and 2p+1 as two 53-bit uniforms in (0,1);
 * element 2p gets R cos(t), element 2p+1 gets R sin(t).  A weight is the float
 * rounding of sigma * z.
 *
 * Block quantiser (weights are stored as int8 blocks of 32 along the input
 * dimension with one fp16 scale per block; when the row length is not a multiple
 * of 32 the last block of each row is partial): amax = max |w| over the block;
 * s = fp16(amax / 127) with round-to-nearest-even (the division in float);
 * q = clamp(rint(w / float(s)), -127, 127); an all-zero block, or one whose
 * scale underflows to zero, gives s = 0 and q = 0.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define SM_GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t sm_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* c-th output of SplitMix64 seeded with k. */
static inline uint64_t sm_draw(uint64_t k, uint64_t c) { return sm_mix(k + (c + 1) * SM_GOLDEN); }

/* Stream key for a tuple of non-negative fields (seed, config, layer, tensor, expert, ...). */
uint64_t synth_key(const int64_t* fields, int n) {
  uint64_t k = 0x243F6A8885A308D3ULL;
  for (int i = 0; i < n; ++i) k = sm_mix(k ^ sm_draw((uint64_t)fields[i], (uint64_t)i));
  return k;
}

static inline double u53(uint64_t r) { return ((double)(r >> 11) + 0.5) * (1.0 / 9007199254740992.0); }

static inline void normal_pair(uint64_t k, uint64_t p, double* z0, double* z1) {
  const double two_pi = 6.283185307179586476925286766559;
  double u1 = u53(sm_draw(k, 2 * p)), u2 = u53(sm_draw(k, 2 * p + 1));
  double r = sqrt(-2.0 * log(u1)), t = two_pi * u2;
  *z0 = r * cos(t);
  *z1 = r * sin(t);
}

/* float -> IEEE binary16 bits, round to nearest even (handles subnormals, overflow to inf). */
static uint16_t f32_to_f16_rne(float f) {
  uint32_t x;
  memcpy(&x, &f, 4);
  uint32_t sign = (x >> 16) & 0x8000u;
  uint32_t ax = x & 0x7FFFFFFFu;
  if (ax >= 0x7F800000u) return (uint16_t)(sign | (ax > 0x7F800000u ? 0x7E00u : 0x7C00u));
  if (ax >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u); /* rounds to >= 65520: inf */
  if (ax < 0x38800000u) {                                     /* below 2^-14: fp16 subnormal or zero */
    if (ax < 0x33000000u) return (uint16_t)sign;              /* below 2^-25: rounds to zero */
    uint32_t e = ax >> 23, m = (ax & 0x7FFFFFu) | 0x800000u;
    uint32_t shift = 126 - e;                                 /* value = m * 2^(e-150); unit 2^-24 */
    uint32_t q = m >> shift, rem = m & ((1u << shift) - 1), half = 1u << (shift - 1);
    if (rem > half || (rem == half && (q & 1u))) q++;
    return (uint16_t)(sign | q);
  }
  uint32_t e = (ax >> 23) - 112, m = ax & 0x7FFFFFu;
  uint32_t q = (e << 10) | (m >> 13), rem = m & 0x1FFFu;
  if (rem > 0x1000u || (rem == 0x1000u && (q & 1u))) q++;
  return (uint16_t)(sign | q);
}

static float f16_to_f32(uint16_t h) {
  uint32_t sign = (uint32_t)(h & 0x8000u) << 16, e = (h >> 10) & 0x1Fu, m = h & 0x3FFu, x;
  if (e == 0) {
    if (m == 0) x = sign;
    else { float v = (float)m * (1.0f / 16777216.0f); memcpy(&x, &v, 4); x |= sign; }
  } else if (e == 31) x = sign | 0x7F800000u | (m << 13);
  else x = sign | ((e + 112) << 23) | (m << 13);
  float f;
  memcpy(&f, &x, 4);
  return f;
}

/* Normal draws sigma*z for elements [start, start+count) of stream k, rounded to float, plus mean. */
void synth_normal_f32(uint64_t k, int64_t start, int64_t count, double sigma, double mean, float* out) {
  int64_t i = 0;
  while (i < count) {
    int64_t e = start + i;
    double z0, z1;
    normal_pair(k, (uint64_t)(e >> 1), &z0, &z1);
    if (e & 1) {
      out[i++] = (float)(mean + sigma * z1);
    } else {
      out[i++] = (float)(mean + sigma * z0);
      if (i < count) out[i++] = (float)(mean + sigma * z1);
    }
  }
}

/* Quantise one block of n <= 32 floats (the last block of a row may be partial). */
static void quant_block(const float* w, int n, int8_t* q, uint16_t* s) {
  float amax = 0.0f;
  for (int j = 0; j < n; ++j) {
    float a = fabsf(w[j]);
    if (a > amax) amax = a;
  }
  volatile float ratio = amax / 127.0f;
  uint16_t sh = f32_to_f16_rne(ratio);
  float sf = f16_to_f32(sh);
  *s = sh;
  for (int j = 0; j < n; ++j) {
    if (sf == 0.0f) { q[j] = 0; continue; }
    volatile float t = w[j] / sf;
    float r = rintf(t);
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    q[j] = (int8_t)r;
  }
}

/* Quantise [rows x cols] floats row by row: blocks of 32 along each row, the last one
 * partial when cols % 32 != 0.  s is [rows x ceil(cols/32)]. */
void synth_quantize(const float* w, int64_t rows, int64_t cols, int8_t* q, uint16_t* s) {
  int64_t nb = (cols + 31) / 32;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < nb; ++b) {
      int n = cols - 32 * b < 32 ? (int)(cols - 32 * b) : 32;
      quant_block(w + r * cols + 32 * b, n, q + r * cols + 32 * b, s + r * nb + b);
    }
}

/* Rows [row0, row0+nrows) of a [rows x cols] N(0, sigma) matrix, quantised; q is [nrows x cols],
 * s is [nrows x ceil(cols/32)]. */
static void q8_rows(uint64_t k, int64_t cols, int64_t row0, int64_t nrows, double sigma, int8_t* q,
                    uint16_t* s) {
  float w[32];
  int64_t nb = (cols + 31) / 32;
  for (int64_t r = 0; r < nrows; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      int n = cols - 32 * b < 32 ? (int)(cols - 32 * b) : 32;
      synth_normal_f32(k, (row0 + r) * cols + 32 * b, n, sigma, 0.0, w);
      quant_block(w, n, q + r * cols + 32 * b, s + r * nb + b);
    }
  }
}

typedef struct {
  uint64_t k;
  int64_t cols, row0, nrows;
  double sigma;
  int8_t* q;
  uint16_t* s;
} q8_job;

static void* q8_worker(void* arg) {
  q8_job* j = (q8_job*)arg;
  q8_rows(j->k, j->cols, j->row0, j->nrows, j->sigma, j->q, j->s);
  return 0;
}

/* Threaded version of q8_rows; the output does not depend on n_threads. */
int synth_q8(uint64_t k, int64_t cols, int64_t row0, int64_t nrows, double sigma, int8_t* q, uint16_t* s,
             int n_threads) {
  if (cols <= 0 || nrows < 0) return -1;
  if (n_threads > 256) n_threads = 256;
  if ((int64_t)n_threads > nrows / 16) n_threads = (int)(nrows / 16);
  if (n_threads < 1) n_threads = 1;
  pthread_t th[256];
  int created[256];
  q8_job jobs[256];
  int64_t per = (nrows + n_threads - 1) / n_threads, nb = (cols + 31) / 32;
  for (int t = 0; t < n_threads; ++t) {
    int64_t a = t * per, b = a + per < nrows ? a + per : nrows;
    if (a > b) a = b;
    jobs[t] = (q8_job){k, cols, row0 + a, b - a, sigma, q + a * cols, s + a * nb};
    created[t] = 0;
  }
  for (int t = 1; t < n_threads; ++t) created[t] = pthread_create(&th[t], 0, q8_worker, &jobs[t]) == 0;
  q8_worker(&jobs[0]);
  for (int t = 1; t < n_threads; ++t) {
    if (created[t]) pthread_join(th[t], 0);
    else q8_worker(&jobs[t]);
  }
  return 0;
}

/* count uniform integers in [0, n) from stream k (Lemire's multiply-shift on the top 32 bits). */
void synth_uniform_int(uint64_t k, int64_t start, int64_t count, int64_t n, int32_t* out) {
  for (int64_t i = 0; i < count; ++i) {
    uint64_t r = sm_draw(k, (uint64_t)(start + i)) >> 32;
    out[i] = (int32_t)((r * (uint64_t)n) >> 32);
  }
}

/* float <-> fp16 helpers exported for the Python side of the generator. */
void synth_f32_to_f16(const float* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_f16_rne(x[i]);
}
