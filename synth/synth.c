/*
 * synth.c -- seeded synthetic inputs for the GEMM tests and benchmark.
 *
 * This module only makes inputs: random matrices with the value
 * distributions of the workloads (uniform, normal, normal with rare large
 * outliers), rounded to BF16, or quantised to FP8 E4M3 with FP32 scale
 * factors.  It holds none of the GEMM's arithmetic.  Both the CUDA library's
 * tests and the CPU oracle read what it writes; neither is imported here.
 *
 * Random numbers are counter based: SplitMix64's output function applied to
 * key + (counter + 1) * 0x9E3779B97F4A7C15, where the key mixes the seed
 * and a tensor id.  Element (r, c) of a rows x cols tensor uses counters
 * derived from its logical index e = r * cols + c only, so any element can
 * be regenerated on its own and the result does not depend on the thread
 * count or the leading dimension of the output.
 *
 *   uniform(lo, hi):  u = (x >> 11) * 2^-53,          value = lo + (hi - lo) u
 *   normal(mu, sd):   Box-Muller on counters 3e, 3e+1:
 *                     u1 = ((x0 >> 11) + 1) 2^-53, u2 = (x1 >> 11) 2^-53,
 *                     z = sqrt(-2 ln u1) cos(2 pi u2),  value = mu + sd z
 *                     outliers: if ((x2 >> 11) 2^-53 < p) value *= factor
 *
 * Values are produced in FP64, rounded once to FP32 (the "FP32 draw" of the
 * workload recipes) and from there to BF16 (round to nearest even) or, after
 * division by a scale, to E4M3 (round to nearest even, saturating at 448).
 * The FP8 scale is amax / 448 over the tensor, over each 1 x 128 row block
 * (A) or over each 128 x 128 block (B); an all-zero block gets scale 1.
 * Scale storage: a_scale[kb * rows + i], b_scale[nb * KB + kb].
 *
 * Portable C11, compiled with -ffp-contract=off.  libm's log/cos may differ
 * by an ulp between hosts, so stored test fixtures never depend on the
 * normal generator.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SYN_UNIFORM 0
#define SYN_NORMAL 1

static const uint64_t kGolden = 0x9E3779B97F4A7C15ull;

static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t synth_key(uint64_t seed, uint64_t tensor) {
  return mix64(mix64(seed + kGolden) ^ (tensor * 0xD1B54A32D192ED03ull));
}

uint64_t synth_draw(uint64_t key, uint64_t ctr) { return mix64(key + (ctr + 1u) * kGolden); }

static double unit53(uint64_t x) { return (double)(x >> 11) * 0x1.0p-53; }

typedef struct {
  int32_t dist;
  int32_t pad_;
  double p0, p1;          /* uniform: lo, hi.  normal: mu, sd */
  double out_prob;        /* normal only: probability of an outlier */
  double out_factor;      /* normal only: outlier multiplier */
} synth_dist;

static double value_at(const synth_dist* d, uint64_t key, uint64_t e) {
  if (d->dist == SYN_UNIFORM) return d->p0 + (d->p1 - d->p0) * unit53(synth_draw(key, e));
  double u1 = ((double)(synth_draw(key, 3 * e) >> 11) + 1.0) * 0x1.0p-53;
  double u2 = unit53(synth_draw(key, 3 * e + 1));
  double z = sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
  double v = d->p0 + d->p1 * z;
  if (d->out_prob > 0.0 && unit53(synth_draw(key, 3 * e + 2)) < d->out_prob) v *= d->out_factor;
  return v;
}

/* ---- value -> storage format ------------------------------------------- */

static uint16_t to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN */
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* E4M3, nearest-even, saturating.  Normals: round the FP32 pattern at bit 20
 * and re-bias the exponent (127 -> 7).  Below 2^-6: the grid is k * 2^-9, so
 * scale by 2^9 (exact) and round to an integer with rint (ties to even in the
 * default rounding mode). */
static uint8_t to_e4m3(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint8_t s = (uint8_t)((u >> 24) & 0x80u);
  uint32_t a = u & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return (uint8_t)(s | 0x7Fu);
  float m;
  memcpy(&m, &a, 4);
  if (m < 0x1.0p-6f) {
    int k = (int)rintf(m * 512.0f); /* 0..8; 8 is the smallest normal 0x08 */
    return (uint8_t)(s | (uint8_t)k);
  }
  if (m >= 464.0f) return (uint8_t)(s | 0x7Eu); /* 464 ties to 448 (even); above saturates */
  uint32_t r = (a + 0x7FFFFu + ((a >> 20) & 1u)) >> 20; /* exponent:8 | mantissa:3 */
  uint32_t e8 = r >> 3, m3 = r & 7u;
  uint32_t e4 = e8 - 127u + 7u;
  if (e4 > 15u || (e4 == 15u && m3 == 7u)) return (uint8_t)(s | 0x7Eu);
  return (uint8_t)(s | (uint8_t)(e4 << 3) | (uint8_t)m3);
}

/* E5M2, nearest-even, saturating at +-57344 (like the E4M3 encoder).
 * Normals: round the FP32 pattern at bit 21 and re-bias the exponent
 * (127 -> 15).  Below 2^-14: the grid is k * 2^-16 (scale by 2^16, exact,
 * and rint).  57344 = 1.75 * 2^15; halfway to 2^16 (61440) and above
 * saturate. */
static uint8_t to_e5m2(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint8_t s = (uint8_t)((u >> 24) & 0x80u);
  uint32_t a = u & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return (uint8_t)(s | 0x7Fu);
  float m;
  memcpy(&m, &a, 4);
  if (m < 0x1.0p-14f) {
    int k = (int)rintf(m * 65536.0f); /* 0..4; 4 is the smallest normal 0x04 */
    return (uint8_t)(s | (uint8_t)k);
  }
  if (m >= 61440.0f) return (uint8_t)(s | 0x7Bu);
  uint32_t r = (a + 0xFFFFFu + ((a >> 21) & 1u)) >> 21; /* exponent:8 | mantissa:2 */
  uint32_t e8 = r >> 2, m2 = r & 3u;
  uint32_t e5 = e8 - 127u + 15u;
  if (e5 > 30u) return (uint8_t)(s | 0x7Bu);
  return (uint8_t)(s | (uint8_t)(e5 << 2) | (uint8_t)m2);
}

/* ---- threaded row loops ------------------------------------------------- */

typedef struct {
  const synth_dist* d;
  uint64_t key;
  int64_t rows, cols, ld;
  int32_t kind; /* 0: float out, 1: bf16 out */
  void* out;
  int64_t r0, r1;
} fill_job;

static void* fill_rows(void* p) {
  fill_job* j = (fill_job*)p;
  for (int64_t r = j->r0; r < j->r1; ++r) {
    for (int64_t c = 0; c < j->cols; ++c) {
      float v = (float)value_at(j->d, j->key, (uint64_t)(r * j->cols + c));
      if (j->kind == 0)
        ((float*)j->out)[r * j->ld + c] = v;
      else
        ((uint16_t*)j->out)[r * j->ld + c] = to_bf16(v);
    }
  }
  return NULL;
}

static void run_fill(const synth_dist* d, uint64_t seed, uint64_t tensor, int64_t rows,
                     int64_t cols, int64_t ld, int32_t kind, void* out, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 128) nthreads = 128;
  if (nthreads > rows) nthreads = rows > 0 ? (int)rows : 1;
  fill_job jobs[128];
  pthread_t th[128];
  int started[128];
  uint64_t key = synth_key(seed, tensor);
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].d = d;
    jobs[t].key = key;
    jobs[t].rows = rows;
    jobs[t].cols = cols;
    jobs[t].ld = ld;
    jobs[t].kind = kind;
    jobs[t].out = out;
    jobs[t].r0 = rows * t / nthreads;
    jobs[t].r1 = rows * (t + 1) / nthreads;
  }
  for (int t = 1; t < nthreads; ++t) started[t] = pthread_create(&th[t], NULL, fill_rows, &jobs[t]) == 0;
  fill_rows(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) {
    if (started[t])
      pthread_join(th[t], NULL);
    else
      fill_rows(&jobs[t]);
  }
}

/* rows x cols FP32 values, row r at out + r * ld. */
void synth_fill_f32(const synth_dist* d, uint64_t seed, uint64_t tensor, int64_t rows, int64_t cols,
                    int64_t ld, float* out, int nthreads) {
  run_fill(d, seed, tensor, rows, cols, ld, 0, out, nthreads);
}

/* rows x cols BF16 bit patterns (FP64 draw -> FP32 -> BF16 nearest even). */
void synth_fill_bf16(const synth_dist* d, uint64_t seed, uint64_t tensor, int64_t rows,
                     int64_t cols, int64_t ld, uint16_t* out, int nthreads) {
  run_fill(d, seed, tensor, rows, cols, ld, 1, out, nthreads);
}

static float scale_of(float amax) { return amax > 0.0f ? amax / 448.0f : 1.0f; }

/* Per-tensor FP8: scale = amax / 448 over the dense rows x cols input x,
 * q = E4M3(x / scale).  q has leading dimension ldq. */
void synth_quant_e4m3_tensor(const float* x, int64_t rows, int64_t cols, int64_t ldq, uint8_t* q,
                             float* scale) {
  float amax = 0.0f;
  for (int64_t i = 0; i < rows * cols; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  float s = scale_of(amax);
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) q[r * ldq + c] = to_e4m3(x[r * cols + c] / s);
  *scale = s;
}

/* FP8 with one scale per 1 x 128 block of each row (the activation side):
 * scale[kb * rows + r] for columns 128kb .. 128kb+127 of row r. */
void synth_quant_e4m3_rowblock(const float* x, int64_t rows, int64_t cols, int64_t ldq,
                               uint8_t* q, float* scale) {
  int64_t KB = (cols + 127) / 128;
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t kb = 0; kb < KB; ++kb) {
      int64_t c0 = kb * 128, c1 = c0 + 128 < cols ? c0 + 128 : cols;
      float amax = 0.0f;
      for (int64_t c = c0; c < c1; ++c) {
        float a = fabsf(x[r * cols + c]);
        if (a > amax) amax = a;
      }
      float s = scale_of(amax);
      scale[kb * rows + r] = s;
      for (int64_t c = c0; c < c1; ++c) q[r * ldq + c] = to_e4m3(x[r * cols + c] / s);
    }
  }
}

/* FP8 with one scale per 128 x 128 block (the weight side, rows = N):
 * scale[nb * KB + kb]. */
void synth_quant_e4m3_block128(const float* x, int64_t rows, int64_t cols, int64_t ldq,
                               uint8_t* q, float* scale) {
  int64_t KB = (cols + 127) / 128, NB = (rows + 127) / 128;
  for (int64_t nb = 0; nb < NB; ++nb) {
    int64_t r0 = nb * 128, r1 = r0 + 128 < rows ? r0 + 128 : rows;
    for (int64_t kb = 0; kb < KB; ++kb) {
      int64_t c0 = kb * 128, c1 = c0 + 128 < cols ? c0 + 128 : cols;
      float amax = 0.0f;
      for (int64_t r = r0; r < r1; ++r)
        for (int64_t c = c0; c < c1; ++c) {
          float a = fabsf(x[r * cols + c]);
          if (a > amax) amax = a;
        }
      float s = scale_of(amax);
      scale[nb * KB + kb] = s;
      for (int64_t r = r0; r < r1; ++r)
        for (int64_t c = c0; c < c1; ++c) q[r * ldq + c] = to_e4m3(x[r * cols + c] / s);
    }
  }
}

/* Element-wise encoders, exposed so tests can compare them with other
 * implementations of the same formats. */
void synth_to_bf16_array(const float* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = to_bf16(x[i]);
}
void synth_to_e4m3_array(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = to_e4m3(x[i]);
}
void synth_to_e5m2_array(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = to_e5m2(x[i]);
}
