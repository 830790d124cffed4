/*
 * oracle.c -- plain, slow CPU reference for the dense tensor-core GEMM
 *
 *     D = alpha * A * B + beta * C
 *
 * with BF16 or FP8 E4M3 operands, computed exactly (up to FP64 rounding).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * under tensor_core_dense_gb300/) may include, link or call this file; only
 * tests/, the smoke check in __graft_entry__.py and bench.py's CPU-baseline
 * leg use it.  It shares no code, header, table or constant with the CUDA
 * path.
 *
 * What it computes, and where that comes from:
 *
 *  - The operation is the multiply-accumulate D = A*B + C with A an M x K
 *    matrix, B a K x N matrix and C, D M x N ("Tensor Cores: Matrix
 *    Instructions, Swizzling and FP8, Measured", Step 1; "Tensor Cores",
 *    "What a Tensor Core does"), extended by the alpha/beta scalars and the
 *    FP8 scale factors of the FP8 recipe ("Tensor cores and low precision",
 *    paragraph on FP8 scaling: scale before the cast, remove the scale after
 *    the multiply).
 *  - B is held N x K with K contiguous, the "TN" layout of the 4,096^3 test
 *    ("Tensor Cores: Matrix Instructions, ...", Step 2): element (k, j) of B
 *    sits at B[j * ldb + k].  A is M x K row-major: A[i * lda + k].
 *  - BF16 is 1 sign / 8 exponent / 7 mantissa bits, the top half of an FP32
 *    word ("Tensor Cores", "Precision: FP16, BF16, TF32, FP8").
 *  - E4M3 is 1 / 4 / 3 bits, no infinities, maximum normal 448 ("Tensor
 *    cores and low precision", paragraph on the two 8-bit encodings).  448 =
 *    1.75 * 2^8 is the largest finite value with exponent field 15 and
 *    mantissa 110, so the exponent bias is 7 and only mantissa 111 at
 *    exponent 15 is NaN.
 *  - E5M2 is 1 / 5 / 2 bits with IEEE 754 behaviour for the special values
 *    and maximum normal 57,344 (same paragraph).  57,344 = 1.75 * 2^15 is the
 *    largest finite value with exponent field 30 (31 is kept for infinity and
 *    NaN, as in IEEE 754), so the bias is 15.  Either operand of an FP8 GEMM
 *    may be E4M3 or E5M2.
 *
 * Accumulation is in FP64.  BF16 x BF16 products are exact in FP64.  For
 * E4M3 the raw code products q_a * q_b (at most 8 significant bits, exponents
 * 2^-18 .. 2^17) are summed per 128-wide K block, which is exact, and only
 * then multiplied by the block's FP64 scale product s_a * s_b (exact, 24+24
 * bits).  With E5M2 operands (exponents 2^-16 .. 2^15) a block sum can span
 * more than 53 bits and is exact only up to FP64 rounding, at most
 * 128 * 2^-53 of the block's sum of |products|.  The sum of |a_ik * b_kj| is
 * returned beside each value as the error bound the tolerances are stated
 * against.
 *
 * The scale layouts for the 128-block mode (the pages name block scaling but
 * give no storage order; this is the library's choice, stated here and in
 * its header):
 *     a_scale[kb * M + i]          scale of A row i, K block kb   (1 x 128)
 *     b_scale[nb * KB + kb]        scale of B rows 128nb.., K block kb
 *                                   (128 x 128), KB = ceil(K / 128)
 *
 * Microscaled FP8 (ORC_SCALE_MX32): the hardware block scaling of "How
 * Blackwell's Tensor Memory Actually Works", section "Quantization became an
 * allocation problem": D = C + (A x SFA)(B x SFB) with one scale factor per
 * group of 32 elements along K, for the MX formats an E8M0 byte, a bare
 * power-of-two exponent (the Open Compute microscaling specification the
 * page names).  Reading: E8M0 code e is 2^(e - 127), the microscaling
 * specification's bias, and 0xFF is NaN.  The products of one 32-wide block
 * are summed exactly (as above), multiplied by 2^(ea - 127) * 2^(eb - 127)
 * (exact: a power of two), and the blocks are added in K order.  The storage
 * of the scale bytes is the library's choice, tiles of 128 rows x 4 K blocks
 * of 512 bytes each (the order the tensor core's scale-factor copy reads):
 *     tile (r / 128, kb / 4) at byte offset ((r/128) * KT + kb/4) * 512,
 *     inside it (r % 32) * 16 + ((r / 32) % 4) * 4 + kb % 4,
 * with KT = ceil(ceil(K / 32) / 4), for A (r = i) and for B (r = j).
 *
 * Portable C11, no intrinsics; compiled with -ffp-contract=off so x86 and
 * Arm hosts round identically.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_IN_BF16 0
#define ORC_IN_E4M3 1
#define ORC_SCALE_NONE 0   /* BF16: no scales */
#define ORC_SCALE_TENSOR 1 /* one scale per operand */
#define ORC_SCALE_BLOCK128 2
#define ORC_SCALE_MX32 3   /* E8M0 per 32-wide K block of every row of A and B */
#define ORC_C_BF16 0
#define ORC_C_F32 1
#define ORC_FP8_E4M3 0
#define ORC_FP8_E5M2 1

/* ------------------------------------------------------------------ codecs */

/* BF16 bits -> value: the 16 bits are the high half of an FP32 word. */
double orc_bf16_decode(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* FP32 -> BF16 with round-to-nearest, ties to even, on the 16 dropped bits.
 * NaN stays a quiet NaN with its sign; overflow rounds to infinity. */
uint16_t orc_bf16_encode(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
    return (uint16_t)(((u >> 16) & 0x8000u) | 0x7FC0u);
  uint32_t dropped = u & 0xFFFFu;
  uint32_t kept = u >> 16;
  if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) kept += 1u;
  return (uint16_t)kept;
}

/* E4M3 bits -> value.  S.EEEE.MMM, bias 7; exponent field 0 is subnormal
 * (M/8 * 2^-6); S.1111.111 is NaN; there is no infinity. */
double orc_e4m3_decode(uint8_t b) {
  int s = (b >> 7) & 1;
  int e = (b >> 3) & 15;
  int m = b & 7;
  if (e == 15 && m == 7) return NAN;
  double mag = (e == 0) ? ldexp((double)m, -9)           /* (m/8) * 2^-6 */
                        : ldexp((double)(8 + m), e - 10); /* (1+m/8) * 2^(e-7) */
  return s ? -mag : mag;
}

/* FP32 -> E4M3, round to nearest even on the E4M3 grid, saturating: any
 * finite or infinite magnitude that rounds above 448 becomes +-448.  NaN ->
 * 0x7F (sign kept).  The rounding is done on integers (the FP32 significand
 * and exponent), with no floating-point arithmetic. */
uint8_t orc_e4m3_encode(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  uint8_t sign = (uint8_t)((u >> 24) & 0x80u);
  uint32_t a = u & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return (uint8_t)(sign | 0x7Fu);
  if (a == 0x7F800000u) return (uint8_t)(sign | 0x7Eu);
  int ef = (int)(a >> 23);
  if (ef == 0) return sign; /* FP32 zero or subnormal (< 2^-126): rounds to 0 */
  uint64_t sig = (uint64_t)((a & 0x7FFFFFu) | 0x800000u); /* value = sig * 2^(E-23) */
  int E = ef - 127;
  /* E4M3 quantum at this magnitude: 2^(E-3) for normals (E >= -6), else the
   * subnormal step 2^-9. */
  int q = (E >= -6) ? E - 3 : -9;
  int shift = 23 + q - E; /* bits of sig below the quantum, >= 20 */
  uint64_t r;             /* magnitude rounded, in units of 2^q */
  if (shift >= 40) {
    r = 0;
  } else {
    uint64_t keep = sig >> shift;
    uint64_t rem = sig & ((1ull << shift) - 1ull);
    uint64_t half = 1ull << (shift - 1);
    r = keep + ((rem > half || (rem == half && (keep & 1ull))) ? 1u : 0u);
  }
  /* Re-express r * 2^q as exponent field / mantissa.  r * 2^q with q = -9 and
   * r < 8 is a subnormal; otherwise normalise so the significand is 8..15. */
  if (q == -9 && r < 8) return (uint8_t)(sign | (uint8_t)r);
  int qq = q;
  while (r >= 16) { /* rounding carried into the next binade */
    r >>= 1;        /* r was even (a multiple of 16), exact */
    qq += 1;
  }
  /* value = r * 2^qq with 8 <= r <= 15, i.e. (1 + (r-8)/8) * 2^(qq+3) */
  int e_unb = qq + 3;
  int efield = e_unb + 7;
  if (efield > 15 || (efield == 15 && (r - 8) >= 7)) return (uint8_t)(sign | 0x7Eu);
  return (uint8_t)(sign | (uint8_t)(efield << 3) | (uint8_t)(r - 8));
}

/* E5M2 bits -> value.  S.EEEEE.MM, bias 15; exponent field 0 is subnormal
 * (M/4 * 2^-14); exponent field 31 is infinity (M = 0) or NaN (M != 0). */
double orc_e5m2_decode(uint8_t b) {
  int s = (b >> 7) & 1;
  int e = (b >> 2) & 31;
  int m = b & 3;
  double mag;
  if (e == 31) {
    if (m != 0) return NAN;
    mag = INFINITY;
  } else {
    mag = (e == 0) ? ldexp((double)m, -16)             /* (m/4) * 2^-14 */
                   : ldexp((double)(4 + m), e - 17);   /* (1+m/4) * 2^(e-15) */
  }
  return s ? -mag : mag;
}

/* FP32 -> E5M2, round to nearest even on the E5M2 grid (2 fraction bits;
 * subnormal step 2^-16 below 2^-14), saturating: a finite or infinite
 * magnitude that rounds above 57344 becomes +-57344 (0x7B).  NaN -> 0x7F
 * (sign kept).  Integer rounding on the FP32 significand, as for E4M3. */
uint8_t orc_e5m2_encode(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  uint8_t sign = (uint8_t)((u >> 24) & 0x80u);
  uint32_t a = u & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return (uint8_t)(sign | 0x7Fu);
  if (a == 0x7F800000u) return (uint8_t)(sign | 0x7Bu);
  int ef = (int)(a >> 23);
  if (ef == 0) return sign; /* below 2^-126: rounds to 0 */
  uint64_t sig = (uint64_t)((a & 0x7FFFFFu) | 0x800000u); /* value = sig * 2^(E-23) */
  int E = ef - 127;
  int q = (E >= -14) ? E - 2 : -16; /* E5M2 quantum at this magnitude */
  int shift = 23 + q - E;           /* >= 21 */
  uint64_t r;
  if (shift >= 40) {
    r = 0;
  } else {
    uint64_t keep = sig >> shift;
    uint64_t rem = sig & ((1ull << shift) - 1ull);
    uint64_t half = 1ull << (shift - 1);
    r = keep + ((rem > half || (rem == half && (keep & 1ull))) ? 1u : 0u);
  }
  if (q == -16 && r < 4) return (uint8_t)(sign | (uint8_t)r); /* subnormal r * 2^-16 */
  int qq = q;
  while (r >= 8) { /* carried into the next binade */
    r >>= 1;
    qq += 1;
  }
  /* value = r * 2^qq, 4 <= r <= 7, i.e. (1 + (r-4)/4) * 2^(qq+2) */
  int efield = qq + 2 + 15;
  if (efield > 30) return (uint8_t)(sign | 0x7Bu);
  return (uint8_t)(sign | (uint8_t)(efield << 2) | (uint8_t)(r - 4));
}

/* E8M0 bits -> value: 2^(e - 127); the code 0xFF is NaN.  No sign, no
 * mantissa, no zero. */
double orc_e8m0_decode(uint8_t e) {
  if (e == 0xFFu) return NAN;
  return ldexp(1.0, (int)e - 127);
}

void orc_e8m0_decode_array(const uint8_t* in, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e8m0_decode(in[i]);
}

/* Byte offset of the scale of row r, 32-wide K block kb in the tiled MX
 * scale layout (header comment), kt = ceil(ceil(K/32) / 4) tiles along K. */
int64_t orc_mx_sf_offset(int64_t r, int64_t kb, int64_t kt) {
  const int64_t tile = (r / 128) * kt + kb / 4;
  return tile * 512 + (r % 32) * 16 + ((r / 32) % 4) * 4 + kb % 4;
}

void orc_e5m2_encode_array(const float* in, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e5m2_encode(in[i]);
}

void orc_e5m2_decode_array(const uint8_t* in, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e5m2_decode(in[i]);
}

void orc_bf16_decode_array(const uint16_t* in, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_decode(in[i]);
}
void orc_bf16_encode_array(const float* in, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_encode(in[i]);
}
void orc_e4m3_decode_array(const uint8_t* in, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_decode(in[i]);
}
void orc_e4m3_encode_array(const float* in, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(in[i]);
}

/* The BF16 output the library is expected to store for an FP64 value v:
 * v rounded to FP32, then to BF16 with ties to even. */
void orc_cast_bf16_array(const double* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_encode((float)v[i]);
}

/* -------------------------------------------------------------------- GEMM */

typedef struct {
  int64_t M, N, K;
  int32_t in_type;    /* ORC_IN_BF16 / ORC_IN_E4M3 */
  int32_t scale_mode; /* ORC_SCALE_* */
  const void* A;
  int64_t lda;
  const void* B;
  int64_t ldb;
  const float* a_scale;
  const float* b_scale;
  const void* C; /* may be NULL when beta == 0 */
  int64_t ldc;
  int32_t c_type; /* ORC_C_BF16 / ORC_C_F32 */
  int32_t pad_;
  double alpha, beta;
  int32_t a_fp8, b_fp8; /* FP8 inputs: ORC_FP8_E4M3 / ORC_FP8_E5M2 per operand */
  const uint8_t* a_sf;  /* ORC_SCALE_MX32: E8M0 scales of A and B, tiled layout */
  const uint8_t* b_sf;
} orc_gemm_args;

static double dec_in(const orc_gemm_args* g, const void* base, int64_t idx, int32_t fp8) {
  if (g->in_type == ORC_IN_BF16) return orc_bf16_decode(((const uint16_t*)base)[idx]);
  uint8_t b = ((const uint8_t*)base)[idx];
  return fp8 == ORC_FP8_E5M2 ? orc_e5m2_decode(b) : orc_e4m3_decode(b);
}

static double dec_c(const orc_gemm_args* g, int64_t i, int64_t j) {
  int64_t idx = i * g->ldc + j;
  if (g->c_type == ORC_C_BF16) return orc_bf16_decode(((const uint16_t*)g->C)[idx]);
  return (double)((const float*)g->C)[idx];
}

/* One output element.  Sums run over k in ascending order. */
static void gemm_one(const orc_gemm_args* g, const double* arow, const double* brow, int64_t i,
                     int64_t j, double* v_out, double* bound_out) {
  const int64_t K = g->K;
  double acc = 0.0, bound = 0.0;
  if (g->scale_mode == ORC_SCALE_MX32) {
    const int64_t KB = (K + 31) / 32, KT = (KB + 3) / 4;
    for (int64_t kb = 0; kb < KB; ++kb) {
      double part = 0.0, apart = 0.0;
      int64_t k1 = (kb + 1) * 32 < K ? (kb + 1) * 32 : K;
      for (int64_t k = kb * 32; k < k1; ++k) {
        double p = arow[k] * brow[k];
        part += p;
        apart += fabs(p);
      }
      double s = orc_e8m0_decode(g->a_sf[orc_mx_sf_offset(i, kb, KT)]) *
                 orc_e8m0_decode(g->b_sf[orc_mx_sf_offset(j, kb, KT)]);
      acc += part * s;
      bound += apart * s;
    }
  } else if (g->scale_mode == ORC_SCALE_BLOCK128) {
    const int64_t KB = (K + 127) / 128;
    const int64_t nb = j / 128;
    for (int64_t kb = 0; kb < KB; ++kb) {
      double part = 0.0, apart = 0.0;
      int64_t k1 = (kb + 1) * 128 < K ? (kb + 1) * 128 : K;
      for (int64_t k = kb * 128; k < k1; ++k) {
        double p = arow[k] * brow[k];
        part += p;
        apart += fabs(p);
      }
      double s = (double)g->a_scale[kb * g->M + i] * (double)g->b_scale[nb * KB + kb];
      acc += part * s;
      bound += apart * fabs(s);
    }
  } else {
    for (int64_t k = 0; k < K; ++k) {
      double p = arow[k] * brow[k];
      acc += p;
      bound += fabs(p);
    }
    if (g->scale_mode == ORC_SCALE_TENSOR) {
      double s = (double)g->a_scale[0] * (double)g->b_scale[0];
      acc *= s;
      bound *= fabs(s);
    }
  }
  double v = g->alpha * acc;
  if (g->beta != 0.0) v += g->beta * dec_c(g, i, j);
  *v_out = v;
  *bound_out = fabs(g->alpha) * bound;
}

/* One rectangular block of outputs: rows i0..i0+mi-1, columns j0..j0+nj-1,
 * written row-major into v[mi*nj] and bound[mi*nj]. */
static int gemm_tile(const orc_gemm_args* g, int64_t i0, int64_t j0, int64_t mi, int64_t nj,
                     double* v, double* bound) {
  const int64_t K = g->K;
  double* arows = (double*)malloc((size_t)(mi * (K > 0 ? K : 1)) * sizeof(double));
  double* brows = (double*)malloc((size_t)(nj * (K > 0 ? K : 1)) * sizeof(double));
  if (!arows || !brows) {
    free(arows);
    free(brows);
    return -1;
  }
  for (int64_t r = 0; r < mi; ++r)
    for (int64_t k = 0; k < K; ++k)
      arows[r * K + k] = dec_in(g, g->A, (i0 + r) * g->lda + k, g->a_fp8);
  for (int64_t c = 0; c < nj; ++c)
    for (int64_t k = 0; k < K; ++k)
      brows[c * K + k] = dec_in(g, g->B, (j0 + c) * g->ldb + k, g->b_fp8);
  for (int64_t r = 0; r < mi; ++r)
    for (int64_t c = 0; c < nj; ++c)
      gemm_one(g, arows + r * K, brows + c * K, i0 + r, j0 + c, &v[r * nj + c], &bound[r * nj + c]);
  free(arows);
  free(brows);
  return 0;
}

typedef struct {
  const orc_gemm_args* g;
  const int64_t* tiles; /* [n][4]: i0, j0, mi, nj */
  const int64_t* offs;  /* output offset of each tile */
  int64_t ntiles;
  int64_t next; /* next tile index to take (guarded by mu) */
  pthread_mutex_t mu;
  double* v;
  double* bound;
  int err;
} work_t;

static void* worker(void* p) {
  work_t* w = (work_t*)p;
  for (;;) {
    pthread_mutex_lock(&w->mu);
    int64_t t = w->next++;
    pthread_mutex_unlock(&w->mu);
    if (t >= w->ntiles) break;
    const int64_t* d = w->tiles + 4 * t;
    if (gemm_tile(w->g, d[0], d[1], d[2], d[3], w->v + w->offs[t], w->bound + w->offs[t]) != 0) {
      pthread_mutex_lock(&w->mu);
      w->err = -1;
      pthread_mutex_unlock(&w->mu);
    }
  }
  return NULL;
}

/* Compute a list of output tiles.  tiles[4*t .. 4*t+3] = (i0, j0, mi, nj);
 * tile t's values land row-major at v + sum_{u<t} mi_u * nj_u (same for
 * bound).  Tiles are taken by `nthreads` worker threads; each tile is
 * computed by one thread, so the result does not depend on nthreads.
 * Returns 0, or -1 on a bad argument or allocation failure. */
int orc_gemm_tiles(const orc_gemm_args* g, int64_t ntiles, const int64_t* tiles, double* v,
                   double* bound, int nthreads) {
  if (!g || ntiles < 0 || (ntiles > 0 && (!tiles || !v || !bound))) return -1;
  if (g->M < 0 || g->N < 0 || g->K < 0) return -1;
  if (g->K > 0 && (!g->A || !g->B)) return -1;
  if (g->beta != 0.0 && !g->C) return -1;
  if ((g->scale_mode == ORC_SCALE_TENSOR || g->scale_mode == ORC_SCALE_BLOCK128) &&
      (!g->a_scale || !g->b_scale))
    return -1;
  if (g->scale_mode == ORC_SCALE_MX32 && (!g->a_sf || !g->b_sf)) return -1;
  if (g->scale_mode < ORC_SCALE_NONE || g->scale_mode > ORC_SCALE_MX32) return -1;
  int64_t* offs = (int64_t*)malloc((size_t)(ntiles > 0 ? ntiles : 1) * sizeof(int64_t));
  if (!offs) return -1;
  int64_t o = 0;
  for (int64_t t = 0; t < ntiles; ++t) {
    const int64_t* d = tiles + 4 * t;
    if (d[0] < 0 || d[1] < 0 || d[2] < 0 || d[3] < 0 || d[0] + d[2] > g->M || d[1] + d[3] > g->N) {
      free(offs);
      return -1;
    }
    offs[t] = o;
    o += d[2] * d[3];
  }
  work_t w;
  w.g = g;
  w.tiles = tiles;
  w.offs = offs;
  w.ntiles = ntiles;
  w.next = 0;
  w.v = v;
  w.bound = bound;
  w.err = 0;
  pthread_mutex_init(&w.mu, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&th[started], NULL, worker, &w) == 0) ++started;
  }
  worker(&w);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  pthread_mutex_destroy(&w.mu);
  free(offs);
  return w.err;
}

/* --------------------------------------------------------------- quantiser */

/* FP8 E4M3 quantisation of a rows x cols matrix X ("Tensor cores and low
 * precision", FP8 paragraph: rescale so that the largest magnitudes land at
 * the format's maximum, 448, then cast; the scale is removed again after the
 * product; "Tensor Cores", "Precision: FP16, BF16, TF32, FP8": the scaling
 * factors are per tensor, per row or per block).  Written as the library stores it: the
 * stored (dequantisation) scale is s = amax / 448 and each code is
 * E4M3(x / s), i.e. the same as multiplying by 448 / amax up to the rounding
 * of that factor.
 *
 * E5M2 (fmt 1) is the same with 57344, E5M2's maximum normal value, in place
 * of 448 and the E5M2 encoder (orc_e5m2_encode).
 *
 * Readings (the pages give the recipe, not these details):
 *  - amax is the largest |x| over the block, NaN entries ignored;
 *  - s = amax / 448 in FP32 (correctly rounded division); a block whose s is
 *    0 (all zeros, or so small that the division underflows) takes s = 1, so
 *    that no code divides by zero;
 *  - each code is the FP32 quotient x / s (correctly rounded) encoded to E4M3
 *    with nearest-even rounding, saturating at +-448 (orc_e4m3_encode); a NaN
 *    quotient is stored as the canonical NaN code 0x7F.
 *
 * Block geometries (mode), matching the GEMM's scale layouts:
 *  ORC_Q_TENSOR    one block, the whole matrix; scale[0]
 *  ORC_Q_ROW128    1 x 128: row r, columns 128kb..128kb+127; scale[kb*rows + r]
 *  ORC_Q_BLOCK128  128 x 128: rows 128rb.., columns 128kb..;
 *                  scale[rb*ceil(cols/128) + kb]
 * A partial last block (cols or rows not a multiple of 128) uses its own
 * amax.  X is FP32 (x_type 0) or BF16 bit patterns (x_type 1), element (r, c)
 * at X[r*ldx + c]; Q holds one byte per element at Q[r*ldq + c]; bytes of Q
 * beyond column cols are not written.  Returns 0, or -1 on a bad argument. */
#define ORC_Q_TENSOR 0
#define ORC_Q_ROW128 1
#define ORC_Q_BLOCK128 2

static float quant_in(const void* X, int32_t x_type, int64_t idx) {
  if (x_type == 0) return ((const float*)X)[idx];
  return (float)orc_bf16_decode(((const uint16_t*)X)[idx]); /* exact: BF16 is FP32's top half */
}

/* Quantise the block rows r0..r1-1 x columns c0..c1-1 to E4M3 (fmt 0, top
 * 448) or E5M2 (fmt 1, top 57344); returns its scale. */
static float quant_block(const void* X, int32_t x_type, int64_t ldx, int64_t r0, int64_t r1,
                         int64_t c0, int64_t c1, uint8_t* Q, int64_t ldq, int32_t fmt) {
  float amax = 0.0f;
  for (int64_t r = r0; r < r1; ++r)
    for (int64_t c = c0; c < c1; ++c) {
      float a = fabsf(quant_in(X, x_type, r * ldx + c));
      if (a > amax) amax = a; /* false for NaN: NaN entries are skipped */
    }
  float s = amax / (fmt == ORC_FP8_E5M2 ? 57344.0f : 448.0f);
  if (s == 0.0f) s = 1.0f;
  for (int64_t r = r0; r < r1; ++r)
    for (int64_t c = c0; c < c1; ++c) {
      float y = quant_in(X, x_type, r * ldx + c) / s;
      Q[r * ldq + c] = (y != y)                ? (uint8_t)0x7Fu
                       : (fmt == ORC_FP8_E5M2) ? orc_e5m2_encode(y)
                                               : orc_e4m3_encode(y);
    }
  return s;
}

int orc_quant_fp8(const void* X, int32_t x_type, int64_t rows, int64_t cols, int64_t ldx,
                  int32_t mode, int32_t fmt, uint8_t* Q, int64_t ldq, float* scale) {
  if (rows < 0 || cols < 0 || (x_type != 0 && x_type != 1) || !scale) return -1;
  if (fmt != ORC_FP8_E4M3 && fmt != ORC_FP8_E5M2) return -1;
  if (rows > 0 && cols > 0 && (!X || !Q || ldx < cols || ldq < cols)) return -1;
  const int64_t KB = (cols + 127) / 128, RB = (rows + 127) / 128;
  if (mode == ORC_Q_TENSOR) {
    scale[0] = quant_block(X, x_type, ldx, 0, rows, 0, cols, Q, ldq, fmt);
  } else if (mode == ORC_Q_ROW128) {
    for (int64_t r = 0; r < rows; ++r)
      for (int64_t kb = 0; kb < KB; ++kb) {
        int64_t c1 = (kb + 1) * 128 < cols ? (kb + 1) * 128 : cols;
        scale[kb * rows + r] = quant_block(X, x_type, ldx, r, r + 1, kb * 128, c1, Q, ldq, fmt);
      }
  } else if (mode == ORC_Q_BLOCK128) {
    for (int64_t rb = 0; rb < RB; ++rb)
      for (int64_t kb = 0; kb < KB; ++kb) {
        int64_t r1 = (rb + 1) * 128 < rows ? (rb + 1) * 128 : rows;
        int64_t c1 = (kb + 1) * 128 < cols ? (kb + 1) * 128 : cols;
        scale[rb * KB + kb] =
            quant_block(X, x_type, ldx, rb * 128, r1, kb * 128, c1, Q, ldq, fmt);
      }
  } else {
    return -1;
  }
  return 0;
}

/* The E4M3 quantiser (fmt 0) under its original name. */
int orc_quant_e4m3(const void* X, int32_t x_type, int64_t rows, int64_t cols, int64_t ldx,
                   int32_t mode, uint8_t* Q, int64_t ldq, float* scale) {
  return orc_quant_fp8(X, x_type, rows, cols, ldx, mode, ORC_FP8_E4M3, Q, ldq, scale);
}
