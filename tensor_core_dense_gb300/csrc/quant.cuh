// quant.cuh -- FP8 quantiser kernels, E4M3 and E5M2 (the C ABI entry points
// quantize_fp8 / quantize_e4m3 and their launch are in tcgemm.cu).
//
// The FP8 recipe of "Tensor cores and low precision" (FP8 paragraph): a
// tensor is rescaled so that its largest magnitudes land at E4M3's maximum
// normal value, 448, then cast; the scale is removed after the product.
// "Tensor Cores" ("Precision: FP16, BF16, TF32, FP8") names the granularities:
// per tensor, per row, per block.  The stored (dequantisation) scale of a
// block is s = amax / top and each code is FP8(x / s) -- the FP32 quotient,
// rounded to nearest even on the format's grid, saturating at +-top -- with
// top = 448 for E4M3 and 57344 for E5M2 (the two encodings' largest normal
// values, same page): exactly the codes and scales gemm_fp8 consumes.
//
// The work is a stream over X (read once, twice for one scale per tensor)
// and Q (written once): HBM-bound, no tensor cores.  A persistent CTA per SM:
// one producer lane moves 64-row x 128-column boxes of X into a 192 KB
// shared-memory ring with TMA (out-of-range elements arrive as zeros, which no
// block maximum can exceed), and sixteen consumer warps take each box out of
// shared memory (warp w: rows 4w..4w+3; lane l: columns 4l..4l+3), so HBM
// stays busy while they reduce, divide and store.  Units of work:
//   BLOCK128  a 128 x 128 block = 2 boxes; CTA-wide maximum, then codes
//   ROW128    one box; each row is its own 1 x 128 block (warp-wide maximum)
//   TENSOR    two launches over boxes: the maxima, folded into scale[0] with
//             an integer atomicMax (bit patterns of non-negative floats order
//             like the floats, and rounding a quotient by the top is monotone, so
//             the largest per-CTA s is s of the global maximum); then codes.
//
// Division.  Each code needs RN(x / s), the correctly rounded FP32 quotient.
// Per block, r = RN(1/s) (one IEEE division) and its remainder term
// r' = RN(RN(1 - s*r) * r) make r + r' = (1/s)(1 + O(2^-46)); per element,
// q0 = RN(x*r + RN(x*r')) is then within one unit in the last place of x / s
// (faithful), and Markstein's correction (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990: if r is RN(1/s) and q0 a faithful approximation of x / s,
// the remainder x - s*q0 is exact in an FMA and RN(q0 + (x - s*q0)*r) is
// RN(x / s)) finishes it: four FMA-pipe instructions instead of a division.
// The premises need no underflow in the remainder, so blocks whose s lies
// outside [2^-60, 2^60] (an infinite maximum, or one below ~2^-51) use the
// IEEE division __fdiv_rn for every element instead.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "gemm_tn.cuh"  // wait_phase, record_timeout, kWaitLimitNs
#include "ptx.cuh"

namespace tcg {

constexpr int kQConsumerWarps = 16;
constexpr int kQThreads = 32 * (kQConsumerWarps + 1);  // + one producer warp
constexpr int kQBoxRows = 64;
constexpr int kQBoxCols = 128;
constexpr int kQRowsPerWarp = kQBoxRows / kQConsumerWarps;  // 4
constexpr int kQBoxesPerBlock = 128 / kQBoxRows;             // boxes of one 128 x 128 block
constexpr uint32_t kQRingBytes = 192u * 1024u;
constexpr uint32_t kQSmemBytes = kQRingBytes + 1024u /*barriers, slots*/ + 1024u /*align*/;

enum QuantKind { kQuantBlock = 0, kQuantAmax = 1, kQuantEncode = 2, kQuantRow = 3 };

struct QuantParams {
  uint8_t* Q;
  float* scale;
  int64_t ldq;
  int32_t rows, cols;
  int32_t KB;     // column blocks: ceil(cols / 128)
  int32_t units;  // BLOCK: ceil(rows/128) * KB; otherwise ceil(rows/kQBoxRows) * KB
};

// Unit u -> first row, first column and number of boxes.
template <int kKind>
__device__ __forceinline__ void quant_unit(const QuantParams& p, int u, int& r0, int& c0,
                                           int& nbox) {
  const int kb = u % p.KB;
  c0 = kb * kQBoxCols;
  if (kKind == kQuantBlock) {
    r0 = (u / p.KB) * 128;
    nbox = min(kQBoxesPerBlock, (p.rows - r0 + kQBoxRows - 1) / kQBoxRows);
  } else {
    r0 = (u / p.KB) * kQBoxRows;
    nbox = 1;
  }
}

__device__ __forceinline__ float abs_max4(const float (&v)[4]) {
  // fmaxf returns the other operand when one is NaN: NaN entries are skipped
  return fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
}

__device__ __forceinline__ float warp_max(float m) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  return m;
}

// Largest normal value of the FP8 format: E4M3 (kFmt 0) 448, E5M2 (1) 57344.
template <int kFmt>
__device__ __forceinline__ constexpr float quant_top() { return kFmt == 0 ? 448.0f : 57344.0f; }

// Dequantisation scale for a block maximum; a zero quotient (all-zero block,
// or underflow) becomes 1.
template <int kFmt>
__device__ __forceinline__ float quant_scale_of(float amax) {
  const float s = __fdiv_rn(amax, quant_top<kFmt>());
  return s == 0.0f ? 1.0f : s;
}

// Per-block constants of the encoder: s, r = RN(1/s), r' (the remainder term
// of the reciprocal), and whether the block needs the IEEE division.
struct QuantDiv {
  float s, r, r2;
  bool exact;
};

__device__ __forceinline__ QuantDiv quant_div(float s) {
  QuantDiv d;
  d.s = s;
  d.exact = !(s >= 0x1p-60f && s <= 0x1p60f);
  d.r = d.exact ? 1.0f : __fdiv_rn(1.0f, s);
  d.r2 = d.exact ? 0.0f : __fmul_rn(__fmaf_rn(-s, d.r, 1.0f), d.r);
  return d;
}

// RN(x / s) for two elements of a block whose s passed quant_div's range
// test: q0 = RN(x*r + RN(x*r')) (faithful), e = x - s*q0 (exact), q1 =
// RN(q0 + e*r) (correctly rounded), each step one packed f32x2 operation
// that rounds every lane exactly as the scalar instruction would.
__device__ __forceinline__ void quant_quotient2(float x0, float x1, const QuantDiv& d, float& y0,
                                                float& y1) {
  const uint64_t x = pack_f32x2(x0, x1);
  const uint64_t r = pack_f32x2(d.r, d.r), r2 = pack_f32x2(d.r2, d.r2);
  const uint64_t ns = pack_f32x2(-d.s, -d.s);
  uint64_t p, q0, e, q1;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(p) : "l"(x), "l"(r2));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q0) : "l"(x), "l"(r), "l"(p));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(e) : "l"(q0), "l"(ns), "l"(x));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q1) : "l"(e), "l"(r), "l"(q0));
  float a, b;
  unpack_f32x2(q1, a, b);
  // the quotient has x's sign (s > 0); this also keeps -0 for x = -0
  y0 = __uint_as_float((__float_as_uint(a) & 0x7FFFFFFFu) | (__float_as_uint(x0) & 0x80000000u));
  y1 = __uint_as_float((__float_as_uint(b) & 0x7FFFFFFFu) | (__float_as_uint(x1) & 0x80000000u));
}

// Four codes FP8(x / s), packed little-endian (first element in the low
// byte).  cvt.rn.satfinite rounds to nearest even, clamps finite overflow and
// infinities to the largest normal value and turns a NaN of either sign into
// the canonical 0x7F (checked on GB300 for +-NaN, +-inf, +-0, subnormal ties
// and the overflow midpoint, both formats).
template <int kFmt>
__device__ __forceinline__ uint32_t quant_encode4(const float (&v)[4], const QuantDiv& d) {
  float y[4];
  if (d.exact) {
#pragma unroll
    for (int e = 0; e < 4; ++e) y[e] = __fdiv_rn(v[e], d.s);
  } else {
    quant_quotient2(v[0], v[1], d, y[0], y[1]);
    quant_quotient2(v[2], v[3], d, y[2], y[3]);
  }
  uint16_t lo, hi;
  if (kFmt == 0) {
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(y[1]), "f"(y[0]));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(y[3]), "f"(y[2]));
  } else {
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(y[1]), "f"(y[0]));
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(y[3]), "f"(y[2]));
  }
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// Stores one row's four codes at columns c..c+3 (those < cols); `full`
// (the whole unit lies inside the matrix) skips the checks.
__device__ __forceinline__ void quant_store4(const QuantParams& p, int r, int c, uint32_t w,
                                             bool full) {
  if (full) {
    *reinterpret_cast<uint32_t*>(p.Q + (int64_t)r * p.ldq + c) = w;
    return;
  }
  if (r >= p.rows || c >= p.cols) return;
  uint8_t* q = p.Q + (int64_t)r * p.ldq + c;
  if (c + 3 < p.cols) {
    *reinterpret_cast<uint32_t*>(q) = w;
  } else {
    for (int e = 0; c + e < p.cols; ++e) q[e] = (uint8_t)(w >> (8 * e));
  }
}

// One box row (this lane's four values) from shared memory.
template <int kIn>
__device__ __forceinline__ void quant_read4(const uint8_t* stage, int row, int lane,
                                            float (&v)[4]) {
  if (kIn == 0) {
    const float4 t = *reinterpret_cast<const float4*>(stage + row * 512 + lane * 16);
    v[0] = t.x;
    v[1] = t.y;
    v[2] = t.z;
    v[3] = t.w;
  } else {
    const uint2 t = *reinterpret_cast<const uint2*>(stage + row * 256 + lane * 8);
    v[0] = __uint_as_float(t.x << 16);
    v[1] = __uint_as_float(t.x & 0xFFFF0000u);
    v[2] = __uint_as_float(t.y << 16);
    v[3] = __uint_as_float(t.y & 0xFFFF0000u);
  }
}

// Bounded wait by every lane of a warp; true only if all lanes saw the phase.
__device__ __forceinline__ bool quant_warp_wait(uint32_t bar, uint32_t parity,
                                                volatile int* abort_flag, uint32_t where) {
  const bool ok = wait_phase(bar, parity, abort_flag, where);
  return __all_sync(0xFFFFFFFFu, ok);
}

template <int kIn, int kKind, int kFmt>
__global__ void __launch_bounds__(kQThreads, 1)
    quant_fp8_kernel(const __grid_constant__ CUtensorMap tmap, const QuantParams p) {
  constexpr uint32_t kStageBytes = kQBoxRows * kQBoxCols * (kIn == 0 ? 4u : 2u);
  constexpr int S = (int)(kQRingBytes / kStageBytes);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kQRingBytes);
  // bars[0..S): full, [S..2S): empty, [2S]: reduction
  float* slots = reinterpret_cast<float*>(bars + 2 * S + 1);  // [2][kQConsumerWarps]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(slots + 2 * kQConsumerWarps);
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + S + s); };
  const uint32_t red_bar = smem_u32(bars + 2 * S);

  const int warp = (int)(threadIdx.x >> 5);
  const int lane = (int)(threadIdx.x & 31u);
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kQConsumerWarps);
    }
    mbar_init(red_bar, kQConsumerWarps);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // the codes pass may start loading while the maxima pass drains: X is not
  // written by it (only scale[0] is, read after the dependency wait)
  if (kKind == kQuantAmax) grid_launch_dependents();
  // Row and block quantisation are launched to overlap the previous kernel's
  // tail (programmatic dependent launch): X, Q and the scales are touched
  // only after it has finished.
  if (kKind == kQuantRow || kKind == kQuantBlock) {
    grid_dependency_wait();
    grid_launch_dependents();
  }

  if (warp == kQConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmap);
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
        int r0, c0, nbox;
        quant_unit<kKind>(p, u, r0, c0, nbox);
        for (int j = 0; j < nbox; ++j, ++it) {
          const int s = (int)(it % S);
          const uint32_t ph = (it / S) & 1u;
          if (!wait_phase(empty_bar(s), ph ^ 1u, abort_flag, 0x41)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(s), kStageBytes);
          tma_load_2d(smem_u32(smem + (uint32_t)s * kStageBytes), &tmap, full_bar(s), c0,
                      r0 + j * kQBoxRows);
        }
      }
      if (!ok) {
        // after an abort, wait (bounded) for the copies still in flight
        const uint32_t first = it > (uint32_t)S ? it - (uint32_t)S : 0u;
        for (uint32_t k = first; k < it; ++k) {
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(full_bar((int)(k % S)), (k / S) & 1u) &&
                 global_timer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    uint32_t it = 0, nunit = 0;
    bool ok = true;
    float run_max = 0.0f;  // maxima pass: this lane's running maximum
    QuantDiv tensor_div{1.0f, 1.0f, false};
    if (kKind == kQuantEncode) {
      grid_dependency_wait();  // scale[0] holds the folded maximum from here on
      const float folded = *reinterpret_cast<volatile const float*>(p.scale);
      // An all-zero tensor left 0 in scale[0]; its scale is 1.  Readers that
      // see either value use 1, so one CTA may overwrite it.
      if (blockIdx.x == 0 && threadIdx.x == 0 && folded == 0.0f) p.scale[0] = 1.0f;
      tensor_div = quant_div(folded == 0.0f ? 1.0f : folded);
    }
    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x, ++nunit) {
      int r0, c0, nbox;
      quant_unit<kKind>(p, u, r0, c0, nbox);
      const int c = c0 + 4 * lane;
      const bool full = r0 + nbox * kQBoxRows <= p.rows && c0 + kQBoxCols <= p.cols &&
                        (kKind != kQuantBlock || nbox == kQBoxesPerBlock);
      if (kKind == kQuantBlock) {
        float v[kQBoxesPerBlock * kQRowsPerWarp][4];
        for (int j = 0; j < kQBoxesPerBlock; ++j) {
          if (j < nbox) {
            const int s = (int)(it % S);
            if (!quant_warp_wait(full_bar(s), (it / S) & 1u, abort_flag, 0x42)) {
              ok = false;
              break;
            }
            const uint8_t* st = smem + (uint32_t)s * kStageBytes;
#pragma unroll
            for (int i = 0; i < kQRowsPerWarp; ++i)
              quant_read4<kIn>(st, warp * kQRowsPerWarp + i, lane, v[j * kQRowsPerWarp + i]);
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(s));
            ++it;
          } else {
#pragma unroll
            for (int i = 0; i < kQRowsPerWarp; ++i)
              v[j * kQRowsPerWarp + i][0] = v[j * kQRowsPerWarp + i][1] =
                  v[j * kQRowsPerWarp + i][2] = v[j * kQRowsPerWarp + i][3] = 0.0f;
          }
        }
        if (!ok) break;
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < kQBoxesPerBlock * kQRowsPerWarp; ++i) m = fmaxf(m, abs_max4(v[i]));
        m = warp_max(m);
        const uint32_t par = nunit & 1u;
        if (lane == 0) {
          slots[par * kQConsumerWarps + warp] = m;
          mbar_arrive(red_bar);
        }
        if (!quant_warp_wait(red_bar, par, abort_flag, 0x43)) {
          ok = false;
          break;
        }
        m = slots[par * kQConsumerWarps];
#pragma unroll
        for (int w = 1; w < kQConsumerWarps; ++w) m = fmaxf(m, slots[par * kQConsumerWarps + w]);
        const QuantDiv d = quant_div(quant_scale_of<kFmt>(m));
        if (threadIdx.x == 0) p.scale[u] = d.s;  // u = rb * KB + kb
#pragma unroll
        for (int j = 0; j < kQBoxesPerBlock; ++j)
#pragma unroll
          for (int i = 0; i < kQRowsPerWarp; ++i)
            quant_store4(p, r0 + j * kQBoxRows + warp * kQRowsPerWarp + i, c,
                         quant_encode4<kFmt>(v[j * kQRowsPerWarp + i], d), full);
      } else {
        const int s = (int)(it % S);
        if (!quant_warp_wait(full_bar(s), (it / S) & 1u, abort_flag, 0x44)) {
          ok = false;
          break;
        }
        const uint8_t* st = smem + (uint32_t)s * kStageBytes;
        float v[kQRowsPerWarp][4];
#pragma unroll
        for (int i = 0; i < kQRowsPerWarp; ++i)
          quant_read4<kIn>(st, warp * kQRowsPerWarp + i, lane, v[i]);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(s));
        ++it;
        const int rw = r0 + warp * kQRowsPerWarp;  // this warp's first row
        if (kKind == kQuantAmax) {
#pragma unroll
          for (int i = 0; i < kQRowsPerWarp; ++i) run_max = fmaxf(run_max, abs_max4(v[i]));
        } else if (kKind == kQuantEncode) {
#pragma unroll
          for (int i = 0; i < kQRowsPerWarp; ++i)
            quant_store4(p, rw + i, c, quant_encode4<kFmt>(v[i], tensor_div), full);
        } else {  // ROW128: every row is a block
          float my_scale = 1.0f;
#pragma unroll
          for (int i = 0; i < kQRowsPerWarp; ++i) {
            const QuantDiv d = quant_div(quant_scale_of<kFmt>(warp_max(abs_max4(v[i]))));
            if (lane == i) my_scale = d.s;
            quant_store4(p, rw + i, c, quant_encode4<kFmt>(v[i], d), full);
          }
          if (lane < kQRowsPerWarp && rw + lane < p.rows)
            p.scale[(int64_t)(u % p.KB) * p.rows + rw + lane] = my_scale;
        }
      }
    }
    if (kKind == kQuantAmax && ok) {
      const float m = warp_max(run_max);
      if (lane == 0) {
        slots[warp] = m;
        mbar_arrive(red_bar);
      }
      if (quant_warp_wait(red_bar, 0, abort_flag, 0x45) && threadIdx.x == 0) {
        float t = slots[0];
        for (int w = 1; w < kQConsumerWarps; ++w) t = fmaxf(t, slots[w]);
        // 0 for an all-zero tensor; the codes pass turns a final 0 into 1
        atomicMax(reinterpret_cast<unsigned int*>(p.scale),
                  __float_as_uint(__fdiv_rn(t, quant_top<kFmt>())));
      }
    }
  }
  __syncwarp();
  __syncthreads();
}

// scale[0] = 1: the per-tensor scale of an empty matrix (its maximum is 0).
__global__ void quant_scale_one_kernel(float* scale) { scale[0] = 1.0f; }

}  // namespace tcg
