// gemm_skinny.cuh -- FP8 E4M3 GEMM with 128-block scales for skinny M (<= 128).
//
//   D[m, n] = alpha * sum_kb sa[kb*M + m] * sb[(n/128)*KB + kb]
//                    * sum_{k in block kb} qa[m, k] * qb[n, k]   (+ beta * C)
//
// The scale granularity is DeepSeek-style fine-grained block scaling ("Tensor
// Cores", "Precision: FP16, BF16, TF32, FP8": FP8 GEMMs need per-tensor,
// per-row or per-block scale factors) with 1 x 128 blocks for the activation
// A and 128 x 128 blocks for the weight B.  A scale that changes every 128
// values of K forces each K block to be summed on its own and promoted into
// an FP32 accumulator, the periodic promotion of "Tensor Cores: Matrix
// Instructions, Swizzling and FP8, Measured", Step 5.
//
// Skinny M (a decode-sized batch) cannot fill UMMA's M >= 64 rows ("How
// Blackwell's Tensor Memory Actually Works", "What this does to serving
// economics"), so the kernel swaps the operands: the tensor core computes
// the 128 x Mp tile of D^T = B * A^T, with a 128-row slab of B as UMMA A and
// the M (padded to Mp, zero-filled by TMA) rows of A as UMMA B.  The work is
// the sequence of (N tile, K block) steps, split into one contiguous range
// per CTA (stream-K), which spreads the B stream (the HBM-bound part) evenly
// over all SMs.  A tile whose K range is split over several CTAs is finished
// through a global FP32 workspace: each CTA writes its partial sums to its
// slot, bumps the tile's counter, and the last one to arrive adds the slots
// in slot order (deterministic) and writes D.
//
// Roles (10 warps): warp 0 TMA producer (one lane), warp 1 TMEM allocator +
// MMA issuer (one lane), warps 2-9 two epilogue warpgroups; warpgroup h
// promotes columns [h*Mp/2, (h+1)*Mp/2) of every partial.  The MMA writes
// each K block's partial into one of four TMEM buffers; the epilogue drains
// it, multiplies by sa*sb and adds it into registers.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "gemm_tn.cuh"
#include "ptx.cuh"

namespace tcg {

constexpr int kSkThreads = 320;
constexpr int kSkNumAcc = 4;                  // TMEM partial buffers
constexpr uint32_t kSkBTileBytes = 128 * 128; // 128 rows of B x 128 K bytes
constexpr int kSkEpiThreads = 256;

template <int kMp>
struct SkinnyCfg {
  static constexpr uint32_t kATileBytes = kMp * 128;
  static constexpr uint32_t kStageBytes = kSkBTileBytes + kATileBytes;
  static constexpr int kStagesRaw = (int)((196u * 1024u) / kStageBytes);
  static constexpr int kStages = kStagesRaw > 10 ? 10 : kStagesRaw;
  static constexpr int kCols = kMp * kSkNumAcc;
  static constexpr int kTmemCols = kCols <= 32 ? 32 : kCols <= 64 ? 64 : kCols <= 128 ? 128
                                   : kCols <= 256 ? 256 : 512;
  static constexpr int kHalf = kMp / 2;  // columns per epilogue warpgroup
  static constexpr int kNumBars = 2 * kStages + 2 * kSkNumAcc + 3;
  static constexpr uint32_t kScaleBytes = 8u * kHalf * 4u;
  static constexpr uint32_t kSmemBytes = kStages * kStageBytes + 1024u + kScaleBytes + 1024u;
  static_assert(kMp % 16 == 0 && kMp >= 16 && kMp <= 128, "UMMA N");
};

struct SkinnyParams {
  int32_t M, N, K;
  int32_t n_tiles, num_kb, total_steps, grid, max_seg;
  const float* a_scale;  // [KB][M]
  const float* b_scale;  // [ceil(N/128)][KB]
  const void* C;
  int64_t ldc;
  void* D;
  int64_t ldd;
  float alpha, beta;
  int32_t out_f32, has_c;
  float* ws;               // [n_tiles][max_seg][Mp][128] partial sums
  unsigned int* counters;  // [n_tiles], zero between calls
};

__host__ __device__ __forceinline__ int64_t sk_range_start(int64_t c, int64_t T, int64_t G) {
  return c * T / G;
}
// The CTA whose range holds step x.
__host__ __device__ __forceinline__ int64_t sk_owner(int64_t x, int64_t T, int64_t G) {
  return ((x + 1) * G - 1) / T;
}

template <int kMp>
__global__ void __launch_bounds__(kSkThreads, 1)
    gemm_fp8_block_skinny_kernel(const __grid_constant__ CUtensorMap tmap_a,
                                 const __grid_constant__ CUtensorMap tmap_b,
                                 const SkinnyParams p) {
  using Cfg = SkinnyCfg<kMp>;
  constexpr int S = Cfg::kStages;
  constexpr int kHalf = Cfg::kHalf;
  constexpr uint32_t kIdesc = make_idesc(0, 0, 128, kMp);  // E4M3 x E4M3 -> F32, M=128, N=Mp

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + S * Cfg::kStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);
  float* scale_area = reinterpret_cast<float*>(gbase + S * Cfg::kStageBytes + 1024);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](uint32_t b) { return bar0 + 8u * (2 * S + b); };
  auto tempty_bar = [&](uint32_t b) { return bar0 + 8u * (2 * S + kSkNumAcc + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 2 * kSkNumAcc);
  const uint32_t seg_bar = bar0 + 8u * (2 * S + 2 * kSkNumAcc + 1);   // 8 epilogue warps done
  const uint32_t flag_bar = bar0 + 8u * (2 * S + 2 * kSkNumAcc + 2);  // last_flag published
  auto b_smem = [&](uint32_t s) { return sbase + s * Cfg::kStageBytes; };
  auto a_smem = [&](uint32_t s) { return sbase + s * Cfg::kStageBytes + kSkBTileBytes; };

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;
  const int64_t T = p.total_steps, G = p.grid;
  const int64_t s0 = sk_range_start(blockIdx.x, T, G);
  const int64_t s1 = sk_range_start(blockIdx.x + 1, T, G);
  const int KB = p.num_kb;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < kSkNumAcc; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 8);  // one arrival per epilogue warp
    }
    mbar_init(drain_bar, 1);
    mbar_init(seg_bar, 8);
    mbar_init(flag_bar, 1);
    *abort_flag = 0;
    *last_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmap_a);
      tma_prefetch_desc(&tmap_b);
      const uint64_t stream_policy = l2_policy_evict_first();  // B is read once
      const uint64_t keep_policy = l2_policy_evict_last();     // A is re-read by every CTA
      uint32_t j = 0;
      bool ok = true;
      for (int64_t st = s0; st < s1; ++st, ++j) {
        const int nt = (int)(st / KB), kb = (int)(st % KB);
        const uint32_t s = j % S, ph = (j / S) & 1u;
        if (!wait_phase(empty_bar(s), ph ^ 1u, abort_flag, 0x11)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(full_bar(s), Cfg::kStageBytes);
        tma_load_2d_hint(b_smem(s), &tmap_b, full_bar(s), kb * 128, nt * 128, stream_policy);
        tma_load_2d_hint(a_smem(s), &tmap_a, full_bar(s), kb * 128, 0, keep_policy);
      }
      if (!ok) {
        const uint32_t n = j < (uint32_t)S ? j : (uint32_t)S;
        for (uint32_t i = j - n; i < j; ++i) {
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(full_bar(i % S), (i / S) & 1u) &&
                 global_timer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t j = 0;
      bool ok = true, issued = false;
      for (int64_t st = s0; st < s1; ++st, ++j) {
        const uint32_t s = j % S, ph = (j / S) & 1u;
        const uint32_t b = j % kSkNumAcc, bph = (j / kSkNumAcc) & 1u;
        if (!wait_phase(tempty_bar(b), bph ^ 1u, abort_flag, 0x12) ||
            !wait_phase(full_bar(s), ph, abort_flag, 0x13)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint64_t ad = smem_desc_k_sw128(b_smem(s));  // UMMA A: 128 rows of B
        const uint64_t bd = smem_desc_k_sw128(a_smem(s));  // UMMA B: Mp rows of A
        const uint32_t d_tmem = tmem_base + b * kMp;
#pragma unroll
        for (int k = 0; k < 4; ++k) mma_e4m3(d_tmem, ad + 2u * k, bd + 2u * k, kIdesc, k != 0);
        issued = true;
        tc_commit(empty_bar(s));
        tc_commit(tfull_bar(b));
      }
      if (!ok && issued) {
        tc_commit(drain_bar);
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(drain_bar, 0) && global_timer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------- epilogue
    const uint32_t ew = warp - 2;   // 0..7
    const uint32_t q = warp & 3u;   // TMEM lane quarter
    const uint32_t h = ew >> 2;     // column half
    const int col0 = (int)h * kHalf;
    const int nloc = (int)(q * 32u + lane);
    float* sc = scale_area + ew * kHalf;  // this warp's scale vector
    uint32_t j = 0, nsplit = 0;
    bool ok = true;
    int64_t st = s0;
    while (ok && st < s1) {
      const int nt = (int)(st / KB);
      const int64_t seg_end = ((int64_t)nt + 1) * KB < s1 ? ((int64_t)nt + 1) * KB : s1;
      const int kb_first = (int)(st - (int64_t)nt * KB);
      float acc[kHalf];
#pragma unroll
      for (int c = 0; c < kHalf; ++c) acc[c] = 0.0f;
      for (; st < seg_end; ++st, ++j) {
        const int kb = (int)(st - (int64_t)nt * KB);
        // this K block's column scales sa[kb, m] * sb[nt, kb]
        const float sbv = p.b_scale[(int64_t)nt * KB + kb];
        for (int c = (int)lane; c < kHalf; c += 32) {
          const int m = col0 + c;
          sc[c] = m < p.M ? p.a_scale[(int64_t)kb * p.M + m] * sbv : 0.0f;
        }
        const uint32_t b = j % kSkNumAcc, bph = (j / kSkNumAcc) & 1u;
        uint32_t got = 0;
        if (lane == 0) got = wait_phase(tfull_bar(b), bph, abort_flag, 0x14) ? 1u : 0u;
        got = __shfl_sync(0xFFFFFFFFu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        uint32_t r[kHalf];
        tmem_load_cols<kHalf>(tmem_base + ((q * 32u) << 16) + b * kMp + (uint32_t)col0, r);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(b));
#pragma unroll
        for (int c = 0; c < kHalf; c += 4) {
          const float4 s4 = *reinterpret_cast<const float4*>(sc + c);
          acc[c + 0] = fmaf(__uint_as_float(r[c + 0]), s4.x, acc[c + 0]);
          acc[c + 1] = fmaf(__uint_as_float(r[c + 1]), s4.y, acc[c + 1]);
          acc[c + 2] = fmaf(__uint_as_float(r[c + 2]), s4.z, acc[c + 2]);
          acc[c + 3] = fmaf(__uint_as_float(r[c + 3]), s4.w, acc[c + 3]);
        }
        __syncwarp();  // sc is rewritten for the next K block
      }
      if (!ok) break;
      // ---- the segment [kb_first, kb_last] of tile nt is summed
      const int kb_last_excl = (int)(seg_end - (int64_t)nt * KB);
      const int n = nt * 128 + nloc;
      auto emit = [&](int m, float val) {
        if (m >= p.M || n >= p.N) return;
        float o = p.alpha * val;
        if (p.out_f32) {
          if (p.has_c) o += p.beta * static_cast<const float*>(p.C)[(int64_t)m * p.ldc + n];
          static_cast<float*>(p.D)[(int64_t)m * p.ldd + n] = o;
        } else {
          if (p.has_c)
            o += p.beta * __uint_as_float(
                              (uint32_t)static_cast<const uint16_t*>(p.C)[(int64_t)m * p.ldc + n]
                              << 16);
          static_cast<uint16_t*>(p.D)[(int64_t)m * p.ldd + n] =
              (uint16_t)(pack_bf16x2(o, 0.0f) & 0xFFFFu);
        }
      };
      if (kb_first == 0 && kb_last_excl == KB) {
#pragma unroll
        for (int c = 0; c < kHalf; ++c) emit(col0 + c, acc[c]);
      } else {
        const int64_t first_owner = sk_owner((int64_t)nt * KB, T, G);
        const int64_t last_owner = sk_owner((int64_t)nt * KB + KB - 1, T, G);
        const int nseg = (int)(last_owner - first_owner + 1);
        const int slot = (int)((int64_t)blockIdx.x - first_owner);
        float* wsp = p.ws + ((int64_t)nt * p.max_seg + slot) * (int64_t)kMp * 128;
#pragma unroll
        for (int c = 0; c < kHalf; ++c) __stcg(wsp + (int64_t)(col0 + c) * 128 + nloc, acc[c]);
        // Publish the partial, then one thread counts arrivals for the tile.
        // The group syncs through mbarriers with bounded waits, so an
        // aborting warp cannot leave the others blocked.
        __threadfence();
        __syncwarp();
        if (lane == 0) mbar_arrive(seg_bar);
        const uint32_t par = nsplit & 1u;
        ++nsplit;
        if (ew == 0 && lane == 0) {
          int last = 0;
          if (wait_phase(seg_bar, par, abort_flag, 0x15)) {
            const unsigned prev = atomicAdd(&p.counters[nt], 1u);
            last = prev == (unsigned)(nseg - 1);
            if (last) p.counters[nt] = 0u;  // ready for the next call
          }
          *last_flag = last;
          mbar_arrive(flag_bar);
        }
        uint32_t got = 0;
        if (lane == 0) got = wait_phase(flag_bar, par, abort_flag, 0x16) ? 1u : 0u;
        got = __shfl_sync(0xFFFFFFFFu, got, 0);
        if (!got || *abort_flag) {
          ok = false;
          break;
        }
        if (*last_flag) {
          __threadfence();
          const float* wt = p.ws + (int64_t)nt * p.max_seg * kMp * 128;
          for (int c = 0; c < kHalf; ++c) {
            float sum = 0.0f;
            for (int sgi = 0; sgi < nseg; ++sgi)
              sum += __ldcg(wt + ((int64_t)sgi * kMp + col0 + c) * 128 + nloc);
            emit(col0 + c, sum);
          }
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

}  // namespace tcg
