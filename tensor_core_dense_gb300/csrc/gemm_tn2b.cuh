// gemm_tn2b.cuh -- FP8 GEMM with 128-block scales on CTA pairs (M > 128).
//
//   D[m, n] = alpha * sum_kb sa[kb*M + m] * sb[(n/128)*KB + kb]
//                    * sum_{k in block kb} qa[m, k] * qb[n, k]   (+ beta * C)
//
// The block scaling of gemm_skinny.cuh (1 x 128 blocks of A, 128 x 128 blocks
// of B, the per-K-block promotion of "Tensor Cores: Matrix Instructions,
// Swizzling and FP8, Measured", Step 5) at the tile shape of gemm_tn2.cuh: a
// 256 x 256 output tile per cluster of two CTAs, the leader issuing
// tcgen05.mma.cta_group::2, each CTA holding rows [128r, 128r+128) of the
// tile.  The 128 x 128 tiles of the chunked skinny kernel need about twice the
// operand bytes per SM per MMA cycle that L2 delivers; the pair tile needs the
// same as the per-tensor FP8 kernel.
//
// Roles: warpgroup 0 = TMA producer (warp 0), MMA issuer (warp 1, leader CTA
// only) and two idle warps, all shrunk to 40 registers; warpgroups 1 and 2 =
// the eight promotion warps at 232 registers.
//
// Per K block kb (one pipeline stage of 128 K bytes) the MMA writes a fresh
// partial (enable-input-d = 0 on the block's first instruction) into one of
// two 256-column TMEM buffers, alternating.  Eight promotion warps, two per
// TMEM lane quarter (warp w reads lanes 32*(w%4)..), each own 128 columns of
// the CTA's 128 x 256 accumulator as FP32 registers: they load the partial
// (tcgen05.ld), add partial * sa[row, kb] * sb[column block, kb] with scalar
// FMAs, and hand the buffer back.  (FP32 work on the SM slows the tensor
// pipe: without the FMAs a K block's MMA completes in about 730 cycles, with
// them about 1170.  Packed f32x2 FMAs, half the instructions, were 1-2 %
// slower than scalar ones.)  A 256-column tile spans two column
// blocks of B's scales; the warps of column half h use block 2*tn + h.  The
// scales come in sets of kPbAhead K blocks: a set is loaded into registers
// one set ahead of use, so a load has kPbAhead K blocks of MMA time to land
// before anything reads its register.  After the tile's last K block the same
// warps apply alpha and beta*C, convert and store; the MMA meanwhile fills
// both buffers with the next tile's first K blocks.
//
// Barriers as in gemm_tn2.cuh, except that tfull/tempty turn over once per K
// block instead of once per tile; tempty[a] counts 16 arrivals (8 warps in
// each CTA), each a CTA-scope release arrive after a tcgen05 fence.  With two
// buffers the MMA of block g+2 waits for both CTAs' promotion of block g, so
// a K block costs about half of (MMA + promotion + the two notification
// latencies); a 256-column partial per buffer leaves no room for a third.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "gemm_tn.cuh"
#include "gemm_tn2.cuh"
#include "ptx.cuh"

namespace tcg {

constexpr int kPbPromoWarps = 8;                     // two per TMEM lane quarter
constexpr int kPbThreads = 128 + 32 * kPbPromoWarps; // warpgroup 0, then two promotion groups
constexpr int kPbAhead = 4;                          // K blocks per scale refill
constexpr int kPbChunk = 64;                         // TMEM columns per tcgen05.ld
// Registers per thread: 168 at launch (three warps per SM sub-partition);
// warpgroup 0 gives up 128 each, the promotion warps take 64 each more:
// 4*32*40 + 8*32*232 = 12*32*168, so the increase is always satisfiable.
constexpr uint32_t kPbRegsLow = 40;
constexpr uint32_t kPbRegsHigh = 232;
static_assert(4 * 32 * kPbRegsLow + kPbPromoWarps * 32 * kPbRegsHigh <= kPbThreads * 168u,
              "register split exceeds the launch budget");

// One promotion chunk of this warp's 32 TMEM lanes (by the chunk width).
__device__ __forceinline__ void pb_tmem_ld(uint32_t taddr, uint32_t (&r)[32]) {
  tmem_ld_32x32b_x32(taddr, r);
}
__device__ __forceinline__ void pb_tmem_ld(uint32_t taddr, uint32_t (&r)[64]) {
  tmem_ld_32x32b_x64(taddr, r);
}

// Bounded wait with cluster-scope acquire (arrivals from the peer CTA).
__device__ __forceinline__ bool wait_phase_cluster(uint32_t bar, uint32_t parity,
                                                   volatile int* abort_flag, uint32_t where) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 31u) == 0u) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        record_timeout(where);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// The scales one promotion thread needs, step by step along its cluster's
// work sequence: sa of its row and sb of its column block, for every K block
// of every work item.  Zero beyond M or N (those outputs are never stored).
struct PbScaleStream {
  PairWorkIter wi;
  const float* pa;  // &sa[row] of the current item, or null
  const float* pb;  // &sb[block * KB] of the current item, or null
  int64_t M;
  int kb, num_kb;
  bool valid;

  __device__ __forceinline__ void item(const Gemm2Params& p, int row_in_tile, int h) {
    WorkItem w;
    valid = wi.next(w);
    kb = 0;
    pa = pb = nullptr;
    if (!valid) return;
    int tm, tn;
    tile_coords(w.tile, p.tiles_m, p.tiles_n, tm, tn);
    const int row = tm * 256 + row_in_tile;
    const int nsub = 256 / w.split;
    const int col = tn * 256 + w.sub * nsub + h * (nsub / 2);
    if (row < p.M) pa = p.a_scale + row;
    if (col < p.N) pb = p.b_scale + (int64_t)(col >> 7) * p.num_kb;
  }
  __device__ __forceinline__ void init(const Gemm2Params& p, int cluster, int clusters,
                                       int row_in_tile, int h) {
    wi.init(p, cluster, clusters);
    M = p.M;
    num_kb = p.num_kb;
    item(p, row_in_tile, h);
  }
  __device__ __forceinline__ void load(float& a, float& b) const {
    a = pa ? __ldg(pa + (int64_t)kb * M) : 0.0f;
    b = pb ? __ldg(pb + kb) : 0.0f;
  }
  __device__ __forceinline__ void advance(const Gemm2Params& p, int row_in_tile, int h) {
    if (!valid) return;
    if (++kb == num_kb) item(p, row_in_tile, h);
  }
};

// kOut: 0 = BF16, 1 = FP32.  kHasC: beta != 0.
template <int kOut, bool kHasC>
__global__ void __launch_bounds__(kPbThreads, 1)
    gemm_fp8_block_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                               const __grid_constant__ CUtensorMap tmap_b, const Gemm2Params p) {
  constexpr uint32_t kIdesc256 = make_idesc(0u, 0u, 256, 256);  // format bits from p.fp8_fmt
  constexpr uint32_t kIdesc128 = make_idesc(0u, 0u, 256, 128);
  constexpr int kMmaPerStage = kBKBytes / 32;
  constexpr int S = kP2Stages;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + S * kP2StageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kP2NumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](uint32_t a) { return bar0 + 8u * (2 * S + a); };
  auto tempty_bar = [&](uint32_t a) { return bar0 + 8u * (2 * S + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);
  auto a_smem = [&](uint32_t s) { return sbase + s * kP2StageBytes; };
  auto b_smem = [&](uint32_t s) { return sbase + s * kP2StageBytes + kP2ATileBytes; };

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = (int)(blockIdx.x >> 1);
  const int clusters = (int)(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 2 * kPbPromoWarps);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers are initialised before any remote use
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
    // warm L2 with this CTA's first stages while the previous kernel drains
    PairWorkIter wi;
    wi.init(p, cluster, clusters);
    WorkItem w;
    if (wi.next(w)) {
      int tm, tn;
      tile_coords(w.tile, p.tiles_m, p.tiles_n, tm, tn);
      const int nsub = 256 / w.split, half = nsub / 2;
      const int brow0 = tn * 256 + w.sub * nsub + (int)rank * half;
      const int arow0 = tm * 256 + (int)rank * 128;
      for (int kb = 0; kb < S && kb < p.num_kb; ++kb) {
        tma_prefetch_l2_2d(&tmap_a, kb * kBKBytes, arow0);
        for (int bx = 0; bx < half / kBBoxRows; ++bx)
          tma_prefetch_l2_2d(&tmap_b, kb * kBKBytes, brow0 + bx * kBBoxRows);
      }
    }
  }
  grid_dependency_wait();  // global memory only after the previous kernel finished

  if (warp < 4) {
    setmaxnreg_dec<kPbRegsLow>();
    if (warp == 0) {
      // ------------------------------------------------------- TMA producer
      if (lane == 0) {
        uint32_t it = 0;
        bool ok = true;
        PairWorkIter wi;
        wi.init(p, cluster, clusters);
        WorkItem w;
        while (ok && wi.next(w)) {
          int tm, tn;
          tile_coords(w.tile, p.tiles_m, p.tiles_n, tm, tn);
          const int nsub = 256 / w.split;
          const int half = nsub / 2;  // rows of B this CTA loads
          const int nboxes = half / kBBoxRows;
          const int brow0 = tn * 256 + w.sub * nsub + (int)rank * half;
          const int arow0 = tm * 256 + (int)rank * 128;
          const uint32_t my_bytes = kP2ATileBytes + (uint32_t)half * kBKBytes;
          for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
            const uint32_t s = it % S, ph = (it / S) & 1u;
            if (!wait_phase(empty_bar(s), ph ^ 1u, abort_flag, 0x31)) {
              ok = false;
              break;
            }
            const uint32_t fb = map_shared_to_cta(full_bar(s), 0);  // the leader's barrier
            if (leader) mbar_arrive_expect_tx(full_bar(s), 2u * my_bytes);
            tma_load_2d_pair(a_smem(s), &tmap_a, fb, kb * kBKBytes, arow0);
            for (int bx = 0; bx < nboxes; ++bx)
              tma_load_2d_pair(b_smem(s) + (uint32_t)bx * kBBoxRows * kBKBytes, &tmap_b, fb,
                               kb * kBKBytes, brow0 + bx * kBBoxRows);
          }
        }
        grid_launch_dependents();  // every load is issued: the next kernel may launch
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------------- MMA issuer (leader)
      if (leader && lane == 0) {
        uint32_t it = 0;  // stage counter
        uint32_t g = 0;   // K-block counter: TMEM buffer g & 1
        bool ok = true, issued = false;
        PairWorkIter wi;
        wi.init(p, cluster, clusters);
        WorkItem w;
        while (ok && wi.next(w)) {
          const uint32_t idesc = (w.split == 1 ? kIdesc256 : kIdesc128) | p.fp8_fmt;
          for (int kb = 0; kb < p.num_kb; ++kb, ++it, ++g) {
            const uint32_t acc = g & 1u, aph = (g >> 1) & 1u;
            // both CTAs' promotion warps have drained this buffer
            if (!wait_phase_cluster(tempty_bar(acc), aph ^ 1u, abort_flag, 0x32)) {
              ok = false;
              break;
            }
            const uint32_t s = it % S, ph = (it / S) & 1u;
            if (!wait_phase(full_bar(s), ph, abort_flag, 0x33)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t d_tmem = tmem_base + acc * kAccCols;
            const uint64_t ad = smem_desc_k_sw128(a_smem(s));
            const uint64_t bd = smem_desc_k_sw128(b_smem(s));
  #pragma unroll
            for (int k = 0; k < kMmaPerStage; ++k)
              mma_e4m3_pair(d_tmem, ad + 2u * k, bd + 2u * k, idesc, k != 0 ? 1u : 0u);
            issued = true;
            tc_commit_pair(empty_bar(s), 0x3);
            tc_commit_pair(tfull_bar(acc), 0x3);
          }
        }
        if (!ok && issued) {
          tc_commit_pair(drain_bar, 0x1);
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(drain_bar, 0) && global_timer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
      __syncwarp();
    }
  } else {
    setmaxnreg_inc<kPbRegsHigh>();
    // ------------------------------------------------------- promotion + epilogue
    const uint32_t q = warp & 3u;                 // TMEM lane quarter
    const int h = (int)(warp - 4u) >> 2;          // column half of the tile
    const int row_in_tile = (int)(rank * 128u + q * 32u + lane);
    PbScaleStream ss;
    ss.init(p, cluster, clusters, row_in_tile, h);
    float ca[kPbAhead], cb[kPbAhead];  // the current set of K blocks
    float na[kPbAhead], nb[kPbAhead];  // the next set, in flight
#pragma unroll
    for (int d = 0; d < kPbAhead; ++d) {
      ss.load(na[d], nb[d]);
      ss.advance(p, row_in_tile, h);
    }
    uint32_t g = 0;
    bool ok = true;
    PairWorkIter wi;
    wi.init(p, cluster, clusters);
    WorkItem w;
    while (ok && wi.next(w)) {
      int tm, tn;
      tile_coords(w.tile, p.tiles_m, p.tiles_n, tm, tn);
      const int nsub = 256 / w.split;
      const int ncols = nsub / 2;  // this warp's columns: 128, or 64 for a half tile
      const int row = tm * 256 + row_in_tile;
      const int col0 = tn * 256 + w.sub * nsub + h * ncols;
      float acc[128];  // this thread's row, this warp's 128 (or 64) columns
#pragma unroll
      for (int j = 0; j < 128; ++j) acc[j] = 0.0f;
      for (int kb = 0; kb < p.num_kb; ++kb, ++g) {
        const uint32_t buf = g & 1u, ph = (g >> 1) & 1u;
        const uint32_t slot = g % kPbAhead;
        if (slot == 0) {
          // the set loaded kPbAhead K blocks ago becomes current; load the next
#pragma unroll
          for (int d = 0; d < kPbAhead; ++d) {
            ca[d] = na[d];
            cb[d] = nb[d];
          }
#pragma unroll
          for (int d = 0; d < kPbAhead; ++d) {
            ss.load(na[d], nb[d]);
            ss.advance(p, row_in_tile, h);
          }
        }
        float sa_k = ca[0], sb_k = cb[0];
#pragma unroll
        for (int d = 1; d < kPbAhead; ++d) {
          if (slot == (uint32_t)d) {
            sa_k = ca[d];
            sb_k = cb[d];
          }
        }
        const float sk = sa_k * sb_k;
        uint32_t got = 0;
        if (lane == 0) got = wait_phase(tfull_bar(buf), ph, abort_flag, 0x34) ? 1u : 0u;
        got = __shfl_sync(0xFFFFFFFFu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t t_row =
            tmem_base + ((q * 32u) << 16) + buf * kAccCols + (uint32_t)(h * ncols);
#pragma unroll
        for (int c = 0; c < 128 / kPbChunk; ++c) {
          if (c * kPbChunk < ncols) {
            uint32_t r[kPbChunk];
            pb_tmem_ld(t_row + (uint32_t)(c * kPbChunk), r);
            tmem_ld_wait_n(r);
#pragma unroll
            for (int j = 0; j < kPbChunk; ++j)
              acc[c * kPbChunk + j] = fmaf(__uint_as_float(r[j]), sk, acc[c * kPbChunk + j]);
          }
        }
        // hand the buffer back to the leader's MMA warp (ordered by the
        // tcgen05 fence; CTA-scope release keeps the arrive from waiting on
        // this thread's scale loads in flight)
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote_cta(map_shared_to_cta(tempty_bar(buf), 0));
      }
      if (!ok) break;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (c * 32 < ncols) {
          float a[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) a[j] = acc[c * 32 + j];
          store_row_chunk2<kOut, kHasC>(p, row, col0 + c * 32, a, p.alpha);
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while the pair may still use its memory
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace tcg
