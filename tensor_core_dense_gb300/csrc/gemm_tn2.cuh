// gemm_tn2.cuh -- the persistent TN GEMM on CTA pairs (tcgen05 cta_group::2).
//
// Same computation, roles and epilogue as gemm_tn.cuh, with a 256 x 256
// output tile per cluster of two CTAs on neighbouring SMs.  CTA r of the pair
// loads rows [128r, 128r+128) of the tile's A block and rows [128r, 128r+128)
// of its B block; the leader (r = 0) issues one tcgen05.mma.cta_group::2 per
// 32 bytes of K, which reads A and B halves from both CTAs' shared memory and
// leaves rows [128r, 128r+128) of the FP32 accumulator in CTA r's Tensor
// Memory.  Per SM and per K block this halves the B bytes that TMA writes and
// the tensor core reads compared with a 128 x 256 tile on one SM, the
// operand-traffic argument of "How Blackwell's Tensor Memory Actually Works",
// "Why it had to be a separate memory" (cta_group::2 halves the per-SM
// operand traffic), with only the leader CTA issuing ("The instruction").
//
// Pair protocol:
//   full[s]    in the leader: armed by the leader's producer with the bytes of
//              both CTAs' copies; both producers' TMA loads credit it
//              (cta_group::2 loads may signal the peer's barrier).
//   empty[s]   in each CTA: the leader's commit multicasts to both.
//   tfull[a]   in each CTA: the leader's commit multicasts to both epilogues.
//   tempty[a]  in the leader: 8 arrivals, 4 local epilogue warps + 4 remote.
// Cluster barriers at start (barriers initialised before any remote use) and
// end (no CTA leaves while its peer may still touch its shared memory).
//
// Epilogue stores go through shared memory and TMA: each epilogue warp turns
// a chunk of its 32 rows x 128 bytes (64 BF16 or 32 FP32 columns) into a
// 128-byte-swizzled buffer (two per warp, reused once the store two chunks
// back has read it) and stores it with one tensor copy; rows and columns
// outside D are clipped by the tensor map.  With beta != 0 the same box of C
// is first loaded into the buffer by TMA.  Per-lane 16-byte stores, one row
// per lane, had put one L2 request per 16 bytes of D (2.1 M of the kernel's
// 7.6 M L2 requests at FP8 4096^3).  A chunk that ends past column N while
// N x element size is not a multiple of 16 bytes keeps the per-lane stores:
// the tensor copy clipped such a row at 16-byte granularity and wrote past N.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "gemm_tn.cuh"
#include "ptx.cuh"

namespace tcg {

constexpr int kP2Stages = 7;
constexpr uint32_t kP2ATileBytes = 128 * kBKBytes;  // this CTA's 128 rows of A
constexpr uint32_t kP2BTileBytes = 128 * kBKBytes;  // up to 128 rows of B (its half)
constexpr uint32_t kP2StageBytes = kP2ATileBytes + kP2BTileBytes;
constexpr int kP2NumBars = 2 * kP2Stages + 5;
constexpr uint32_t kP2SmemBytes = kP2Stages * kP2StageBytes + 1024 + 1024;
// gemm_tn2_kernel itself: one stage fewer (7 -> 6 measured the same) for the
// epilogue's staging buffers, 2 x 4 KB per epilogue warp
constexpr int kP2DStages = 6;
constexpr uint32_t kP2DStageOut = 32 * 128;  // one store chunk: 32 rows x 128 bytes
constexpr uint32_t kP2DOutBytes = 4 * 2 * kP2DStageOut;
constexpr int kP2DNumBars = 2 * kP2DStages + 5 + 4;  // + one C-load barrier per epilogue warp
constexpr uint32_t kP2DSmemBytes = kP2DStages * kP2StageBytes + kP2DOutBytes + 1024 + 1024;

struct Gemm2Params {
  int32_t M, N, K;
  int32_t tiles_m, tiles_n, num_kb, num_tiles;  // tiles are 256 x 256
  int32_t dp_waves, dp_end, split;              // as GemmParams; split 1 or 2
  uint32_t fp8_fmt;                             // as GemmParams
  const void* C;
  int64_t ldc;
  void* D;
  int64_t ldd;
  float alpha, beta;
  const float* a_scale;
  const float* b_scale;
};

// Work sequence of one cluster (b = cluster index, G = clusters).
struct PairWorkIter {
  int b, G, i, j, dp_waves, dp_end, split, tail_units;
  __device__ __forceinline__ void init(const Gemm2Params& p, int cluster, int clusters) {
    b = cluster;
    G = clusters;
    i = j = 0;
    dp_waves = p.dp_waves;
    dp_end = p.dp_end;
    split = p.split;
    tail_units = (p.num_tiles - p.dp_end) * p.split;
  }
  __device__ __forceinline__ bool next(WorkItem& w) {
    while (i < dp_waves) {
      const int t = b + i * G;
      ++i;
      if (t < dp_end) {
        w.tile = t;
        w.sub = 0;
        w.split = 1;
        return true;
      }
    }
    const int u = b + j * G;
    if (u < tail_units) {
      ++j;
      w.tile = dp_end + u / split;
      w.sub = u % split;
      w.split = split;
      return true;
    }
    return false;
  }
};

template <int kOut, bool kHasC>
__device__ __forceinline__ void store_row_chunk2(const Gemm2Params& p, int row, int col0,
                                                 const float (&acc)[32], float scale) {
  GemmParams q;
  q.M = p.M;
  q.N = p.N;
  q.C = p.C;
  q.ldc = p.ldc;
  q.D = p.D;
  q.ldd = p.ldd;
  q.beta = p.beta;
  store_row_chunk<kOut, kHasC>(q, row, col0, acc, scale);
}

template <int kIn, int kOut, bool kHasC>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tn2_kernel(const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_d,
                    const __grid_constant__ CUtensorMap tmap_c, const Gemm2Params p) {
  constexpr int kBKElems = kIn == 0 ? kBKBytes / 2 : kBKBytes;
  constexpr uint32_t kFmt = kIn == 0 ? 1u : 0u;
  constexpr uint32_t kIdesc256 = make_idesc(kFmt, kFmt, 256, 256);
  constexpr uint32_t kIdesc128 = make_idesc(kFmt, kFmt, 256, 128);
  constexpr int kMmaPerStage = kBKBytes / 32;
  constexpr int S = kP2DStages;
  constexpr int kCW = kOut == 0 ? 64 : 32;  // columns per 128-byte store chunk

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  const uint32_t out_base = sbase + S * kP2StageBytes;  // staging buffers, 1024-aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + S * kP2StageBytes + kP2DOutBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kP2DNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](uint32_t a) { return bar0 + 8u * (2 * S + a); };
  auto tempty_bar = [&](uint32_t a) { return bar0 + 8u * (2 * S + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);
  auto cload_bar = [&](uint32_t e) { return bar0 + 8u * (2 * S + 5 + e); };
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
      mbar_init(tempty_bar(a), 8);  // 4 epilogue warps in each CTA of the pair
    }
    mbar_init(drain_bar, 1);
    for (int e = 0; e < 4; ++e) mbar_init(cload_bar(e), 1);
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
    tma_prefetch_desc(&tmap_d);
    if (kHasC) tma_prefetch_desc(&tmap_c);
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
        tma_prefetch_l2_2d(&tmap_a, kb * kBKElems, arow0);
        for (int bx = 0; bx < half / kBBoxRows; ++bx)
          tma_prefetch_l2_2d(&tmap_b, kb * kBKElems, brow0 + bx * kBBoxRows);
      }
    }
  }
  grid_dependency_wait();  // global memory only after the previous kernel finished

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
        const int nsub = 256 / w.split;              // tile columns of this unit
        const int half = nsub / 2;                   // rows of B this CTA loads
        const int nboxes = half / kBBoxRows;         // 2 or 1
        const int brow0 = tn * 256 + w.sub * nsub + (int)rank * half;
        const int arow0 = tm * 256 + (int)rank * 128;
        const uint32_t my_bytes = kP2ATileBytes + (uint32_t)half * kBKBytes;
        for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
          const uint32_t s = it % S, ph = (it / S) & 1u;
          if (!wait_phase(empty_bar(s), ph ^ 1u, abort_flag, 0x21)) {
            ok = false;
            break;
          }
          const uint32_t fb = map_shared_to_cta(full_bar(s), 0);  // the leader's barrier
          if (leader) mbar_arrive_expect_tx(full_bar(s), 2u * my_bytes);
          tma_load_2d_pair(a_smem(s), &tmap_a, fb, kb * kBKElems, arow0);
          for (int bx = 0; bx < nboxes; ++bx)
            tma_load_2d_pair(b_smem(s) + (uint32_t)bx * kBBoxRows * kBKBytes, &tmap_b, fb,
                             kb * kBKElems, brow0 + bx * kBBoxRows);
        }
      }
      grid_launch_dependents();  // every load is issued: the next kernel may launch
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer (leader)
    if (leader && lane == 0) {
      uint32_t it = 0, lt = 0;
      bool ok = true, issued = false;
      PairWorkIter wi;
      wi.init(p, cluster, clusters);
      WorkItem w;
      for (; ok && wi.next(w); ++lt) {
        const uint32_t acc = lt & 1u, aph = (lt >> 1) & 1u;
        // both CTAs' epilogues have drained this accumulator
        bool free_ok = mbar_try_wait_cluster(tempty_bar(acc), aph ^ 1u);
        if (!free_ok) {
          const uint64_t t0 = global_timer_ns();
          for (uint32_t i = 1; !free_ok; ++i) {
            free_ok = mbar_try_wait_cluster(tempty_bar(acc), aph ^ 1u);
            if (!free_ok && (i & 31u) == 0u) {
              if (*abort_flag) break;
              if (global_timer_ns() - t0 > kWaitLimitNs) {
                record_timeout(0x22);
                *abort_flag = 1;
                break;
              }
            }
          }
        }
        if (!free_ok) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * kAccCols;
        const uint32_t idesc = (w.split == 1 ? kIdesc256 : kIdesc128) | (kIn == 1 ? p.fp8_fmt : 0u);
        static_assert(kMmaPerStage == 4, "one K step is four 32-byte MMAs");
        // The unit's first K step is waited for here; every later one was
        // tested while the step before it was issued (see
        // mma_step4_pair_test_next) and is waited for only if that test failed.
        bool ready = false;
        for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
          const uint32_t s = it % S, ph = (it / S) & 1u;
          if (!ready && !wait_phase(full_bar(s), ph, abort_flag, 0x23)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t ad = smem_desc_k_sw128(a_smem(s));
          const uint64_t bd = smem_desc_k_sw128(b_smem(s));
          // test the next step of this unit; at the last step, a phase that is
          // already complete (the result is not used)
          const bool more = kb + 1 < p.num_kb;
          const uint32_t s1 = (it + 1u) % S, ph1 = ((it + 1u) / S) & 1u;
          const uint32_t got = mma_step4_pair_test_next<kIn>(
              d_tmem, ad, bd, idesc, kb != 0 ? 1u : 0u, empty_bar(s), more ? full_bar(s1) : full_bar(s),
              more ? ph1 : ph);
          ready = more && got != 0u;
          issued = true;
        }
        if (ok) tc_commit_pair(tfull_bar(acc), 0x3);
      }
      if (!ok && issued) {
        tc_commit_pair(drain_bar, 0x1);
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(drain_bar, 0) && global_timer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------- epilogue
    const uint32_t q = warp & 3u;   // TMEM lane quarter: rows 32q..32q+31 of this CTA's half
    const uint32_t ew = warp - 2u;  // epilogue warp 0..3: its staging buffers and C barrier
    float scale = p.alpha;
    if (kIn == 1) scale = p.a_scale[0] * p.b_scale[0] * p.alpha;
    uint32_t lt = 0, nst = 0, cph = 0;  // units, chunks stored, C-barrier phase
    bool ok_all = true;
    PairWorkIter wi;
    wi.init(p, cluster, clusters);
    WorkItem w;
    for (; ok_all && wi.next(w); ++lt) {
      const uint32_t acc = lt & 1u, aph = (lt >> 1) & 1u;
      uint32_t ok = 0;
      if (lane == 0) ok = wait_phase(tfull_bar(acc), aph, abort_flag, 0x24) ? 1u : 0u;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after_sync();
      int tm, tn;
      tile_coords(w.tile, p.tiles_m, p.tiles_n, tm, tn);
      const int row0 = tm * 256 + (int)(rank * 128u + q * 32u);  // this warp's first row
      const int nsub = 256 / w.split;
      const int col_base = tn * 256 + w.sub * nsub;
      const int nchunks = nsub / kCW;
      const uint32_t t_row = tmem_base + ((q * 32u) << 16) + acc * kAccCols;
      constexpr int kOutBytes = kOut == 0 ? 2 : 4;
      const bool n_aligned = ((int64_t)p.N * kOutBytes) % 16 == 0;
#pragma unroll 1
      for (int c = 0; c < nchunks; ++c) {
        const int col = col_base + c * kCW;
        const bool last = c == nchunks - 1;
        if (col >= p.N && !last) continue;  // nothing of D in this chunk (its TMEM stays unread)
        if (!n_aligned && col + kCW > p.N) {
          // ragged right edge: per-lane stores, clipped per element
          uint32_t r[64];
          __syncwarp();
          tmem_ld_32x32b_x32(t_row + (uint32_t)(c * kCW), *reinterpret_cast<uint32_t(*)[32]>(r));
          if (kCW == 64)
            tmem_ld_32x32b_x32(t_row + (uint32_t)(c * kCW + 32),
                               *reinterpret_cast<uint32_t(*)[32]>(r + 32));
          tmem_ld_wait_n<64>(r);
          if (last) {
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote_cta(map_shared_to_cta(tempty_bar(acc), 0));
          }
#pragma unroll
          for (int h = 0; h < kCW / 32; ++h) {
            float a[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) a[j] = __uint_as_float(r[32 * h + j]);
            store_row_chunk2<kOut, kHasC>(p, row0 + (int)lane, col + 32 * h, a, scale);
          }
          continue;
        }
        if (col >= p.N) {
          // the last chunk lies past N: only the hand-back is left
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote_cta(map_shared_to_cta(tempty_bar(acc), 0));
          continue;
        }
        const uint32_t buf = out_base + (ew * 2u + (nst & 1u)) * kP2DStageOut;
        uint8_t* gbuf = gbase + (buf - sbase);
        ++nst;
        // the store two chunks back read this buffer; with C, load its box
        if (lane == 0) {
          if (nst >= 3) bulk_wait_group_read<1>();
          if (kHasC) {
            mbar_arrive_expect_tx(cload_bar(ew), kP2DStageOut);
            tma_load_2d(buf, &tmap_c, cload_bar(ew), col, row0);
          }
        }
        uint32_t r[64];
        __syncwarp();
        tmem_ld_32x32b_x32(t_row + (uint32_t)(c * kCW), *reinterpret_cast<uint32_t(*)[32]>(r));
        if (kCW == 64)
          tmem_ld_32x32b_x32(t_row + (uint32_t)(c * kCW + 32),
                             *reinterpret_cast<uint32_t(*)[32]>(r + 32));
        tmem_ld_wait_n<64>(r);
        if (last) {
          // hand the accumulator back to the leader's MMA warp (ordered by
          // the tcgen05 fence; a CTA-scope release does not wait for this
          // thread's earlier stores)
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote_cta(map_shared_to_cta(tempty_bar(acc), 0));
        }
        if (kHasC) {
          uint32_t got = 0;
          if (lane == 0) got = wait_phase(cload_bar(ew), cph, abort_flag, 0x25) ? 1u : 0u;
          cph ^= 1u;
          got = __shfl_sync(0xFFFFFFFFu, got, 0);
          if (!got) {
            ok_all = false;
            break;
          }
        }
        // lane = row; 16-byte piece j of the row sits at j ^ (row % 8)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint4* piece = reinterpret_cast<uint4*>(gbuf + lane * 128u + ((j ^ (lane & 7u)) << 4));
          if (kOut == 0) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = scale * __uint_as_float(r[8 * j + e]);
            if (kHasC) {
              const uint4 cv = *piece;
              v[0] += p.beta * bf16_lo_to_f32(cv.x);
              v[1] += p.beta * bf16_hi_to_f32(cv.x);
              v[2] += p.beta * bf16_lo_to_f32(cv.y);
              v[3] += p.beta * bf16_hi_to_f32(cv.y);
              v[4] += p.beta * bf16_lo_to_f32(cv.z);
              v[5] += p.beta * bf16_hi_to_f32(cv.z);
              v[6] += p.beta * bf16_lo_to_f32(cv.w);
              v[7] += p.beta * bf16_hi_to_f32(cv.w);
            }
            *piece = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
          } else {
            float4 o = make_float4(scale * __uint_as_float(r[4 * j + 0]),
                                   scale * __uint_as_float(r[4 * j + 1]),
                                   scale * __uint_as_float(r[4 * j + 2]),
                                   scale * __uint_as_float(r[4 * j + 3]));
            if (kHasC) {
              const float4 cv = *reinterpret_cast<const float4*>(piece);
              o.x += p.beta * cv.x;
              o.y += p.beta * cv.y;
              o.z += p.beta * cv.z;
              o.w += p.beta * cv.w;
            }
            *reinterpret_cast<float4*>(piece) = o;
          }
        }
        fence_proxy_async_shared();  // the writes above, before the TMA store reads them
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmap_d, buf, col, row0);
          bulk_commit_group();
        }
      }
    }
    if (lane == 0) bulk_wait_group<0>();  // every store has finished before the CTA exits
    __syncwarp();
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
