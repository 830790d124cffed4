// gemm_tn.cuh -- persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
//   D[M x N] = scale * A[M x K] * B[N x K]^T (+ beta * C)
//
// A and B are K-major (the "TN" layout, "Tensor Cores: Matrix Instructions,
// Swizzling and FP8, Measured", Step 2).  Operands are BF16 (kind::f16) or
// FP8 E4M3 (kind::f8f6f4); accumulation is FP32 in Tensor Memory.
//
// One CTA per SM loops over 128 x 256 output tiles (persistent scheduler,
// grouped raster for L2 reuse).  Whole waves of tiles run one tile per CTA.
// The tiles of a last, partial wave (or of a grid smaller than the GPU) are
// cut along N into 2 or 4 sub-tiles of 128 or 64 columns (UMMA N = 128 / 64)
// so that the last wave keeps every SM busy for a half or a quarter of a tile
// time instead of leaving most SMs idle for a whole one.  Each output element
// is still produced by exactly one CTA from all of K: no workspace, no
// reduction, bit-identical results from run to run.  Its six warps have fixed
// roles:
//   warp 0     one lane issues TMA loads of 128-byte-swizzled A/B K-blocks
//              into a kStages-deep ring of shared-memory stages, each stage
//              guarded by a `full` mbarrier (TMA transaction bytes) and an
//              `empty` mbarrier (released by tcgen05.commit);
//   warp 1     allocates Tensor Memory (512 columns = two 128 x 256 FP32
//              accumulators), then one lane issues four tcgen05.mma per
//              stage and commits; at the end of a tile it commits to the
//              tile's `tmem_full` barrier;
//   warps 2-5  the epilogue warpgroup: each warp drains its 32 TMEM lanes
//              (tcgen05.ld 32x32b.x32), applies scale/alpha/beta, converts,
//              and stores with 16-byte vector stores; it then frees the
//              accumulator buffer (`tmem_empty`), so the epilogue of tile i
//              overlaps the main loop of tile i+1.
//
// This is the producer/consumer warp specialisation of "Tensor cores and
// low precision" (H100 worklog paragraph), re-expressed for tcgen05: the MMA
// is issued by a single thread and its accumulator lives in Tensor Memory
// ("How Blackwell's Tensor Memory Actually Works", "What Tensor Memory
// actually is"); latency is hidden by the in-CTA ring, not by occupancy
// (same page, "Occupancy stops meaning what it meant").
//
// Every mbarrier wait is bounded (kWaitLimitNs).  A wait that runs out
// records TCG_ERR_TIMEOUT in the device status word, raises a shared abort
// flag so that the other roles stop too, drains the work already in flight
// (bounded again) and frees Tensor Memory before the CTA exits.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "ptx.cuh"

namespace tcg {

constexpr int kBM = 128;               // tile rows (UMMA M)
constexpr int kBN = 256;               // tile columns (UMMA N)
constexpr int kBKBytes = 128;          // K bytes per stage: one 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr int kAccCols = kBN;          // TMEM columns per accumulator buffer
constexpr int kTmemCols = 2 * kAccCols;
constexpr uint32_t kATileBytes = kBM * kBKBytes;
constexpr uint32_t kBTileBytes = kBN * kBKBytes;
constexpr uint32_t kStageBytes = kATileBytes + kBTileBytes;
constexpr int kNumBars = 2 * kStages + 5;  // full, empty, tmem_full x2, tmem_empty x2, drain
constexpr int kBBoxRows = 64;              // B is loaded as 64-row boxes (1, 2 or 4 per stage)
constexpr uint32_t kSmemBytes = kStages * kStageBytes + 1024 /*barriers*/ + 1024 /*align*/;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kGroupM = 16;            // raster: tile-rows per group

// Error word shared by all kernels of the library on one device: 0, or
// 0x80000000 | (code of the first wait that timed out).
__device__ unsigned int g_tcg_status = 0;

struct GemmParams {
  int32_t M, N, K;
  int32_t tiles_m, tiles_n, num_kb, num_tiles;
  // schedule: CTA b takes whole tiles b + i*gridDim.x (i < dp_waves, tile <
  // dp_end), then sub-tile units u = b + j*gridDim.x (u < (num_tiles -
  // dp_end) * split) of the remaining tiles, each split into `split` pieces
  // along N.
  int32_t dp_waves, dp_end, split;
  uint32_t fp8_fmt;  // FP8: A/B format fields of the instruction descriptor
  // Rows of A per TMA box: 128, or M rounded up to 8 when M < 128 (a box
  // reaching far past a few-row A made every stage slower: M = 1, N = 28672,
  // K = 8192 BF16 112 us against 78).  The MMA still reads 128 rows; the rest
  // hold stale data and feed only output rows >= M, which are never stored.
  uint32_t a_rows;
  const void* C;
  int64_t ldc;
  void* D;
  int64_t ldd;
  float alpha, beta;
  const float* a_scale;  // FP8 per-tensor scales (device), else null
  const float* b_scale;
};

__device__ __forceinline__ void record_timeout(uint32_t where) {
  atomicCAS(&g_tcg_status, 0u, 0x80000000u | where);
}

// Bounded wait for phase `parity` of `bar`; false on timeout or when another
// role has already aborted.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           uint32_t where) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
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

// Tile t -> (tile row, tile column).  Tiles run down a band of kGroupM tile
// rows before moving to the next column, so a wave of CTAs shares A rows and
// B columns in L2.
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int& tm, int& tn) {
  const int group_tiles = kGroupM * tiles_n;
  const int g = t / group_tiles;
  const int first_m = g * kGroupM;
  const int gm = min(tiles_m - first_m, kGroupM);
  const int local = t - g * group_tiles;
  tm = first_m + local % gm;
  tn = local / gm;
}

// One unit of work: columns [sub*256/split, (sub+1)*256/split) of tile `tile`.
struct WorkItem {
  int tile, sub, split;
};

// The sequence of work items of one CTA; every role walks the same sequence.
struct WorkIter {
  int b, G, i, j, dp_waves, dp_end, split, tail_units;
  __device__ __forceinline__ void init(const GemmParams& p) {
    b = blockIdx.x;
    G = gridDim.x;
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

// Scales 32 accumulator values of one row, adds beta*C, converts and stores
// them at D[row, col0 .. col0+31] (columns >= N are skipped).
template <int kOut, bool kHasC>
__device__ __forceinline__ void store_row_chunk(const GemmParams& p, int row, int col0,
                                                const float (&acc)[32], float scale) {
  if (row >= p.M || col0 >= p.N) return;
  const bool full_chunk = col0 + 32 <= p.N;
  const float beta = p.beta;
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = scale * acc[j];
  if (kOut == 1) {
    float* drow = static_cast<float*>(p.D) + (int64_t)row * p.ldd + col0;
    const float* crow =
        kHasC ? static_cast<const float*>(p.C) + (int64_t)row * p.ldc + col0 : nullptr;
    if (full_chunk) {
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        float4 o = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        if (kHasC) {
          const float4 cv = *reinterpret_cast<const float4*>(crow + j);
          o.x += beta * cv.x;
          o.y += beta * cv.y;
          o.z += beta * cv.z;
          o.w += beta * cv.w;
        }
        *reinterpret_cast<float4*>(drow + j) = o;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (col0 + j < p.N) {
          float o = v[j];
          if (kHasC) o += beta * crow[j];
          drow[j] = o;
        }
      }
    }
  } else {
    uint16_t* drow = static_cast<uint16_t*>(p.D) + (int64_t)row * p.ldd + col0;
    const uint16_t* crow =
        kHasC ? static_cast<const uint16_t*>(p.C) + (int64_t)row * p.ldc + col0 : nullptr;
    if (full_chunk) {
#pragma unroll
      for (int j = 0; j < 32; j += 8) {
        if (kHasC) {
          const uint4 cv = *reinterpret_cast<const uint4*>(crow + j);
          v[j + 0] += beta * bf16_lo_to_f32(cv.x);
          v[j + 1] += beta * bf16_hi_to_f32(cv.x);
          v[j + 2] += beta * bf16_lo_to_f32(cv.y);
          v[j + 3] += beta * bf16_hi_to_f32(cv.y);
          v[j + 4] += beta * bf16_lo_to_f32(cv.z);
          v[j + 5] += beta * bf16_hi_to_f32(cv.z);
          v[j + 6] += beta * bf16_lo_to_f32(cv.w);
          v[j + 7] += beta * bf16_hi_to_f32(cv.w);
        }
        uint4 o;
        o.x = pack_bf16x2(v[j + 0], v[j + 1]);
        o.y = pack_bf16x2(v[j + 2], v[j + 3]);
        o.z = pack_bf16x2(v[j + 4], v[j + 5]);
        o.w = pack_bf16x2(v[j + 6], v[j + 7]);
        *reinterpret_cast<uint4*>(drow + j) = o;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (col0 + j < p.N) {
          float o = v[j];
          if (kHasC) o += beta * __uint_as_float((uint32_t)crow[j] << 16);
          drow[j] = (uint16_t)(pack_bf16x2(o, 0.0f) & 0xFFFFu);
        }
      }
    }
  }
}

// kIn: 0 = BF16, 1 = E4M3.  kOut: 0 = BF16, 1 = FP32.  kHasC: beta != 0.
template <int kIn, int kOut, bool kHasC>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tn_kernel(const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ CUtensorMap tmap_b, const GemmParams p) {
  constexpr int kBKElems = kIn == 0 ? kBKBytes / 2 : kBKBytes;
  // BF16 -> format 1 of kind::f16; E4M3 -> format 0 of kind::f8f6f4.
  constexpr uint32_t kFmt = kIn == 0 ? 1u : 0u;
  constexpr uint32_t kIdesc256 = make_idesc(kFmt, kFmt, kBM, 256);
  constexpr uint32_t kIdesc128 = make_idesc(kFmt, kFmt, kBM, 128);
  constexpr uint32_t kIdesc64 = make_idesc(kFmt, kFmt, kBM, 64);
  // Each MMA consumes 32 bytes of K (16 BF16 or 32 E4M3 values); the
  // descriptor start address advances by 32 bytes (2 in its >>4 units)
  // inside the 128-byte swizzled row.
  constexpr int kMmaPerStage = kBKBytes / 32;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + kStages * kStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (kStages + s); };
  auto tfull_bar = [&](uint32_t a) { return bar0 + 8u * (2 * kStages + a); };
  auto tempty_bar = [&](uint32_t a) { return bar0 + 8u * (2 * kStages + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 4);
  auto a_smem = [&](uint32_t s) { return sbase + s * kStageBytes; };
  auto b_smem = [&](uint32_t s) { return sbase + s * kStageBytes + kATileBytes; };

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4);  // one arrival per epilogue warp
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
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
      {  // warm L2 with the first stages while the previous kernel drains
        WorkIter wi;
        wi.init(p);
        WorkItem w;
        if (wi.next(w)) {
          int tm, tn;
          tile_coords(w.tile, p.tiles_m, p.tiles_n, tm, tn);
          const int nboxes = (kBN / kBBoxRows) / w.split;
          const int brow0 = tn * kBN + w.sub * (kBN / w.split);
          for (int kb = 0; kb < kStages && kb < p.num_kb; ++kb) {
            tma_prefetch_l2_2d(&tmap_a, kb * kBKElems, tm * kBM);
            for (int bx = 0; bx < nboxes; ++bx)
              tma_prefetch_l2_2d(&tmap_b, kb * kBKElems, brow0 + bx * kBBoxRows);
          }
        }
      }
    }
  }
  // The set-up above may overlap the previous kernel's tail; global memory
  // is read or written only after it has finished.
  grid_dependency_wait();

  if (warp == 0) {
    // ------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      WorkIter wi;
      wi.init(p);
      WorkItem w;
      while (ok && wi.next(w)) {
        int tm, tn;
        tile_coords(w.tile, p.tiles_m, p.tiles_n, tm, tn);
        const int nboxes = (kBN / kBBoxRows) / w.split;
        const int brow0 = tn * kBN + w.sub * (kBN / w.split);
        const uint32_t bytes = p.a_rows * kBKBytes + (uint32_t)nboxes * kBBoxRows * kBKBytes;
        for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
          if (!wait_phase(empty_bar(s), ph ^ 1u, abort_flag, 1)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(s), bytes);
          tma_load_2d(a_smem(s), &tmap_a, full_bar(s), kb * kBKElems, tm * kBM);
          for (int bx = 0; bx < nboxes; ++bx)
            tma_load_2d(b_smem(s) + (uint32_t)bx * kBBoxRows * kBKBytes, &tmap_b, full_bar(s),
                        kb * kBKElems, brow0 + bx * kBBoxRows);
        }
      }
      grid_launch_dependents();  // every load is issued: the next kernel may launch
      if (!ok) {
        // Let the copies already issued land before the CTA can exit.
        const uint32_t n = it < (uint32_t)kStages ? it : (uint32_t)kStages;
        for (uint32_t j = it - n; j < it; ++j) {
          const uint32_t s = j % kStages, ph = (j / kStages) & 1u;
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(full_bar(s), ph) && global_timer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
    __syncwarp();  // reconverge before the CTA barrier
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t it = 0, lt = 0;
      bool ok = true, issued = false;
      WorkIter wi;
      wi.init(p);
      WorkItem w;
      for (; ok && wi.next(w); ++lt) {
        const uint32_t acc = lt & 1u, aph = (lt >> 1) & 1u;
        if (!wait_phase(tempty_bar(acc), aph ^ 1u, abort_flag, 2)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * kAccCols;
        const uint32_t idesc = (w.split == 1 ? kIdesc256 : w.split == 2 ? kIdesc128 : kIdesc64) |
                               (kIn == 1 ? p.fp8_fmt : 0u);
        static_assert(kMmaPerStage == 4, "one K step is four 32-byte MMAs");
        // the unit's first K step is waited for here; every later one was
        // tested while the step before it was issued (mma_step4_test_next)
        bool ready = false;
        for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
          if (!ready && !wait_phase(full_bar(s), ph, abort_flag, 3)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t ad = smem_desc_k_sw128(a_smem(s));
          const uint64_t bd = smem_desc_k_sw128(b_smem(s));
          const bool more = kb + 1 < p.num_kb;
          const uint32_t s1 = (it + 1u) % kStages, ph1 = ((it + 1u) / kStages) & 1u;
          const uint32_t got = mma_step4_test_next<kIn>(d_tmem, ad, bd, idesc, kb != 0 ? 1u : 0u,
                                                        empty_bar(s), more ? full_bar(s1) : full_bar(s),
                                                        more ? ph1 : ph);
          ready = more && got != 0u;
          issued = true;
        }
        if (ok) tc_commit(tfull_bar(acc));
      }
      if (!ok && issued) {
        // Wait (bounded) for this thread's MMAs before TMEM is freed.
        tc_commit(drain_bar);
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(drain_bar, 0) && global_timer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------- epilogue
    const uint32_t q = warp & 3u;  // TMEM lane quarter this warp may access
    const int row_in_tile = (int)(q * 32u + lane);
    float scale = p.alpha;
    if (kIn == 1) scale = p.a_scale[0] * p.b_scale[0] * p.alpha;
    uint32_t lt = 0;
    WorkIter wi;
    wi.init(p);
    WorkItem w;
    for (; wi.next(w); ++lt) {
      const uint32_t acc = lt & 1u, aph = (lt >> 1) & 1u;
      uint32_t ok = 0;
      if (lane == 0) ok = wait_phase(tfull_bar(acc), aph, abort_flag, 4) ? 1u : 0u;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after_sync();
      int tm, tn;
      tile_coords(w.tile, p.tiles_m, p.tiles_n, tm, tn);
      const int row = tm * kBM + row_in_tile;
      const int col_base = tn * kBN + w.sub * (kBN / w.split);
      const int nchunks = (kBN / 32) / w.split;
      const uint32_t t_row = tmem_base + ((q * 32u) << 16) + acc * kAccCols;
#pragma unroll 1
      for (int c = 0; c < nchunks; ++c) {
        uint32_t r[32];
        __syncwarp();  // tcgen05.ld is .sync.aligned: reconverge after the stores
        tmem_ld_32x32b_x32(t_row + (uint32_t)(c * 32), r);
        tmem_ld_wait(r);
        if (c == nchunks - 1) {
          // Accumulator fully read: hand the buffer back to the MMA warp.
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty_bar(acc));
        }
        float a[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) a[j] = __uint_as_float(r[j]);
        store_row_chunk<kOut, kHasC>(p, row, col_base + c * 32, a, scale);
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace tcg
