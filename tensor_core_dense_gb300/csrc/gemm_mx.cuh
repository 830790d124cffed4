// gemm_mx.cuh -- microscaled FP8 GEMM on CTA pairs: the hardware block
// scaling of tcgen05.mma kind::mxf8f6f4.
//
//   D = alpha * sum_kb (SFA[i,kb] SFB[j,kb]) * sum_{k in block kb} a_ik b_kj (+ beta * C)
//
// with one E8M0 scale (a power of two, 2^(e - 127)) per row and 32-wide K
// block of A and of B.  This is the block-scaled MMA of "How Blackwell's
// Tensor Memory Actually Works", "Quantization became an allocation
// problem": D = C + (A x SFA)(B x SFB), the scale factors consumed by the
// tensor core from Tensor Memory as it runs, not folded in before or applied
// after, so the K loop has no promotion step (compare gemm_tn2b.cuh).
//
// Structure: the 256 x 256 CTA-pair tile, roles and schedule of gemm_tn2.cuh.
// What the scales change ("the largest accumulator takes half, block scale
// factors take a few more", same page, the Tensor Memory ledger):
//   * each stage carries, beside A and B, this CTA's A scales (one 512-byte
//     tile: 128 rows x 4 blocks) and the B scales of all 256 columns of the
//     pair's tile (two such tiles: the tensor core of each SM reads the scales
//     of every column from its own Tensor Memory), loaded by TMA on the
//     stage's mbarrier, tiles past the last row tile reading as zeros: A
//     through a 3-D tensor map (128 words x K tiles x row tiles), B through a
//     4-D one whose second dimension repeats each tile 4 times (stride 0), so
//     the two B tiles land as the 128-row x 32-byte image, each lane quarter
//     holding the 32-row pattern, that one copy spreads over 8 columns;
//   * the MMA thread copies them to Tensor Memory, 12 columns per stage after
//     the accumulator (A at +0 with tcgen05.cp 32x128b.warpx4, B at +4..+11
//     with one 128x256b), issued before the stage's MMAs, which it orders.
//     Each copy costs about 70 tensor cycles in the MMA stream whatever its
//     size (three per stage measured 57.2 us at 4096^3, none 46.4), so the
//     copies are as few and as large as the layout allows;
//   * the accumulator takes 256 columns and the scale slots 72, so there is a
//     single accumulator: eight epilogue warps read all of it into registers
//     (128 columns each), hand it back, and only then scale, convert and
//     store, so the next tile's MMAs wait only for the Tensor Memory reads.
//
// Scale layout in global memory (E8M0 bytes): tiles of 128 rows x 4 blocks
// of 512 bytes, tile (r / 128, kb / 4) at ((r / 128) * KT + kb / 4) * 512,
// KT = ceil(K / 128); inside a tile, row r % 32 owns 16 bytes, (r / 32) % 4
// picks 4 of them and kb % 4 the byte.  That is the order tcgen05.cp's
// 32x128b.warpx4 shape writes Tensor Memory in (32 lanes x 16 bytes,
// repeated for the four lane quarters), and the instruction descriptor's
// scale-factor ids select the byte (the block within the 4).
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "gemm_tn.cuh"
#include "gemm_tn2.cuh"
#include "ptx.cuh"

namespace tcg {

constexpr int kMxStages = 6;
constexpr uint32_t kMxATileBytes = 128 * kBKBytes;     // this CTA's 128 rows of A
constexpr uint32_t kMxBTileBytes = 128 * kBKBytes;     // its half of the B block
constexpr uint32_t kMxSfaBytes = 512;                  // A scales of 128 rows x 4 blocks
constexpr uint32_t kMxSfbBytes = 4096;  // B scales of 256 rows x 4 blocks, each tile 4 times
constexpr uint32_t kMxStageBytes = kMxATileBytes + kMxBTileBytes;  // operand part (1024-aligned)
constexpr int kMxThreads = 320;                        // producer, MMA, 8 epilogue warps
constexpr int kMxNumBars = 2 * kMxStages + 3;          // full, empty, tfull, tempty, drain
constexpr uint32_t kMxSfColBase = 256;                 // TMEM columns after the accumulator
constexpr uint32_t kMxSfColsPerStage = 16;             // A 4 + B 8, rounded to 16
constexpr uint32_t kMxSmemBytes = kMxStages * (kMxStageBytes + kMxSfaBytes + kMxSfbBytes) +
                                  1024 + 1024;

struct MxParams {
  int32_t M, N, K;
  int32_t tiles_m, tiles_n, num_kb, num_tiles;  // 256 x 256 tiles; num_kb = KT
  int32_t dp_waves, dp_end, split;              // the schedule of gemm_tn2.cuh
  uint32_t fp8_fmt;                             // A / B format fields (E4M3 0, E5M2 1)
  const void* C;
  int64_t ldc;
  void* D;
  int64_t ldd;
  float alpha, beta;
};

// Shared-memory descriptor of one 512-byte scale tile as tcgen05.cp reads it:
// 32 rows of 16 bytes, no swizzle, 8-row core matrices 128 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sf_tile(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(128u >> 4) << 16;
  d |= static_cast<uint64_t>(128u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  return d;  // layout 0: no swizzle
}

// Copies a 512-byte scale tile from shared memory into 4 Tensor Memory
// columns of all 128 lanes, in each CTA of the pair from its own shared
// memory (same offsets).
__device__ __forceinline__ void tmem_cp_sf_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// Shared-memory descriptor of the B-scale image as tcgen05.cp's 128x256b
// shape reads it: 128 rows x 32 bytes, no swizzle, the rows' first 16 bytes
// (the first tile, 4 times) in one 2 KB block and the second 16 bytes 2 KB
// further (leading byte offset), 8-row core matrices 128 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sf_image(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(2048u >> 4) << 16;
  d |= static_cast<uint64_t>(128u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  return d;
}

// Copies the 4 KB B-scale image into 8 Tensor Memory columns of all 128
// lanes (each CTA of the pair from its own shared memory).
__device__ __forceinline__ void tmem_cp_sf_image_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Instruction descriptor of kind::mxf8f6f4 with E8M0 scales, both operands
// K-major: scale ids of B (bits 4-5) and A (29-30) pick the byte, i.e. the
// 32-wide block within the 4 of a Tensor Memory column; bit 23 = E8M0; N / 8
// at 17, M / 16 at 24; A / B formats at 7 / 10.
__host__ __device__ constexpr uint32_t make_idesc_mx(uint32_t M, uint32_t N, uint32_t sf_id) {
  return (sf_id << 4) | ((N >> 3) << 17) | (1u << 23) | ((M >> 4) << 24) | (sf_id << 29);
}

__device__ __forceinline__ void mma_mx_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// One K step of the pair: the stage's A and B scales into Tensor Memory, the
// four block-scaled MMAs of its 32-wide K blocks (block k: descriptors + 2k,
// scale id k in the instruction descriptor and in bits 30-31 of both scale
// addresses), and the commit of the stage to `done_bar` in both CTAs. As in
// mma_step4_pair_test_next, the test of the next step's barrier is issued
// first and its result read last, so that the issuing thread never waits on a
// read-back with an empty tcgen05 queue; `idesc` is block 0's descriptor.
__device__ __forceinline__ uint32_t mx_step_pair_test_next(
    uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t sfa_tmem,
    uint32_t sfb_tmem, uint64_t sfa_sdesc, uint64_t sfb_sdesc, uint32_t accumulate,
    uint32_t done_bar, uint32_t next_bar, uint32_t next_par) {
  uint32_t ready;
  asm volatile(
      "{\n\t.reg .pred rdy, acc, one;\n\t"
      ".reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
      ".reg .b32 i1, i2, i3, sa1, sa2, sa3, sb1, sb2, sb3;\n\t"
      "setp.ne.b32 acc, %9, 0;\n\t"
      "setp.eq.b32 one, 0, 0;\n\t"
      "add.s64 a1, %2, 2;\n\t"
      "add.s64 a2, %2, 4;\n\t"
      "add.s64 a3, %2, 6;\n\t"
      "add.s64 b1, %3, 2;\n\t"
      "add.s64 b2, %3, 4;\n\t"
      "add.s64 b3, %3, 6;\n\t"
      "or.b32 i1, %4, 0x20000010;\n\t"
      "or.b32 i2, %4, 0x40000020;\n\t"
      "or.b32 i3, %4, 0x60000030;\n\t"
      "or.b32 sa1, %5, 0x40000000;\n\t"
      "or.b32 sa2, %5, 0x80000000;\n\t"
      "or.b32 sa3, %5, 0xC0000000;\n\t"
      "or.b32 sb1, %6, 0x40000000;\n\t"
      "or.b32 sb2, %6, 0x80000000;\n\t"
      "or.b32 sb3, %6, 0xC0000000;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 rdy, [%11], %12;\n\t"
      "tcgen05.cp.cta_group::2.32x128b.warpx4 [%5], %7;\n\t"
      "tcgen05.cp.cta_group::2.128x256b [%6], %8;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%1], %2, %3, %4, [%5], [%6], acc;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%1], a1, b1, i1, [sa1], [sb1], one;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%1], a2, b2, i2, [sa2], [sb2], one;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%1], a3, b3, i3, [sa3], [sb3], one;\n\t"
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%10], %13;\n\t"
      "selp.u32 %0, 1, 0, rdy;\n\t}"
      : "=r"(ready)
      : "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem),
        "l"(sfa_sdesc), "l"(sfb_sdesc), "r"(accumulate), "r"(done_bar), "r"(next_bar),
        "r"(next_par), "h"((uint16_t)0x3)
      : "memory");
  return ready;
}

template <int kOut, bool kHasC>
__global__ void __launch_bounds__(kMxThreads, 1)
    gemm_mx_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_b,
                        const __grid_constant__ CUtensorMap tmap_sfa,
                        const __grid_constant__ CUtensorMap tmap_sfb, const MxParams p) {
  constexpr int S = kMxStages;
  constexpr int kMmaPerStage = kBKBytes / 32;  // 4 blocks of 32 FP8 values

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  const uint32_t sf_base = sbase + S * kMxStageBytes;  // S x (A scales, B scales)
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(gbase + S * (kMxStageBytes + kMxSfaBytes + kMxSfbBytes));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kMxNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (S + s); };
  const uint32_t tfull_bar = bar0 + 8u * (2 * S);
  const uint32_t tempty_bar = bar0 + 8u * (2 * S + 1);
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 2);
  auto a_smem = [&](uint32_t s) { return sbase + s * kMxStageBytes; };
  auto b_smem = [&](uint32_t s) { return sbase + s * kMxStageBytes + kMxATileBytes; };
  auto sfa_smem = [&](uint32_t s) { return sf_base + s * (kMxSfaBytes + kMxSfbBytes); };
  auto sfb_smem = [&](uint32_t s) { return sfa_smem(s) + kMxSfaBytes; };

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = (int)(blockIdx.x >> 1);
  const int clusters = (int)(gridDim.x >> 1);
  // Gemm2Params view of the schedule for the shared work iterator
  Gemm2Params sched{};
  sched.num_tiles = p.num_tiles;
  sched.dp_waves = p.dp_waves;
  sched.dp_end = p.dp_end;
  sched.split = p.split;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, 16);  // 8 epilogue warps in each CTA of the pair
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
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
    tma_prefetch_desc(&tmap_sfa);
    tma_prefetch_desc(&tmap_sfb);
  }
  grid_dependency_wait();  // global memory only after the previous kernel finished

  if (warp == 0) {
    // ------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      PairWorkIter wi;
      wi.init(sched, cluster, clusters);
      WorkItem w;
      while (ok && wi.next(w)) {
        int tm, tn;
        tile_coords(w.tile, p.tiles_m, p.tiles_n, tm, tn);
        const int nsub = 256 / w.split;              // tile columns of this unit
        const int half = nsub / 2;                   // rows of B this CTA loads
        const int nboxes = half / kBBoxRows;         // 2 or 1
        const int col0 = tn * 256 + w.sub * nsub;    // first column of the unit
        const int brow0 = col0 + (int)rank * half;
        const int arow0 = tm * 256 + (int)rank * 128;
        // scale tiles: this CTA's 128 rows of A, and the two 128-row tiles
        // from the unit's first column of B (the second unused by a unit of
        // 128 columns; tiles past M or N read as zeros and only feed outputs
        // that are never stored)
        const uint32_t my_bytes =
            kMxATileBytes + (uint32_t)half * kBKBytes + kMxSfaBytes + kMxSfbBytes;
        for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
          const uint32_t s = it % S, ph = (it / S) & 1u;
          if (!wait_phase(empty_bar(s), ph ^ 1u, abort_flag, 0x41)) {
            ok = false;
            break;
          }
          const uint32_t fb = map_shared_to_cta(full_bar(s), 0);  // the leader's barrier
          if (leader) mbar_arrive_expect_tx(full_bar(s), 2u * my_bytes);
          tma_load_2d_pair(a_smem(s), &tmap_a, fb, kb * kBKBytes, arow0);
          for (int bx = 0; bx < nboxes; ++bx)
            tma_load_2d_pair(b_smem(s) + (uint32_t)bx * kBBoxRows * kBKBytes, &tmap_b, fb,
                             kb * kBKBytes, brow0 + bx * kBBoxRows);
          tma_load_3d_pair(sfa_smem(s), &tmap_sfa, fb, 0, kb, arow0 / 128);
          tma_load_4d_pair(sfb_smem(s), &tmap_sfb, fb, 0, 0, kb, col0 / 128);
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
      wi.init(sched, cluster, clusters);
      WorkItem w;
      for (; ok && wi.next(w); ++lt) {
        // both CTAs' epilogues have read the accumulator of the previous unit
        if (lt > 0) {
          bool free_ok = mbar_try_wait_cluster(tempty_bar, (lt - 1u) & 1u);
          if (!free_ok) {
            const uint64_t t0 = global_timer_ns();
            for (uint32_t i = 1; !free_ok; ++i) {
              free_ok = mbar_try_wait_cluster(tempty_bar, (lt - 1u) & 1u);
              if (!free_ok && (i & 31u) == 0u) {
                if (*abort_flag) break;
                if (global_timer_ns() - t0 > kWaitLimitNs) {
                  record_timeout(0x42);
                  *abort_flag = 1;
                  break;
                }
              }
            }
          }
          if (!free_ok) break;
        }
        tc_fence_after_sync();
        const uint32_t nsub = 256u / (uint32_t)w.split;
        static_assert(kMmaPerStage == 4, "one K step is four 32-wide scale blocks");
        const uint32_t idesc0 = make_idesc_mx(256, nsub, 0u) | p.fp8_fmt;
        // The unit's first K step is waited for here; every later one was
        // tested while the step before it was issued.
        bool ready = false;
        for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
          const uint32_t s = it % S, ph = (it / S) & 1u;
          if (!ready && !wait_phase(full_bar(s), ph, abort_flag, 0x43)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          // scales of this stage into its Tensor Memory slot; the slot was
          // last read by the MMAs of stage it - S, which completed before the
          // producer could refill the stage
          const uint32_t sfa_t = tmem_base + kMxSfColBase + s * kMxSfColsPerStage;
          const uint32_t sfb_t = sfa_t + 4u;
          const uint64_t ad = smem_desc_k_sw128(a_smem(s));
          const uint64_t bd = smem_desc_k_sw128(b_smem(s));
          const bool more = kb + 1 < p.num_kb;
          const uint32_t s1 = (it + 1u) % S, ph1 = ((it + 1u) / S) & 1u;
          const uint32_t got = mx_step_pair_test_next(
              tmem_base, ad, bd, idesc0, sfa_t, sfb_t, smem_desc_sf_tile(sfa_smem(s)),
              smem_desc_sf_image(sfb_smem(s)), kb != 0 ? 1u : 0u, empty_bar(s),
              more ? full_bar(s1) : full_bar(s), more ? ph1 : ph);
          ready = more && got != 0u;
          issued = true;
        }
        if (ok) tc_commit_pair(tfull_bar, 0x3);
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
    // warps 2..9: TMEM lane quarter q, column half h of the unit
    const uint32_t q = warp & 3u;
    const uint32_t h = (warp - 2u) >> 2;
    const int row_in_tile = (int)(rank * 128u + q * 32u + lane);
    const uint32_t leader_tempty = map_shared_to_cta(tempty_bar, 0);
    Gemm2Params st{};  // store view of D and C
    st.M = p.M;
    st.N = p.N;
    st.C = p.C;
    st.ldc = p.ldc;
    st.D = p.D;
    st.ldd = p.ldd;
    st.beta = p.beta;
    uint32_t lt = 0;
    PairWorkIter wi;
    wi.init(sched, cluster, clusters);
    WorkItem w;
    for (; wi.next(w); ++lt) {
      uint32_t ok = 0;
      if (lane == 0) ok = wait_phase(tfull_bar, lt & 1u, abort_flag, 0x44) ? 1u : 0u;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after_sync();
      int tm, tn;
      tile_coords(w.tile, p.tiles_m, p.tiles_n, tm, tn);
      const int nsub = 256 / w.split;
      const int row = tm * 256 + row_in_tile;
      const int c0 = (int)h * (nsub / 2);  // this warp's first column in the unit
      const int col_base = tn * 256 + w.sub * nsub + c0;
      const uint32_t t_row = tmem_base + ((q * 32u) << 16) + (uint32_t)c0;
      if (nsub == 256) {
        uint32_t r0[64], r1[64];
        tmem_ld_32x32b_x64(t_row, r0);
        tmem_ld_32x32b_x64(t_row + 64u, r1);
        tmem_ld_wait_n<64>(r0);
        tmem_ld_wait_n<64>(r1);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote_cta(leader_tempty);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float a[32];
#pragma unroll
          for (int j = 0; j < 32; ++j)
            a[j] = __uint_as_float(c < 2 ? r0[32 * c + j] : r1[32 * (c - 2) + j]);
          store_row_chunk2<kOut, kHasC>(st, row, col_base + 32 * c, a, p.alpha);
        }
      } else {
        uint32_t r0[64];
        tmem_ld_32x32b_x64(t_row, r0);
        tmem_ld_wait_n<64>(r0);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote_cta(leader_tempty);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float a[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) a[j] = __uint_as_float(r0[32 * c + j]);
          store_row_chunk2<kOut, kHasC>(st, row, col_base + 32 * c, a, p.alpha);
        }
      }
      __syncwarp();  // tcgen05.ld is .sync.aligned: reconverge after the stores
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while the pair may still use its memory
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

}  // namespace tcg
