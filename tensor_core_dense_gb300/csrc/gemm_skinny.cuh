// gemm_skinny.cuh -- swap-AB GEMM for skinny M: FP8 with 128-block scales (M
// <= 128 in one chunk, larger M in chunks of 128 rows), and for M <= 128 also
// per-tensor FP8 and BF16 (one scale product for every step, or 1).
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
// Larger M is cut into chunks of 128 rows of A: a tile is then (N tile, M
// chunk), a 128 x 128 block of D, with the same steps and promotion.
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
// slot as soon as its part is summed, and only at the end of its range (so
// the pipeline never stops in the middle) bumps the tiles' counters; the last
// CTA to arrive at a tile adds the slots in slot order (deterministic) and
// writes D.  Only the first and the last piece of a CTA's range can be
// partial tiles.
//
// When every tile is split into exactly kJoin = 2 or 3 pieces (N tiles *
// kJoin <= SMs, e.g. N = 8192 in two, N <= 6400 in three), the CTAs of a tile
// form a cluster instead: each leaves its FP32 partial in its own shared
// memory, and after a cluster barrier CTA r adds the pieces (lowest K range
// first, so the result is the same every run) for its share of the tile's
// outputs, reading the others' partials over distributed shared memory -- no
// workspace, no atomics, no global round trip at the end.
//
// Roles: warp 0 TMA producer (one lane), warp 1 TMEM allocator + MMA issuer
// (one lane), then two (Mp <= 32) or four (Mp >= 64) epilogue warpgroups;
// warpgroup h promotes its own slice of Mp/2 or Mp/4 columns of every
// partial.  The MMA writes
// each K block's partial into one of four (Mp = 128) or eight TMEM buffers;
// the epilogue drains it, multiplies by sa*sb (read from a shared-memory table
// of the CTA's scale products, filled once with all its loads in flight) and
// adds it into registers.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "gemm_tn.cuh"
#include "ptx.cuh"

namespace tcg {


constexpr uint32_t kSkBTileBytes = 128 * 128; // 128 rows of B x 128 K bytes
constexpr int kSkMaxSeg = 4;                  // CTAs sharing one tile, at most

template <int kMp>
struct SkinnyCfg {
  static constexpr uint32_t kATileBytes = kMp * 128;
  static constexpr uint32_t kStageBytes = kSkBTileBytes + kATileBytes;
  // scale-product table: kTabSteps K blocks x kMp columns of sa*sb
  static constexpr uint32_t kTabBytes = 16u * 1024u;
  static constexpr int kTabSteps = (int)(kTabBytes / (kMp * 4u));
  static constexpr int kStagesRaw = (int)((224u * 1024u - kTabBytes - 2048u) / kStageBytes);
  static constexpr int kStages = kStagesRaw > 10 ? 10 : kStagesRaw;
  static constexpr int kNumAcc = kMp >= 128 ? 4 : 8;  // TMEM partial buffers
  static constexpr int kCols = kMp * kNumAcc;
  static constexpr int kTmemCols = kCols <= 32 ? 32 : kCols <= 64 ? 64 : kCols <= 128 ? 128
                                   : kCols <= 256 ? 256 : 512;
  // epilogue: kEpiWG warpgroups, warpgroup h promotes columns
  // [h*kCols, (h+1)*kCols) of every partial
  static constexpr int kEpiWG = kMp >= 64 ? 4 : 2;
  static constexpr int kEpiWarps = 4 * kEpiWG;
  static constexpr int kEpiThreads = 32 * kEpiWarps;
  static constexpr int kThreads = 64 + kEpiThreads;
  static constexpr int kHalf = kMp / kEpiWG;  // columns per epilogue warp
  static constexpr int kNumBars = 2 * kStages + 2 * kNumAcc + 4;
  static constexpr uint32_t kSmemBytes = kStages * kStageBytes + 1024u + kTabBytes + 1024u;
  static_assert(kMp % 16 == 0 && kMp >= 16 && kMp <= 128, "UMMA N");
};

struct SkinnyParams {
  int32_t M, N, K;
  int32_t n_tiles, num_kb, total_steps, grid, max_seg;
  int32_t m_tiles;   // M in chunks of kMp rows (1 when M <= 128)
  // 1: CTA c takes whole tiles [c*tiles/grid, (c+1)*tiles/grid), all of K,
  // so no tile is split and ws / counters are never touched; 0: the steps
  // are cut into grid equal ranges (stream-K)
  int32_t whole_tiles;
  const float* a_scale;  // [KB][M]
  const float* b_scale;  // [ceil(N/128)][KB]
  const void* C;
  int64_t ldc;
  void* D;
  int64_t ldd;
  float alpha, beta;
  int32_t out_f32, has_c;
  uint32_t fp8_fmt;  // UMMA A (= B, the weights) / UMMA B (= A) format fields
  int32_t pad_;
  float* ws;               // [grid][2][Mp][128] partial sums: a CTA's first and last piece
  unsigned int* counters;  // [n_tiles * m_tiles], zero between calls
};

// Tile t (of n_tiles * m_tiles) -> N tile and M chunk.  Tiles that share an
// N tile (the same slab of B, the HBM stream) are consecutive, so CTAs working
// on different M chunks of one slab read it at about the same time.
__host__ __device__ __forceinline__ void sk_tile(int t, int m_tiles, int& ntile, int& mt) {
  ntile = t / m_tiles;
  mt = t - ntile * m_tiles;
}

__host__ __device__ __forceinline__ int64_t sk_range_start(int64_t c, int64_t T, int64_t G) {
  return c * T / G;
}
// The CTA whose range holds step x.
__host__ __device__ __forceinline__ int64_t sk_owner(int64_t x, int64_t T, int64_t G) {
  return ((x + 1) * G - 1) / T;
}

// D[m, n] = alpha * val (+ beta * C[m, n]), skipping the padding rows and
// columns (m >= M, n >= N).
__device__ __forceinline__ void emit_one(const SkinnyParams& p, int m, int n, float val) {
  if (m >= p.M || n >= p.N) return;
  float o = p.alpha * val;
  if (p.out_f32) {
    if (p.has_c) o += p.beta * static_cast<const float*>(p.C)[(int64_t)m * p.ldc + n];
    static_cast<float*>(p.D)[(int64_t)m * p.ldd + n] = o;
  } else {
    if (p.has_c)
      o += p.beta *
           __uint_as_float((uint32_t)static_cast<const uint16_t*>(p.C)[(int64_t)m * p.ldc + n]
                           << 16);
    static_cast<uint16_t*>(p.D)[(int64_t)m * p.ldd + n] =
        (uint16_t)(pack_bf16x2(o, 0.0f) & 0xFFFFu);
  }
}

// Four consecutive outputs D[m, n .. n+3] (n a multiple of 4): one vector
// store when all four are inside the matrix.
__device__ __forceinline__ void emit_four(const SkinnyParams& p, int m, int n, float4 v) {
  if (m >= p.M || n >= p.N) return;
  if (n + 4 > p.N) {
    emit_one(p, m, n + 0, v.x);
    emit_one(p, m, n + 1, v.y);
    emit_one(p, m, n + 2, v.z);
    emit_one(p, m, n + 3, v.w);
    return;
  }
  float o[4] = {p.alpha * v.x, p.alpha * v.y, p.alpha * v.z, p.alpha * v.w};
  if (p.out_f32) {
    float* d = static_cast<float*>(p.D) + (int64_t)m * p.ldd + n;
    if (p.has_c) {
      const float4 c = *reinterpret_cast<const float4*>(static_cast<const float*>(p.C) +
                                                        (int64_t)m * p.ldc + n);
      o[0] += p.beta * c.x;
      o[1] += p.beta * c.y;
      o[2] += p.beta * c.z;
      o[3] += p.beta * c.w;
    }
    *reinterpret_cast<float4*>(d) = make_float4(o[0], o[1], o[2], o[3]);
  } else {
    uint16_t* d = static_cast<uint16_t*>(p.D) + (int64_t)m * p.ldd + n;
    if (p.has_c) {
      const uint2 c = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.C) +
                                                      (int64_t)m * p.ldc + n);
      o[0] += p.beta * bf16_lo_to_f32(c.x);
      o[1] += p.beta * bf16_hi_to_f32(c.x);
      o[2] += p.beta * bf16_lo_to_f32(c.y);
      o[3] += p.beta * bf16_hi_to_f32(c.y);
    }
    *reinterpret_cast<uint2*>(d) = make_uint2(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]));
  }
}

// kMChunks: M > 128, A in chunks of kMp = 128 rows.  Without it m_tiles is the
// constant 1, so the chunk index folds away (M <= 128 keeps its lean code).
// kIn: 1 = FP8 (kind::f8f6f4, 128 K elements per step), 0 = BF16 (kind::f16,
// 64 K elements per step: a step is 128 bytes of K either way).
// kJoin: 0 = partial tiles through the global workspace; 2 or 3 = every tile
// is split into kJoin pieces computed by the CTAs of one cluster, which join
// them in distributed shared memory.
// kScalar: one scale for the whole problem, a_scale[0] * b_scale[0] (per-
// tensor FP8; 1 for a null pointer, as for BF16): no scale table.  With Mp =
// 128, where nothing changes across K, the MMA also accumulates a CTA's whole
// piece of a tile in Tensor Memory and the epilogue drains it once instead of
// promoting every step (N = K = 8192: BF16 36.3 -> 34.2 us); for smaller Mp
// the MMAs into one accumulator serialise (BF16 M = 16: 26.1 -> 29.5 us), so
// those keep one buffer per step and promote with the one scale.
template <int kMp, int kJoin, bool kMChunks, int kIn = 1, bool kScalar = false>
__global__ void __launch_bounds__(SkinnyCfg<kMp>::kThreads, 1)
    gemm_fp8_block_skinny_kernel(const __grid_constant__ CUtensorMap tmap_a,
                                 const __grid_constant__ CUtensorMap tmap_b,
                                 const SkinnyParams p) {
  using Cfg = SkinnyCfg<kMp>;
  constexpr int kKElems = kIn == 1 ? 128 : 64;  // K elements per 128-byte step
  constexpr bool kAccTmem = kScalar && kMp == 128;  // a piece accumulates in TMEM
  constexpr int S = Cfg::kStages;
  constexpr int kHalf = Cfg::kHalf;
  constexpr int kSkNumAcc = Cfg::kNumAcc;
  constexpr int kSkEpiThreads = Cfg::kEpiThreads;
  constexpr uint32_t kEpiWarps = Cfg::kEpiWarps;
  // FP8 x FP8 (formats from p.fp8_fmt) or BF16 x BF16 -> F32, M=128, N=Mp
  const uint32_t kIdesc =
      kIn == 1 ? make_idesc(0, 0, 128, kMp) | p.fp8_fmt : make_idesc(1, 1, 128, kMp);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + S * Cfg::kStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [2]
  float* stab = reinterpret_cast<float*>(gbase + S * Cfg::kStageBytes + 1024);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](uint32_t b) { return bar0 + 8u * (2 * S + b); };
  auto tempty_bar = [&](uint32_t b) { return bar0 + 8u * (2 * S + kSkNumAcc + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 2 * kSkNumAcc);
  const uint32_t seg_bar = bar0 + 8u * (2 * S + 2 * kSkNumAcc + 1);   // epilogue warps done
  const uint32_t flag_bar = bar0 + 8u * (2 * S + 2 * kSkNumAcc + 2);  // last_flag published
  const uint32_t tab_bar = bar0 + 8u * (2 * S + 2 * kSkNumAcc + 3);   // epilogue group sync
  auto b_smem = [&](uint32_t s) { return sbase + s * Cfg::kStageBytes; };
  auto a_smem = [&](uint32_t s) { return sbase + s * Cfg::kStageBytes + kSkBTileBytes; };

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;
  const int64_t T = p.total_steps, G = p.grid;
  const int KB = p.num_kb;
  const int64_t s0 = p.whole_tiles ? sk_range_start(blockIdx.x, T / KB, G) * KB
                                   : sk_range_start(blockIdx.x, T, G);
  const int64_t s1 = p.whole_tiles ? sk_range_start(blockIdx.x + 1, T / KB, G) * KB
                                   : sk_range_start(blockIdx.x + 1, T, G);
  const int32_t m_tiles = kMChunks ? p.m_tiles : 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < kSkNumAcc; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), kEpiWarps);  // one arrival per epilogue warp
    }
    mbar_init(drain_bar, 1);
    mbar_init(seg_bar, kEpiWarps);
    mbar_init(flag_bar, 1);
    mbar_init(tab_bar, kEpiWarps);
    *abort_flag = 0;
    last_flag[0] = last_flag[1] = 0;
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
  if (warp == 0 && lane == 0) {
    // (no L2 prefetch of the first B tiles here: issuing it delayed the
    // producer's own first loads by about 1.7 us, more than it saved)
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  grid_dependency_wait();  // global memory only after the previous kernel finished

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
        const int q = (int)st / KB;  // steps fit in 32 bits (checked at launch)
        const int kb = (int)st - q * KB;
        int nt, mt;
        sk_tile(q, m_tiles, nt, mt);
        const uint32_t s = j % S, ph = (j / S) & 1u;
        if (!wait_phase(empty_bar(s), ph ^ 1u, abort_flag, 0x11)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(full_bar(s), Cfg::kStageBytes);
        tma_load_2d_hint(b_smem(s), &tmap_b, full_bar(s), kb * kKElems, nt * 128, stream_policy);
        tma_load_2d_hint(a_smem(s), &tmap_a, full_bar(s), kb * kKElems, mt * kMp, keep_policy);
      }
      grid_launch_dependents();  // every load is issued: the next kernel may launch
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
    __syncwarp();  // reconverge before the CTA barrier
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t j = 0;
      uint32_t pc = 0;  // kAccTmem: pieces (a CTA's part of one tile) so far
      bool ok = true, issued = false;
      // Each step's stage and (at a piece start) buffer were tested while the
      // step before it was issued (mma_step4_test2_next) and are waited for
      // only if a test failed. Not in the block-scaled Mp = 128 form: there the
      // promotion warps bound the loop, and an MMA thread freed from its stalls
      // only spins longer on their buffers, next to them (2 % slower).
      constexpr bool kLookAhead = kScalar || kMp < 128;
      bool rdy_full = false, rdy_free = false;
      for (int64_t st = s0; st < s1; ++st, ++j) {
        const uint32_t s = j % S, ph = (j / S) & 1u;
        const int kbs = (int)st - ((int)st / KB) * KB;
        const bool piece_start = !kAccTmem || st == s0 || kbs == 0;
        const bool piece_end = !kAccTmem || kbs == KB - 1 || st == s1 - 1;
        const uint32_t slot = kAccTmem ? pc : j;  // TMEM buffer sequence number
        const uint32_t b = slot % kSkNumAcc, bph = (slot / kSkNumAcc) & 1u;
        if ((piece_start && !rdy_free && !wait_phase(tempty_bar(b), bph ^ 1u, abort_flag, 0x12)) ||
            (!rdy_full && !wait_phase(full_bar(s), ph, abort_flag, 0x13))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint64_t ad = smem_desc_k_sw128(b_smem(s));  // UMMA A: 128 rows of B
        const uint64_t bd = smem_desc_k_sw128(a_smem(s));  // UMMA B: Mp rows of A
        const uint32_t d_tmem = tmem_base + b * kMp;
        // The next step's stage and, if it starts a piece, its buffer. A test
        // that is not needed reads this step's stage, whose phase cannot
        // move before this step's own commit.
        const bool more = kLookAhead && st + 1 < s1;
        const bool next_start = !kAccTmem || (kbs + 1 == KB);
        const uint32_t s_n = (j + 1u) % S, ph_n = ((j + 1u) / S) & 1u;
        const uint32_t slot_n = kAccTmem ? pc + (piece_end ? 1u : 0u) : j + 1u;
        const uint32_t b_n = slot_n % kSkNumAcc, bph_n = (slot_n / kSkNumAcc) & 1u;
        const bool test_free = more && next_start;
        const uint32_t got = mma_step4_test2_next<kIn>(
            d_tmem, ad, bd, kIdesc, piece_start ? 0u : 1u, more ? full_bar(s_n) : full_bar(s),
            more ? ph_n : ph, test_free ? tempty_bar(b_n) : full_bar(s), test_free ? bph_n ^ 1u : ph,
            piece_end ? 1u : 0u, empty_bar(s), tfull_bar(b));
        rdy_full = more && (got & 1u) != 0u;
        rdy_free = test_free && (got & 2u) != 0u;
        issued = true;
        if (piece_end) ++pc;
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
    const uint32_t ew = warp - 2;   // 0 .. kEpiWarps-1
    const uint32_t q = warp & 3u;   // TMEM lane quarter
    const uint32_t h = ew >> 2;     // column group
    const int col0 = (int)h * kHalf;
    const int nloc = (int)(q * 32u + lane);
    const int etid = (int)(ew * 32u + lane);  // 0 .. kSkEpiThreads-1
    uint32_t tab_phase = 0;
    // The epilogue warps meet on an mbarrier with a bounded wait, so a warp
    // that aborts cannot leave the others blocked.
    auto group_sync = [&](uint32_t where) -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(tab_bar);
      uint32_t okg = 0;
      if (lane == 0) okg = wait_phase(tab_bar, tab_phase & 1u, abort_flag, where) ? 1u : 0u;
      ++tab_phase;
      return __shfl_sync(0xFFFFFFFFu, okg, 0) != 0;
    };
    uint32_t j = 0;
    uint32_t pc = 0;  // kAccTmem: pieces drained so far
    int pend_nt[2];  // partial tiles of this range (its first and last piece)
    int npend = 0;
    bool ok = true;
    int64_t st = s0, tab_begin = s0, tab_end = s0;
    float acc[kHalf];
#pragma unroll
    for (int c = 0; c < kHalf; ++c) acc[c] = 0.0f;
    float s_scalar = 1.0f;  // kScalar: the one scale product (1 for BF16)
    if (kScalar)
      s_scalar = (p.a_scale ? __ldg(p.a_scale) : 1.0f) * (p.b_scale ? __ldg(p.b_scale) : 1.0f);
    for (; ok && st < s1; ++st, ++j) {
      if (!kScalar && st == tab_end) {
        // Next chunk of the scale-product table: every load in flight at once.
        if (st != s0 && !group_sync(0x17)) {  // everyone is done with the old chunk
          ok = false;
          break;
        }
        tab_begin = st;
        tab_end = s1 - st < Cfg::kTabSteps ? s1 : st + Cfg::kTabSteps;
        const int n = (int)(tab_end - tab_begin) * kMp;
        // 8 entries per thread per round, every load issued before any store
        for (int base = 0; base < n; base += 8 * kSkEpiThreads) {
          float va[8], vb[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int idx = base + e * kSkEpiThreads + etid;
            va[e] = 0.0f;
            vb[e] = 0.0f;
            if (idx < n) {
              const int gst = (int)tab_begin + idx / kMp;
              const int q = gst / KB;
              const int tkb = gst - q * KB;
              int tnt, tmt;
              sk_tile(q, m_tiles, tnt, tmt);
              const int m = tmt * kMp + idx % kMp;
              if (m < p.M) {
                va[e] = __ldg(p.a_scale + (int64_t)tkb * p.M + m);
                vb[e] = __ldg(p.b_scale + (int64_t)tnt * KB + tkb);
              }
            }
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int idx = base + e * kSkEpiThreads + etid;
            if (idx < n) stab[idx] = va[e] * vb[e];
          }
        }
        if (!group_sync(0x18)) {
          ok = false;
          break;
        }
      }
      const int nt = (int)st / KB;  // tile index (N tile and M chunk)
      const int kb = (int)st - nt * KB;
      if (kAccTmem && !(kb == KB - 1 || st == s1 - 1)) continue;  // the MMA keeps accumulating
      const uint32_t slot = kAccTmem ? pc : j;  // TMEM buffer sequence number
      const uint32_t b = slot % kSkNumAcc, bph = (slot / kSkNumAcc) & 1u;
      uint32_t got = 0;
      if (lane == 0) got = wait_phase(tfull_bar(b), bph, abort_flag, 0x14) ? 1u : 0u;
      got = __shfl_sync(0xFFFFFFFFu, got, 0);
      if (!got) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const float* sc = kScalar ? stab : stab + (st - tab_begin) * kMp + col0;  // (no table)
      // Drain the partial in pieces of at most 32 columns (register budget).
      constexpr int kPiece = kHalf < 32 ? kHalf : 32;
      if constexpr (kAccTmem) {
        // the whole piece's sum, once: acc (zero here) = sum * scale
#pragma unroll
        for (int c1 = 0; c1 < kHalf; c1 += kPiece) {
          uint32_t r[kPiece];
          tmem_load_cols<kPiece>(
              tmem_base + ((q * 32u) << 16) + b * kMp + (uint32_t)(col0 + c1), r);
#pragma unroll
          for (int c = 0; c < kPiece; ++c)
            acc[c1 + c] = fmaf(__uint_as_float(r[c]), s_scalar, acc[c1 + c]);
        }
        ++pc;
      } else {
#pragma unroll
        for (int c1 = 0; c1 < kHalf; c1 += kPiece) {
          uint32_t r[kPiece];
          tmem_load_cols<kPiece>(
              tmem_base + ((q * 32u) << 16) + b * kMp + (uint32_t)(col0 + c1), r);
#pragma unroll
          for (int c = 0; c < kPiece; c += 4) {
            // acc += partial * scale product, two columns per packed f32x2 FMA
            // (each lane rounded as fmaf)
            const float4 s4 = kScalar ? make_float4(s_scalar, s_scalar, s_scalar, s_scalar)
                                      : *reinterpret_cast<const float4*>(sc + c1 + c);
            fma_f32x2_pair(acc[c1 + c + 0], acc[c1 + c + 1], r[c + 0], r[c + 1], s4.x, s4.y);
            fma_f32x2_pair(acc[c1 + c + 2], acc[c1 + c + 3], r[c + 2], r[c + 3], s4.z, s4.w);
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(b));
      const bool seg_done = kb == KB - 1 || st == s1 - 1;
      if (!seg_done) continue;
      // ---- this CTA's K range of tile nt is summed
      const int64_t tile_first = st - kb;
      const int kb_first = (int)((tile_first > s0 ? tile_first : s0) - tile_first);
      if (kJoin > 0) {
        // park this piece's partial in this CTA's shared memory (every MMA
        // and TMA copy of the range is complete: the stages are free)
        float* part = reinterpret_cast<float*>(gbase);
#pragma unroll
        for (int c = 0; c < kHalf; ++c) part[(col0 + c) * 128 + nloc] = acc[c];
      } else if (kb_first == 0 && kb == KB - 1) {
        int ntile, mt;
        sk_tile(nt, m_tiles, ntile, mt);
        const int n = ntile * 128 + nloc;
#pragma unroll
        for (int c = 0; c < kHalf; ++c) emit_one(p, mt * kMp + col0 + c, n, acc[c]);
      } else {
        // partial tile: park it in this CTA's workspace slot (0 for the
        // first tile of its range, 1 for the last); the handshake waits for
        // the end of the range
        const int slot = nt == (int)s0 / KB ? 0 : 1;
        float* wsp = p.ws + ((int64_t)blockIdx.x * 2 + slot) * kMp * 128;
#pragma unroll
        for (int c = 0; c < kHalf; ++c) __stcg(wsp + (int64_t)(col0 + c) * 128 + nloc, acc[c]);
        pend_nt[npend++] = nt;
      }
#pragma unroll
      for (int c = 0; c < kHalf; ++c) acc[c] = 0.0f;
    }
    // ---- end of the range: count this CTA's partial tiles in, and finish
    // the tiles it is the last contributor to.
    if (kJoin == 0 && ok && npend > 0) {
      __threadfence();
      __syncwarp();
      if (lane == 0) mbar_arrive(seg_bar);
      if (ew == 0 && lane < (uint32_t)npend) {
        const int tnt = pend_nt[lane];
        const int64_t tf = (int64_t)tnt * KB;
        const int nseg = (int)(sk_owner(tf + KB - 1, T, G) - sk_owner(tf, T, G) + 1);
        int last = 0;
        if (wait_phase(seg_bar, 0, abort_flag, 0x15)) {
          const unsigned prev = atomicAdd(&p.counters[tnt], 1u);
          last = prev == (unsigned)(nseg - 1);
          if (last) p.counters[tnt] = 0u;  // ready for the next call
        }
        last_flag[lane] = last;
      }
      __syncwarp();
      if (ew == 0 && lane == 0) mbar_arrive(flag_bar);
      uint32_t gotf = 0;
      if (lane == 0) gotf = wait_phase(flag_bar, 0, abort_flag, 0x16) ? 1u : 0u;
      gotf = __shfl_sync(0xFFFFFFFFu, gotf, 0);
      if (gotf && !*abort_flag) {
        __threadfence();
        for (int i = 0; i < npend; ++i) {
          if (!last_flag[i]) continue;
          const int tnt = pend_nt[i];
          const int64_t tf = (int64_t)tnt * KB;
          const int64_t first_owner = sk_owner(tf, T, G);
          const int nseg = (int)(sk_owner(tf + KB - 1, T, G) - first_owner + 1);
          // contributor sgi is CTA first_owner + sgi; its slot for this tile
          // is 0 if the tile is the first of its range, else 1
          const float4* src[kSkMaxSeg];
#pragma unroll
          for (int sgi = 0; sgi < kSkMaxSeg; ++sgi) {
            const int64_t c = first_owner + (sgi < nseg ? sgi : 0);
            const int slot = tnt == (int)sk_range_start(c, T, G) / KB ? 0 : 1;
            src[sgi] = reinterpret_cast<const float4*>(p.ws + (c * 2 + slot) * kMp * 128);
          }
          // All epilogue threads sum the slots (in slot order) over float4
          // units of the Mp x 128 tile: a warp covers 32 consecutive units (one
          // row m), kU units x all slots in flight per thread.
          constexpr int kUnits = kMp * 32;  // float4 units per slot
          constexpr int kU = kMp >= 64 ? 4 : 2;
          static_assert(kUnits % (kSkEpiThreads * kU) == 0, "reduction tiling");
          for (int u0 = 0; u0 < kUnits; u0 += kSkEpiThreads * kU) {
            float4 part[kSkMaxSeg][kU];
#pragma unroll
            for (int sgi = 0; sgi < kSkMaxSeg; ++sgi)
#pragma unroll
              for (int v = 0; v < kU; ++v)
                part[sgi][v] = sgi < nseg ? __ldcg(src[sgi] + u0 + v * kSkEpiThreads + etid)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int v = 0; v < kU; ++v) {
              float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
              for (int sgi = 0; sgi < kSkMaxSeg; ++sgi) {
                if (sgi < nseg) {
                  sum.x += part[sgi][v].x;
                  sum.y += part[sgi][v].y;
                  sum.z += part[sgi][v].z;
                  sum.w += part[sgi][v].w;
                }
              }
              const int u = u0 + v * kSkEpiThreads + etid;
              int ntile, mt;
              sk_tile(tnt, m_tiles, ntile, mt);
              emit_four(p, mt * kMp + (u >> 5), ntile * 128 + (u & 31) * 4, sum);
            }
          }
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if constexpr (kJoin > 0) {
    cluster_sync_all();  // every piece's partial is in shared memory
    if (warp >= 2 && !*abort_flag) {
      // CTA r finishes float4 units [r*kPer, (r+1)*kPer) of the Mp x 128 tile
      // (a unit is 4 consecutive n of one row m), adding the pieces in
      // cluster-rank order, which is K order: the same result every run
      constexpr int kUnits = kMp * 32;
      constexpr int kPer = (kUnits + kJoin - 1) / kJoin;
      const uint32_t rank = cluster_ctarank();
      const uint32_t local = smem_u32(gbase);
      uint32_t piece[kJoin];
#pragma unroll
      for (int r = 0; r < kJoin; ++r) piece[r] = map_shared_to_cta(local, (uint32_t)r);
      int tnt, tmt;
      sk_tile((int)s0 / KB, m_tiles, tnt, tmt);
      const int etid = (int)((warp - 2) * 32u + lane);
      const int u_end = ((int)rank + 1) * kPer < kUnits ? ((int)rank + 1) * kPer : kUnits;
      for (int u = (int)rank * kPer + etid; u < u_end; u += kSkEpiThreads) {
        float4 sum = ld_shared_cluster_v4(piece[0] + 16u * (uint32_t)u);
#pragma unroll
        for (int r = 1; r < kJoin; ++r) {
          const float4 v = ld_shared_cluster_v4(piece[r] + 16u * (uint32_t)u);
          sum = make_float4(sum.x + v.x, sum.y + v.y, sum.z + v.z, sum.w + v.w);
        }
        emit_four(p, tmt * kMp + (u >> 5), tnt * 128 + (u & 31) * 4, sum);
      }
    }
    cluster_sync_all();  // the other CTAs have finished reading this CTA's partial
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

}  // namespace tcg
