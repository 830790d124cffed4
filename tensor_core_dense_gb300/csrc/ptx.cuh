// ptx.cuh -- inline-PTX wrappers for the sm_103a data path: mbarriers, TMA
// bulk-tensor loads, and the tcgen05 family (Tensor Memory allocation, MMA,
// commit, loads).
//
// The protocol follows "Tensor cores and low precision", "How a TMA copy says
// it is done": one thread arms an mbarrier with the byte count of the tile
// (arrive + expect_tx), the TMA copy credits its bytes against the same
// barrier, and consumers wait on the barrier's phase parity, which flips at
// every reuse.  Tensor Memory and tcgen05 rules follow "How Blackwell's Tensor
// Memory Actually Works", "What Tensor Memory actually is" (allocation by
// power-of-two column counts >= 32, base address returned through shared
// memory, dealloc from the allocating warp, warp w of a warpgroup reaches
// lanes 32w..32w+31) and "What the compiler actually emits" (single-thread
// MMA issue, commit through an mbarrier in the .shared::cluster space).
#pragma once

#include <stdint.h>

namespace tcg {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lane_id() {
  uint32_t l;
  asm volatile("mov.u32 %0, %%laneid;" : "=r"(l));
  return l;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// True once the phase with parity `parity` has completed.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// ------------------------------------------------- programmatic launch

// Waits until the grids this one depends on (the previous kernel in the
// stream, when launched with programmatic stream serialisation) have finished
// and their memory is visible.  A no-op otherwise.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next kernel in the stream start launching (its CTAs take SMs as
// this grid's CTAs exit) before this grid has finished.
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ----------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load of one box into shared memory; completion is credited to
// `bar` as transaction bytes.  x is the innermost (contiguous) coordinate in
// elements, y the row.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* map, uint32_t bar, int32_t x,
                                            int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Same, with an L2 cache policy (e.g. evict-first for a streamed operand).
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const void* map, uint32_t bar,
                                                 int32_t x, int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// 2-D tiled store of one box from this CTA's shared memory to global memory
// (elements outside the tensor are not written), tracked as a bulk group of
// the issuing thread.
__device__ __forceinline__ void tma_store_2d(const void* map, uint32_t src, int32_t x,
                                             int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
}

// Closes this thread's group of bulk copies issued since the last commit.
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until at most kN of this thread's bulk groups still read their
// shared-memory source (the buffers of the others may be reused).
template <int kN>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kN) : "memory");
}

// Waits until at most kN of this thread's bulk groups are incomplete.
template <int kN>
__device__ __forceinline__ void bulk_wait_group() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(kN) : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory writes before
// later async-proxy accesses (a TMA store reading them).
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Hint: bring one box of a tensor into L2 (no shared memory, no barrier).
// L2 is coherent for the whole GPU, so this is safe before the grid
// dependency wait even if the previous kernel is still writing the tensor.
__device__ __forceinline__ void tma_prefetch_l2_2d(const void* map, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive (once) on `bar` when every tcgen05 operation this thread issued
// before it has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, both K-major; accumulate != 0 adds to D.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 128 bytes, 8-row (1024-byte) swizzle atoms
// stacked along M/N.  Fields: start address >> 4 (bits 0-13), leading byte
// offset >> 4 (16-29, not used by swizzled K-major layouts), stride byte
// offset >> 4 (32-45: 1024 bytes between 8-row groups), the fixed version
// bits 46-48 = 0b001, base offset 0 (bits 49-51; tiles are 1024-byte
// aligned), layout 2 = 128-byte swizzle (61-63).
__device__ __forceinline__ uint64_t smem_desc_k_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(16u >> 4) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Instruction descriptor for kind::f16 / kind::f8f6f4 with an FP32
// accumulator and both operands K-major.  fmt: BF16 = 1 (kind::f16); E4M3 =
// 0, E5M2 = 1 (kind::f8f6f4, where A and B may differ).  N in steps of 16
// (M = 128), M in steps of 16.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t a_fmt, uint32_t b_fmt, uint32_t M,
                                                  uint32_t N) {
  return (1u << 4)              // D format: F32
         | (a_fmt << 7)         // A format
         | (b_fmt << 10)        // B format
         | (0u << 15)           // A K-major
         | (0u << 16)           // B K-major
         | ((N >> 3) << 17)     // N / 8
         | ((M >> 4) << 24);    // M / 16
}

// 32 lanes x 32 columns of 32-bit TMEM cells -> 32 registers per thread
// (thread t of the warp gets lane base+t, columns col..col+31).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// 32 lanes x 64 columns -> 64 registers per thread.
__device__ __forceinline__ void tmem_ld_32x32b_x64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
      "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
      "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]),
        "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]),
        "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]),
        "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]),
        "=r"(r[62]), "=r"(r[63])
      : "r"(taddr));
}

// 32 lanes x 8 columns -> r[0..7] (thread t of the warp gets lane base+t).
__device__ __forceinline__ void tmem_ld_32x32b_x8(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr));
}

__device__ __forceinline__ void pin_regs8(uint32_t* r) {
  asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                    "+r"(r[6]), "+r"(r[7]));
}

// Waits for this thread's outstanding tcgen05.ld and pins n registers (a
// multiple of 8) after the wait.
template <int kN>
__device__ __forceinline__ void tmem_ld_wait_n(uint32_t (&r)[kN]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < kN / 8; ++i) pin_regs8(&r[8 * i]);
}

// Loads kCols consecutive TMEM columns (a multiple of 8) of this warp's 32
// lanes, waits for them, and pins the registers after the wait.
template <int kCols>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, uint32_t (&r)[kCols]) {
  static_assert(kCols % 8 == 0, "columns in steps of 8");
#pragma unroll
  for (int i = 0; i < kCols / 8; ++i) tmem_ld_32x32b_x8(taddr + 8u * i, &r[8 * i]);
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < kCols / 8; ++i) pin_regs8(&r[8 * i]);
}

// Waits for this thread's outstanding tcgen05.ld, then pins the 32 loaded
// registers after the wait so no use of them is scheduled before it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31]));
}

// Two FP32 values as one 64-bit register pair, and back (the operand form of
// Blackwell's packed f32x2 arithmetic).
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t v;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(lo), "f"(hi));
  return v;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// Per-warpgroup register budget changes (every warp of the warpgroup executes
// the same one).  An increase waits until the block's pool has the registers,
// so the decreases and increases of one kernel must balance against the
// registers it was launched with.
template <uint32_t kRegs>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
}
template <uint32_t kRegs>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
}

// (a0, a1) += (p0, p1) * (s0, s1) in one packed instruction (p0, p1: FP32 bit
// patterns); each lane is rounded exactly as a scalar fmaf.
__device__ __forceinline__ void fma_f32x2_pair(float& a0, float& a1, uint32_t p0, uint32_t p1,
                                               float s0, float s1) {
  uint64_t pp, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(pp) : "r"(p0), "r"(p1));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(pp), "l"(pack_f32x2(s0, s1)),
      "l"(pack_f32x2(a0, a1)));
  unpack_f32x2(d, a0, a1);
}

// Two FP32 -> packed BF16x2, round to nearest even (lo in bits 0-15).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ float bf16_lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi_to_f32(uint32_t v) {
  return __uint_as_float(v & 0xFFFF0000u);
}

}  // namespace tcg

// ------------------------------------------------------ CTA pairs (clusters)
//
// A cluster of two CTAs on neighbouring SMs can run one tcgen05.mma with
// cta_group::2: the pair computes a 256-row tile, each CTA holding half of A
// (its 128 rows) and half of B (N/2 rows) in its own shared memory and the
// accumulator rows of its half in its own Tensor Memory ("How Blackwell's
// Tensor Memory Actually Works", "The instruction": only the leader CTA of
// the pair issues the MMA; "Why it had to be a separate memory": the pair
// halves the operand traffic each SM serves).

namespace tcg {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory offset in CTA `cta` of the cluster.
__device__ __forceinline__ uint32_t map_shared_to_cta(uint32_t addr, uint32_t cta) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(cta));
  return r;
}

// 16-byte load from a shared::cluster address (this CTA's or a peer's).
__device__ __forceinline__ float4 ld_shared_cluster_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on an mbarrier in another CTA of the cluster with CTA-scope release:
// for hand-backs whose ordering comes from a tcgen05 fence (a drained TMEM
// buffer), so the arrive does not wait for this thread's outstanding global
// loads and stores as a cluster-scope release does.
__device__ __forceinline__ void mbar_arrive_remote_cta(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// try_wait with cluster-scope acquire (arrivals from the peer CTA).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// TMA load into this CTA's shared memory whose completion is credited to an
// mbarrier in either CTA of the pair (bar is a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* map, uint32_t bar,
                                                 int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// 3-D tiled load into this CTA's shared memory, completion credited to an
// mbarrier in either CTA of the pair (x innermost).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const void* map, uint32_t bar,
                                                 int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// 4-D tiled load into this CTA's shared memory, completion credited to an
// mbarrier in either CTA of the pair (x innermost).
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const void* map, uint32_t bar,
                                                 int32_t x, int32_t y, int32_t z, int32_t w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Arrive once on the mbarrier at offset `bar` in every CTA of `cta_mask`
// when this thread's earlier tcgen05 operations have completed.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_e4m3_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Four MMAs D (+)= A * B^T over the consecutive 32-byte K slices of one
// 128-byte K step: operand descriptors + 0, 2, 4, 6 (16-byte units), the
// first slice accumulating into D when `acc`, the rest always. Expects the
// predicates acc / one and the 64-bit registers a1..a3 / b1..b3 of
// TCG_STEP4_SETUP; operands %1 (D), %2 (A), %3 (B), %4 (instruction desc.).
// TCG_COMMIT_PAIR arrives on a barrier in both CTAs of the pair (mask: %8).
#define TCG_STEP4_SETUP(ACC_OPERAND)                              \
  ".reg .pred rdy, acc, one;\n\t"                                 \
  ".reg .b64 a1, a2, a3, b1, b2, b3;\n\t"                         \
  "setp.ne.b32 acc, " ACC_OPERAND ", 0;\n\t"                      \
  "setp.eq.b32 one, 0, 0;\n\t"                                    \
  "add.s64 a1, %2, 2;\n\tadd.s64 a2, %2, 4;\n\tadd.s64 a3, %2, 6;\n\t" \
  "add.s64 b1, %3, 2;\n\tadd.s64 b2, %3, 4;\n\tadd.s64 b3, %3, 6;\n\t"
#define TCG_STEP4_MMAS(GROUP, KIND)                                        \
  "tcgen05.mma.cta_group::" GROUP ".kind::" KIND " [%1], %2, %3, %4, acc;\n\t" \
  "tcgen05.mma.cta_group::" GROUP ".kind::" KIND " [%1], a1, b1, %4, one;\n\t" \
  "tcgen05.mma.cta_group::" GROUP ".kind::" KIND " [%1], a2, b2, %4, one;\n\t" \
  "tcgen05.mma.cta_group::" GROUP ".kind::" KIND " [%1], a3, b3, %4, one;\n\t"
#define TCG_COMMIT_PAIR(BAR) \
  "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [" BAR "], %8;\n\t"

// One K step of a CTA pair: the four MMAs of the step, then a commit of the
// step's operands to `done_bar` in both CTAs. Before the MMAs it tests
// (without suspending) whether `next_bar` has completed the phase of parity
// `next_par`, and returns that result at the end.
//
// The order matters for the tensor pipe's occupancy. Any value the issuing
// thread reads back -- an mbarrier test or wait, even a plain shared-memory
// load -- reaches it only after the tcgen05 instructions it issued before
// have been handed to the tensor core. A thread that reads the next step's
// barrier after issuing this step's MMAs therefore stalls until the queue is
// empty, and the pipe idles while its next MMAs are issued (measured at
// 4096^3: 11 % of every K step). Issued first and read last, the test's
// result comes back while this step's MMAs are still queued behind it.
template <int kKind>  // 0: kind::f16 (BF16), 1: kind::f8f6f4 (FP8)
__device__ __forceinline__ uint32_t mma_step4_pair_test_next(uint32_t d_tmem, uint64_t a_desc,
                                                             uint64_t b_desc, uint32_t idesc,
                                                             uint32_t accumulate, uint32_t done_bar,
                                                             uint32_t next_bar,
                                                             uint32_t next_par) {
  uint32_t ready;
  if (kKind == 0) {
    asm volatile("{\n\t" TCG_STEP4_SETUP("%5")
                 "mbarrier.test_wait.parity.shared::cta.b64 rdy, [%6], %7;\n\t"
                 TCG_STEP4_MMAS("2", "f16") TCG_COMMIT_PAIR("%9")
                 "selp.u32 %0, 1, 0, rdy;\n\t}"
                 : "=r"(ready)
                 : "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate),
                   "r"(next_bar), "r"(next_par), "h"((uint16_t)0x3), "r"(done_bar)
                 : "memory");
  } else {
    asm volatile("{\n\t" TCG_STEP4_SETUP("%5")
                 "mbarrier.test_wait.parity.shared::cta.b64 rdy, [%6], %7;\n\t"
                 TCG_STEP4_MMAS("2", "f8f6f4") TCG_COMMIT_PAIR("%9")
                 "selp.u32 %0, 1, 0, rdy;\n\t}"
                 : "=r"(ready)
                 : "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate),
                   "r"(next_bar), "r"(next_par), "h"((uint16_t)0x3), "r"(done_bar)
                 : "memory");
  }
  return ready;
}

// A skinny-kernel K step on one SM: four MMAs over the step's 32-byte K
// slices (the first accumulating when `accumulate`), a commit to `done_bar`
// and, when `commit_full` is nonzero, one to `full_tmem_bar`. Ahead of them it
// tests the next step's operand barrier (`next_bar`, parity `next_par`) and
// Tensor Memory buffer barrier (`free_bar`, parity `free_par`); returns bit 0
// / bit 1 for them -- the ordering of mma_step4_pair_test_next.
template <int kKind>  // 0: kind::f16 (BF16), 1: kind::f8f6f4 (FP8)
__device__ __forceinline__ uint32_t mma_step4_test2_next(uint32_t d_tmem, uint64_t a_desc,
                                                         uint64_t b_desc, uint32_t idesc,
                                                         uint32_t accumulate, uint32_t next_bar,
                                                         uint32_t next_par, uint32_t free_bar,
                                                         uint32_t free_par, uint32_t commit_full,
                                                         uint32_t done_bar,
                                                         uint32_t full_tmem_bar) {
  uint32_t ready;
  if (kKind == 0) {
    asm volatile("{\n\t" TCG_STEP4_SETUP("%5")
                 ".reg .pred fre, ctf;\n\t"
                 ".reg .b32 fb;\n\t"
                 "setp.ne.b32 ctf, %10, 0;\n\t"
                 "mbarrier.test_wait.parity.shared::cta.b64 rdy, [%6], %7;\n\t"
                 "mbarrier.test_wait.parity.shared::cta.b64 fre, [%8], %9;\n\t"
                 TCG_STEP4_MMAS("1", "f16")
                 "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%11];\n\t"
                 "@ctf tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%12];\n\t"
                 "selp.u32 fb, 2, 0, fre;\n\t"
                 "selp.u32 %0, 1, 0, rdy;\n\t"
                 "or.b32 %0, %0, fb;\n\t}"
                 : "=r"(ready)
                 : "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate),
                   "r"(next_bar), "r"(next_par), "r"(free_bar), "r"(free_par), "r"(commit_full),
                   "r"(done_bar), "r"(full_tmem_bar)
                 : "memory");
  } else {
    asm volatile("{\n\t" TCG_STEP4_SETUP("%5")
                 ".reg .pred fre, ctf;\n\t"
                 ".reg .b32 fb;\n\t"
                 "setp.ne.b32 ctf, %10, 0;\n\t"
                 "mbarrier.test_wait.parity.shared::cta.b64 rdy, [%6], %7;\n\t"
                 "mbarrier.test_wait.parity.shared::cta.b64 fre, [%8], %9;\n\t"
                 TCG_STEP4_MMAS("1", "f8f6f4")
                 "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%11];\n\t"
                 "@ctf tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%12];\n\t"
                 "selp.u32 fb, 2, 0, fre;\n\t"
                 "selp.u32 %0, 1, 0, rdy;\n\t"
                 "or.b32 %0, %0, fb;\n\t}"
                 : "=r"(ready)
                 : "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate),
                   "r"(next_bar), "r"(next_par), "r"(free_bar), "r"(free_par), "r"(commit_full),
                   "r"(done_bar), "r"(full_tmem_bar)
                 : "memory");
  }
  return ready;
}

// One K step on one SM: four MMAs over the step's 32-byte K slices (the
// first accumulating when `accumulate`), then a commit to `done_bar`, with a
// test of `next_bar` (parity `next_par`) issued ahead of them and read after
// -- the ordering of mma_step4_pair_test_next, for the same reason.
template <int kKind>  // 0: kind::f16 (BF16), 1: kind::f8f6f4 (FP8)
__device__ __forceinline__ uint32_t mma_step4_test_next(uint32_t d_tmem, uint64_t a_desc,
                                                        uint64_t b_desc, uint32_t idesc,
                                                        uint32_t accumulate, uint32_t done_bar,
                                                        uint32_t next_bar, uint32_t next_par) {
  uint32_t ready;
  if (kKind == 0) {
    asm volatile("{\n\t" TCG_STEP4_SETUP("%5")
                 "mbarrier.test_wait.parity.shared::cta.b64 rdy, [%6], %7;\n\t"
                 TCG_STEP4_MMAS("1", "f16")
                 "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%8];\n\t"
                 "selp.u32 %0, 1, 0, rdy;\n\t}"
                 : "=r"(ready)
                 : "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate),
                   "r"(next_bar), "r"(next_par), "r"(done_bar)
                 : "memory");
  } else {
    asm volatile("{\n\t" TCG_STEP4_SETUP("%5")
                 "mbarrier.test_wait.parity.shared::cta.b64 rdy, [%6], %7;\n\t"
                 TCG_STEP4_MMAS("1", "f8f6f4")
                 "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%8];\n\t"
                 "selp.u32 %0, 1, 0, rdy;\n\t}"
                 : "=r"(ready)
                 : "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate),
                   "r"(next_bar), "r"(next_par), "r"(done_bar)
                 : "memory");
  }
  return ready;
}

}  // namespace tcg
