/*
 * tcgemm.h -- dense tensor-core GEMM for NVIDIA GB300 (sm_103a), C ABI.
 *
 *     D = alpha * A * B + beta * C          (FP32 accumulation)
 *
 * The operation is the matrix multiply-accumulate D = A*B + C, A M x K, B
 * K x N, C and D M x N ("Tensor Cores: Matrix Instructions, Swizzling and
 * FP8, Measured", Step 1), on BF16 operands ("Tensor Cores", "Precision:
 * FP16, BF16, TF32, FP8") or FP8 E4M3 operands carrying FP32 scale factors
 * that are removed after the product ("Tensor cores and low precision", the
 * FP8 scaling paragraph).
 *
 * Layouts (all row-major with an explicit leading dimension, in elements):
 *   A  M x K, element (i, k) at A[i * lda + k]            (K contiguous)
 *   B  stored N x K, element (k, j) at B[j * ldb + k]     (K contiguous; the
 *      "TN" layout of the 4,096^3 test in the page above, Step 2)
 *   C  M x N, (i, j) at C[i * ldc + j]; same dtype as D; read only if beta != 0
 *   D  M x N, (i, j) at D[i * ldd + j]; BF16 (round to nearest even) or FP32
 *
 * Every pointer is a device pointer owned by the caller.  A call enqueues
 * work on `stream` and returns without synchronising; D is valid once the
 * stream has reached that point.  No entry point allocates device memory:
 * the library keeps a process-wide cache of TMA tensor maps (host memory),
 * and gemm_fp8_e4m3_block_noalloc keeps a fixed scratch array in the
 * library's device code (below).  Calls on different streams may run
 * concurrently and are independent of one another, except calls of
 * gemm_fp8_e4m3_block_noalloc, which share that array.
 *
 * No exception or abort crosses this boundary: every entry point returns a
 * tcg_status.  Argument errors are detected on the host before anything is
 * enqueued.  A device-side wait that exceeds its time limit (which would
 * indicate a bug, never a slow GPU) makes the kernel exit early and records
 * TCG_ERR_TIMEOUT in a device status word read by tcg_last_device_status().
 */
#ifndef TCGEMM_H
#define TCGEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* tcg_stream;

typedef enum {
  TCG_OK = 0,
  TCG_ERR_INVALID_ARG = 1, /* negative size, ld too small, NULL pointer, ... */
  TCG_ERR_ALIGNMENT = 2,   /* base not 16-byte aligned or row pitch not a multiple of 16 bytes */
  TCG_ERR_UNSUPPORTED = 3, /* an enum value or size this library does not handle */
  TCG_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed (launch, tensor-map encode) */
  TCG_ERR_TIMEOUT = 5      /* a device-side wait ran out (reported by tcg_last_device_status) */
} tcg_status;

typedef enum { TCG_OUT_BF16 = 0, TCG_OUT_F32 = 1 } tcg_out_dtype;

typedef enum {
  /* a_scale[0] and b_scale[0]: one FP32 scale per operand */
  TCG_SCALE_TENSOR = 0,
  /* one FP32 scale per 1 x 128 block of A (row i, K block kb) at
   * a_scale[kb * M + i], and per 128 x 128 block of B (N block nb, K block
   * kb) at b_scale[nb * ceil(K/128) + kb] */
  TCG_SCALE_BLOCK128 = 1
} tcg_scale_mode;

/*
 * gemm_bf16 -- D = alpha * A * B + beta * C with BF16 A and B.
 *
 * M, N, K      sizes, >= 0.  M == 0 or N == 0: nothing is done.  K == 0:
 *              D = beta * C (zero when beta == 0).
 * A, lda       BF16, M x K, lda >= K.  B, ldb: BF16, N x K, ldb >= K.
 * C, ldc       dtype given by out_dtype; may be NULL iff beta == 0; ldc >= N.
 *              C may alias D only exactly (C == D and ldc == ldd).
 * D, ldd       out_dtype, M x N, ldd >= N.
 * Alignment    A, B, C, D 16-byte aligned; lda*2, ldb*2, ldc*size, ldd*size
 *              multiples of 16 bytes (a TMA requirement for A and B; vector
 *              stores for C and D).
 * Numerics     products accumulate in FP32 on the tensor cores; alpha and beta
 *              are applied in FP32; BF16 output rounds to nearest even.
 * Kernels      tile kernels by shape; decode-sized calls (M <= 128, with
 *              ceil(N/128) * 2 <= SMs) run swap-AB with K split over clusters
 *              of two or three CTAs whose FP32 partial sums are added in a
 *              fixed order.  Every path is deterministic and none allocates.
 */
tcg_status gemm_bf16(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                     int64_t ldb, const void* C, int64_t ldc, void* D, int64_t ldd,
                     tcg_out_dtype out_dtype, float alpha, float beta, tcg_stream stream);

/*
 * gemm_fp8_e4m3 -- D = alpha * (sA . A) * (sB . B) + beta * C with E4M3 bytes
 * in A and B and FP32 dequantisation scales (device pointers).
 *
 * Layouts and alignment as gemm_bf16 with one byte per element of A and B
 * (lda, ldb multiples of 16).  mode selects the scale granularity above; the
 * scales must be finite.
 * TCG_SCALE_TENSOR   the per-tensor product a_scale[0]*b_scale[0] multiplies
 *                    the FP32 sums once, in the epilogue (on the decode-sized
 *                    path with M <= 64, every 128-byte K step's partial sum
 *                    before it is added), then alpha.
 * TCG_SCALE_BLOCK128 every 128-wide K block is accumulated on its own and
 *                    promoted into an FP32 register accumulator with its
 *                    scales sa[i,kb] * sb[j/128,kb] ("promotion": partial sums
 *                    moved to FP32 at intervals, "Tensor Cores: Matrix
 *                    Instructions, Swizzling and FP8, Measured", Step 5).
 *                    Any M: M <= 128 (the skinny, decode-sized shape) runs
 *                    swap-AB with A in one chunk; larger M runs on 256 x 256
 *                    CTA-pair tiles, or, when those would leave more than
 *                    half the SMs idle, in chunks of 128 rows of A (128 x 128
 *                    output tiles).  The swap-AB kernel splits each tile's K
 *                    range over a cluster of two or three CTAs when the
 *                    tiles fill at most half (a third) of the SMs, and
 *                    otherwise gives each CTA whole tiles; no tile is ever
 *                    finished through global memory.  The result does not
 *                    depend on the choice beyond FP32 rounding order, and
 *                    repeats bit for bit for the same call.
 */
tcg_status gemm_fp8_e4m3(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                         const void* B, int64_t ldb, const float* a_scale, const float* b_scale,
                         tcg_scale_mode mode, const void* C, int64_t ldc, void* D, int64_t ldd,
                         tcg_out_dtype out_dtype, float alpha, float beta, tcg_stream stream);

/* The two 8-bit floating-point encodings ("Tensor cores and low precision",
 * FP8 paragraph): E4M3 (1/4/3 bits, bias 7, no infinity, maximum 448) and
 * E5M2 (1/5/2 bits, bias 15, IEEE infinities and NaNs, maximum 57,344). */
typedef enum { TCG_FP8_E4M3 = 0, TCG_FP8_E5M2 = 1 } tcg_fp8_format;

/*
 * gemm_fp8 -- gemm_fp8_e4m3 with the encoding of each operand given
 * separately: E4M3 x E4M3, E5M2 x E5M2, or mixed (E4M3 activations or weights
 * against E5M2 gradients, the pages' suggested split between the formats).
 * Arguments, layouts, scale modes, alignment and numerics are those of
 * gemm_fp8_e4m3; codes must be finite (no E5M2 infinities or NaNs).  An
 * unknown format returns TCG_ERR_UNSUPPORTED.  gemm_fp8_e4m3(...) is
 * gemm_fp8 with a_format = b_format = TCG_FP8_E4M3.
 */
tcg_status gemm_fp8(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                    tcg_fp8_format a_format, const void* B, int64_t ldb, tcg_fp8_format b_format,
                    const float* a_scale, const float* b_scale, tcg_scale_mode mode,
                    const void* C, int64_t ldc, void* D, int64_t ldd, tcg_out_dtype out_dtype,
                    float alpha, float beta, tcg_stream stream);

/*
 * gemm_fp8_e4m3_block_noalloc -- the TCG_SCALE_BLOCK128 GEMM on the skinny
 * kernel's stream-K form, whose scratch memory is a fixed array inside the
 * library, so that nothing is allocated.  The pages have no counterpart to
 * this entry point.
 *
 * Why it exists: past the sizes where a tile's K range splits over a
 * cluster, gemm_fp8_e4m3 gives every CTA whole tiles, which leaves SMs idle
 * when the tiles do not divide evenly over them (160 tiles on 152 SMs: 8
 * CTAs take two).  The stream-K form cuts the K steps of all tiles into
 * equal ranges and finishes tiles split between CTAs through global scratch
 * (FP32 partial sums and per-tile counters).  A library that allocated that
 * scratch itself would call cudaMalloc, which some callers cannot allow: a
 * serving runtime or framework whose own allocator reserves all of device
 * memory up front (an outside cudaMalloc fails, or fragments its pool), and
 * latency-critical loops that cannot absorb the device-wide synchronisation
 * cudaMalloc and cudaFree may imply.  Here the scratch is a file-scope
 * __device__ array of 32 MiB, present on every device that loads the
 * library until the process exits; the caller still provides A, B, the
 * scales, C and D.
 *
 * Arguments, layouts, alignment and numerics are those of gemm_fp8_e4m3 with
 * mode = TCG_SCALE_BLOCK128.  Kernel choice differs from gemm_fp8_e4m3 in
 * two ways: M > 128 always runs the CTA-pair kernel (no scratch), even where
 * gemm_fp8_e4m3 takes the 128-row chunks because few 256 x 256 tiles would
 * leave SMs idle (such shapes may run slower here); M <= 128 runs the
 * cluster-join form (no scratch) when ceil(N/128) * 2 <= SMs and K > 128,
 * and the stream-K form otherwise.  A stream-K problem whose scratch would
 * exceed 32 MiB is rejected with TCG_ERR_UNSUPPORTED before anything is
 * enqueued: counters take ceil(N/128) 4-byte words rounded up to 256 bytes,
 * partial sums two Mp x 128 FP32 tiles per CTA of the launch (Mp = M rounded
 * up to 16/32/64/128; at most SMs x 128 KB).
 *
 * The first call on a device looks up the array's device address (with that
 * device current) and raises the kernels' shared-memory limits; make that
 * first call before any stream capture.  A stream-K call clears the tile
 * counters (a memset on `stream`), then launches one kernel; every other
 * call launches one kernel.  All calls on a device share the one array and
 * it keeps what the last call left: calls whose executions overlap on the
 * GPU (different streams without ordering between them) race on it and give
 * wrong results.
 */
tcg_status gemm_fp8_e4m3_block_noalloc(int64_t M, int64_t N, int64_t K, const void* A,
                                       int64_t lda, const void* B, int64_t ldb,
                                       const float* a_scale, const float* b_scale, const void* C,
                                       int64_t ldc, void* D, int64_t ldd, tcg_out_dtype out_dtype,
                                       float alpha, float beta, tcg_stream stream);

/*
 * gemm_mxfp8 -- D = alpha * sum over 32-wide K blocks kb of SFA[i,kb] *
 * SFB[j,kb] * sum_{k in kb} A[i,k] B[k,j] + beta * C, with FP8 A and B (E4M3
 * or E5M2 per operand, as gemm_fp8) and one E8M0 scale per row and 32-wide
 * K block of each: the hardware block scaling of "How Blackwell's Tensor
 * Memory Actually Works", section "Quantization became an allocation
 * problem" (D = C + (A x SFA)(B x SFB), scale factors consumed by the tensor
 * core; blocks of 32 with E8M0 scales, the microscaling format).  E8M0 code
 * e is the scale 2^(e - 127).
 *
 * Layouts, C/D, alpha/beta, alignment and errors are those of gemm_fp8.
 * a_sf, b_sf  device pointers to E8M0 bytes, 16-byte aligned, in tiles of
 *             128 rows x 4 blocks (512 bytes): the scale of row r and block kb
 *             is at byte ((r / 128) * KT + kb / 4) * 512 + (r % 32) * 16 +
 *             ((r / 32) % 4) * 4 + kb % 4, KT = ceil(K / 128), for A with r =
 *             i (ceil(M/128) * KT tiles) and for B with r = j (ceil(N/128) *
 *             KT tiles).  Bytes of padding rows and blocks (r >= M or N, kb
 *             >= ceil(K/32)) are read; those of padding blocks must not be
 *             0xFF (NaN), which would reach real outputs through products
 *             with the zero padding of A and B.
 * Kernels     256 x 256 CTA-pair tiles; every product and scale is applied
 *             by the tensor core, accumulation in FP32.  Nothing is
 *             allocated; calls on different streams are independent.
 * Errors      as gemm_fp8; NULL a_sf or b_sf: TCG_ERR_INVALID_ARG; a_sf or
 *             b_sf not 16-byte aligned: TCG_ERR_ALIGNMENT.
 */
tcg_status gemm_mxfp8(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                      tcg_fp8_format a_format, const void* B, int64_t ldb,
                      tcg_fp8_format b_format, const uint8_t* a_sf, const uint8_t* b_sf,
                      const void* C, int64_t ldc, void* D, int64_t ldd, tcg_out_dtype out_dtype,
                      float alpha, float beta, tcg_stream stream);

/* Element type of the quantiser's input. */
typedef enum { TCG_IN_F32 = 0, TCG_IN_BF16 = 1 } tcg_in_dtype;

/* Scale granularity of the quantiser, in the layouts gemm_fp8_e4m3 reads. */
typedef enum {
  /* one scale for the whole matrix: scale[0] */
  TCG_QUANT_TENSOR = 0,
  /* 1 x 128 blocks (row r, columns 128kb..128kb+127): scale[kb * rows + r];
   * the A-operand layout of TCG_SCALE_BLOCK128 with rows = M */
  TCG_QUANT_ROW128 = 1,
  /* 128 x 128 blocks: scale[rb * ceil(cols/128) + kb]; the B-operand layout
   * of TCG_SCALE_BLOCK128 with rows = N */
  TCG_QUANT_BLOCK128 = 2
} tcg_quant_mode;

/*
 * quantize_e4m3 -- FP8 E4M3 codes and FP32 dequantisation scales for a
 * rows x cols matrix X, the step before gemm_fp8_e4m3.
 *
 * The recipe is FP8 scaling as "Tensor cores and low precision" gives it
 * (FP8 paragraph): rescale so that the largest magnitude of a block sits at
 * 448, E4M3's maximum normal value, then cast; the scale is removed after the
 * product.  Scales per tensor, per row or per block ("Tensor Cores",
 * "Precision: FP16, BF16, TF32, FP8").  For each block:
 *     amax = max |x| over the block (NaN entries ignored)
 *     s    = amax / 448 in FP32, correctly rounded; s = 1 if that is 0
 *     Q    = E4M3(x / s): FP32 division, then round to nearest even,
 *            saturating at +-448; a NaN quotient gives 0x7F
 * and scale[...] = s, so that x is approximately decode(Q) * s.  A partial
 * last block (rows or cols not a multiple of 128) uses its own amax.
 *
 * rows, cols   >= 0.  rows == 0 or cols == 0: with TCG_QUANT_TENSOR,
 *              scale[0] = 1 is written; otherwise nothing is done.
 * X, ldx       device pointer, element (r, c) at X[r * ldx + c], FP32 or BF16
 *              (x_dtype); ldx >= cols; X 16-byte aligned, ldx * element size
 *              a multiple of 16 bytes.
 * Q, ldq       device pointer, one byte per element at Q[r * ldq + c];
 *              ldq >= cols, Q 16-byte aligned, ldq a multiple of 16 (so Q can
 *              be gemm_fp8_e4m3's A or B directly).  Bytes at columns >= cols
 *              are not written.
 * scale        device pointer, 4-byte aligned, FP32: 1 value (TENSOR),
 *              rows * ceil(cols/128) (ROW128) or ceil(rows/128) *
 *              ceil(cols/128) (BLOCK128) values.  With TCG_QUANT_TENSOR it
 *              also serves as the running maximum while the call runs (it is
 *              cleared on `stream`, then raised, then read).
 * Errors       TCG_ERR_INVALID_ARG for negative sizes, NULL pointers or short
 *              leading dimensions; TCG_ERR_ALIGNMENT as above;
 *              TCG_ERR_UNSUPPORTED for an unknown x_dtype or mode, or rows or
 *              cols >= 2^31.  Checked on the host before anything is enqueued.
 * Work         ROW128 and BLOCK128: one kernel.  TENSOR: a 4-byte memset and
 *              two kernels (block maxima, then codes).  Nothing is allocated.
 */
tcg_status quantize_e4m3(int64_t rows, int64_t cols, const void* X, int64_t ldx,
                         tcg_in_dtype x_dtype, tcg_quant_mode mode, void* Q, int64_t ldq,
                         float* scale, tcg_stream stream);

/*
 * quantize_fp8 -- quantize_e4m3 with the FP8 encoding chosen: TCG_FP8_E4M3
 * (exactly quantize_e4m3) or TCG_FP8_E5M2, for which the scale is amax /
 * 57344 (E5M2's largest normal value, "Tensor cores and low precision", FP8
 * paragraph) and each code is the E5M2 value of the FP32 quotient, nearest
 * even, saturating at +-57344; a NaN quotient gives 0x7F.  The pages suggest
 * E5M2 for gradients.  Arguments, layouts, errors and work as quantize_e4m3;
 * an unknown format returns TCG_ERR_UNSUPPORTED.
 */
tcg_status quantize_fp8(int64_t rows, int64_t cols, const void* X, int64_t ldx,
                        tcg_in_dtype x_dtype, tcg_fp8_format format, tcg_quant_mode mode,
                        void* Q, int64_t ldq, float* scale, tcg_stream stream);

/* A static, human-readable name for a status code. */
const char* tcg_status_string(tcg_status status);

/*
 * Synchronises `stream`, then reads and clears this device's status word.
 * Returns TCG_ERR_TIMEOUT if any kernel of this library on the current
 * device gave up on a wait since the last call, TCG_ERR_CUDA if the
 * synchronisation failed, else TCG_OK.  Meant for tests and debugging.
 */
tcg_status tcg_last_device_status(tcg_stream stream);

/*
 * tcg_debug_timeout_probe -- exercises the failure path every kernel's waits
 * share, for tests.  Enqueues one CTA whose only work is a bounded wait on an
 * mbarrier that nothing signals: after the library's wait limit (2 s) it
 * records TCG_ERR_TIMEOUT in the device status word and returns (no trap, no
 * fault; the context stays usable).  tcg_last_device_status(stream) then
 * reports TCG_ERR_TIMEOUT once.  The pages have no counterpart: it tests the
 * bounded waits the build adds because a spinning wait on a shared GPU must
 * end.
 */
tcg_status tcg_debug_timeout_probe(tcg_stream stream);

/* Number of kernels this library has launched in this process (all devices). */
uint64_t tcg_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* TCGEMM_H */
