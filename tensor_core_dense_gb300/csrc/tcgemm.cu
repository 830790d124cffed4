// tcgemm.cu -- host side of the C ABI declared in include/tcgemm.h:
// argument validation, TMA tensor-map encoding (cached), kernel selection and
// launch.  The kernels themselves are in gemm_tn2.cuh / gemm_tn.cuh (BF16 and
// per-tensor FP8), gemm_skinny.cuh (decode-sized shapes and block-scaled FP8
// in 128-row chunks) and gemm_tn2b.cuh (block-scaled FP8 on pair tiles); the
// FP8 quantiser's are in quant.cuh.  No entry point allocates device memory;
// gemm_fp8_e4m3_block_noalloc keeps a fixed scratch array in this module.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <utility>

#include "gemm_mx.cuh"
#include "gemm_skinny.cuh"
#include "gemm_tn.cuh"
#include "gemm_tn2.cuh"
#include "gemm_tn2b.cuh"
#include "quant.cuh"
#include "tcgemm.h"

namespace tcg {
namespace {

std::atomic<uint64_t> g_launches{0};

// ---------------------------------------------------------------- K == 0

// D = beta * C (or 0): the product has no terms.
__global__ void scale_c_kernel(int64_t M, int64_t N, const void* C, int64_t ldc, void* D,
                               int64_t ldd, float beta, int out_f32, int has_c) {
  const int64_t total = M * N;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = e / N, j = e % N;
    float v = 0.0f;
    if (out_f32) {
      if (has_c) v = beta * static_cast<const float*>(C)[i * ldc + j];
      static_cast<float*>(D)[i * ldd + j] = v;
    } else {
      if (has_c)
        v = beta * __uint_as_float((uint32_t)static_cast<const uint16_t*>(C)[i * ldc + j] << 16);
      static_cast<uint16_t*>(D)[i * ldd + j] = (uint16_t)(pack_bf16x2(v, 0.0f) & 0xFFFFu);
    }
  }
}

// ------------------------------------------------------ timeout probe

// One CTA waits on an mbarrier that nothing arrives on, with the library's
// bounded wait: it must give up after kWaitLimitNs, record TCG_ERR_TIMEOUT
// in the status word and return, leaving the context usable.
__global__ void wait_timeout_probe_kernel() {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)wait_phase(smem_u32(&bar), 0, &abort_flag, 0x7E);
  __syncthreads();
}

// ---------------------------------------------------------------- devices

struct DeviceInfo {
  int sms = 0;
  bool init = false;
};
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

tcg_status current_device(int* dev, int* sms) {
  if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) return TCG_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[*dev];
  if (!d.init) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess)
      return TCG_ERR_CUDA;
    d.init = true;
  }
  *sms = d.sms;
  return TCG_OK;
}

// Raises a kernel's dynamic shared-memory limit once per (kernel, device).
std::mutex g_attr_mu;
std::unordered_map<uint64_t, bool> g_attr_done;

template <typename F>
tcg_status ensure_smem(F* fn, uint32_t bytes, int dev) {
  const uint64_t key = (uint64_t)(uintptr_t)fn * 131u + (uint64_t)dev;
  std::lock_guard<std::mutex> lk(g_attr_mu);
  if (g_attr_done.count(key)) return TCG_OK;
  if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)bytes) != cudaSuccess)
    return TCG_ERR_CUDA;
  g_attr_done[key] = true;
  return TCG_OK;
}

// ------------------------------------------------------------ tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// A tensor map's identity; the planes fields are 0 for 2-D maps.
struct MapKey {
  uint64_t ptr, inner, rows, ld_bytes;
  uint32_t dtype, box_inner, box_rows, swizzle;
  uint64_t planes = 0, plane_bytes = 0;
  uint32_t box_planes = 0;
  uint64_t cubes = 0, cube_bytes = 0;  // 4-D maps: fourth dimension
  uint32_t box_cubes = 0;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && inner == o.inner && rows == o.rows && ld_bytes == o.ld_bytes &&
           dtype == o.dtype && box_inner == o.box_inner && box_rows == o.box_rows &&
           swizzle == o.swizzle && planes == o.planes && plane_bytes == o.plane_bytes &&
           box_planes == o.box_planes && cubes == o.cubes && cube_bytes == o.cube_bytes &&
           box_cubes == o.box_cubes;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    uint64_t h = 1469598103934665603ull;
    const uint64_t v[14] = {k.ptr,       k.inner,       k.rows,       k.ld_bytes, k.dtype,
                            k.box_inner, k.box_rows,    k.swizzle,    k.planes,   k.plane_bytes,
                            k.box_planes, k.cubes,      k.cube_bytes, k.box_cubes};
    for (uint64_t x : v) h = (h ^ x) * 1099511628211ull;
    return (size_t)h;
  }
};
std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;
constexpr size_t kMaxCachedMaps = 4096;

// A 2-D row-major matrix (rows x inner elements, pitch ld_bytes) read in
// boxes of box_rows x box_inner with 128-byte swizzling (or `swizzle`);
// out-of-range elements read as zero.
tcg_status tensor_map(CUtensorMap* out, CUtensorMapDataType dtype, const void* ptr,
                      uint64_t inner, uint64_t rows, uint64_t ld_bytes, uint32_t box_inner,
                      uint32_t box_rows,
                      CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  const MapKey key{(uint64_t)(uintptr_t)ptr, inner,     rows,     ld_bytes,
                   (uint32_t)dtype,          box_inner, box_rows, (uint32_t)swizzle};
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    auto it = g_maps.find(key);
    if (it != g_maps.end()) {
      *out = it->second;
      return TCG_OK;
    }
  }
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return TCG_ERR_CUDA;
  CUtensorMap m;
  std::memset(&m, 0, sizeof m);
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {ld_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(&m, dtype, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return TCG_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_map_mu);
  if (g_maps.size() >= kMaxCachedMaps) g_maps.clear();
  g_maps.emplace(key, m);
  *out = m;
  return TCG_OK;
}

// A 3-D tensor (inner x rows x planes elements, row pitch ld_bytes, plane
// pitch plane_bytes) read in boxes of box_inner x box_rows x box_planes,
// without swizzling; out-of-range elements read as zero.
tcg_status tensor_map_3d(CUtensorMap* out, CUtensorMapDataType dtype, const void* ptr,
                         uint64_t inner, uint64_t rows, uint64_t planes, uint64_t ld_bytes,
                         uint64_t plane_bytes, uint32_t box_inner, uint32_t box_rows,
                         uint32_t box_planes) {
  MapKey key{(uint64_t)(uintptr_t)ptr, inner,     rows,     ld_bytes,
             (uint32_t)dtype,          box_inner, box_rows, (uint32_t)CU_TENSOR_MAP_SWIZZLE_NONE};
  key.planes = planes;
  key.plane_bytes = plane_bytes;
  key.box_planes = box_planes;
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    auto it = g_maps.find(key);
    if (it != g_maps.end()) {
      *out = it->second;
      return TCG_OK;
    }
  }
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return TCG_ERR_CUDA;
  CUtensorMap m;
  std::memset(&m, 0, sizeof m);
  const cuuint64_t dims[3] = {inner, rows, planes};
  const cuuint64_t strides[2] = {ld_bytes, plane_bytes};
  const cuuint32_t box[3] = {box_inner, box_rows, box_planes};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(&m, dtype, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return TCG_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_map_mu);
  if (g_maps.size() >= kMaxCachedMaps) g_maps.clear();
  g_maps.emplace(key, m);
  *out = m;
  return TCG_OK;
}

// A 4-D tensor (inner x rows x planes x cubes elements; pitches ld_bytes,
// plane_bytes, cube_bytes, any of them may be 0 to repeat the data) read in
// boxes without swizzling; out-of-range elements read as zero.
tcg_status tensor_map_4d(CUtensorMap* out, CUtensorMapDataType dtype, const void* ptr,
                         const uint64_t (&dims)[4], const uint64_t (&pitch)[3],
                         const uint32_t (&box)[4]) {
  MapKey key{(uint64_t)(uintptr_t)ptr, dims[0], dims[1], pitch[0],
             (uint32_t)dtype,          box[0],  box[1],  (uint32_t)CU_TENSOR_MAP_SWIZZLE_NONE};
  key.planes = dims[2];
  key.plane_bytes = pitch[1];
  key.box_planes = box[2];
  key.cubes = dims[3];
  key.cube_bytes = pitch[2];
  key.box_cubes = box[3];
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    auto it = g_maps.find(key);
    if (it != g_maps.end()) {
      *out = it->second;
      return TCG_OK;
    }
  }
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return TCG_ERR_CUDA;
  CUtensorMap m;
  std::memset(&m, 0, sizeof m);
  const cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
  const cuuint64_t st[3] = {pitch[0], pitch[1], pitch[2]};
  const cuuint32_t b[4] = {box[0], box[1], box[2], box[3]};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = enc(&m, dtype, 4, const_cast<void*>(ptr), d, st, b, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return TCG_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_map_mu);
  if (g_maps.size() >= kMaxCachedMaps) g_maps.clear();
  g_maps.emplace(key, m);
  *out = m;
  return TCG_OK;
}

// ------------------------------------------------------------- validation

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

struct Common {
  int64_t M, N, K;
  const void *A, *B, *C;
  int64_t lda, ldb, ldc, ldd;
  void* D;
  int out;  // tcg_out_dtype
  float alpha, beta;
  int a_fp8 = 0, b_fp8 = 0;  // tcg_fp8_format of A and B (FP8 entry points)
};

// FP8 operand formats as the instruction descriptor's A and B fields.
uint32_t fp8_fmt_bits(int umma_a, int umma_b) {
  return ((uint32_t)umma_a << 7) | ((uint32_t)umma_b << 10);
}

// Checks shared by both entry points; in_bytes = bytes per A/B element.
tcg_status validate(const Common& a, int in_bytes) {
  if (a.M < 0 || a.N < 0 || a.K < 0) return TCG_ERR_INVALID_ARG;
  if (a.out != TCG_OUT_BF16 && a.out != TCG_OUT_F32) return TCG_ERR_UNSUPPORTED;
  if (a.M == 0 || a.N == 0) return TCG_OK;
  if (a.M > INT32_MAX || a.N > INT32_MAX || a.K > INT32_MAX) return TCG_ERR_UNSUPPORTED;
  const int out_bytes = a.out == TCG_OUT_F32 ? 4 : 2;
  if (!a.D || a.ldd < a.N) return TCG_ERR_INVALID_ARG;
  if (a.beta != 0.0f && (!a.C || a.ldc < a.N)) return TCG_ERR_INVALID_ARG;
  if (a.K > 0 && (!a.A || !a.B || a.lda < a.K || a.ldb < a.K)) return TCG_ERR_INVALID_ARG;
  if (!aligned16(a.D) || (a.ldd * out_bytes) % 16 != 0) return TCG_ERR_ALIGNMENT;
  if (a.beta != 0.0f && (!aligned16(a.C) || (a.ldc * out_bytes) % 16 != 0))
    return TCG_ERR_ALIGNMENT;
  if (a.K > 0 && (!aligned16(a.A) || !aligned16(a.B) || (a.lda * in_bytes) % 16 != 0 ||
                  (a.ldb * in_bytes) % 16 != 0))
    return TCG_ERR_ALIGNMENT;
  return TCG_OK;
}

tcg_status launch_k0(const Common& a, cudaStream_t stream) {
  const int64_t total = a.M * a.N;
  const int threads = 256;
  const int64_t want = (total + threads - 1) / threads;
  const int blocks = (int)(want < 4096 ? want : 4096);
  scale_c_kernel<<<blocks, threads, 0, stream>>>(a.M, a.N, a.beta != 0.0f ? a.C : nullptr, a.ldc,
                                                 a.D, a.ldd, a.beta, a.out == TCG_OUT_F32,
                                                 a.beta != 0.0f);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError() == cudaSuccess ? TCG_OK : TCG_ERR_CUDA;
}

// Launches a GEMM kernel with programmatic stream serialisation, so that its
// CTAs may start (and run their set-up) while the previous kernel in the
// stream drains; the kernels wait for that kernel before touching global
// memory.  cluster_x > 1 launches clusters of that many CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_gemm_kernel(void (*fn)(KArgs...), int grid, int block, uint32_t smem,
                               cudaStream_t stream, int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3((unsigned)block, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = (unsigned)n;
  return cudaLaunchKernelEx(&cfg, fn, std::forward<Args>(args)...);
}

template <int kIn, int kOut, bool kHasC>
tcg_status launch_tn_inst(const CUtensorMap& ma, const CUtensorMap& mb, const GemmParams& p,
                          int grid, int dev, cudaStream_t stream) {
  auto* fn = &gemm_tn_kernel<kIn, kOut, kHasC>;
  if (tcg_status s = ensure_smem(fn, kSmemBytes, dev); s != TCG_OK) return s;
  if (launch_gemm_kernel(fn, grid, kThreads, kSmemBytes, stream, 1, ma, mb, p) != cudaSuccess)
    return TCG_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError() == cudaSuccess ? TCG_OK : TCG_ERR_CUDA;
}

// Kernel choice for the dense path: the CTA-pair kernel for problems with at
// least one full 256 x 256 tile; for M <= 128 the swap-AB skinny kernel where
// skinny_pays says so; else the one-SM kernel.  For block-scaled FP8: the pair
// kernel for M > 128 (see gemm_fp8), else the skinny one.  TCG_KERNEL=1cta,
// 2cta or skinny in the environment forces one of them (for tests and
// measurements).
int forced_kernel() {
  const char* e = std::getenv("TCG_KERNEL");
  if (!e) return 0;
  if (std::strcmp(e, "1cta") == 0) return 1;
  if (std::strcmp(e, "2cta") == 0) return 2;
  if (std::strcmp(e, "skinny") == 0) return 3;
  return 0;
}

template <int kIn, int kOut, bool kHasC>
tcg_status launch_tn2_inst(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& md,
                           const CUtensorMap& mc, const Gemm2Params& p, int grid, int dev,
                           cudaStream_t stream) {
  auto* fn = &gemm_tn2_kernel<kIn, kOut, kHasC>;
  if (tcg_status s = ensure_smem(fn, kP2DSmemBytes, dev); s != TCG_OK) return s;
  if (launch_gemm_kernel(fn, grid, kThreads, kP2DSmemBytes, stream, 2, ma, mb, md, mc, p) !=
      cudaSuccess)
    return TCG_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError() == cudaSuccess ? TCG_OK : TCG_ERR_CUDA;
}

tcg_status pair_schedule(const Common& a, int in_bytes, int sms, Gemm2Params* pp, int* grid);

// Tensor maps and the persistent schedule of the 256 x 256 pair-tile kernels:
// whole tiles in waves of SMs/2 clusters, the rest split into two 256 x 128
// halves when that still fits one wave.  Returns the grid (CTAs).
tcg_status pair_setup(const Common& a, int in_bytes, int sms, CUtensorMap* ma, CUtensorMap* mb,
                      Gemm2Params* pp, int* grid) {
  const CUtensorMapDataType dt =
      in_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const uint32_t box_k = kBKBytes / in_bytes;
  if (tcg_status s = tensor_map(ma, dt, a.A, a.K, a.M, a.lda * in_bytes, box_k, 128); s != TCG_OK)
    return s;
  if (tcg_status s = tensor_map(mb, dt, a.B, a.K, a.N, a.ldb * in_bytes, box_k, kBBoxRows);
      s != TCG_OK)
    return s;
  return pair_schedule(a, in_bytes, sms, pp, grid);
}

// The schedule part of pair_setup (no tensor maps, no host-side tables).
tcg_status pair_schedule(const Common& a, int in_bytes, int sms, Gemm2Params* pp, int* grid) {
  Gemm2Params& p = *pp;
  p = Gemm2Params{};
  p.M = (int32_t)a.M;
  p.N = (int32_t)a.N;
  p.K = (int32_t)a.K;
  p.tiles_m = (int32_t)((a.M + 255) / 256);
  p.tiles_n = (int32_t)((a.N + 255) / 256);
  p.num_kb = (int32_t)((a.K * in_bytes + kBKBytes - 1) / kBKBytes);
  const int64_t tiles = (int64_t)p.tiles_m * p.tiles_n;
  if (tiles > INT32_MAX) return TCG_ERR_UNSUPPORTED;
  p.num_tiles = (int32_t)tiles;
  const int clusters_max = sms / 2;
  int clusters = clusters_max;
  int64_t rest;
  if (tiles >= clusters_max) {
    p.dp_waves = (int32_t)(tiles / clusters_max);
    rest = tiles % clusters_max;
  } else {
    p.dp_waves = 0;
    rest = tiles;
  }
  const int split = (rest > 0 && rest * 2 <= clusters_max) ? 2 : 1;
  if (tiles < clusters_max) clusters = (int)(rest * split);
  p.dp_end = (int32_t)(tiles - rest);
  p.split = split;
  p.C = a.beta != 0.0f ? a.C : nullptr;
  p.ldc = a.ldc;
  p.D = a.D;
  p.ldd = a.ldd;
  p.alpha = a.alpha;
  p.beta = a.beta;
  p.fp8_fmt = fp8_fmt_bits(a.a_fp8, a.b_fp8);
  *grid = 2 * clusters;
  return TCG_OK;
}

// The persistent 256 x 256 pair-tile kernel.
template <int kIn>
tcg_status launch_tn2(const Common& a, const float* a_scale, const float* b_scale,
                      cudaStream_t stream, int dev, int sms) {
  CUtensorMap ma, mb;
  Gemm2Params p;
  int grid;
  if (tcg_status s = pair_setup(a, kIn == 0 ? 2 : 1, sms, &ma, &mb, &p, &grid); s != TCG_OK)
    return s;
  p.a_scale = a_scale;
  p.b_scale = b_scale;
  const bool has_c = a.beta != 0.0f;
  // D (and C) as 2-D tensors for the epilogue's TMA stores (loads): boxes of
  // 128 bytes (64 BF16 or 32 FP32 columns) x 32 rows, 128-byte swizzle
  const bool bf16 = a.out == TCG_OUT_BF16;
  const CUtensorMapDataType dto = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const int osz = bf16 ? 2 : 4;
  CUtensorMap md, mc;
  if (tcg_status s = tensor_map(&md, dto, a.D, a.N, a.M, a.ldd * osz, 128 / osz, 32); s != TCG_OK)
    return s;
  mc = md;
  if (has_c) {
    if (tcg_status s = tensor_map(&mc, dto, a.C, a.N, a.M, a.ldc * osz, 128 / osz, 32);
        s != TCG_OK)
      return s;
  }
  if (bf16)
    return has_c ? launch_tn2_inst<kIn, 0, true>(ma, mb, md, mc, p, grid, dev, stream)
                 : launch_tn2_inst<kIn, 0, false>(ma, mb, md, mc, p, grid, dev, stream);
  return has_c ? launch_tn2_inst<kIn, 1, true>(ma, mb, md, mc, p, grid, dev, stream)
               : launch_tn2_inst<kIn, 1, false>(ma, mb, md, mc, p, grid, dev, stream);
}

template <int kOut, bool kHasC>
tcg_status launch_block_pair_inst(const CUtensorMap& ma, const CUtensorMap& mb,
                                  const Gemm2Params& p, int grid, int dev, cudaStream_t stream) {
  auto* fn = &gemm_fp8_block_pair_kernel<kOut, kHasC>;
  if (tcg_status s = ensure_smem(fn, kP2SmemBytes, dev); s != TCG_OK) return s;
  if (launch_gemm_kernel(fn, grid, kPbThreads, kP2SmemBytes, stream, 2, ma, mb, p) != cudaSuccess)
    return TCG_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError() == cudaSuccess ? TCG_OK : TCG_ERR_CUDA;
}

// Block-scaled FP8 on 256 x 256 pair tiles (the schedule of launch_tn2).
tcg_status launch_block_pair(const Common& a, const float* a_scale, const float* b_scale,
                             cudaStream_t stream, int dev, int sms) {
  CUtensorMap ma, mb;
  Gemm2Params p;
  int grid;
  if (tcg_status s = pair_setup(a, 1, sms, &ma, &mb, &p, &grid); s != TCG_OK) return s;
  p.a_scale = a_scale;
  p.b_scale = b_scale;
  const bool has_c = a.beta != 0.0f;
  if (a.out == TCG_OUT_BF16)
    return has_c ? launch_block_pair_inst<0, true>(ma, mb, p, grid, dev, stream)
                 : launch_block_pair_inst<0, false>(ma, mb, p, grid, dev, stream);
  return has_c ? launch_block_pair_inst<1, true>(ma, mb, p, grid, dev, stream)
               : launch_block_pair_inst<1, false>(ma, mb, p, grid, dev, stream);
}

template <int kIn>
tcg_status launch_skinny(const Common& a, const float* sa, const float* sb, bool scalar,
                         cudaStream_t stream);

template <int kOut, bool kHasC>
tcg_status launch_mx_inst(const CUtensorMap (&maps)[4], const MxParams& p, int grid, int dev,
                          cudaStream_t stream) {
  auto* fn = &gemm_mx_pair_kernel<kOut, kHasC>;
  if (tcg_status s = ensure_smem(fn, kMxSmemBytes, dev); s != TCG_OK) return s;
  if (launch_gemm_kernel(fn, grid, kMxThreads, kMxSmemBytes, stream, 2, maps[0], maps[1], maps[2],
                         maps[3], p) != cudaSuccess)
    return TCG_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError() == cudaSuccess ? TCG_OK : TCG_ERR_CUDA;
}

// Microscaled FP8 on 256 x 256 pair tiles (the schedule of launch_tn2): A
// and B maps as the FP8 pair kernel's, and 3-D maps over the tiled E8M0
// scales (128 four-byte words per 512-byte tile x K tiles x row tiles).
tcg_status launch_mx(const Common& a, const uint8_t* a_sf, const uint8_t* b_sf,
                     cudaStream_t stream) {
  int dev, sms;
  if (tcg_status s = current_device(&dev, &sms); s != TCG_OK) return s;
  CUtensorMap maps[4];
  Gemm2Params g;
  int grid;
  if (tcg_status s = pair_setup(a, 1, sms, &maps[0], &maps[1], &g, &grid); s != TCG_OK) return s;
  const uint64_t kt = (uint64_t)((a.K + 127) / 128);
  const uint64_t rta = (uint64_t)((a.M + 127) / 128), rtb = (uint64_t)((a.N + 127) / 128);
  if (tcg_status s = tensor_map_3d(&maps[2], CU_TENSOR_MAP_DATA_TYPE_UINT32, a_sf, 128, kt, rta,
                                   512, kt * 512, 128, 1, 1);
      s != TCG_OK)
    return s;
  // B: each 512-byte tile read 4 times (a stride-0 dimension), two row tiles
  // per box: the 128 x 32-byte image of one 128x256b Tensor Memory copy
  if (tcg_status s = tensor_map_4d(&maps[3], CU_TENSOR_MAP_DATA_TYPE_UINT32, b_sf,
                                   {128, 4, kt, rtb}, {0, 512, kt * 512}, {128, 4, 1, 2});
      s != TCG_OK)
    return s;
  MxParams p{};
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.tiles_m = g.tiles_m;
  p.tiles_n = g.tiles_n;
  p.num_kb = g.num_kb;
  p.num_tiles = g.num_tiles;
  p.dp_waves = g.dp_waves;
  p.dp_end = g.dp_end;
  p.split = g.split;
  p.fp8_fmt = g.fp8_fmt;
  p.C = g.C;
  p.ldc = g.ldc;
  p.D = g.D;
  p.ldd = g.ldd;
  p.alpha = g.alpha;
  p.beta = g.beta;
  const bool has_c = a.beta != 0.0f;
  if (a.out == TCG_OUT_BF16)
    return has_c ? launch_mx_inst<0, true>(maps, p, grid, dev, stream)
                 : launch_mx_inst<0, false>(maps, p, grid, dev, stream);
  return has_c ? launch_mx_inst<1, true>(maps, p, grid, dev, stream)
               : launch_mx_inst<1, false>(maps, p, grid, dev, stream);
}

// Decode-sized problems (M <= 128) are streams of B: the swap-AB skinny
// kernel spreads them over the SMs in K, where the 128 x 256 tile kernel has
// only ceil(N/256) tiles.  It is taken when every N tile splits into two or
// three pieces joined by a cluster in shared memory (N tiles * 2 <= SMs, at
// least two K steps): that form uses no workspace, so these calls keep the
// dense entry points' properties (no allocation, calls on concurrent streams
// independent).  Measured on GB300: BF16 M = 16, N = K = 8192 (pairs): 26.1
// us against 40.4; N = 2048, K = 4096 (clusters of three): 11.0 against 20.2;
// M = 128, N = 4096, K = 4096: 15.8 against 21.3; per-tensor FP8 M = 64,
// N = 2048, K = 2048: 6.8 against 7.2.
bool skinny_pays(const Common& a, int in_bytes, int sms) {
  const int64_t n_tiles = (a.N + 127) / 128;
  const int64_t steps = (a.K * in_bytes + 127) / 128;
  return n_tiles * 2 <= sms && steps >= 2;
}

// The persistent 128 x 256 tile kernel (BF16, or per-tensor FP8).
template <int kIn>
tcg_status launch_tn(const Common& a, const float* a_scale, const float* b_scale,
                     cudaStream_t stream) {
  int dev, sms;
  if (tcg_status s = current_device(&dev, &sms); s != TCG_OK) return s;
  const int fk = forced_kernel();
  if (fk == 2 || (fk == 0 && a.M >= 256 && a.N >= 256))
    return launch_tn2<kIn>(a, a_scale, b_scale, stream, dev, sms);
  if (a.M <= 128 && (fk == 3 || (fk == 0 && skinny_pays(a, kIn == 0 ? 2 : 1, sms))))
    return launch_skinny<kIn>(a, a_scale, b_scale, true, stream);
  const int in_bytes = kIn == 0 ? 2 : 1;
  const CUtensorMapDataType dt =
      kIn == 0 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const uint32_t box_k = kBKBytes / in_bytes;
  CUtensorMap ma, mb;
  const uint32_t a_rows = a.M < kBM ? (uint32_t)((a.M + 7) / 8 * 8) : (uint32_t)kBM;
  if (tcg_status s = tensor_map(&ma, dt, a.A, a.K, a.M, a.lda * in_bytes, box_k, a_rows);
      s != TCG_OK)
    return s;
  if (tcg_status s = tensor_map(&mb, dt, a.B, a.K, a.N, a.ldb * in_bytes, box_k, kBBoxRows);
      s != TCG_OK)
    return s;
  GemmParams p{};
  p.a_rows = a_rows;
  p.M = (int32_t)a.M;
  p.N = (int32_t)a.N;
  p.K = (int32_t)a.K;
  p.tiles_m = (int32_t)((a.M + kBM - 1) / kBM);
  p.tiles_n = (int32_t)((a.N + kBN - 1) / kBN);
  p.num_kb = (int32_t)((a.K * in_bytes + kBKBytes - 1) / kBKBytes);
  const int64_t tiles = (int64_t)p.tiles_m * p.tiles_n;
  if (tiles > INT32_MAX) return TCG_ERR_UNSUPPORTED;
  p.num_tiles = (int32_t)tiles;
  p.C = a.beta != 0.0f ? a.C : nullptr;
  p.ldc = a.ldc;
  p.D = a.D;
  p.ldd = a.ldd;
  p.alpha = a.alpha;
  p.beta = a.beta;
  p.a_scale = a_scale;
  p.fp8_fmt = fp8_fmt_bits(a.a_fp8, a.b_fp8);
  p.b_scale = b_scale;
  // Schedule: whole waves of tiles run one tile per CTA; the tiles left for a
  // last partial wave (or all tiles, when there are fewer than SMs) are cut
  // along N into 2 or 4 sub-tiles when that still fits in one wave.
  int grid;
  int64_t rest;
  if (tiles >= sms) {
    grid = sms;
    p.dp_waves = (int32_t)(tiles / sms);
    rest = tiles % sms;
  } else {
    p.dp_waves = 0;
    rest = tiles;
  }
  int split = 1;
  if (rest > 0) {
    if (rest * 4 <= sms) split = 4;
    else if (rest * 2 <= sms) split = 2;
  }
  if (tiles < sms) grid = (int)(rest * split);
  p.dp_end = (int32_t)(tiles - rest);
  p.split = split;
  const bool has_c = a.beta != 0.0f;
  if (a.out == TCG_OUT_BF16)
    return has_c ? launch_tn_inst<kIn, 0, true>(ma, mb, p, grid, dev, stream)
                 : launch_tn_inst<kIn, 0, false>(ma, mb, p, grid, dev, stream);
  return has_c ? launch_tn_inst<kIn, 1, true>(ma, mb, p, grid, dev, stream)
               : launch_tn_inst<kIn, 1, false>(ma, mb, p, grid, dev, stream);
}

// The skinny kernel with its tiles split over clusters of kJoin CTAs.
template <int kMp, int kJoin, int kIn, bool kScalar>
tcg_status launch_skinny_join(bool chunks, const CUtensorMap& ma, const CUtensorMap& mb,
                              const SkinnyParams& p, cudaStream_t stream, int dev) {
  using Cfg = SkinnyCfg<kMp>;
  constexpr bool kChunks = kMp == 128 && kIn == 1 && !kScalar;  // M > 128: block scales only
  auto* fn = chunks ? &gemm_fp8_block_skinny_kernel<kMp, kJoin, kChunks, kIn, kScalar>
                    : &gemm_fp8_block_skinny_kernel<kMp, kJoin, false, kIn, kScalar>;
  if (tcg_status s = ensure_smem(fn, Cfg::kSmemBytes, dev); s != TCG_OK) return s;
  if (launch_gemm_kernel(fn, p.grid, Cfg::kThreads, Cfg::kSmemBytes, stream, kJoin, ma, mb, p) !=
      cudaSuccess)
    return TCG_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError() == cudaSuccess ? TCG_OK : TCG_ERR_CUDA;
}

// Whether `tiles` clusters of three skinny CTAs can be resident at once (a
// cluster must fit in one GPC, so fewer than SMs/3 may fit); asked once per
// kernel and device.
template <int kMp, int kIn, bool kScalar>
bool skinny_trio_fits(bool chunks, int64_t tiles, int dev) {
  using Cfg = SkinnyCfg<kMp>;
  static int max_clusters[2][kMaxDevices] = {};
  constexpr bool kChunks = kMp == 128 && kIn == 1 && !kScalar;
  auto* fn = chunks ? &gemm_fp8_block_skinny_kernel<kMp, 3, kChunks, kIn, kScalar>
                    : &gemm_fp8_block_skinny_kernel<kMp, 3, false, kIn, kScalar>;
  std::lock_guard<std::mutex> lk(g_attr_mu);
  int& n = max_clusters[chunks ? 1 : 0][dev];
  if (n == 0) {
    if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)Cfg::kSmemBytes) != cudaSuccess)
      return false;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(3, 1, 1);
    cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 3;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n <= 0) {
      n = -1;  // unknown: use pairs
      cudaGetLastError();
    }
  }
  return n > 0 && tiles <= n;
}

// kIn: 1 = FP8 (block scales, or one scale per tensor with kScalar), 0 = BF16
// (M <= 128, no scales, kScalar).
template <int kMp, int kIn, bool kScalar>
tcg_status launch_skinny_inst(const Common& a, const float* sa, const float* sb,
                              cudaStream_t stream, int dev, int sms) {
  using Cfg = SkinnyCfg<kMp>;
  constexpr bool kChunks = kMp == 128 && kIn == 1 && !kScalar;
  if (kScalar && a.M > kMp) return TCG_ERR_UNSUPPORTED;  // one chunk of A only
  constexpr int in_bytes = kIn == 1 ? 1 : 2;
  const CUtensorMapDataType dt =
      kIn == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap ma, mb;
  if (tcg_status s = tensor_map(&ma, dt, a.A, a.K, a.M, a.lda * in_bytes, 128 / in_bytes, kMp);
      s != TCG_OK)
    return s;
  if (tcg_status s = tensor_map(&mb, dt, a.B, a.K, a.N, a.ldb * in_bytes, 128 / in_bytes, 128);
      s != TCG_OK)
    return s;
  SkinnyParams p{};
  p.M = (int32_t)a.M;
  p.N = (int32_t)a.N;
  p.K = (int32_t)a.K;
  p.n_tiles = (int32_t)((a.N + 127) / 128);
  p.m_tiles = (int32_t)((a.M + kMp - 1) / kMp);  // 1 unless M > 128 (kMp = 128)
  p.num_kb = (int32_t)((a.K * in_bytes + 127) / 128);  // 128-byte steps of K
  const int64_t tiles = (int64_t)p.n_tiles * p.m_tiles;
  const int64_t T = tiles * p.num_kb;
  if (T > INT32_MAX) return TCG_ERR_UNSUPPORTED;
  p.total_steps = (int32_t)T;
  // A tile's K range is cut into two or three pieces, one per CTA of a
  // cluster that joins them in shared memory, when the tiles fill at most
  // half (a third) of the SMs; otherwise every CTA takes whole tiles (grid =
  // min(tiles, SMs), contiguous tile ranges) and writes D directly.  Neither
  // form has a partial tile that crosses CTAs through global memory, so this
  // entry point needs no workspace and calls on concurrent streams stay
  // independent.
  int64_t split = tiles < sms ? sms / tiles : 1;
  if (split > 3) split = 3;
  if (split > p.num_kb) split = p.num_kb;
  p.a_scale = sa;
  p.fp8_fmt = fp8_fmt_bits(a.b_fp8, a.a_fp8);  // swap-AB: UMMA A is B
  p.b_scale = sb;
  p.C = a.beta != 0.0f ? a.C : nullptr;
  p.ldc = a.ldc;
  p.D = a.D;
  p.ldd = a.ldd;
  p.alpha = a.alpha;
  p.beta = a.beta;
  p.out_f32 = a.out == TCG_OUT_F32;
  p.has_c = a.beta != 0.0f;
  if (split == 3 && !skinny_trio_fits<kMp, kIn, kScalar>(p.m_tiles > 1, tiles, dev))
    split = 2;  // fewer clusters of three fit at once than there are tiles
  if (split == 2 || split == 3) {
    // two or three pieces per tile: a cluster of their CTAs joins them in
    // shared memory (no workspace)
    p.grid = (int32_t)(tiles * split);
    if (split == 2)
      return launch_skinny_join<kMp, 2, kIn, kScalar>(p.m_tiles > 1, ma, mb, p, stream, dev);
    return launch_skinny_join<kMp, 3, kIn, kScalar>(p.m_tiles > 1, ma, mb, p, stream, dev);
  }
  p.whole_tiles = 1;
  p.grid = (int32_t)(tiles < sms ? tiles : sms);
  p.max_seg = 1;
  auto* fn = p.m_tiles > 1 ? &gemm_fp8_block_skinny_kernel<kMp, 0, kChunks, kIn, kScalar>
                           : &gemm_fp8_block_skinny_kernel<kMp, 0, false, kIn, kScalar>;
  if (tcg_status s = ensure_smem(fn, Cfg::kSmemBytes, dev); s != TCG_OK) return s;
  if (launch_gemm_kernel(fn, p.grid, Cfg::kThreads, Cfg::kSmemBytes, stream, 1, ma, mb, p) !=
      cudaSuccess)
    return TCG_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError() == cudaSuccess ? TCG_OK : TCG_ERR_CUDA;
}

template <int kIn, bool kScalar>
tcg_status launch_skinny_mp(const Common& a, const float* sa, const float* sb,
                            cudaStream_t stream) {
  int dev, sms;
  if (tcg_status s = current_device(&dev, &sms); s != TCG_OK) return s;
  if (a.M <= 16) return launch_skinny_inst<16, kIn, kScalar>(a, sa, sb, stream, dev, sms);
  if (a.M <= 32) return launch_skinny_inst<32, kIn, kScalar>(a, sa, sb, stream, dev, sms);
  if (a.M <= 64) return launch_skinny_inst<64, kIn, kScalar>(a, sa, sb, stream, dev, sms);
  return launch_skinny_inst<128, kIn, kScalar>(a, sa, sb, stream, dev, sms);
}

// scalar: one scale for the problem (per-tensor FP8, or BF16).
template <int kIn>
tcg_status launch_skinny(const Common& a, const float* sa, const float* sb, bool scalar,
                         cudaStream_t stream) {
  if constexpr (kIn == 1) {
    if (!scalar) return launch_skinny_mp<1, false>(a, sa, sb, stream);
  }
  return launch_skinny_mp<kIn, true>(a, sa, sb, stream);
}

// ------------------------------------------------------------ quantiser

template <int kIn, int kKind, int kFmt>
tcg_status launch_quant_inst(const CUtensorMap& map, const QuantParams& p, int grid, int dev,
                             cudaStream_t stream, bool pdl) {
  auto* fn = &quant_fp8_kernel<kIn, kKind, kFmt>;
  if (tcg_status s = ensure_smem(fn, kQSmemBytes, dev); s != TCG_OK) return s;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kQThreads, 1, 1);
  cfg.dynamicSmemBytes = kQSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, fn, map, p) != cudaSuccess) return TCG_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError() == cudaSuccess ? TCG_OK : TCG_ERR_CUDA;
}

template <int kIn, int kFmt>
tcg_status launch_quant(int64_t rows, int64_t cols, const void* X, int64_t ldx,
                        tcg_quant_mode mode, void* Q, int64_t ldq, float* scale,
                        cudaStream_t stream) {
  int dev, sms;
  if (tcg_status s = current_device(&dev, &sms); s != TCG_OK) return s;
  const int64_t esize = kIn == 0 ? 4 : 2;
  CUtensorMap map;
  if (tcg_status s = tensor_map(&map,
                                kIn == 0 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                         : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                X, (uint64_t)cols, (uint64_t)rows, (uint64_t)(ldx * esize),
                                kQBoxCols, kQBoxRows, CU_TENSOR_MAP_SWIZZLE_NONE);
      s != TCG_OK)
    return s;
  QuantParams p{};
  p.Q = static_cast<uint8_t*>(Q);
  p.scale = scale;
  p.ldq = ldq;
  p.rows = (int32_t)rows;
  p.cols = (int32_t)cols;
  p.KB = (int32_t)((cols + 127) / 128);
  const int64_t row_units =
      mode == TCG_QUANT_BLOCK128 ? (rows + 127) / 128 : (rows + kQBoxRows - 1) / kQBoxRows;
  const int64_t units = row_units * p.KB;
  if (units > INT32_MAX) return TCG_ERR_UNSUPPORTED;
  p.units = (int32_t)units;
  const int grid = (int)(units < sms ? units : sms);
  if (mode == TCG_QUANT_BLOCK128)
    return launch_quant_inst<kIn, kQuantBlock, kFmt>(map, p, grid, dev, stream, true);
  if (mode == TCG_QUANT_ROW128)
    return launch_quant_inst<kIn, kQuantRow, kFmt>(map, p, grid, dev, stream, true);
  // per tensor: clear the running maximum, fold the per-CTA maxima, encode.
  // (Loading X with an evict-last policy in the first pass did not keep it in
  // L2 for the second on GB300; both passes read it from HBM.)
  if (cudaMemsetAsync(scale, 0, sizeof(float), stream) != cudaSuccess) return TCG_ERR_CUDA;
  if (tcg_status s = launch_quant_inst<kIn, kQuantAmax, kFmt>(map, p, grid, dev, stream, false);
      s != TCG_OK)
    return s;
  return launch_quant_inst<kIn, kQuantEncode, kFmt>(map, p, grid, dev, stream, true);
}

}  // namespace
}  // namespace tcg

using namespace tcg;

extern "C" {

tcg_status gemm_bf16(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                     int64_t ldb, const void* C, int64_t ldc, void* D, int64_t ldd,
                     tcg_out_dtype out_dtype, float alpha, float beta, tcg_stream stream) {
  const Common a{M, N, K, A, B, C, lda, ldb, ldc, ldd, D, (int)out_dtype, alpha, beta};
  if (tcg_status s = validate(a, 2); s != TCG_OK) return s;
  if (M == 0 || N == 0) return TCG_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return launch_k0(a, st);
  return launch_tn<0>(a, nullptr, nullptr, st);
}

tcg_status gemm_fp8(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                    tcg_fp8_format a_format, const void* B, int64_t ldb, tcg_fp8_format b_format,
                    const float* a_scale, const float* b_scale, tcg_scale_mode mode,
                    const void* C, int64_t ldc, void* D, int64_t ldd, tcg_out_dtype out_dtype,
                    float alpha, float beta, tcg_stream stream) {
  Common a{M, N, K, A, B, C, lda, ldb, ldc, ldd, D, (int)out_dtype, alpha, beta};
  if (mode != TCG_SCALE_TENSOR && mode != TCG_SCALE_BLOCK128) return TCG_ERR_UNSUPPORTED;
  if ((a_format != TCG_FP8_E4M3 && a_format != TCG_FP8_E5M2) ||
      (b_format != TCG_FP8_E4M3 && b_format != TCG_FP8_E5M2))
    return TCG_ERR_UNSUPPORTED;
  a.a_fp8 = (int)a_format;
  a.b_fp8 = (int)b_format;
  if (tcg_status s = validate(a, 1); s != TCG_OK) return s;
  if (M == 0 || N == 0) return TCG_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return launch_k0(a, st);
  if (!a_scale || !b_scale) return TCG_ERR_INVALID_ARG;
  if (mode == TCG_SCALE_TENSOR) return launch_tn<1>(a, a_scale, b_scale, st);
  // Block scales: M <= 128 on the swap-AB skinny kernel; larger M on pair
  // tiles when their work units (256 x 256 tiles, or halves of them when few)
  // keep at least half the SMs busy, else on the skinny kernel with A in
  // 128-row chunks (more, smaller tiles).
  const int fk = forced_kernel();
  if (fk != 3 && M > 128) {
    int dev, sms;
    if (tcg_status s = current_device(&dev, &sms); s != TCG_OK) return s;
    const int64_t tiles = ((M + 255) / 256) * ((N + 255) / 256);
    const int64_t clusters = sms / 2;
    const int64_t units = tiles >= clusters ? tiles : (tiles * 2 <= clusters ? tiles * 2 : tiles);
    if (fk == 2 || units * 2 >= sms / 2)
      return launch_block_pair(a, a_scale, b_scale, st, dev, sms);
  } else if (fk == 2) {
    int dev, sms;
    if (tcg_status s = current_device(&dev, &sms); s != TCG_OK) return s;
    return launch_block_pair(a, a_scale, b_scale, st, dev, sms);
  }
  return launch_skinny<1>(a, a_scale, b_scale, false, st);
}

tcg_status gemm_fp8_e4m3(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                         const void* B, int64_t ldb, const float* a_scale, const float* b_scale,
                         tcg_scale_mode mode, const void* C, int64_t ldc, void* D, int64_t ldd,
                         tcg_out_dtype out_dtype, float alpha, float beta, tcg_stream stream) {
  return gemm_fp8(M, N, K, A, lda, TCG_FP8_E4M3, B, ldb, TCG_FP8_E4M3, a_scale, b_scale, mode, C,
                  ldc, D, ldd, out_dtype, alpha, beta, stream);
}

tcg_status gemm_mxfp8(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                      tcg_fp8_format a_format, const void* B, int64_t ldb,
                      tcg_fp8_format b_format, const uint8_t* a_sf, const uint8_t* b_sf,
                      const void* C, int64_t ldc, void* D, int64_t ldd, tcg_out_dtype out_dtype,
                      float alpha, float beta, tcg_stream stream) {
  Common a{M, N, K, A, B, C, lda, ldb, ldc, ldd, D, (int)out_dtype, alpha, beta};
  if ((a_format != TCG_FP8_E4M3 && a_format != TCG_FP8_E5M2) ||
      (b_format != TCG_FP8_E4M3 && b_format != TCG_FP8_E5M2))
    return TCG_ERR_UNSUPPORTED;
  a.a_fp8 = (int)a_format;
  a.b_fp8 = (int)b_format;
  if (tcg_status s = validate(a, 1); s != TCG_OK) return s;
  if (M == 0 || N == 0) return TCG_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return launch_k0(a, st);
  if (!a_sf || !b_sf) return TCG_ERR_INVALID_ARG;
  if (!aligned16(a_sf) || !aligned16(b_sf)) return TCG_ERR_ALIGNMENT;
  return launch_mx(a, a_sf, b_sf, st);
}

const char* tcg_status_string(tcg_status status) {
  switch (status) {
    case TCG_OK: return "ok";
    case TCG_ERR_INVALID_ARG: return "invalid argument";
    case TCG_ERR_ALIGNMENT: return "misaligned pointer or leading dimension";
    case TCG_ERR_UNSUPPORTED: return "unsupported argument";
    case TCG_ERR_CUDA: return "CUDA error";
    case TCG_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

tcg_status tcg_last_device_status(tcg_stream stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return TCG_ERR_CUDA;
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_tcg_status, sizeof v) != cudaSuccess) return TCG_ERR_CUDA;
  if (v == 0) return TCG_OK;
  if (cudaMemcpyToSymbol(g_tcg_status, &zero, sizeof zero) != cudaSuccess) return TCG_ERR_CUDA;
  return TCG_ERR_TIMEOUT;
}

uint64_t tcg_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

tcg_status tcg_debug_timeout_probe(tcg_stream stream) {
  wait_timeout_probe_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>();
  if (cudaGetLastError() != cudaSuccess) return TCG_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return TCG_OK;
}

tcg_status quantize_fp8(int64_t rows, int64_t cols, const void* X, int64_t ldx,
                        tcg_in_dtype x_dtype, tcg_fp8_format format, tcg_quant_mode mode,
                        void* Q, int64_t ldq, float* scale, tcg_stream stream) {
  if (x_dtype != TCG_IN_F32 && x_dtype != TCG_IN_BF16) return TCG_ERR_UNSUPPORTED;
  if (format != TCG_FP8_E4M3 && format != TCG_FP8_E5M2) return TCG_ERR_UNSUPPORTED;
  if (mode != TCG_QUANT_TENSOR && mode != TCG_QUANT_ROW128 && mode != TCG_QUANT_BLOCK128)
    return TCG_ERR_UNSUPPORTED;
  if (rows < 0 || cols < 0) return TCG_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (rows == 0 || cols == 0) {
    if (mode != TCG_QUANT_TENSOR) return TCG_OK;  // no blocks, no scales
    if (!scale) return TCG_ERR_INVALID_ARG;
    if ((uintptr_t)scale % 4 != 0) return TCG_ERR_ALIGNMENT;
    quant_scale_one_kernel<<<1, 1, 0, st>>>(scale);  // the maximum of nothing is 0: scale 1
    if (cudaGetLastError() != cudaSuccess) return TCG_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return TCG_OK;
  }
  if (!X || !Q || !scale || ldx < cols || ldq < cols) return TCG_ERR_INVALID_ARG;
  const int64_t esize = x_dtype == TCG_IN_F32 ? 4 : 2;
  if (!aligned16(X) || (ldx * esize) % 16 != 0 || !aligned16(Q) || ldq % 16 != 0 ||
      (uintptr_t)scale % 4 != 0)
    return TCG_ERR_ALIGNMENT;
  if (rows > INT32_MAX || cols > INT32_MAX) return TCG_ERR_UNSUPPORTED;
  if (format == TCG_FP8_E4M3)
    return x_dtype == TCG_IN_F32 ? launch_quant<0, 0>(rows, cols, X, ldx, mode, Q, ldq, scale, st)
                                 : launch_quant<1, 0>(rows, cols, X, ldx, mode, Q, ldq, scale, st);
  return x_dtype == TCG_IN_F32 ? launch_quant<0, 1>(rows, cols, X, ldx, mode, Q, ldq, scale, st)
                               : launch_quant<1, 1>(rows, cols, X, ldx, mode, Q, ldq, scale, st);
}

tcg_status quantize_e4m3(int64_t rows, int64_t cols, const void* X, int64_t ldx,
                         tcg_in_dtype x_dtype, tcg_quant_mode mode, void* Q, int64_t ldq,
                         float* scale, tcg_stream stream) {
  return quantize_fp8(rows, cols, X, ldx, x_dtype, TCG_FP8_E4M3, mode, Q, ldq, scale, stream);
}

}  // extern "C"

// ------------------------------------------------------------------------
// Allocation-free stream-K variant of the block-scaled skinny FP8 path.
//
// The regular entry points never need scratch: a tile's K range is split
// only over the CTAs of one cluster, else each CTA takes whole tiles, which
// leaves SMs idle when the tiles do not divide evenly over them.  The
// stream-K form of the skinny kernel balances that by finishing tiles split
// between any CTAs through global scratch.  Allocating it would mean calling
// cudaMalloc, which some callers cannot allow: runtimes whose allocator owns
// all of device memory, and latency-critical loops that cannot absorb the
// device-wide synchronisation of cudaMalloc/cudaFree.  So this entry point
// keeps the scratch in a fixed array that is part of the loaded module.
namespace tcg {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB per device

// Scratch for the allocation-free entry point: tile counters first (zeroed by
// every call), then the FP32 partial-sum slots.  Every device that loads this
// library holds it until the process exits.  In host code this name is only a
// stand-in for the symbol; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

void* g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
tcg_status noalloc_scratch(int dev, void** out) {
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return TCG_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return TCG_OK;
}

// Encodes a tensor map on the stack (the cached path would insert into a
// host-side table, which allocates).
tcg_status encode_map_uncached(CUtensorMap* out, const void* ptr, uint64_t inner, uint64_t rows,
                               uint64_t ld_bytes, uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return TCG_ERR_CUDA;
  std::memset(out, 0, sizeof *out);
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {ld_bytes};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? TCG_OK
             : TCG_ERR_CUDA;
}

// The cluster-join forms of the skinny kernel without the host-side table
// (a per-device flag raises the shared-memory limit).
template <int kMp, int kJoin>
tcg_status launch_skinny_join_noalloc(const CUtensorMap& ma, const CUtensorMap& mb,
                                      const SkinnyParams& p, cudaStream_t stream, int dev) {
  using Cfg = SkinnyCfg<kMp>;
  auto* fn = &gemm_fp8_block_skinny_kernel<kMp, kJoin, false>;
  {
    static bool raised[kMaxDevices] = {};
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!raised[dev]) {
      if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)Cfg::kSmemBytes) != cudaSuccess)
        return TCG_ERR_CUDA;
      raised[dev] = true;
    }
  }
  if (launch_gemm_kernel(fn, p.grid, Cfg::kThreads, Cfg::kSmemBytes, stream, kJoin, ma, mb, p) !=
      cudaSuccess)
    return TCG_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError() == cudaSuccess ? TCG_OK : TCG_ERR_CUDA;
}

template <int kMp>
tcg_status launch_skinny_noalloc(const Common& a, const float* sa, const float* sb,
                                 cudaStream_t stream, int dev, int sms) {
  using Cfg = SkinnyCfg<kMp>;
  SkinnyParams p{};
  p.M = (int32_t)a.M;
  p.N = (int32_t)a.N;
  p.K = (int32_t)a.K;
  p.n_tiles = (int32_t)((a.N + 127) / 128);
  p.m_tiles = 1;  // M <= 128 on this path
  p.num_kb = (int32_t)((a.K + 127) / 128);
  const int64_t T = (int64_t)p.n_tiles * p.num_kb;
  if (T > INT32_MAX) return TCG_ERR_UNSUPPORTED;
  p.total_steps = (int32_t)T;
  // With fewer N tiles than SMs, each tile's K range is cut into
  // floor(SMs / tiles) equal pieces (at most 3), one per CTA, so a tile has
  // few partial sums to add; otherwise the steps are spread over all SMs and
  // every CTA gets at least ceil(KB/3) of them.  Either way at most kSkMaxSeg
  // (4) CTAs share a tile.
  int64_t split = 0;
  {
    int64_t g;
    if (p.n_tiles < sms) {
      split = sms / p.n_tiles;
      if (split > 3) split = 3;
      if (split > p.num_kb) split = p.num_kb;
      g = p.n_tiles * split;
    } else {
      const int64_t min_steps = (p.num_kb + 2) / 3;
      g = T / min_steps;
      if (g > sms) g = sms;
    }
    p.grid = (int32_t)(g < 1 ? 1 : g);
  }
  if (split == 3 && !skinny_trio_fits<kMp, 1, false>(false, p.n_tiles, dev)) {
    split = 2;
    p.grid = (int32_t)(p.n_tiles * 2);
  }
  if (split == 2 || split == 3) {  // cluster join: no scratch at all
    CUtensorMap ma, mb;
    if (tcg_status s = encode_map_uncached(&ma, a.A, a.K, a.M, a.lda, kMp); s != TCG_OK) return s;
    if (tcg_status s = encode_map_uncached(&mb, a.B, a.K, a.N, a.ldb, 128); s != TCG_OK) return s;
    p.a_scale = sa;
    p.b_scale = sb;
    p.C = a.beta != 0.0f ? a.C : nullptr;
    p.ldc = a.ldc;
    p.D = a.D;
    p.ldd = a.ldd;
    p.alpha = a.alpha;
    p.beta = a.beta;
    p.out_f32 = a.out == TCG_OUT_F32;
    p.has_c = a.beta != 0.0f;
    return split == 2 ? launch_skinny_join_noalloc<kMp, 2>(ma, mb, p, stream, dev)
                      : launch_skinny_join_noalloc<kMp, 3>(ma, mb, p, stream, dev);
  }
  const int64_t min_range = T / p.grid;
  p.max_seg = (int32_t)((p.num_kb + min_range - 1) / min_range + 1);
  if (p.max_seg > p.grid) p.max_seg = p.grid;
  const size_t counter_bytes = ((size_t)p.n_tiles * sizeof(unsigned int) + 255) & ~size_t(255);
  const size_t partial_bytes = (size_t)p.grid * 2 * kMp * 128 * sizeof(float);
  if (counter_bytes + partial_bytes > kNoAllocScratchBytes) return TCG_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (tcg_status s = noalloc_scratch(dev, &scratch); s != TCG_OK) return s;
  p.counters = static_cast<unsigned int*>(scratch);
  p.ws = reinterpret_cast<float*>(static_cast<char*>(scratch) + counter_bytes);
  // The array keeps whatever the previous call left; the counters must
  // start at zero.
  if (cudaMemsetAsync(scratch, 0, counter_bytes, stream) != cudaSuccess) return TCG_ERR_CUDA;
  CUtensorMap ma, mb;
  if (tcg_status s = encode_map_uncached(&ma, a.A, a.K, a.M, a.lda, kMp); s != TCG_OK) return s;
  if (tcg_status s = encode_map_uncached(&mb, a.B, a.K, a.N, a.ldb, 128); s != TCG_OK) return s;
  p.a_scale = sa;
  p.b_scale = sb;
  p.C = a.beta != 0.0f ? a.C : nullptr;
  p.ldc = a.ldc;
  p.D = a.D;
  p.ldd = a.ldd;
  p.alpha = a.alpha;
  p.beta = a.beta;
  p.out_f32 = a.out == TCG_OUT_F32;
  p.has_c = a.beta != 0.0f;
  auto* fn = &gemm_fp8_block_skinny_kernel<kMp, 0, false>;  // M <= 128: one chunk
  {  // raise the shared-memory limit once per device (no host-side table)
    static bool raised[kMaxDevices] = {};
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!raised[dev]) {
      if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)Cfg::kSmemBytes) != cudaSuccess)
        return TCG_ERR_CUDA;
      raised[dev] = true;
    }
  }
  fn<<<p.grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(ma, mb, p);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError() == cudaSuccess ? TCG_OK : TCG_ERR_CUDA;
}

// Block-scaled FP8 for M > 128 on the pair-tile kernel, which needs no
// scratch: stack-encoded tensor maps, a per-device flag for the shared-memory
// limit instead of the host-side table.
template <int kOut, bool kHasC>
tcg_status launch_block_pair_noalloc_inst(const Common& a, const float* sa, const float* sb,
                                          cudaStream_t stream, int dev, int sms) {
  CUtensorMap ma, mb;
  if (tcg_status s = encode_map_uncached(&ma, a.A, a.K, a.M, a.lda, 128); s != TCG_OK) return s;
  if (tcg_status s = encode_map_uncached(&mb, a.B, a.K, a.N, a.ldb, kBBoxRows); s != TCG_OK)
    return s;
  Gemm2Params p;
  int grid;
  if (tcg_status s = pair_schedule(a, 1, sms, &p, &grid); s != TCG_OK) return s;
  p.a_scale = sa;
  p.b_scale = sb;
  auto* fn = &gemm_fp8_block_pair_kernel<kOut, kHasC>;
  {
    static bool raised[kMaxDevices] = {};
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!raised[dev]) {
      if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kP2SmemBytes) != cudaSuccess)
        return TCG_ERR_CUDA;
      raised[dev] = true;
    }
  }
  if (launch_gemm_kernel(fn, grid, kPbThreads, kP2SmemBytes, stream, 2, ma, mb, p) != cudaSuccess)
    return TCG_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError() == cudaSuccess ? TCG_OK : TCG_ERR_CUDA;
}

tcg_status launch_block_pair_noalloc(const Common& a, const float* sa, const float* sb,
                                     cudaStream_t stream, int dev, int sms) {
  const bool has_c = a.beta != 0.0f;
  if (a.out == TCG_OUT_BF16)
    return has_c ? launch_block_pair_noalloc_inst<0, true>(a, sa, sb, stream, dev, sms)
                 : launch_block_pair_noalloc_inst<0, false>(a, sa, sb, stream, dev, sms);
  return has_c ? launch_block_pair_noalloc_inst<1, true>(a, sa, sb, stream, dev, sms)
               : launch_block_pair_noalloc_inst<1, false>(a, sa, sb, stream, dev, sms);
}

}  // namespace
}  // namespace tcg

extern "C" tcg_status gemm_fp8_e4m3_block_noalloc(int64_t M, int64_t N, int64_t K, const void* A,
                                                  int64_t lda, const void* B, int64_t ldb,
                                                  const float* a_scale, const float* b_scale,
                                                  const void* C, int64_t ldc, void* D,
                                                  int64_t ldd, tcg_out_dtype out_dtype,
                                                  float alpha, float beta, tcg_stream stream) {
  const Common a{M, N, K, A, B, C, lda, ldb, ldc, ldd, D, (int)out_dtype, alpha, beta};
  if (tcg_status s = validate(a, 1); s != TCG_OK) return s;
  if (M == 0 || N == 0) return TCG_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return launch_k0(a, st);
  if (!a_scale || !b_scale) return TCG_ERR_INVALID_ARG;
  int dev, sms;
  if (tcg_status s = current_device(&dev, &sms); s != TCG_OK) return s;
  if (M > 128) return launch_block_pair_noalloc(a, a_scale, b_scale, st, dev, sms);
  if (M <= 16) return launch_skinny_noalloc<16>(a, a_scale, b_scale, st, dev, sms);
  if (M <= 32) return launch_skinny_noalloc<32>(a, a_scale, b_scale, st, dev, sms);
  if (M <= 64) return launch_skinny_noalloc<64>(a, a_scale, b_scale, st, dev, sms);
  return launch_skinny_noalloc<128>(a, a_scale, b_scale, st, dev, sms);
}
