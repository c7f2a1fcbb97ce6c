// C ABI of the fp8bs library: host-side argument checks, TMA descriptor
// encoding and kernel launches.  Declarations and the full contract are in
// include/fp8bs.h.  Nothing here allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/fp8bs.h"
#include "gemm_kernel.cuh"
#include "gemm_mx_kernel.cuh"
#include "gemm_pair_kernel.cuh"
#include "quant_kernels.cuh"

// Scratch of fp8bs_gemm_static_ws, for callers that cannot allocate device
// memory: the FP32 partials of the split last wave live here instead of in a
// caller workspace.  Every GPU that loads the library holds these 20 MiB until
// the process exits; every call shares them (see include/fp8bs.h).
static __device__ __align__(256) unsigned char fp8bs_static_ws[20u << 20];

namespace fp8bs {
namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kStaticWsBytes = sizeof(fp8bs_static_ws);

// Device address of fp8bs_static_ws on the current device, looked up once per
// device (with that device current).  In host code the array's name is only a
// host-side stand-in, never a device address.
void* g_static_ws_addr[kMaxDevices] = {};

fp8bs_status static_workspace(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP8BS_ERR_CUDA;
  static std::mutex m;
  std::lock_guard<std::mutex> lock(m);
  if (g_static_ws_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, fp8bs_static_ws) != cudaSuccess || ptr == nullptr)
      return FP8BS_ERR_CUDA;
    g_static_ws_addr[dev] = ptr;
  }
  *out = g_static_ws_addr[dev];
  return FP8BS_OK;
}

struct DeviceInfo {
  bool init = false;
  int num_sms = 0;
  int pair_clusters = 0;   // co-resident 2-CTA clusters of the pair GEMM
  int l2_bytes = 0;
};

std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

fp8bs_status device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP8BS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo& d = g_dev[dev];
  if (!d.init) {
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
      return FP8BS_ERR_CUDA;
    d.init = true;
  }
  *out = d;
  return FP8BS_OK;
}

// How many 2-CTA clusters of `kernel` fit on the device at once (queried once
// per device; all pair-kernel variants have the same shape and resources).
template <typename K>
int pair_clusters(K kernel) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo& d = g_dev[dev];
  if (d.pair_clusters == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 512, 1, 1);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = pair_smem_bytes<256>();
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) return 0;
    d.pair_clusters = n;
  }
  return d.pair_clusters;
}

// How many 2-CTA clusters of the MX pair GEMM fit on the device at once
// (queried once per device).
template <typename K>
int mx_pair_clusters(K kernel) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  static int cached[kMaxDevices] = {};
  std::lock_guard<std::mutex> lock(g_mutex);
  if (cached[dev] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 512, 1, 1);
    cfg.blockDim = dim3(kMxThreads, 1, 1);
    cfg.dynamicSmemBytes = kMxPairSmemBytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

fp8bs_status encode_fn(PFN_cuTensorMapEncodeTiled_v12000* out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return FP8BS_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *out = g_encode;
  return FP8BS_OK;
}

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline size_t dtype_size(fp8bs_dtype t) { return t == FP8BS_F32 ? 4 : 2; }

inline bool valid_dtype(fp8bs_dtype t) { return t == FP8BS_F32 || t == FP8BS_BF16; }

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

fp8bs_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? FP8BS_OK : FP8BS_ERR_CUDA;
}

// 2D u8 map over rows x inner bytes, box 128 x box_rows, 128-byte swizzle.
fp8bs_status make_map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                         uint64_t row_stride, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  fp8bs_status st = encode_fn(&enc);
  if (st != FP8BS_OK) return st;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_stride};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FP8BS_OK : FP8BS_ERR_CUDA;
}

// 3D u8 map over [E][rows][inner], box 128 x box_rows x 1.
fp8bs_status make_map_3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                         uint64_t E, uint64_t row_stride, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  fp8bs_status st = encode_fn(&enc);
  if (st != FP8BS_OK) return st;
  cuuint64_t dims[3] = {inner, rows, E};
  cuuint64_t strides[2] = {row_stride, row_stride * rows};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kBK), box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FP8BS_OK : FP8BS_ERR_CUDA;
}

// Output map of the pair GEMM's TMA-store epilogue: [rows][ldc] of fp32 or
// bf16, box = 64 bytes x 32 rows with the 64-byte swizzle.
fp8bs_status make_map_out(CUtensorMap* m, void* base, fp8bs_dtype ct, uint64_t cols,
                          uint64_t rows, uint64_t ld_elems) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  fp8bs_status st = encode_fn(&enc);
  if (st != FP8BS_OK) return st;
  const uint64_t esz = dtype_size(ct);
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld_elems * esz};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(64 / esz), 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, ct == FP8BS_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                   2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FP8BS_OK : FP8BS_ERR_CUDA;
}

// Map over the MX exponent words [KB][ld_words] (uint32, `rows` used per K
// block), box = box_rows words x 1 K block, no swizzle.
fp8bs_status make_map_sf(CUtensorMap* m, const void* base, uint64_t rows, uint64_t KB,
                         uint64_t ld_words, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  fp8bs_status st = encode_fn(&enc);
  if (st != FP8BS_OK) return st;
  cuuint64_t dims[2] = {rows, KB};
  cuuint64_t strides[1] = {ld_words * 4};
  cuuint32_t box[2] = {box_rows, 1};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FP8BS_OK : FP8BS_ERR_CUDA;
}

// Shared checks of the dense and grouped GEMM (all on the host, before any launch).
fp8bs_status check_gemm(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda,
                        const float* sa, int64_t ldsa, const uint8_t* B, int64_t ldb,
                        const float* sb, fp8bs_bscale sb_mode, int64_t ldsb, const void* C,
                        fp8bs_dtype ct, int64_t ldc) {
  if (M < 0 || N < 0 || K < 0) return FP8BS_ERR_INVALID_ARG;
  if (!valid_dtype(ct)) return FP8BS_ERR_INVALID_ARG;
  if (sb_mode != FP8BS_SB_BLOCK_NK && sb_mode != FP8BS_SB_BLOCK_KN && sb_mode != FP8BS_SB_PERCOL)
    return FP8BS_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return FP8BS_OK;
  if (K % kBK != 0) return FP8BS_ERR_UNSUPPORTED;
  if (sb_mode == FP8BS_SB_PERCOL ? (N % 16 != 0) : (N % 128 != 0)) return FP8BS_ERR_UNSUPPORTED;
  if (M > INT_MAX - kBM || N > INT_MAX - kBN || K / kBK > INT_MAX) return FP8BS_ERR_UNSUPPORTED;
  if (((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN) > INT_MAX) return FP8BS_ERR_UNSUPPORTED;
  if (C == nullptr || ldc < N) return FP8BS_ERR_INVALID_ARG;
  if (!aligned(C, 16) || (ldc * static_cast<int64_t>(dtype_size(ct))) % 16 != 0)
    return FP8BS_ERR_MISALIGNED;
  if (K == 0) return FP8BS_OK;
  if (A == nullptr || B == nullptr || sa == nullptr || sb == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (lda < K || ldb < K || ldsa < M) return FP8BS_ERR_INVALID_ARG;
  if (sb_mode == FP8BS_SB_BLOCK_NK && ldsb < K / 128) return FP8BS_ERR_INVALID_ARG;
  if (sb_mode == FP8BS_SB_BLOCK_KN && ldsb < N / 128) return FP8BS_ERR_INVALID_ARG;
  if (sb_mode == FP8BS_SB_PERCOL && ldsb < N) return FP8BS_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(B, 16) || lda % 16 != 0 || ldb % 16 != 0)
    return FP8BS_ERR_MISALIGNED;
  if (!aligned(sa, 4) || !aligned(sb, 4)) return FP8BS_ERR_MISALIGNED;
  if (sb_mode == FP8BS_SB_PERCOL && (!aligned(sb, 16) || ldsb % 4 != 0))
    return FP8BS_ERR_MISALIGNED;
  return FP8BS_OK;
}

// Launch of the CTA-pair GEMM: a persistent grid of as many 2-CTA clusters
// as can be resident at once (at most one per tile).
// Co-resident 2-CTA clusters of the pair GEMM on the current device (all its
// variants have the same shape and resources).
fp8bs_status pair_cluster_count(int* clusters) {
  auto kernel = fp8bs_gemm_pair_kernel<256, kSbBlock, true>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(pair_smem_bytes<256>())) != cudaSuccess)
    return FP8BS_ERR_CUDA;
  *clusters = pair_clusters(kernel);
  return *clusters > 0 ? FP8BS_OK : FP8BS_ERR_CUDA;
}

// Split of the last, partial wave: its `tail` tiles are cut into `splits`
// K-ranges so that every cluster has work; the FP32 partials need
// tail * splits pair tiles of workspace.  ws_avail limits the split count
// (SIZE_MAX: no limit).  No split when it would give fewer than 2 ranges.
struct SplitPlan {
  int full_tiles, splits, units, tail;
  size_t ws_bytes;
};
constexpr int kMaxSplits = 32;
// m tiles per group of the pair GEMM's tile walk (see pair_tile_mn), measured on
// the layer's GEMMs: one group of all m tiles when the whole of A fits in a
// quarter of L2 (its panels then stay there from wave to wave and every B
// panel is read once: Fprop, A = 29 MB, 0.385 -> 0.380 ms against groups of 8;
// Wgrad, A = 29 MB, 0.6205 -> 0.610 ms), else groups of 8 (Dgrad, A = 75 MB:
// 0.528 -> 0.438 ms against one group; 4, 6, 12 and 16 slower).
constexpr int kPairGroupM = 8;

// Tile width of the pair GEMM.  256 for every mode: measured on the layer's
// GEMMs, the 128-wide tile (four TMEM buffers, 45 % more operand bytes per
// FLOP) was slower everywhere (Fprop 0.42 -> 0.69 ms, Dgrad 0.53 -> 1.05 ms,
// Wgrad 0.62 -> 0.89 ms), so the kernel's BN = 128 form is not instantiated.
int pair_tile_n(fp8bs_bscale /*mode*/) { return 256; }

SplitPlan plan_split(int tiles, int KB, int clusters, size_t ws_avail, int bn) {
  const size_t kPartialTileBytes = static_cast<size_t>(kPairTileM) * bn * sizeof(float);
  SplitPlan sp{tiles, 1, tiles, 0, 0};
  if (tiles <= 0 || clusters <= 0) return sp;
  const int tail = tiles % clusters;
  if (tail == 0) return sp;
  int n = clusters / tail;
  if (n > KB) n = KB;
  if (n > kMaxSplits) n = kMaxSplits;
  const size_t per_split = static_cast<size_t>(tail) * kPartialTileBytes;
  if (ws_avail != SIZE_MAX && static_cast<size_t>(n) > ws_avail / per_split)
    n = static_cast<int>(ws_avail / per_split);
  if (n < 2) return sp;
  sp.full_tiles = tiles - tail;
  sp.splits = n;
  sp.units = sp.full_tiles + tail * n;
  sp.tail = tail;
  sp.ws_bytes = per_split * n;
  return sp;
}

template <int BN>
fp8bs_status launch_gemm_pair(GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                              const CUtensorMap& tc, const CUtensorMap& tws, const float* ws,
                              int tail, int clusters, int sb_kind, fp8bs_dtype ct, bool acc,
                              cudaStream_t stream) {
  constexpr size_t smem = pair_smem_bytes<BN>();
  auto run = [&](auto kernel) -> fp8bs_status {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return FP8BS_ERR_CUDA;
    const int grid_clusters = p.units < clusters ? p.units : clusters;
    kernel<<<2 * grid_clusters, kGemmThreads, smem, stream>>>(p, ta, tb, tc, tws);
    fp8bs_status st = launch_status();
    if (st != FP8BS_OK || tail == 0) return st;
    const unsigned blocks = static_cast<unsigned>(tail) * (kPairTileM * (BN / 4) / 256);
    if (ct == FP8BS_BF16)
      split_fixup_kernel<BN, true><<<blocks, 256, 0, stream>>>(ws, p, tail);
    else if (acc)
      split_fixup_kernel<BN, false, true><<<blocks, 256, 0, stream>>>(ws, p, tail);
    else
      split_fixup_kernel<BN, false><<<blocks, 256, 0, stream>>>(ws, p, tail);
    return launch_status();
  };
  const bool bf16 = ct == FP8BS_BF16;
  if (acc)   // FP32 output only
    return sb_kind == kSbBlock ? run(fp8bs_gemm_pair_kernel<BN, kSbBlock, false, true>)
                               : run(fp8bs_gemm_pair_kernel<BN, kSbPerCol, false, true>);
  if (sb_kind == kSbBlock)
    return bf16 ? run(fp8bs_gemm_pair_kernel<BN, kSbBlock, true>)
                : run(fp8bs_gemm_pair_kernel<BN, kSbBlock, false>);
  return bf16 ? run(fp8bs_gemm_pair_kernel<BN, kSbPerCol, true>)
              : run(fp8bs_gemm_pair_kernel<BN, kSbPerCol, false>);
}

// Launch of the single-CTA grouped GEMM: one persistent CTA per SM (at most one per tile).
fp8bs_status launch_grouped(GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                            const CUtensorMap& tc, int sb_kind, fp8bs_dtype ct,
                            cudaStream_t stream) {
  DeviceInfo di;
  fp8bs_status st = device_info(&di);
  if (st != FP8BS_OK) return st;
  const int tiles = p.num_m_tiles * p.num_n_tiles;
  const int grid = tiles < di.num_sms ? tiles : di.num_sms;
  auto run = [&](auto kernel) -> fp8bs_status {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kGemmSmemBytes)) != cudaSuccess)
      return FP8BS_ERR_CUDA;
    kernel<<<grid, kGemmThreads, kGemmSmemBytes, stream>>>(p, ta, tb, tc);
    return launch_status();
  };
  const bool bf16 = ct == FP8BS_BF16;
  if (sb_kind == kSbBlock)
    return bf16 ? run(fp8bs_gemm_kernel<kSbBlock, true>)
                : run(fp8bs_gemm_kernel<kSbBlock, false>);
  return bf16 ? run(fp8bs_gemm_kernel<kSbPerCol, true>)
              : run(fp8bs_gemm_kernel<kSbPerCol, false>);
}

void fill_scale_strides(GemmParams& p, fp8bs_bscale mode, int64_t ldsb) {
  p.ldsb = ldsb;
  if (mode == FP8BS_SB_BLOCK_NK) {
    p.sb_k_stride = 1;
    p.sb_n_stride = ldsb;
  } else if (mode == FP8BS_SB_BLOCK_KN) {
    p.sb_k_stride = ldsb;
    p.sb_n_stride = 1;
  } else {
    p.sb_k_stride = 0;
    p.sb_n_stride = 0;
  }
}

// Zero-fill of C for K == 0 (the empty contraction).
__global__ void zero_fill_kernel(unsigned char* C, int64_t row_bytes, int64_t ld_bytes,
                                 int64_t rows) {
  const int64_t r = blockIdx.x;
  if (r >= rows) return;
  uint4* dst = reinterpret_cast<uint4*>(C + r * ld_bytes);
  for (int64_t i = threadIdx.x; i < row_bytes / 16; i += blockDim.x) dst[i] = make_uint4(0, 0, 0, 0);
}

fp8bs_status zero_fill(void* C, fp8bs_dtype ct, int64_t rows, int64_t N, int64_t ldc,
                       cudaStream_t stream) {
  // N is a multiple of 16 here, so a row is a whole number of 16-byte words.
  int64_t done = 0;
  while (done < rows) {
    const int64_t chunk = rows - done < 65535 * 1024 ? rows - done : 65535 * 1024;
    const int64_t esz = static_cast<int64_t>(dtype_size(ct));
    zero_fill_kernel<<<static_cast<unsigned>(chunk), 256, 0, stream>>>(
        static_cast<unsigned char*>(C) + done * ldc * esz, N * esz, ldc * esz, chunk);
    fp8bs_status st = launch_status();
    if (st != FP8BS_OK) return st;
    done += chunk;
  }
  return FP8BS_OK;
}

// Ask for the maximum shared-memory carveout once per kernel, so that several
// staging CTAs fit on an SM (the default carveout left room for only three).
template <typename K>
void prefer_max_shared(K kernel) {
  cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                       static_cast<int>(cudaSharedmemCarveoutMaxShared));
}

// Grid-stride launch of the 1x128 quantizer: at most 8 blocks of 256 threads per SM.
template <typename TIn, int kUnroll>
void launch_quant_1x128(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                        int64_t ldq, float* s, int64_t lds, const DeviceInfo& di,
                        cudaStream_t stream) {
  const int64_t tiles = M * (K / 128);
  const int64_t tiles_per_block = 8 /* warps */ * 8 /* tiles per warp step */ * kUnroll;
  int64_t blocks = (tiles + tiles_per_block - 1) / tiles_per_block;
  const int64_t max_blocks = static_cast<int64_t>(di.num_sms) * 8;
  if (blocks > max_blocks) blocks = max_blocks;
  quant_1x128_kernel<TIn, kUnroll><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      static_cast<const TIn*>(x), static_cast<uint32_t>(M), static_cast<uint32_t>(K / 128), ldx,
      q, ldq, s, lds);
}

// Dense GEMM on CTA pairs; with a workspace, the tail tiles are split along K.
fp8bs_status gemm_dense(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda,
                        const float* sa, int64_t ldsa, const uint8_t* B, int64_t ldb,
                        const float* sb, fp8bs_bscale sb_mode, int64_t ldsb, void* C,
                        fp8bs_dtype ct, int64_t ldc, float* ws, size_t ws_bytes, void* stream,
                        bool acc = false) {
  fp8bs_status st = check_gemm(M, N, K, A, lda, sa, ldsa, B, ldb, sb, sb_mode, ldsb, C, ct, ldc);
  if (st != FP8BS_OK || M == 0 || N == 0) return st;
  if (K == 0) return acc ? FP8BS_OK : zero_fill(C, ct, M, N, ldc, as_stream(stream));
  const int bn = pair_tile_n(sb_mode);
  CUtensorMap ta, tb, tc;
  if ((st = make_map_2d(&ta, A, K, M, lda, kBM)) != FP8BS_OK) return st;
  if ((st = make_map_2d(&tb, B, K, N, ldb, bn / 2)) != FP8BS_OK) return st;
  if ((st = make_map_out(&tc, C, ct, N, M, ldc)) != FP8BS_OK) return st;
  GemmParams p{};
  p.M = static_cast<int32_t>(M);
  p.N = static_cast<int32_t>(N);
  p.KB = static_cast<int32_t>(K / kBK);
  p.num_m_tiles = static_cast<int32_t>((M + kPairTileM - 1) / kPairTileM);
  p.num_n_tiles = static_cast<int32_t>((N + bn - 1) / bn);
  p.E = 1;
  p.sa = sa;
  p.ldsa = ldsa;
  p.sb = sb;
  fill_scale_strides(p, sb_mode, ldsb);
  p.sb_e_stride = 0;
  p.C = C;
  p.ldc = ldc;
  p.offsets = nullptr;
  int clusters = 0;
  if ((st = pair_cluster_count(&clusters)) != FP8BS_OK) return st;
  DeviceInfo di;
  if ((st = device_info(&di)) != FP8BS_OK) return st;
  p.group_m = (p.num_m_tiles < kPairGroupM || M * K <= di.l2_bytes / 4) ? p.num_m_tiles
                                                                       : kPairGroupM;
  {
    // operand panels a wave of clusters reads: its group's A panels and the
    // B panels of its n tiles, each 256 rows x K bytes
    const int64_t n_per_wave = (clusters + p.group_m - 1) / p.group_m;
    const int64_t wave_bytes = (p.group_m + n_per_wave) * static_cast<int64_t>(kPairTileM) * K;
    p.k_order = wave_bytes > di.l2_bytes / 2 ? kKOrderSerpentine : kKOrderForward;
  }
  const SplitPlan sp = plan_split(p.num_m_tiles * p.num_n_tiles, p.KB, clusters,
                                  ws != nullptr ? ws_bytes : 0, bn);
  p.full_tiles = sp.full_tiles;
  p.splits = sp.splits;
  p.units = sp.units;
  CUtensorMap tws = tc;   // unused without a split
  if (sp.tail > 0 &&
      (st = make_map_out(&tws, ws, FP8BS_F32, bn,
                         static_cast<uint64_t>(sp.tail) * sp.splits * kPairTileM, bn)) != FP8BS_OK)
    return st;
  const int sb_kind = sb_mode == FP8BS_SB_PERCOL ? kSbPerCol : kSbBlock;
  return launch_gemm_pair<256>(p, ta, tb, tc, tws, ws, sp.tail, clusters, sb_kind, ct, acc,
                               as_stream(stream));
}

}  // namespace
}  // namespace fp8bs

using namespace fp8bs;

extern "C" {

fp8bs_status fp8bs_quant_act_1x128(const void* x, fp8bs_dtype xt, int64_t M, int64_t K,
                                   int64_t ldx, uint8_t* q, int64_t ldq, float* s, int64_t lds,
                                   void* stream) {
  if (M < 0 || K < 0 || !valid_dtype(xt)) return FP8BS_ERR_INVALID_ARG;
  if (K % 128 != 0) return FP8BS_ERR_UNSUPPORTED;
  if (M == 0 || K == 0) return FP8BS_OK;
  if (M * (K / 128) > INT_MAX) return FP8BS_ERR_UNSUPPORTED;
  if (x == nullptr || q == nullptr || s == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (ldx < K || ldq < K || lds < M) return FP8BS_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(q, 16) || (ldx * static_cast<int64_t>(dtype_size(xt))) % 16 ||
      ldq % 16 || !aligned(s, 4))
    return FP8BS_ERR_MISALIGNED;
  DeviceInfo di;
  fp8bs_status st = device_info(&di);
  if (st != FP8BS_OK) return st;
  if (xt == FP8BS_BF16)
    launch_quant_1x128<__nv_bfloat16, 2>(x, M, K, ldx, q, ldq, s, lds, di, as_stream(stream));
  else
    launch_quant_1x128<float, 1>(x, M, K, ldx, q, ldq, s, lds, di, as_stream(stream));
  return launch_status();
}

fp8bs_status fp8bs_quant_act_128x1(const void* x, fp8bs_dtype xt, int64_t T, int64_t C,
                                   int64_t ldx, uint8_t* qT, int64_t ldq, float* s, int64_t lds,
                                   void* stream) {
  if (T < 0 || C < 0 || !valid_dtype(xt)) return FP8BS_ERR_INVALID_ARG;
  if (T % 128 != 0 || C % 16 != 0) return FP8BS_ERR_UNSUPPORTED;
  if (T == 0 || C == 0) return FP8BS_OK;
  if (T / 128 > 65535) return FP8BS_ERR_UNSUPPORTED;
  if (x == nullptr || qT == nullptr || s == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (ldx < C || ldq < T || lds < C) return FP8BS_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(qT, 16) || (ldx * static_cast<int64_t>(dtype_size(xt))) % 16 ||
      ldq % 16 || !aligned(s, 4))
    return FP8BS_ERR_MISALIGNED;
  const int64_t cb = xt == FP8BS_BF16 ? 128 : 64;
  dim3 grid(static_cast<unsigned>((C + cb - 1) / cb), static_cast<unsigned>(T / 128));
  auto run = [&](auto kernel, size_t smem, auto* xin) -> fp8bs_status {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return FP8BS_ERR_CUDA;
    prefer_max_shared(kernel);
    kernel<<<grid, 256, smem, as_stream(stream)>>>(xin, C, ldx, qT, ldq, s, lds);
    return launch_status();
  };
  if (xt == FP8BS_BF16)
    return run(quant_128x1_kernel<__nv_bfloat16>, quant_128x1_smem_bytes<__nv_bfloat16>(),
               static_cast<const __nv_bfloat16*>(x));
  return run(quant_128x1_kernel<float>, quant_128x1_smem_bytes<float>(),
             static_cast<const float*>(x));
}

fp8bs_status fp8bs_quant_act_dual(const void* x, fp8bs_dtype xt, int64_t T, int64_t C,
                                  int64_t ldx, uint8_t* q, int64_t ldq, float* s, int64_t lds,
                                  uint8_t* qT, int64_t ldqT, float* sT, int64_t ldsT,
                                  void* stream) {
  if (T < 0 || C < 0 || !valid_dtype(xt)) return FP8BS_ERR_INVALID_ARG;
  if (T % 128 != 0 || C % 128 != 0) return FP8BS_ERR_UNSUPPORTED;
  if (T == 0 || C == 0) return FP8BS_OK;
  if (T / 128 > 65535 || C / 128 > INT_MAX) return FP8BS_ERR_UNSUPPORTED;
  if (x == nullptr || q == nullptr || s == nullptr || qT == nullptr || sT == nullptr)
    return FP8BS_ERR_INVALID_ARG;
  if (ldx < C || ldq < C || lds < T || ldqT < T || ldsT < C) return FP8BS_ERR_INVALID_ARG;
  if (!aligned(x, 16) || (ldx * static_cast<int64_t>(dtype_size(xt))) % 16 || !aligned(q, 16) ||
      ldq % 16 || !aligned(qT, 16) || ldqT % 16 || !aligned(s, 4) || !aligned(sT, 4))
    return FP8BS_ERR_MISALIGNED;
  dim3 grid(static_cast<unsigned>(C / 128), static_cast<unsigned>(T / 128));
  // staged input tile + the transposed codes (128 x 128 bytes)
  const size_t smem = 128 * 128 * dtype_size(xt) + 128 * 128;
  if (xt == FP8BS_BF16) {
    if (cudaFuncSetAttribute(quant_dual_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return FP8BS_ERR_CUDA;
    prefer_max_shared(quant_dual_kernel<__nv_bfloat16>);
    quant_dual_kernel<__nv_bfloat16><<<grid, 256, smem, as_stream(stream)>>>(
        static_cast<const __nv_bfloat16*>(x), ldx, q, ldq, s, lds, qT, ldqT, sT, ldsT);
  } else {
    if (cudaFuncSetAttribute(quant_dual_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return FP8BS_ERR_CUDA;
    prefer_max_shared(quant_dual_kernel<float>);
    quant_dual_kernel<float><<<grid, 256, smem, as_stream(stream)>>>(
        static_cast<const float*>(x), ldx, q, ldq, s, lds, qT, ldqT, sT, ldsT);
  }
  return launch_status();
}

fp8bs_status fp8bs_quant_dispatch(const void* x, fp8bs_dtype xt, int64_t T, int64_t K,
                                  int64_t ldx, const int32_t* expert, int32_t E, uint8_t* q,
                                  int64_t ldq, float* s, int64_t lds, int64_t M_cap,
                                  int32_t* offsets, int32_t* counts, int32_t* token_row,
                                  int32_t* row_token, void* stream) {
  if (T < 0 || K < 0 || M_cap < 0 || !valid_dtype(xt)) return FP8BS_ERR_INVALID_ARG;
  if (E < 1 || E > kDispatchMaxExperts) return FP8BS_ERR_UNSUPPORTED;
  if (K <= 0 || K % 128 != 0 || M_cap % 128 != 0) return FP8BS_ERR_UNSUPPORTED;
  if (M_cap < T + 127 * static_cast<int64_t>(E)) return FP8BS_ERR_INVALID_ARG;   // worst-case padding
  if (T * (K / 128) > INT_MAX || M_cap > INT_MAX) return FP8BS_ERR_UNSUPPORTED;
  if ((T + kRankChunk - 1) / kRankChunk * E > kPlanMaxChunkCounts) return FP8BS_ERR_UNSUPPORTED;
  if (offsets == nullptr || counts == nullptr || (T > 0 && (expert == nullptr || token_row == nullptr)))
    return FP8BS_ERR_INVALID_ARG;
  if (x == nullptr || q == nullptr || s == nullptr || row_token == nullptr)
    return FP8BS_ERR_INVALID_ARG;
  if (ldx < K || ldq < K || lds < M_cap) return FP8BS_ERR_INVALID_ARG;
  if (!aligned(x, 16) || (ldx * static_cast<int64_t>(dtype_size(xt))) % 16 || !aligned(q, 16) ||
      ldq % 16 || !aligned(s, 4))
    return FP8BS_ERR_MISALIGNED;
  if (!aligned(offsets, 4) || !aligned(counts, 4)) return FP8BS_ERR_MISALIGNED;
  cudaStream_t st = as_stream(stream);
  DeviceInfo di;
  fp8bs_status rc = device_info(&di);
  if (rc != FP8BS_OK) return rc;
  // row_token's first chunks * E entries hold the chunk counts between the rank
  // and plan launches (M_cap >= T + 127 E >= chunks * E for E <= 256)
  const int64_t chunks = (T + kRankChunk - 1) / kRankChunk;
  if (chunks > 0)
    dispatch_rank_kernel<<<static_cast<unsigned>(chunks), kRankChunk, 0, st>>>(expert, T, E, token_row,
                                                                              row_token);
  if ((rc = launch_status()) != FP8BS_OK) return rc;
  const size_t plan_smem = static_cast<size_t>(chunks * E) * sizeof(int32_t);
  if (plan_smem > 48 * 1024 &&
      cudaFuncSetAttribute(dispatch_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kPlanMaxChunkCounts * sizeof(int32_t))) != cudaSuccess)
    return FP8BS_ERR_CUDA;
  dispatch_plan_kernel<<<1, 1024, plan_smem, st>>>(expert, T, E, static_cast<int>(chunks), row_token,
                                                   token_row, counts, offsets);
  if ((rc = launch_status()) != FP8BS_OK || T == 0) return rc;
  const int64_t tiles = T * (K / 128);
  int64_t blocks = (tiles + 63) / 64;
  if (blocks > static_cast<int64_t>(di.num_sms) * 8) blocks = static_cast<int64_t>(di.num_sms) * 8;
  if (xt == FP8BS_BF16)
    quant_dispatch_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(x), static_cast<uint32_t>(T),
        static_cast<uint32_t>(K / 128), ldx, token_row, E, counts, offsets, q, ldq, s, lds,
        row_token);
  else
    quant_dispatch_kernel<float><<<static_cast<unsigned>(blocks), 256, 0, st>>>(
        static_cast<const float*>(x), static_cast<uint32_t>(T), static_cast<uint32_t>(K / 128),
        ldx, token_row, E, counts, offsets, q, ldq, s, lds, row_token);
  return launch_status();
}

fp8bs_status fp8bs_quant_w_128x128(const void* w, fp8bs_dtype wt, int64_t R, int64_t C,
                                   int64_t ldw, uint8_t* q, int64_t ldq, uint8_t* qT,
                                   int64_t ldqT, float* s, int64_t lds, void* stream) {
  if (R < 0 || C < 0 || !valid_dtype(wt)) return FP8BS_ERR_INVALID_ARG;
  if (R % 128 != 0 || C % 128 != 0) return FP8BS_ERR_UNSUPPORTED;
  if (R == 0 || C == 0) return FP8BS_OK;
  if (R / 128 > 65535 || C / 128 > INT_MAX) return FP8BS_ERR_UNSUPPORTED;
  if (w == nullptr || s == nullptr || (q == nullptr && qT == nullptr)) return FP8BS_ERR_INVALID_ARG;
  if (ldw < C || (q && ldq < C) || (qT && ldqT < R) || lds < C / 128) return FP8BS_ERR_INVALID_ARG;
  if (!aligned(w, 16) || (ldw * static_cast<int64_t>(dtype_size(wt))) % 16 || !aligned(s, 4))
    return FP8BS_ERR_MISALIGNED;
  if (q && (!aligned(q, 16) || ldq % 16)) return FP8BS_ERR_MISALIGNED;
  if (qT && (!aligned(qT, 16) || ldqT % 16)) return FP8BS_ERR_MISALIGNED;
  dim3 grid(static_cast<unsigned>(C / 128), static_cast<unsigned>(R / 128));
  // staged block, plus the transposed codes (128 x 128 bytes) when qT is asked for
  const size_t smem = 128 * 128 * dtype_size(wt) + (qT != nullptr ? 128 * 128 : 0);
  if (wt == FP8BS_BF16) {
    if (cudaFuncSetAttribute(quant_128x128_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return FP8BS_ERR_CUDA;
    prefer_max_shared(quant_128x128_kernel<__nv_bfloat16>);
    quant_128x128_kernel<__nv_bfloat16><<<grid, 256, smem, as_stream(stream)>>>(
        static_cast<const __nv_bfloat16*>(w), ldw, q, ldq, qT, ldqT, s, lds);
  } else {
    if (cudaFuncSetAttribute(quant_128x128_kernel<float>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return FP8BS_ERR_CUDA;
    prefer_max_shared(quant_128x128_kernel<float>);
    quant_128x128_kernel<float><<<grid, 256, smem, as_stream(stream)>>>(
        static_cast<const float*>(w), ldw, q, ldq, qT, ldqT, s, lds);
  }
  return launch_status();
}

fp8bs_status fp8bs_gemm(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda,
                        const float* sa, int64_t ldsa, const uint8_t* B, int64_t ldb,
                        const float* sb, fp8bs_bscale sb_mode, int64_t ldsb, void* C,
                        fp8bs_dtype ct, int64_t ldc, void* stream) {
  return gemm_dense(M, N, K, A, lda, sa, ldsa, B, ldb, sb, sb_mode, ldsb, C, ct, ldc, nullptr, 0,
                    stream);
}

fp8bs_status fp8bs_gemm_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes) {
  if (bytes == nullptr || M < 0 || N < 0 || K < 0) return FP8BS_ERR_INVALID_ARG;
  *bytes = 0;
  if (M == 0 || N == 0 || K == 0) return FP8BS_OK;
  if (K % kBK != 0 || M > INT_MAX - kPairTileM || N > INT_MAX - kBN) return FP8BS_ERR_UNSUPPORTED;
  int clusters = 0;
  fp8bs_status st = pair_cluster_count(&clusters);
  if (st != FP8BS_OK) return st;
  for (int bn : {256}) {
    const int64_t tiles = ((M + kPairTileM - 1) / kPairTileM) * ((N + bn - 1) / bn);
    if (tiles > INT_MAX) return FP8BS_ERR_UNSUPPORTED;
    const size_t need =
        plan_split(static_cast<int>(tiles), static_cast<int>(K / kBK), clusters, SIZE_MAX, bn).ws_bytes;
    if (need > *bytes) *bytes = need;
  }
  return FP8BS_OK;
}

fp8bs_status fp8bs_gemm_ws(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda,
                           const float* sa, int64_t ldsa, const uint8_t* B, int64_t ldb,
                           const float* sb, fp8bs_bscale sb_mode, int64_t ldsb, void* C,
                           fp8bs_dtype ct, int64_t ldc, void* workspace, size_t workspace_bytes,
                           void* stream) {
  if (workspace != nullptr && !aligned(workspace, 256)) return FP8BS_ERR_MISALIGNED;
  return gemm_dense(M, N, K, A, lda, sa, ldsa, B, ldb, sb, sb_mode, ldsb, C, ct, ldc,
                    static_cast<float*>(workspace), workspace ? workspace_bytes : 0, stream);
}

fp8bs_status fp8bs_gemm_accumulate(int64_t M, int64_t N, int64_t K, const uint8_t* A,
                                   int64_t lda, const float* sa, int64_t ldsa, const uint8_t* B,
                                   int64_t ldb, const float* sb, fp8bs_bscale sb_mode,
                                   int64_t ldsb, float* C, int64_t ldc, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  if (workspace != nullptr && !aligned(workspace, 256)) return FP8BS_ERR_MISALIGNED;
  return gemm_dense(M, N, K, A, lda, sa, ldsa, B, ldb, sb, sb_mode, ldsb, C, FP8BS_F32, ldc,
                    static_cast<float*>(workspace), workspace ? workspace_bytes : 0, stream,
                    /*acc=*/true);
}

fp8bs_status fp8bs_gemm_static_ws(int64_t M, int64_t N, int64_t K, const uint8_t* A,
                                  int64_t lda, const float* sa, int64_t ldsa, const uint8_t* B,
                                  int64_t ldb, const float* sb, fp8bs_bscale sb_mode, int64_t ldsb,
                                  void* C, fp8bs_dtype ct, int64_t ldc, void* stream) {
  // The argument checks of fp8bs_gemm_ws come first, on the host, so a bad
  // call returns the same status and touches no device state.
  fp8bs_status st = check_gemm(M, N, K, A, lda, sa, ldsa, B, ldb, sb, sb_mode, ldsb, C, ct, ldc);
  if (st != FP8BS_OK || M == 0 || N == 0) return st;
  if (K == 0)   // nothing to split: the contraction is empty and C is zero-filled
    return gemm_dense(M, N, K, A, lda, sa, ldsa, B, ldb, sb, sb_mode, ldsb, C, ct, ldc, nullptr, 0,
                      stream);
  size_t need = 0;
  if ((st = fp8bs_gemm_workspace_size(M, N, K, &need)) != FP8BS_OK) return st;
  if (need > kStaticWsBytes) return FP8BS_ERR_UNSUPPORTED;   // more scratch than the array holds
  void* ws = nullptr;
  if ((st = static_workspace(&ws)) != FP8BS_OK) return st;
  return gemm_dense(M, N, K, A, lda, sa, ldsa, B, ldb, sb, sb_mode, ldsb, C, ct, ldc,
                    static_cast<float*>(ws), kStaticWsBytes, stream);
}

fp8bs_status fp8bs_grouped_gemm(int32_t E, const int32_t* offsets, int64_t M_cap, int64_t N,
                                int64_t K, const uint8_t* A, int64_t lda, const float* sa,
                                int64_t ldsa, const uint8_t* B, int64_t ldb, const float* sb,
                                fp8bs_bscale sb_mode, int64_t ldsb, int64_t sb_estride, void* C,
                                fp8bs_dtype ct, int64_t ldc, void* stream) {
  if (E < 1 || E > kMaxExperts || offsets == nullptr || !aligned(offsets, 4))
    return FP8BS_ERR_INVALID_ARG;
  if (M_cap < 0 || M_cap % 128 != 0) return FP8BS_ERR_UNSUPPORTED;
  if (sb_estride < 0) return FP8BS_ERR_INVALID_ARG;
  fp8bs_status st =
      check_gemm(M_cap, N, K, A, lda, sa, ldsa, B, ldb, sb, sb_mode, ldsb, C, ct, ldc);
  if (st != FP8BS_OK || M_cap == 0 || N == 0) return st;
  if (sb_mode == FP8BS_SB_PERCOL && sb_estride % 4 != 0) return FP8BS_ERR_MISALIGNED;
  if (K == 0) return FP8BS_ERR_UNSUPPORTED;  // expert rows are only known on the device
  CUtensorMap ta, tb, tc;
  if ((st = make_map_2d(&ta, A, K, M_cap, lda, kBM)) != FP8BS_OK) return st;
  if ((st = make_map_3d(&tb, B, K, N, E, ldb, kBN)) != FP8BS_OK) return st;
  if ((st = make_map_out(&tc, C, ct, N, M_cap, ldc)) != FP8BS_OK) return st;
  GemmParams p{};
  p.M = static_cast<int32_t>(M_cap);
  p.N = static_cast<int32_t>(N);
  p.KB = static_cast<int32_t>(K / kBK);
  p.num_m_tiles = static_cast<int32_t>(M_cap / kBM);
  p.num_n_tiles = static_cast<int32_t>((N + kBN - 1) / kBN);
  p.E = E;
  p.sa = sa;
  p.ldsa = ldsa;
  p.sb = sb;
  fill_scale_strides(p, sb_mode, ldsb);
  p.sb_e_stride = sb_estride;
  p.C = C;
  p.ldc = ldc;
  p.offsets = offsets;
  return launch_grouped(p, ta, tb, tc, sb_mode == FP8BS_SB_PERCOL ? kSbPerCol : kSbBlock, ct,
                        as_stream(stream));
}

fp8bs_status fp8bs_sync_status(void* stream) {
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return FP8BS_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpyFromSymbol(&word, g_device_error, sizeof(word)) != cudaSuccess)
    return FP8BS_ERR_CUDA;
  if (word != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess)
      return FP8BS_ERR_CUDA;
    if (word & kDevErrTimeout) return FP8BS_ERR_DEVICE_TIMEOUT;
    if (word & kDevErrBadRouting) return FP8BS_ERR_DEVICE_BAD_ROUTING;
    return FP8BS_ERR_DEVICE_BAD_OFFSETS;
  }
  return FP8BS_OK;
}

const char* fp8bs_status_string(fp8bs_status status) {
  switch (status) {
    case FP8BS_OK: return "ok";
    case FP8BS_ERR_INVALID_ARG: return "invalid argument";
    case FP8BS_ERR_MISALIGNED: return "misaligned pointer or leading dimension";
    case FP8BS_ERR_UNSUPPORTED: return "unsupported shape";
    case FP8BS_ERR_CUDA: return "CUDA error";
    case FP8BS_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case FP8BS_ERR_DEVICE_BAD_OFFSETS: return "grouped GEMM offsets failed device validation";
    case FP8BS_ERR_DEVICE_BAD_ROUTING: return "expert id outside [0, E) in dispatch";
  }
  return "unknown status";
}

fp8bs_status fp8bs_probe_mma_f8f6f4(const uint8_t* a, const uint8_t* b, int64_t K, float* d,
                                    void* stream) {
  if (a == nullptr || b == nullptr || d == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (K < 32 || K > 128 || K % 32 != 0) return FP8BS_ERR_UNSUPPORTED;
  if (!aligned(d, 4)) return FP8BS_ERR_MISALIGNED;
  if (cudaFuncSetAttribute(fp8bs_mma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kProbeSmemBytes)) != cudaSuccess)
    return FP8BS_ERR_CUDA;
  fp8bs_mma_probe_kernel<<<1, 128, kProbeSmemBytes, as_stream(stream)>>>(a, b, static_cast<int>(K),
                                                                         d);
  return launch_status();
}

fp8bs_status fp8bs_mx_quant_1x32(const void* x, fp8bs_dtype xt, int64_t R, int64_t K, int64_t ldx,
                                 uint8_t* q, int64_t ldq, uint32_t* sf, int64_t ldsf,
                                 void* stream) {
  if (R < 0 || K < 0 || !valid_dtype(xt)) return FP8BS_ERR_INVALID_ARG;
  if (K % 128 != 0) return FP8BS_ERR_UNSUPPORTED;
  if (R == 0 || K == 0) return FP8BS_OK;
  if ((R + 7) / 8 > INT_MAX || (K + 1023) / 1024 > 65535) return FP8BS_ERR_UNSUPPORTED;
  if (x == nullptr || q == nullptr || sf == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (ldx < K || ldq < K || ldsf < R) return FP8BS_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(q, 16) || (ldx * static_cast<int64_t>(dtype_size(xt))) % 16 ||
      ldq % 16 || !aligned(sf, 4))
    return FP8BS_ERR_MISALIGNED;
  const dim3 grid(static_cast<unsigned>((R + 7) / 8), static_cast<unsigned>((K + 1023) / 1024));
  if (xt == FP8BS_BF16)
    mx_quant_1x32_kernel<__nv_bfloat16><<<grid, 256, 0, as_stream(stream)>>>(
        static_cast<const __nv_bfloat16*>(x), R, K, ldx, q, ldq, sf, ldsf);
  else
    mx_quant_1x32_kernel<float><<<grid, 256, 0, as_stream(stream)>>>(
        static_cast<const float*>(x), R, K, ldx, q, ldq, sf, ldsf);
  return launch_status();
}

fp8bs_status fp8bs_mx_gemm(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda,
                           const uint32_t* sfa, int64_t ldsfa, const uint8_t* B, int64_t ldb,
                           const uint32_t* sfb, int64_t ldsfb, void* C, fp8bs_dtype ct,
                           int64_t ldc, void* stream) {
  if (M < 0 || N < 0 || K < 0 || !valid_dtype(ct)) return FP8BS_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return FP8BS_OK;
  if (K % kBK != 0 || N % 16 != 0) return FP8BS_ERR_UNSUPPORTED;
  if (M > INT_MAX - kBM || N > INT_MAX - kBN || K / kBK > INT_MAX) return FP8BS_ERR_UNSUPPORTED;
  if (((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN) > INT_MAX) return FP8BS_ERR_UNSUPPORTED;
  if (C == nullptr || ldc < N) return FP8BS_ERR_INVALID_ARG;
  if (!aligned(C, 16) || (ldc * static_cast<int64_t>(dtype_size(ct))) % 16 != 0)
    return FP8BS_ERR_MISALIGNED;
  if (K == 0) return zero_fill(C, ct, M, N, ldc, as_stream(stream));
  if (A == nullptr || B == nullptr || sfa == nullptr || sfb == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (lda < K || ldb < K || ldsfa < M || ldsfb < N) return FP8BS_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(B, 16) || lda % 16 != 0 || ldb % 16 != 0)
    return FP8BS_ERR_MISALIGNED;
  if (!aligned(sfa, 16) || !aligned(sfb, 16) || ldsfa % 4 != 0 || ldsfb % 4 != 0)
    return FP8BS_ERR_MISALIGNED;
  DeviceInfo di;
  fp8bs_status st = device_info(&di);
  if (st != FP8BS_OK) return st;
  CUtensorMap ta, tb, tsa, tsb, tc;
  const int64_t KB = K / kBK;
  // CTA pairs: each CTA loads its 128 rows of A and half of the B tile
  if ((st = make_map_2d(&ta, A, K, M, lda, kBM)) != FP8BS_OK) return st;
  if ((st = make_map_2d(&tb, B, K, N, ldb, kBN / 2)) != FP8BS_OK) return st;
  if ((st = make_map_sf(&tsa, sfa, M, KB, ldsfa, kBM)) != FP8BS_OK) return st;
  if ((st = make_map_sf(&tsb, sfb, N, KB, ldsfb, kBN)) != FP8BS_OK) return st;
  if ((st = make_map_out(&tc, C, ct, N, M, ldc)) != FP8BS_OK) return st;
  MxParams p{};
  p.M = static_cast<int32_t>(M);
  p.N = static_cast<int32_t>(N);
  p.KB = static_cast<int32_t>(KB);
  p.num_m_tiles = static_cast<int32_t>((M + kPairTileM - 1) / kPairTileM);
  p.num_n_tiles = static_cast<int32_t>((N + kBN - 1) / kBN);
  const int tiles = p.num_m_tiles * p.num_n_tiles;
  auto run = [&](auto kernel) -> fp8bs_status {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kMxPairSmemBytes)) != cudaSuccess)
      return FP8BS_ERR_CUDA;
    const int clusters = mx_pair_clusters(kernel);
    if (clusters <= 0) return FP8BS_ERR_CUDA;
    const int grid_clusters = tiles < clusters ? tiles : clusters;
    kernel<<<2 * grid_clusters, kMxThreads, kMxPairSmemBytes, as_stream(stream)>>>(p, ta, tb, tsa,
                                                                                   tsb, tc);
    return launch_status();
  };
  return ct == FP8BS_BF16 ? run(fp8bs_mx_gemm_pair_kernel<true>)
                          : run(fp8bs_mx_gemm_pair_kernel<false>);

}

fp8bs_status fp8bs_debug_timeout_probe(int64_t limit_ns, void* stream) {
  if (limit_ns < 1000 || limit_ns > 10000000000LL) return FP8BS_ERR_INVALID_ARG;
  fp8bs_timeout_probe_kernel<<<1, 32, 0, as_stream(stream)>>>(static_cast<uint64_t>(limit_ns));
  return launch_status();
}

}  // extern "C"
