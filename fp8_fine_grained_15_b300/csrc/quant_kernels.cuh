// Fine-grained E4M3 quantizers (1x128, 128x1 transposed, 128x128 with an
// optional transposed copy).
//
// Method: "Should Fixing Deepseek Take 60 Steps?", Figure 7 (a) passage (tile
// and block granularity) and max-abs scaling passage; page at
// why-be.why-be.co.kr, online-amax passage; E4M3 on all tensors (untitled page
// at jp-study.kr, hybrid-format passage).
//
// Per tile: amax = max|x| (exact), r = 448/amax and s = amax/448 as IEEE
// binary32 divisions (r not finite -> s = r = 1), code = cvt.rn.satfinite
// E4M3(x * r).  All three kernels are HBM-bound streams: 16-byte vector loads
// with no L1 allocation, several independent loads in flight per thread, warp
// shuffles for the 1x128 amax, shared-memory staging where the output is the
// transpose of the input.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cstdint>

#include "ptx.cuh"

namespace fp8bs {

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Elements of a 16-byte vector widened to fp32 (exact for bf16).
template <typename T>
struct Vec16;

template <>
struct Vec16<float> {
  static constexpr int kN = 4;
  __device__ __forceinline__ static void widen(const uint4& v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
};

template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int kN = 8;
  __device__ __forceinline__ static void widen(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};

template <typename T>
__device__ __forceinline__ float widen1(T v);
template <>
__device__ __forceinline__ float widen1<float>(float v) { return v; }
template <>
__device__ __forceinline__ float widen1<__nv_bfloat16>(__nv_bfloat16 v) {
  return __uint_as_float(static_cast<uint32_t>(__bfloat16_as_ushort(v)) << 16);
}

// Scale and multiplier of a tile with max-abs amax.
__device__ __forceinline__ void tile_scale(float amax, float& s, float& r) {
  r = __fdiv_rn(448.0f, amax);
  if (isinf(r)) {
    s = 1.0f;
    r = 1.0f;
  } else {
    s = __fdiv_rn(amax, 448.0f);
  }
}

// Two values -> two E4M3 codes (lo in the low byte), RNE with saturation.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi, float r) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(
      make_float2(__fmul_rn(lo, r), __fmul_rn(hi, r)), __NV_SATFINITE, __NV_E4M3));
}

// Four values -> four codes packed little-endian in a word.
__device__ __forceinline__ uint32_t e4m3x4(const float* f, float r) {
  return e4m3x2(f[0], f[1], r) | (e4m3x2(f[2], f[3], r) << 16);
}

// ---------------------------------------------------------------- 1 x 128
// Four lanes share a 128-element tile, 32 elements each, so the per-tile work
// (two IEEE divisions, two shuffle steps, index arithmetic) is spread over 32
// elements per lane.  Load i of a lane covers elements [i*4v + l*v, +v) of its
// tile (v = 16 bytes of input), so the four lanes of a tile read 64 contiguous
// bytes per instruction.  A warp covers 8 tiles per step and kUnroll steps per
// iteration; tiles are numbered row-major (m, kb).
template <typename TIn, int kUnroll>
__global__ void __launch_bounds__(256) quant_1x128_kernel(const TIn* __restrict__ x, uint32_t M,
                                                          uint32_t KB, int64_t ldx,
                                                          uint8_t* __restrict__ q, int64_t ldq,
                                                          float* __restrict__ s, int64_t lds) {
  constexpr int kVec = Vec16<TIn>::kN;         // elements per 16-byte load
  constexpr int kLoads = 128 / (4 * kVec);     // 16-byte loads per lane per tile
  constexpr int kTilesPerIter = 8 * kUnroll;
  const int lane = threadIdx.x & 31;
  const int sub = lane >> 2;                   // tile within the warp step
  const int l = lane & 3;                      // lane within the tile
  const uint32_t total = M * KB;
  const uint32_t warp_id = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t num_warps = (gridDim.x * blockDim.x) >> 5;

  for (uint32_t base = warp_id * kTilesPerIter; base < total; base += num_warps * kTilesPerIter) {
    uint4 v[kUnroll][kLoads];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t t = base + u * 8 + sub;
      if (t < total) {
        const uint32_t m = t / KB, kb = t - m * KB;
        const TIn* src = x + static_cast<int64_t>(m) * ldx + kb * 128 + l * kVec;
#pragma unroll
        for (int i = 0; i < kLoads; ++i) v[u][i] = ld_stream16(src + i * 4 * kVec);
      } else {
#pragma unroll
        for (int i = 0; i < kLoads; ++i) v[u][i] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t t = base + u * 8 + sub;
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < kLoads; ++i) {
        float f[kVec];
        Vec16<TIn>::widen(v[u][i], f);
#pragma unroll
        for (int j = 0; j < kVec; ++j) amax = fmaxf(amax, fabsf(f[j]));
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      float sc, r;
      tile_scale(amax, sc, r);
      if (t < total) {
        const uint32_t m = t / KB, kb = t - m * KB;
        uint8_t* dst = q + static_cast<int64_t>(m) * ldq + kb * 128 + l * kVec;
#pragma unroll
        for (int i = 0; i < kLoads; ++i) {
          float f[kVec];
          Vec16<TIn>::widen(v[u][i], f);
          if constexpr (kVec == 8) {
            *reinterpret_cast<uint2*>(dst + i * 4 * kVec) =
                make_uint2(e4m3x4(f, r), e4m3x4(f + 4, r));
          } else {
            *reinterpret_cast<uint32_t*>(dst + i * 4 * kVec) = e4m3x4(f, r);
          }
        }
        if (l == 0) s[static_cast<int64_t>(kb) * lds + m] = sc;
      }
    }
  }
}

// ---------------------------------------------------------------- 128 x 1
// One CTA per (128 tokens) x (256 bytes of channels).  The block is staged in
// shared memory with cp.async (no register round trip, L1 bypassed).  Each
// thread then owns one 32-bit channel group (two bf16 channels or one fp32
// channel) and 32 consecutive tokens: 32 conflict-free word reads, a
// per-channel partial amax combined across the four token parts through shared
// memory, then 32 codes per channel (words re-read from shared memory) written
// as two 16-byte chunks of that channel's 128-byte output row, staged in
// shared memory (chunk j of row c at j ^ ((c / channels-per-word) & 7):
// conflict-free for the writers).  Eight consecutive lanes then store each
// whole row, so every warp store covers four complete 128-byte lines.
template <typename TIn>
constexpr size_t quant_128x1_smem_bytes() {
  return 128 * 64 * 4 /* staged tile: 128 tokens x 64 words */ +
         (256 / sizeof(TIn)) * 128 /* transposed codes: channels x 128 tokens */;
}

// Coalesced store of staged transposed codes: rows [0, rows) of 128 bytes,
// chunk j of row c at position j ^ ((c / kCh) & 7), to dst_row(c) + 16 j.
template <int kCh>
__device__ __forceinline__ void store_transposed_rows(const uint4* outT, int rows, int64_t c_limit,
                                                      uint8_t* base, int64_t ld) {
  for (int i = threadIdx.x; i < rows * 8; i += blockDim.x) {
    const int c = i >> 3, j = i & 7;
    if (c < c_limit)
      *reinterpret_cast<uint4*>(base + static_cast<int64_t>(c) * ld + j * 16) =
          outT[c * 8 + (j ^ ((c / kCh) & 7))];
  }
}

template <typename TIn>
__global__ void __launch_bounds__(256, 4) quant_128x1_kernel(const TIn* __restrict__ x, int64_t C,
                                                             int64_t ldx, uint8_t* __restrict__ qT,
                                                             int64_t ldq, float* __restrict__ s,
                                                             int64_t lds) {
  constexpr int kVec = Vec16<TIn>::kN;
  constexpr int kCB = 256 / sizeof(TIn);       // channels per CTA (256 bytes per row)
  constexpr int kVecPerRow = kCB / kVec;       // 16
  constexpr int kRowsPerPass = 256 / kVecPerRow;
  constexpr int kLoads = 128 / kRowsPerPass;   // 16-byte copies per thread
  constexpr int kCh = 4 / sizeof(TIn);         // channels per 32-bit word
  constexpr int kGroups = kCB / kCh;           // 64 word columns
  constexpr int kParts = 256 / kGroups;        // 4 token parts
  constexpr int kTok = 128 / kParts;           // 32 tokens per thread
  static_assert(kGroups == 64 && kTok == 32, "layout of quant_128x1_smem_bytes");
  extern __shared__ __align__(16) unsigned char q128x1_smem[];
  uint32_t (*tile)[kGroups] = reinterpret_cast<uint32_t (*)[kGroups]>(q128x1_smem);
  uint4* outT = reinterpret_cast<uint4*>(q128x1_smem + 128 * kGroups * 4);   // [kCB][8]
  __shared__ float part_amax[kParts][kCB];

  const int64_t tb = blockIdx.y;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kCB;
  const int tid = threadIdx.x;
  {
    const int vc = tid % kVecPerRow;
    const int r0 = tid / kVecPerRow;
    const int64_t col = c0 + vc * kVec;
#pragma unroll
    for (int i = 0; i < kLoads; ++i) {
      const int64_t row = tb * 128 + r0 + i * kRowsPerPass;
      uint32_t* dst = &tile[r0 + i * kRowsPerPass][vc * 4];
      if (col < C) {
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)),
                     "l"(x + row * ldx + col)
                     : "memory");
      } else {
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
      }
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
  }
  __syncthreads();

  const int g = tid % kGroups;
  const int part = tid / kGroups;
  float amax[kCh];
#pragma unroll
  for (int k = 0; k < kCh; ++k) amax[k] = 0.0f;
#pragma unroll 8
  for (int t = 0; t < kTok; ++t) {
    const uint32_t w = tile[part * kTok + t][g];
    if constexpr (kCh == 2) {
      amax[0] = fmaxf(amax[0], fabsf(__uint_as_float(w << 16)));
      amax[1] = fmaxf(amax[1], fabsf(__uint_as_float(w & 0xFFFF0000u)));
    } else {
      amax[0] = fmaxf(amax[0], fabsf(__uint_as_float(w)));
    }
  }
#pragma unroll
  for (int k = 0; k < kCh; ++k) part_amax[part][g * kCh + k] = amax[k];
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kCh; ++k) {
    float a = part_amax[0][g * kCh + k];
#pragma unroll
    for (int p = 1; p < kParts; ++p) a = fmaxf(a, part_amax[p][g * kCh + k]);
    float sc, r;
    tile_scale(a, sc, r);
    const int cl = g * kCh + k;   // channel within the CTA's block
#pragma unroll 1
    for (int t = 0; t < kTok; t += 16) {   // words re-read from shared memory (no spills)
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float f[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t wv = tile[part * kTok + t + 4 * j + i][g];
          f[i] = __uint_as_float(kCh == 1 ? wv : (k == 0 ? (wv << 16) : (wv & 0xFFFF0000u)));
        }
        o[j] = e4m3x4(f, r);
      }
      const int chunk = (part * kTok + t) >> 4;
      outT[cl * 8 + (chunk ^ (g & 7))] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (part == 0 && c0 + cl < C) s[tb * lds + c0 + cl] = sc;
  }
  __syncthreads();
  store_transposed_rows<kCh>(outT, kCB, C - c0, qT + c0 * ldq + tb * 128, ldq);
}

// -------------------------------------------------------------- 128 x 128
// One CTA per 128 x 128 block, staged in shared memory with cp.async (32 KB
// for bf16, 64 KB for fp32).  Each thread owns one 32-bit word column (two
// bf16 channels or one fp32 channel) over a run of rows: it reduces its part of
// the block amax from those words (then warp shuffles + shared memory), and
// later re-reads them 16 rows at a time to form that column's transposed
// codes, staged as 128-byte output rows in shared memory (swizzled as in the
// 128x1 kernel) and stored as whole rows by consecutive lanes.  The row-major
// codes come from 16-byte shared-memory reads.  Both copies use the same
// multiply and conversion, so they hold identical codes.
template <typename TIn>
__global__ void __launch_bounds__(256, 5) quant_128x128_kernel(const TIn* __restrict__ w,
                                                               int64_t ldw,
                                                               uint8_t* __restrict__ q,
                                                               int64_t ldq,
                                                               uint8_t* __restrict__ qT,
                                                               int64_t ldqT,
                                                               float* __restrict__ s,
                                                               int64_t lds) {
  constexpr int kVec = Vec16<TIn>::kN;                      // elements per 16 bytes
  constexpr int kWordsPerRow = 128 * sizeof(TIn) / 4;       // 64 (bf16) or 128 (fp32)
  constexpr int kVecPerRow = 128 / kVec;                    // 16 or 32
  constexpr int kCh = 4 / sizeof(TIn);                      // channels per word
  constexpr int kParts = 256 / kWordsPerRow;                // 4 or 2 row parts
  constexpr int kRows = 128 / kParts;                       // 32 or 64 rows per thread
  extern __shared__ __align__(16) unsigned char dyn_smem[];
  uint32_t* tile = reinterpret_cast<uint32_t*>(dyn_smem);   // [128][kWordsPerRow]
  // with qT: the transposed codes [128 channels][8 chunks of 16 rows]
  uint4* outT = reinterpret_cast<uint4*>(dyn_smem + 128 * kWordsPerRow * 4);
  __shared__ float warp_amax[8];

  const int64_t rb = blockIdx.y, cb = blockIdx.x;
  const int tid = threadIdx.x;
  const TIn* src = w + rb * 128 * ldw + cb * 128;
#pragma unroll
  for (int i = tid; i < 128 * kVecPerRow; i += 256) {
    const int row = i / kVecPerRow, vc = i % kVecPerRow;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     smem_u32(tile + row * kWordsPerRow + vc * 4)),
                 "l"(src + row * ldw + vc * kVec)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
  __syncthreads();

  const int g = tid % kWordsPerRow;
  const int part = tid / kWordsPerRow;
  const uint32_t* col = tile + part * kRows * kWordsPerRow + g;   // this thread's word column
  float amax = 0.0f;
#pragma unroll 8
  for (int t = 0; t < kRows; ++t) {
    const uint32_t v = col[t * kWordsPerRow];
    if constexpr (kCh == 2) {
      amax = fmaxf(amax, fabsf(__uint_as_float(v << 16)));
      amax = fmaxf(amax, fabsf(__uint_as_float(v & 0xFFFF0000u)));
    } else {
      amax = fmaxf(amax, fabsf(__uint_as_float(v)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((tid & 31) == 0) warp_amax[tid >> 5] = amax;
  __syncthreads();
  amax = warp_amax[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, warp_amax[i]);
  float sc, r;
  tile_scale(amax, sc, r);
  if (tid == 0) s[rb * lds + cb] = sc;

  if (qT != nullptr) {
    // 16 rows at a time: 16 words -> 16 codes for each channel of the word
#pragma unroll 1
    for (int t = 0; t < kRows; t += 16) {
      uint32_t v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = col[(t + i) * kWordsPerRow];
#pragma unroll
      for (int k = 0; k < kCh; ++k) {
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float f[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t x = v[4 * j + i];
            f[i] = __uint_as_float(kCh == 1 ? x : (k == 0 ? (x << 16) : (x & 0xFFFF0000u)));
          }
          o[j] = e4m3x4(f, r);
        }
        const int chunk = (part * kRows + t) >> 4;
        outT[(g * kCh + k) * 8 + (chunk ^ (g & 7))] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    __syncthreads();
    store_transposed_rows<kCh>(outT, 128, 128, qT + cb * 128 * ldqT + rb * 128, ldqT);
  }
  if (q != nullptr) {
    uint8_t* dst = q + rb * 128 * ldq + cb * 128;
#pragma unroll
    for (int i = tid; i < 128 * kVecPerRow; i += 256) {
      const int row = i / kVecPerRow, vc = i % kVecPerRow;
      const uint4 v = *reinterpret_cast<const uint4*>(tile + row * kWordsPerRow + vc * 4);
      float f[kVec];
      Vec16<TIn>::widen(v, f);
      uint8_t* d = dst + row * ldq + vc * kVec;
      if constexpr (kVec == 8) {
        *reinterpret_cast<uint2*>(d) = make_uint2(e4m3x4(f, r), e4m3x4(f + 4, r));
      } else {
        *reinterpret_cast<uint32_t*>(d) = e4m3x4(f, r);
      }
    }
  }
}

// ------------------------------------------------------------ dual 1x128 + 128x1
// One read of a 128-token x 128-channel block of X gives both granularities the
// layer step needs: the 1x128 codes (row-major, the A operand of Fprop / Dgrad)
// and the 128x1 codes (transposed, the operand of Wgrad), each bit-identical to
// the single-granularity kernels.  The block is staged in shared memory with
// cp.async; its 16-byte chunks are XOR-swizzled by row (chunk ^ (row & 7)) so
// that both the row pass (4 lanes per row, 8 rows per warp) and the column
// pass (32 consecutive words of one row per warp) read without bank conflicts.
template <typename TIn>
__global__ void __launch_bounds__(256) quant_dual_kernel(const TIn* __restrict__ x, int64_t ldx,
                                                         uint8_t* __restrict__ q, int64_t ldq,
                                                         float* __restrict__ s, int64_t lds,
                                                         uint8_t* __restrict__ qT, int64_t ldqT,
                                                         float* __restrict__ sT, int64_t ldsT) {
  constexpr int kVec = Vec16<TIn>::kN;                      // elements per 16 bytes
  constexpr int kChunksPerRow = 128 / kVec;                 // 16 (bf16) or 32 (fp32)
  constexpr int kWordsPerRow = kChunksPerRow * 4;
  constexpr int kCh = 4 / sizeof(TIn);                      // channels per 32-bit word
  constexpr int kParts = 256 / kWordsPerRow;                // 4 or 2 token parts
  constexpr int kRows = 128 / kParts;                       // 32 or 64 tokens per thread
  extern __shared__ __align__(16) unsigned char dual_smem[];
  uint32_t* tile = reinterpret_cast<uint32_t*>(dual_smem);  // [128][kWordsPerRow], swizzled
  // transposed codes [128 channels][8 chunks of 16 tokens], chunk j of channel c
  // at j ^ ((c / kCh) & 7), stored as whole 128-byte rows at the end
  uint4* outT = reinterpret_cast<uint4*>(dual_smem + 128 * kWordsPerRow * 4);
  __shared__ float part_amax[kParts][128];

  const int64_t tb = blockIdx.y, cb = blockIdx.x;
  const int tid = threadIdx.x;
  auto chunk_at = [](int row, int chunk) { return row * kChunksPerRow + (chunk ^ (row & 7)); };
  {
    const TIn* src = x + tb * 128 * ldx + cb * 128;
#pragma unroll 4
    for (int i = tid; i < 128 * kChunksPerRow; i += 256) {
      const int row = i / kChunksPerRow, ch = i % kChunksPerRow;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                       smem_u32(tile + chunk_at(row, ch) * 4)),
                   "l"(src + row * ldx + ch * kVec)
                   : "memory");
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
  }
  __syncthreads();

  // ---- 1x128: four lanes per token row; load i of lane l is chunk i*4 + l
  {
    const int warp = tid >> 5, lane = tid & 31;
    const int l = lane & 3;
    constexpr int kLoads = kChunksPerRow / 4;
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
      const int row = warp * 16 + pass * 8 + (lane >> 2);
      uint4 v[kLoads];
#pragma unroll
      for (int i = 0; i < kLoads; ++i)
        v[i] = *reinterpret_cast<const uint4*>(tile + chunk_at(row, i * 4 + l) * 4);
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < kLoads; ++i) {
        float f[kVec];
        Vec16<TIn>::widen(v[i], f);
#pragma unroll
        for (int j = 0; j < kVec; ++j) amax = fmaxf(amax, fabsf(f[j]));
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      float sc, r;
      tile_scale(amax, sc, r);
      uint8_t* dst = q + (tb * 128 + row) * ldq + cb * 128 + l * kVec;
#pragma unroll
      for (int i = 0; i < kLoads; ++i) {
        float f[kVec];
        Vec16<TIn>::widen(v[i], f);
        if constexpr (kVec == 8) {
          *reinterpret_cast<uint2*>(dst + i * 4 * kVec) = make_uint2(e4m3x4(f, r), e4m3x4(f + 4, r));
        } else {
          *reinterpret_cast<uint32_t*>(dst + i * 4 * kVec) = e4m3x4(f, r);
        }
      }
      if (l == 0) s[cb * lds + tb * 128 + row] = sc;
    }
  }

  // ---- 128x1: thread (g, part) owns word column g over its run of token rows
  const int g = tid % kWordsPerRow;
  const int part = tid / kWordsPerRow;
  auto word_at = [&](int row) {
    return tile[chunk_at(row, g >> 2) * 4 + (g & 3)];
  };
  {
    float amax[kCh];
#pragma unroll
    for (int k = 0; k < kCh; ++k) amax[k] = 0.0f;
#pragma unroll 8
    for (int t = 0; t < kRows; ++t) {
      const uint32_t w = word_at(part * kRows + t);
      if constexpr (kCh == 2) {
        amax[0] = fmaxf(amax[0], fabsf(__uint_as_float(w << 16)));
        amax[1] = fmaxf(amax[1], fabsf(__uint_as_float(w & 0xFFFF0000u)));
      } else {
        amax[0] = fmaxf(amax[0], fabsf(__uint_as_float(w)));
      }
    }
#pragma unroll
    for (int k = 0; k < kCh; ++k) part_amax[part][g * kCh + k] = amax[k];
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kCh; ++k) {
    const int c = g * kCh + k;
    float a = part_amax[0][c];
#pragma unroll
    for (int p2 = 1; p2 < kParts; ++p2) a = fmaxf(a, part_amax[p2][c]);
    float sc, r;
    tile_scale(a, sc, r);
#pragma unroll 1
    for (int t = 0; t < kRows; t += 16) {
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float f[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t wv = word_at(part * kRows + t + 4 * j + i);
          f[i] = __uint_as_float(kCh == 1 ? wv : (k == 0 ? (wv << 16) : (wv & 0xFFFF0000u)));
        }
        o[j] = e4m3x4(f, r);
      }
      const int chunk = (part * kRows + t) >> 4;
      outT[c * 8 + (chunk ^ (g & 7))] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (part == 0) sT[tb * ldsT + cb * 128 + c] = sc;
  }
  __syncthreads();
  store_transposed_rows<kCh>(outT, 128, 128, qT + cb * 128 * ldqT + tb * 128, ldqT);
}

// ------------------------------------------------ quantize-then-dispatch (MoE)
// Activations quantized 1x128 straight into expert-grouped rows: expert e owns
// rows offsets[e] .. offsets[e+1]-1 (its token count padded to a multiple of
// 128), its tokens in increasing token order, then zero padding rows (codes 0,
// scale 1: what quantizing a zero row gives).  Source: untitled page at
// jp-study.kr, MoE passage (activations quantized to FP8 before the up-
// projection and dispatched in FP8).
constexpr int kDispatchMaxExperts = 256;

// The plan (which row each token lands in) takes two small launches:
//  dispatch_rank_kernel   one CTA per chunk of kRankChunk tokens: each token's
//                         rank among the chunk's earlier tokens of its expert
//                         (warp match, then a prefix of the per-warp counts over
//                         the chunk's warps) into token_row[t], and the chunk's
//                         per-expert counts into row_token[chunk * E + e] (the
//                         start of row_token serves as scratch: it is rewritten
//                         by the quantize kernel);
//  dispatch_plan_kernel   one CTA: the chunk counts, read into shared memory,
//                         give each chunk's first rank per expert (prefix over
//                         the chunks), the expert counts and the padded offsets;
//                         every token's row = offset + chunk base + rank goes to
//                         token_row[t].
// Tokens keep their order inside an expert.  (A single CTA ranking all 16384
// tokens of the MoE workload was issue-bound at ~21 us.)
constexpr int kRankChunk = 1024;
constexpr int kPlanMaxChunkCounts = 51200;  // chunks * E the plan CTA holds in shared memory (200 KB)

// Lanes of the warp holding the same expert id as this lane (ids < 256; -1 =
// no expert, matched with the other lanes holding none), from nine ballots.
__device__ __forceinline__ unsigned match_expert(int e) {
  const bool has = e >= 0;
  const unsigned v = __ballot_sync(0xffffffffu, has);
  unsigned m = has ? v : ~v;
  const int bits = has ? e : 0;
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    const bool on = (bits >> b) & 1;
    const unsigned w = __ballot_sync(0xffffffffu, on);
    m &= on ? w : ~w;
  }
  return m;
}

__global__ void __launch_bounds__(kRankChunk) dispatch_rank_kernel(const int32_t* __restrict__ expert,
                                                                   int64_t T, int E,
                                                                   int32_t* __restrict__ token_row,
                                                                   int32_t* __restrict__ chunk_counts) {
  __shared__ int32_t cnt[kDispatchMaxExperts][33];   // [expert][warp], padded rows
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kRankChunk + tid;
  int e = t < T ? expert[t] : -1;
  if (t < T && (e < 0 || e >= E)) {   // routing outside [0, E): the token is dropped
    atomicOr(&g_device_error, kDevErrBadRouting);
    e = -1;
  }
  for (int i = tid; i < 32 * E; i += kRankChunk) cnt[i >> 5][i & 31] = 0;
  __syncthreads();
  const unsigned m = match_expert(e);
  const unsigned lower = m & ((1u << lane) - 1u);
  if (e >= 0 && lower == 0) cnt[e][warp] = __popc(m);
  __syncthreads();
  for (int x = warp; x < E; x += 32) {   // exclusive prefix over the warps, per expert
    const int c = cnt[x][lane];
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    cnt[x][lane] = incl - c;
    if (lane == 31) chunk_counts[static_cast<int64_t>(blockIdx.x) * E + x] = incl;
  }
  __syncthreads();
  if (t < T) token_row[t] = e >= 0 ? cnt[e][warp] + static_cast<int>(__popc(lower)) : -1;
}

__global__ void __launch_bounds__(1024) dispatch_plan_kernel(const int32_t* __restrict__ expert,
                                                             int64_t T, int E, int chunks,
                                                             const int32_t* __restrict__ chunk_counts,
                                                             int32_t* __restrict__ token_row,
                                                             int32_t* __restrict__ counts,
                                                             int32_t* __restrict__ offsets) {
  extern __shared__ int32_t base[];   // [chunk][expert]: first rank, then + offset (dynamic)
  __shared__ int32_t off_s[kDispatchMaxExperts + 1];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < chunks * E; i += blockDim.x) base[i] = chunk_counts[i];
  __syncthreads();
  for (int x = tid; x < E; x += blockDim.x) {   // prefix over the chunks, one thread per expert
    int run = 0;
    for (int c = 0; c < chunks; ++c) {
      const int v = base[c * E + x];
      base[c * E + x] = run;
      run += v;
    }
    counts[x] = run;
    off_s[x] = (run + 127) / 128 * 128;   // padded size, scanned below
  }
  __syncthreads();
  if (warp == 0) {   // exclusive scan of the padded sizes (E <= 256: 8 per lane)
    constexpr int kPer = kDispatchMaxExperts / 32;
    int v[kPer], sum = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int x = lane * kPer + i;
      v[i] = x < E ? off_s[x] : 0;
      sum += v[i];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    int run = incl - sum;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int x = lane * kPer + i;
      if (x < E) {
        off_s[x] = run;
        offsets[x] = run;
      }
      run += v[i];
    }
    if (lane == 31) offsets[E] = incl;
  }
  __syncthreads();
  for (int i = tid; i < chunks * E; i += blockDim.x) base[i] += off_s[i % E];
  __syncthreads();
  constexpr int kBatch = 8;   // tokens per thread in flight
  for (int64_t t0 = tid; t0 < T; t0 += kBatch * static_cast<int64_t>(blockDim.x)) {
    int e[kBatch], r[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int64_t t = t0 + j * static_cast<int64_t>(blockDim.x);
      e[j] = t < T ? expert[t] : -1;
      r[j] = t < T ? token_row[t] : 0;
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int64_t t = t0 + j * static_cast<int64_t>(blockDim.x);
      if (e[j] >= 0 && e[j] < E)   // dropped tokens keep token_row -1
        token_row[t] = base[static_cast<int>(t / kRankChunk) * E + e[j]] + r[j];
    }
  }
}

// 1x128 quantization of token t's row into row token_row[t] (four lanes per
// 128-element tile, as in quant_1x128_kernel), with row_token[row] = t;
// dropped tokens (row -1) are skipped.  Then the padding rows, one warp per
// (expert, padding slot): codes 0, scales 1, row_token -1.
template <typename TIn>
__global__ void __launch_bounds__(256) quant_dispatch_kernel(
    const TIn* __restrict__ x, uint32_t T, uint32_t KB, int64_t ldx,
    const int32_t* __restrict__ token_row, int E, const int32_t* __restrict__ counts,
    const int32_t* __restrict__ offsets, uint8_t* __restrict__ q, int64_t ldq,
    float* __restrict__ s, int64_t lds, int32_t* __restrict__ row_token) {
  constexpr int kVec = Vec16<TIn>::kN;
  constexpr int kLoads = 128 / (4 * kVec);
  const int lane = threadIdx.x & 31;
  const int sub = lane >> 2, l = lane & 3;
  const uint32_t total = T * KB;
  const uint32_t warp_id = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t num_warps = (gridDim.x * blockDim.x) >> 5;
  for (uint32_t base = warp_id * 8; base < total; base += num_warps * 8) {
    const uint32_t tile = base + sub;
    const bool valid = tile < total;
    const uint32_t t = valid ? tile / KB : 0, kb = valid ? tile - t * KB : 0;
    const int32_t row32 = valid ? token_row[t] : -1;
    const bool routed = row32 >= 0;
    uint4 v[kLoads];
    const TIn* src = x + static_cast<int64_t>(t) * ldx + kb * 128 + l * kVec;
#pragma unroll
    for (int i = 0; i < kLoads; ++i) v[i] = routed ? ld_stream16(src + i * 4 * kVec) : make_uint4(0, 0, 0, 0);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < kLoads; ++i) {
      float f[kVec];
      Vec16<TIn>::widen(v[i], f);
#pragma unroll
      for (int j = 0; j < kVec; ++j) amax = fmaxf(amax, fabsf(f[j]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    float sc, r;
    tile_scale(amax, sc, r);
    if (routed) {
      const int64_t row = row32;
      uint8_t* dst = q + row * ldq + kb * 128 + l * kVec;
#pragma unroll
      for (int i = 0; i < kLoads; ++i) {
        float f[kVec];
        Vec16<TIn>::widen(v[i], f);
        if constexpr (kVec == 8) {
          *reinterpret_cast<uint2*>(dst + i * 4 * kVec) = make_uint2(e4m3x4(f, r), e4m3x4(f + 4, r));
        } else {
          *reinterpret_cast<uint32_t*>(dst + i * 4 * kVec) = e4m3x4(f, r);
        }
      }
      if (l == 0) {
        s[static_cast<int64_t>(kb) * lds + row] = sc;
        if (kb == 0) row_token[row] = static_cast<int32_t>(t);
      }
    }
  }
  // padding rows: slot j of expert e is row offsets[e] + counts[e] + j when
  // that is below offsets[e + 1] (at most 127 per expert)
  for (uint32_t u = warp_id; u < static_cast<uint32_t>(E) * 127u; u += num_warps) {
    const int e = static_cast<int>(u / 127u);
    const int64_t r = static_cast<int64_t>(offsets[e]) + counts[e] + (u % 127u);
    if (r >= offsets[e + 1]) continue;
    uint4* dst = reinterpret_cast<uint4*>(q + r * ldq);
    for (uint32_t i = lane; i < KB * 8u; i += 32) dst[i] = make_uint4(0, 0, 0, 0);
    for (uint32_t kb = lane; kb < KB; kb += 32) s[static_cast<int64_t>(kb) * lds + r] = 1.0f;
    if (lane == 0) row_token[r] = -1;
  }
}

// ------------------------------------------------------------ MX 1 x 32
// Microscaling variant ("Should Fixing Deepseek Take 60 Steps?", Figure 7 (a)
// passage and the page at why-be.why-be.co.kr, accumulation-precision passage:
// group scaling by the tensor cores is where fine-grained quantization goes
// next).  Groups of 32 along K; a group's scale is the power of two 2^e with
// the smallest e such that amax <= 448 * 2^e, clamped to [-127, 127] (0 for an
// all-zero group), stored as the UE8M0 byte e + 127; code = cvt.rn.satfinite
// E4M3(x * 2^-e).  The four bytes of a row inside one 128-wide K block form
// one 32-bit word (group 4kb + j in byte j), words at sf[kb * ldsf + row].

// e for a group with max-abs amax.  amax = (1 + m / 2^23) * 2^E for a normal
// amax and 448 = 1.75 * 2^8, so e = E - 8 when the significand is at most
// 1.75 and E - 7 above it; a subnormal amax is below 448 * 2^-127 and clamps.
__device__ __forceinline__ int mx_exponent(float amax) {
  if (amax == 0.0f) return 0;
  const uint32_t bits = __float_as_uint(amax);
  const int biased = static_cast<int>(bits >> 23);
  if (biased == 0) return -127;
  const int e = biased - 127 - 8 + ((bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  return e < -127 ? -127 : e;   // e <= 120 for any finite amax
}

// One warp per row and 1024-column chunk (lane l: the 32 columns of group l,
// 64 or 128 contiguous bytes), 8 rows per CTA.  The exponent words of the 8
// rows are gathered in shared memory and written as 32-byte runs.
template <typename TIn>
__global__ void __launch_bounds__(256) mx_quant_1x32_kernel(const TIn* __restrict__ x, int64_t R,
                                                            int64_t K, int64_t ldx,
                                                            uint8_t* __restrict__ q, int64_t ldq,
                                                            uint32_t* __restrict__ sf,
                                                            int64_t ldsf) {
  constexpr int kV = Vec16<TIn>::kN;       // elements per 16-byte load
  constexpr int kLoads = 32 / kV;
  __shared__ uint32_t words[8][8];         // [128-column block of the chunk][row of the CTA]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  const int64_t col = static_cast<int64_t>(blockIdx.y) * 1024 + lane * 32;
  uint32_t ebyte = 0;
  if (r < R && col < K) {
    const TIn* src = x + r * ldx + col;
    uint4 v[kLoads];
#pragma unroll
    for (int i = 0; i < kLoads; ++i) v[i] = ld_stream16(src + i * kV);
    float f[32];
#pragma unroll
    for (int i = 0; i < kLoads; ++i) {
      float w[kV];
      Vec16<TIn>::widen(v[i], w);
#pragma unroll
      for (int j = 0; j < kV; ++j) f[i * kV + j] = w[j];
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
    const int e = mx_exponent(amax);
    const float mult = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);   // 2^-e, exact
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = e4m3x4(f + 4 * j, mult);
    uint4* dst = reinterpret_cast<uint4*>(q + r * ldq + col);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    ebyte = static_cast<uint32_t>(e + 127);
  }
  // lanes 4j .. 4j+3 hold the four groups of 128-column block j
  const uint32_t b1 = __shfl_down_sync(0xffffffffu, ebyte, 1);
  const uint32_t b2 = __shfl_down_sync(0xffffffffu, ebyte, 2);
  const uint32_t b3 = __shfl_down_sync(0xffffffffu, ebyte, 3);
  if ((lane & 3) == 0) words[lane >> 2][warp] = ebyte | (b1 << 8) | (b2 << 16) | (b3 << 24);
  __syncthreads();
  if (threadIdx.x < 64) {
    const int kbl = threadIdx.x >> 3, rr = threadIdx.x & 7;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + rr;
    const int64_t kb = static_cast<int64_t>(blockIdx.y) * 8 + kbl;
    if (row < R && kb * 128 < K) sf[kb * ldsf + row] = words[kbl][rr];
  }
}

}  // namespace fp8bs
