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
// One CTA per (128 tokens) x (256 bytes of channels): the block is staged in
// shared memory with coalesced 16-byte row loads, then each thread owns one
// channel and a contiguous run of tokens: it reduces the amax (combined across
// the token parts through shared memory), quantizes, and writes its tokens as
// contiguous 16-byte runs of the transposed output.
template <typename TIn>
__global__ void __launch_bounds__(256) quant_128x1_kernel(const TIn* __restrict__ x, int64_t C,
                                                          int64_t ldx, uint8_t* __restrict__ qT,
                                                          int64_t ldq, float* __restrict__ s,
                                                          int64_t lds) {
  constexpr int kVec = Vec16<TIn>::kN;
  constexpr int kCB = 256 / sizeof(TIn);       // channels per CTA (256 bytes per row)
  constexpr int kVecPerRow = kCB / kVec;       // 16
  constexpr int kRowsPerPass = 256 / kVecPerRow;
  constexpr int kLoads = 128 / kRowsPerPass;   // 16-byte loads per thread
  constexpr int kParts = 256 / kCB;            // token parts per channel
  constexpr int kTok = 128 / kParts;           // tokens per thread
  __shared__ __align__(16) TIn tile[128][kCB];
  __shared__ float part_amax[kParts][kCB];

  const int64_t tb = blockIdx.y;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kCB;
  const int tid = threadIdx.x;
  {
    const int vc = tid % kVecPerRow;
    const int r0 = tid / kVecPerRow;
    const int64_t col = c0 + vc * kVec;
    uint4 v[kLoads];
#pragma unroll
    for (int i = 0; i < kLoads; ++i) {
      const int64_t row = tb * 128 + r0 + i * kRowsPerPass;
      v[i] = (col < C) ? ld_stream16(x + row * ldx + col) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kLoads; ++i)
      *reinterpret_cast<uint4*>(&tile[r0 + i * kRowsPerPass][vc * kVec]) = v[i];
  }
  __syncthreads();

  const int c = tid % kCB;
  const int part = tid / kCB;
  float f[kTok];
  float amax = 0.0f;
#pragma unroll
  for (int t = 0; t < kTok; ++t) {
    f[t] = widen1<TIn>(tile[part * kTok + t][c]);
    amax = fmaxf(amax, fabsf(f[t]));
  }
  part_amax[part][c] = amax;
  __syncthreads();
#pragma unroll
  for (int p = 0; p < kParts; ++p) amax = fmaxf(amax, part_amax[p][c]);
  float sc, r;
  tile_scale(amax, sc, r);
  if (c0 + c < C) {
    uint8_t* dst = qT + (c0 + c) * ldq + tb * 128 + part * kTok;
#pragma unroll
    for (int t = 0; t < kTok; t += 16) {
      uint4 o;
      o.x = e4m3x4(f + t, r);
      o.y = e4m3x4(f + t + 4, r);
      o.z = e4m3x4(f + t + 8, r);
      o.w = e4m3x4(f + t + 12, r);
      *reinterpret_cast<uint4*>(dst + t) = o;
    }
    if (part == 0) s[tb * lds + c0 + c] = sc;
  }
}

// -------------------------------------------------------------- 128 x 128
// One CTA per 128 x 128 block.  Each thread loads its 16-byte vectors once;
// the block amax is reduced through warp shuffles and shared memory.  The
// row-major codes are written from registers; the transposed copy is read
// column-wise from the staged block (dynamic shared memory: 32 KB for bf16,
// 64 KB for fp32).  Both copies come from the same multiply and conversion.
template <typename TIn>
__global__ void __launch_bounds__(256) quant_128x128_kernel(const TIn* __restrict__ w,
                                                            int64_t ldw, uint8_t* __restrict__ q,
                                                            int64_t ldq, uint8_t* __restrict__ qT,
                                                            int64_t ldqT, float* __restrict__ s,
                                                            int64_t lds) {
  constexpr int kVec = Vec16<TIn>::kN;
  constexpr int kVecPerRow = 128 / kVec;       // 16 (bf16) or 32 (fp32)
  constexpr int kRowsPerPass = 256 / kVecPerRow;
  constexpr int kLoads = 128 / kRowsPerPass;   // 8 or 16
  extern __shared__ __align__(16) unsigned char dyn_smem[];
  TIn(*tile)[128] = reinterpret_cast<TIn(*)[128]>(dyn_smem);
  __shared__ float warp_amax[8];

  const int64_t rb = blockIdx.y, cb = blockIdx.x;
  const int tid = threadIdx.x;
  const int vc = tid % kVecPerRow;
  const int r0 = tid / kVecPerRow;
  const TIn* src = w + rb * 128 * ldw + cb * 128 + vc * kVec;
  uint4 v[kLoads];
#pragma unroll
  for (int i = 0; i < kLoads; ++i) v[i] = ld_stream16(src + (r0 + i * kRowsPerPass) * ldw);

  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < kLoads; ++i) {
    float f[kVec];
    Vec16<TIn>::widen(v[i], f);
#pragma unroll
    for (int j = 0; j < kVec; ++j) amax = fmaxf(amax, fabsf(f[j]));
    if (qT != nullptr)
      *reinterpret_cast<uint4*>(&tile[r0 + i * kRowsPerPass][vc * kVec]) = v[i];
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

  if (q != nullptr) {
    uint8_t* dst = q + rb * 128 * ldq + cb * 128 + vc * kVec;
#pragma unroll
    for (int i = 0; i < kLoads; ++i) {
      float f[kVec];
      Vec16<TIn>::widen(v[i], f);
      uint8_t* d = dst + (r0 + i * kRowsPerPass) * ldq;
      if constexpr (kVec == 8) {
        *reinterpret_cast<uint2*>(d) = make_uint2(e4m3x4(f, r), e4m3x4(f + 4, r));
      } else {
        *reinterpret_cast<uint32_t*>(d) = e4m3x4(f, r);
      }
    }
  }
  if (qT != nullptr) {
    // thread -> (column c, 64 consecutive rows)
    const int c = tid & 127;
    const int part = tid >> 7;
    uint8_t* d = qT + (cb * 128 + c) * ldqT + rb * 128 + part * 64;
#pragma unroll
    for (int t = 0; t < 64; t += 16) {
      float f[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) f[j] = widen1<TIn>(tile[part * 64 + t + j][c]);
      uint4 o;
      o.x = e4m3x4(f, r);
      o.y = e4m3x4(f + 4, r);
      o.z = e4m3x4(f + 8, r);
      o.w = e4m3x4(f + 12, r);
      *reinterpret_cast<uint4*>(d + t) = o;
    }
  }
}

}  // namespace fp8bs
