// Block-scaled FP8 GEMM with promotion of every 128-deep K-slab into FP32
// registers on CUDA cores.
//
// Method: "Should Fixing Deepseek Take 60 Steps?", Figure 6 passage (Fprop,
// Dgrad, Wgrad in FP8; FP8 inputs, BF16 / FP32 outputs) and Figure 7 (a)
// passage (1x128 activation tiles, 128x128 weight blocks); untitled page at
// jp-study.kr, Figure 7 (b) passage (partial sums promoted to FP32 on CUDA
// cores with the scales applied; MMA and promotion overlap so the tensor cores
// stay busy).
//
// This single-CTA kernel serves the grouped (MoE expert) GEMM, whose experts
// are padded to 128 rows: a 256-row pair tile would straddle two experts, and
// the pair form that loads zeros for such halves measured slower (its
// block-scale promotion spills at the register limit).  The dense GEMM runs on
// the CTA-pair kernel (gemm_pair_kernel.cuh), which reuses the helpers here.
//
// B300 design (one CTA per SM, persistent):
//   warp 0      TMA producer: A tile 128x128 B and B tile 256x128 B per K-slab,
//               128-byte swizzle, into a kStages-deep shared-memory ring.
//   warp 1      MMA issuer: 4 x tcgen05.mma kind::f8f6f4 (M=128, N=256, K=32)
//               per slab into one of two TMEM slab buffers (256 columns each);
//               commits release the smem stage and publish the slab.
//   warps 2,3   scale loaders: every slab's A and B scales into a shared-memory
//               ring (one entry per operand stage) with cp.async, ahead of
//               the promotion warps
//   warps 4..11 promotion + epilogue: tcgen05.ld the slab (32 rows x 128
//               columns per warp), acc += P * (sa[row] * sb) in FP32 registers
//               (packed f32x2 FMAs), release the TMEM buffer; after the last
//               slab convert and store the 128 x 256 output tile.
// The double-buffered TMEM slab lets the tensor cores run slab k+1 while the
// CUDA cores promote slab k -- the overlap the pages get from two WGMMA
// warpgroups on H800.
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

#include "ptx.cuh"

namespace fp8bs {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 128;  // one promotion slab, one scale group
constexpr int kStages = 4;
constexpr int kStageABytes = kBM * kBK;
constexpr int kStageBBytes = kBN * kBK;
constexpr int kStageBytes = kStageABytes + kStageBBytes;
constexpr int kTmemCols = 512;         // two slab buffers of kBN columns
constexpr int kGemmThreads = 384;      // 3 warpgroups
constexpr int kEpiWarps = 8;
// Register split: launch budget 168 x 384; the producer warpgroup gives up all
// but 56 per thread so the two promotion warpgroups can hold 224 each
// (128 x 56 + 256 x 224 = 64512 = 168 x 384).
constexpr uint32_t kProducerRegs = 56;
constexpr uint32_t kEpilogueRegs = 224;
static_assert(128 * kProducerRegs + 256 * kEpilogueRegs <= 168 * kGemmThreads,
              "register split exceeds the launch budget");
constexpr int kMaxExperts = 1024;

enum SbKind : int { kSbBlock = 0, kSbPerCol = 1 };
constexpr int kEpiStageBytes = 32 * 64;   // one warp's output chunk: 32 rows x 64 B
constexpr int kScaleThreads = 64;         // warps 2 and 3: the scale loaders

struct GemmParams {
  int32_t M;            // rows of A / C (M_cap for the grouped call)
  int32_t N;
  int32_t KB;           // K / 128
  int32_t num_m_tiles;
  int32_t num_n_tiles;
  int32_t E;            // experts (1 for the dense call)
  const float* sa;      // sa[kb*ldsa + row]
  int64_t ldsa;
  const float* sb;
  int64_t sb_k_stride;  // block modes: element stride per K-slab
  int64_t sb_n_stride;  // block modes: element stride per 128-column block
  int64_t ldsb;         // per-column mode: stride per K-slab
  int64_t sb_e_stride;  // per expert
  void* C;
  int64_t ldc;          // elements
  const int32_t* offsets;  // grouped: device offsets[E+1]
  // pair kernel work units: tiles [0, full_tiles) whole, then each remaining
  // tile as `splits` K-ranges whose FP32 partials go to a workspace
  int32_t full_tiles;
  int32_t splits;
  int32_t units;
  int32_t group_m;   // pair kernel: m tiles per group of the tile walk (>= 1)
  int32_t k_order;   // pair kernel, whole tiles: kKOrderForward or kKOrderSerpentine
};

// Order in which the pair kernel's whole tiles take their K slabs.
// Serpentine: every odd wave of the persistent walk takes them last to first,
// so a wave starts on the slabs of its A panels that the previous wave (same
// m group) read last, still in L2 when a wave's panels are too large to stay
// there whole (the K = 18432 Dgrad: 0.453 -> 0.416 ms, DRAM reads 700 -> 481
// MB, measured).  The promotion's FP32 sum then runs over the slabs in that
// order.
constexpr int32_t kKOrderForward = 0;
constexpr int32_t kKOrderSerpentine = 1;

struct GemmSmem {
  alignas(1024) unsigned char epi_stage[kEpiWarps][kEpiStageBytes];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t bad_offsets;
  int32_t num_tiles;   // dense: m tiles x n tiles; grouped: tile_base[E]
  int32_t offsets[kMaxExperts + 1];
  // grouped: first tile index of each expert; expert e owns tiles
  // tile_base[e] .. tile_base[e+1]-1, its m tiles fastest, then its n tiles
  int32_t tile_base[kMaxExperts + 1];
  // scale ring, one entry per operand stage: warps 2 and 3 copy each slab's
  // A scales (the tile's 128 rows) and B scales (its 256 columns, per-column
  // mode, or its two column blocks, block mode) ahead of the promotion warps
  uint64_t scl_full[kStages];   // the copies of an entry have landed (64 arrivals)
  uint64_t scl_free[kStages];   // the promotion warps read it (kEpiWarps arrivals)
  alignas(16) float scl_sa[kStages][kBM];
  alignas(16) float scl_sb[kStages][kBN];
};

constexpr size_t kGemmSmemBytes =
    1024 /* alignment slack */ + static_cast<size_t>(kStages) * kStageBytes + sizeof(GemmSmem);

struct TileCoord {
  int32_t m0, n0, e;
};

// Output tile t of the persistent walk: expert by expert, and within an
// expert its m tiles fastest, so an expert's rows of A are re-read from L2
// across its n tiles instead of from HBM.
__device__ __forceinline__ TileCoord tile_coord(int t, const GemmParams& p, const GemmSmem& sm) {
  TileCoord c;
  // owner: the last e with tile_base[e] <= t (it has at least one tile)
  int lo = 0, hi = p.E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sm.tile_base[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int l = t - sm.tile_base[lo];
  const int mte = (sm.offsets[lo + 1] - sm.offsets[lo]) / kBM;
  c.e = lo;
  c.m0 = sm.offsets[lo] + (l % mte) * kBM;
  c.n0 = (l / mte) * kBN;
  return c;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// acc[j] += P[j] * scale for 32 columns held as 32 raw fp32 words.
__device__ __forceinline__ void promote32(float2* acc, const uint32_t (&r)[32], float2 sc2) {
#pragma unroll
  for (int i = 0; i < 16; ++i)
    acc[i] = __ffma2_rn(make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])),
                        sc2, acc[i]);
}

// acc[j] += (P[j] * sb[j]) * sa for 32 columns; sb[] read from shared memory
// (every lane reads the same addresses: broadcast).
__device__ __forceinline__ void promote32_percol(float2* acc, const uint32_t (&r)[32],
                                                 const float* sbv, float2 sa2) {
  const float4* sb4 = reinterpret_cast<const float4*>(sbv);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 b = sb4[i];
    const float2 p0 = make_float2(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]));
    const float2 p1 = make_float2(__uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
    acc[2 * i] = __ffma2_rn(__fmul2_rn(p0, make_float2(b.x, b.y)), sa2, acc[2 * i]);
    acc[2 * i + 1] = __ffma2_rn(__fmul2_rn(p1, make_float2(b.z, b.w)), sa2, acc[2 * i + 1]);
  }
}

// Write box c of this warp's accumulators (32 rows x 64 bytes: FP32 columns
// 16c .. 16c+15, or BF16 rounded to nearest even, columns 32c .. 32c+31) into
// 2 KB of shared memory at dst: row `lane` at 64 * lane, its 16-byte unit j at
// position j ^ ((lane >> 1) & 3) (the 64-byte swizzle of the output maps).
template <bool kBf16>
__device__ __forceinline__ void stage_box(const float2* acc, uint32_t dst0, int lane, int c) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {   // 16-byte unit j of this row's 64 bytes
    const uint32_t dst = dst0 + static_cast<uint32_t>(lane) * 64u +
                         ((static_cast<uint32_t>(j) ^ ((static_cast<uint32_t>(lane) >> 1) & 3u)) << 4);
    if constexpr (kBf16) {
      const int k = c * 16 + 4 * j;   // float2 index of column c*32 + 8j
      st_shared_v4(dst, make_uint4(pack_bf16x2(acc[k].x, acc[k].y),
                                   pack_bf16x2(acc[k + 1].x, acc[k + 1].y),
                                   pack_bf16x2(acc[k + 2].x, acc[k + 2].y),
                                   pack_bf16x2(acc[k + 3].x, acc[k + 3].y)));
    } else {
      // two 8-byte stores straight from the accumulator register pairs
      const int k = c * 8 + 2 * j;    // float2 index of column c*16 + 4j
      st_shared_v2f(dst, acc[k]);
      st_shared_v2f(dst + 8, acc[k + 1]);
    }
  }
}

// Store this warp's 32 rows x kCols accumulator columns (row `lane` per
// thread) through a 2 KB shared buffer and 64-byte-wide TMA boxes at (col, row)
// of `tmap`: FP32 (16 columns per box) or BF16 rounded to nearest even (32).
// kAdd: the FP32 boxes are added into the existing values instead.  kCols:
// accumulator columns of the warp (128, or 64 for the 128-wide pair tile).
template <bool kBf16, bool kAdd = false, int kCols = 128>
__device__ __forceinline__ void store_rows_tma(const float2* acc, uint32_t stg, int lane,
                                               const CUtensorMap* tmap, int col, int row) {
  constexpr int kChunkCols = kBf16 ? 32 : 16;   // 64 bytes of output per row
#pragma unroll
  for (int c = 0; c < kCols / kChunkCols; ++c) {
    // the previous bulk store of this buffer must have read it
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
    stage_box<kBf16>(acc, stg, lane, c);
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
      if constexpr (kAdd)
        tma_reduce_add_2d(tmap, col + c * kChunkCols, row, stg);
      else
        tma_store_2d(tmap, col + c * kChunkCols, row, stg);
      bulk_commit_group();
    }
  }
}

// Park this warp's 32 rows x kCols accumulator columns in shared memory (one
// 2 KB box after the other from `park`) and issue their TMA stores as one
// bulk group without waiting for them: the stores drain while the warp goes on
// with its next tile.  The previous parked group must have been read before
// the area is rewritten; the wait at the start covers it (and every earlier
// store of this thread).
template <bool kBf16, bool kAdd = false, int kCols = 64>
__device__ __forceinline__ void park_rows_tma(const float2* acc, uint32_t park, int lane,
                                              const CUtensorMap* tmap, int col, int row) {
  constexpr int kChunkCols = kBf16 ? 32 : 16;
  constexpr int kBoxes = kCols / kChunkCols;
  if (lane == 0) bulk_wait_read_all();
  __syncwarp();
#pragma unroll
  for (int c = 0; c < kBoxes; ++c) stage_box<kBf16>(acc, park + c * 2048u, lane, c);
  fence_proxy_async_shared();
  __syncwarp();
  if (lane == 0) {
#pragma unroll
    for (int c = 0; c < kBoxes; ++c) {
      if constexpr (kAdd)
        tma_reduce_add_2d(tmap, col + c * kChunkCols, row, park + c * 2048u);
      else
        tma_store_2d(tmap, col + c * kChunkCols, row, park + c * 2048u);
    }
    bulk_commit_group();
  }
}

template <int kSb, bool kOutBf16>
__global__ void __launch_bounds__(kGemmThreads, 1)
    fp8bs_gemm_kernel(const __grid_constant__ GemmParams p,
                      const __grid_constant__ CUtensorMap tmap_a,
                      const __grid_constant__ CUtensorMap tmap_b,
                      const __grid_constant__ CUtensorMap tmap_c) {
  extern __shared__ __align__(1024) unsigned char gemm_smem_raw[];
  // 1024-byte aligned operand ring (the 128-byte swizzle atoms need it)
  const uint32_t raw_addr = smem_u32(gemm_smem_raw);
  unsigned char* ring = gemm_smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  GemmSmem& sm = *reinterpret_cast<GemmSmem*>(ring + static_cast<size_t>(kStages) * kStageBytes);
  const uint32_t ring_addr = smem_u32(ring);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &sm.abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.tfull[b], 1);
      mbar_init(&sm.tempty[b], kEpiWarps);
    }
    for (int e = 0; e < kStages; ++e) {
      mbar_init(&sm.scl_full[e], kScaleThreads);
      mbar_init(&sm.scl_free[e], kEpiWarps);
    }
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    sm.bad_offsets = 0;
    sm.num_tiles = p.num_m_tiles * p.num_n_tiles;
    fence_mbarrier_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
    tma_prefetch_desc(&tmap_c);
  }
  {
    // Stage and validate the expert offsets (every CTA, so none depends on another).
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) sm.offsets[i] = p.offsets[i];
    __syncthreads();
    if (warp == 0) {
      // Validate, and scan the per-expert tile counts into tile_base: each
      // lane takes a contiguous chunk of experts, then a warp prefix sum.
      const int chunk = (p.E + 31) / 32;
      const int e0 = lane * chunk < p.E ? lane * chunk : p.E;
      const int e1 = e0 + chunk < p.E ? e0 + chunk : p.E;
      bool ok = true;
      int count = 0;
      for (int e = e0; e < e1; ++e) {
        const int rows = sm.offsets[e + 1] - sm.offsets[e];
        ok = ok && rows >= 0 && (sm.offsets[e + 1] % kBM) == 0;
        count += (rows / kBM) * p.num_n_tiles;
      }
      ok = __all_sync(0xffffffffu, ok) && sm.offsets[0] == 0 && sm.offsets[p.E] <= p.M;
      int incl = count;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int run = incl - count;
      for (int e = e0; e < e1; ++e) {
        sm.tile_base[e] = run;
        run += ((sm.offsets[e + 1] - sm.offsets[e]) / kBM) * p.num_n_tiles;
      }
      if (lane == 31) sm.tile_base[p.E] = incl;
      if (lane == 0) {
        if (!ok) {
          sm.bad_offsets = 1;
          if (blockIdx.x == 0) atomicOr(&g_device_error, kDevErrBadOffsets);
        }
      }
      if (lane == 31) sm.num_tiles = ok ? incl : 0;
    }
  }
  if (warp == 1) tmem_alloc(&sm.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sm.tmem_base;
  const bool skip_all = sm.bad_offsets != 0;
  // (re-read per tile rather than held in a register: the promotion warps
  // have none to spare)
#define FP8BS_NUM_TILES (sm.num_tiles)

  if (warp < 4) {
    regs_dealloc<kProducerRegs>();
  if (!skip_all && warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA
    const uint64_t policy = l2_policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0, parity_mask = 0;
    for (int t = blockIdx.x; t < FP8BS_NUM_TILES; t += gridDim.x) {
      const TileCoord tc = tile_coord(t, p, sm);
      for (int kb = 0; kb < p.KB; ++kb) {
        if (!bounded_wait(&sm.empty[stage], phase ^ 1u, abort_flag)) goto producer_done;
        mbar_arrive_expect_tx(&sm.full[stage], kStageBytes);
        const uint32_t sa_addr = ring_addr + stage * kStageBytes;
        tma_load_2d(sa_addr, &tmap_a, kb * kBK, tc.m0, &sm.full[stage], policy);
        tma_load_3d(sa_addr + kStageABytes, &tmap_b, kb * kBK, tc.n0, tc.e, &sm.full[stage],
                    policy);
        issued_mask |= 1u << stage;
        parity_mask = (parity_mask & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  producer_done:
    // Every load issued must land before the CTA may exit.
    for (int s = 0; s < kStages; ++s)
      if (issued_mask & (1u << s))
        bounded_wait_noabort(&sm.full[s], (parity_mask >> s) & 1u, kSpinLimitNs);
  } else if (!skip_all && warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA
    constexpr uint32_t idesc = idesc_e4m3_f32(kBM, kBN);
    int stage = 0, buf = 0;
    uint32_t phase = 0, tphase = 0;
    bool issued = false;
    for (int t = blockIdx.x; t < FP8BS_NUM_TILES; t += gridDim.x) {
      const TileCoord tc = tile_coord(t, p, sm);
      for (int kb = 0; kb < p.KB; ++kb) {
        if (!bounded_wait(&sm.full[stage], phase, abort_flag)) goto mma_done;
        if (!bounded_wait(&sm.tempty[buf], tphase ^ 1u, abort_flag)) goto mma_done;
        tc_fence_after();
        const uint32_t a_addr = ring_addr + stage * kStageBytes;
        const uint64_t adesc = smem_desc_k_sw128(a_addr);
        const uint64_t bdesc = smem_desc_k_sw128(a_addr + kStageABytes);
        const uint32_t d = tmem_base + static_cast<uint32_t>(buf * kBN);
#pragma unroll
        for (int kk = 0; kk < kBK / 32; ++kk)  // 32 bytes = 32 E4M3 values per MMA
          mma_f8f6f4(d, adesc + 2u * kk, bdesc + 2u * kk, idesc, kk > 0 ? 1u : 0u);
        mma_commit(&sm.empty[stage]);
        mma_commit(&sm.tfull[buf]);
        issued = true;
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
        if (++buf == 2) {
          buf = 0;
          tphase ^= 1u;
        }
      }
    }
  mma_done:
    if (issued) {  // all MMAs must finish before TMEM is released
      mma_commit(&sm.drain);
      bounded_wait_noabort(&sm.drain, 0, kSpinLimitNs);
    }
  } else if (!skip_all && warp >= 2) {
    // ---------------------------------------------------------------- scales
    // Every slab's scales into the next free ring entry with asynchronous
    // copies that arrive on the entry's barrier when they land: thread lt
    // copies the A scales of rows lt and 64 + lt, and 4 B scales (per-column
    // mode) or one column block's scale (block mode, threads 0 and 1).  Rows
    // past M and columns past N get zeros.
    const int lt = static_cast<int>(threadIdx.x) - 64;
    int e = 0;
    uint32_t ephase = 0;
    for (int t = blockIdx.x; t < FP8BS_NUM_TILES; t += gridDim.x) {
      const TileCoord tc = tile_coord(t, p, sm);
      const float* sbe = p.sb + static_cast<int64_t>(tc.e) * p.sb_e_stride;
      const int cb = tc.n0 / 128 + (lt < kBN / 128 ? lt : 0);
      const bool cb_ok = cb * 128 < p.N;
      const float* sb_k = sbe + static_cast<int64_t>(cb_ok ? cb : 0) * p.sb_n_stride;
      for (int kb = 0; kb < p.KB; ++kb) {
        if (!bounded_wait(&sm.scl_free[e], ephase ^ 1u, abort_flag)) goto scales_done;
        const float* sa_k = p.sa + static_cast<int64_t>(kb) * p.ldsa;
#pragma unroll
        for (int r = lt; r < kBM; r += kScaleThreads) {
          const bool ok = tc.m0 + r < p.M;
          cp_async_4(smem_u32(&sm.scl_sa[e][r]), sa_k + (ok ? tc.m0 + r : 0), ok ? 4u : 0u);
        }
        if constexpr (kSb == kSbPerCol) {
#pragma unroll
          for (int j = lt * 4; j < kBN; j += 4 * kScaleThreads) {
            // N is a multiple of 16: columns n0+j .. n0+j+3 are all in or all out
            const bool ok = tc.n0 + j < p.N;
            cp_async_16(smem_u32(&sm.scl_sb[e][j]),
                        sbe + static_cast<int64_t>(kb) * p.ldsb + (ok ? tc.n0 + j : 0),
                        ok ? 16u : 0u);
          }
        } else {
          if (lt < kBN / 128)
            cp_async_4(smem_u32(&sm.scl_sb[e][lt]), sb_k + static_cast<int64_t>(kb) * p.sb_k_stride,
                       cb_ok ? 4u : 0u);
        }
        cp_async_arrive(&sm.scl_full[e]);
        if (++e == kStages) {
          e = 0;
          ephase ^= 1u;
        }
      }
    }
  scales_done:
    cp_async_wait_all();   // this thread's copies have landed before the CTA may exit
  }
  } else {
    regs_alloc<kEpilogueRegs>();
    if (!skip_all) {
    // ------------------------------------------------- promotion + epilogue
    const int g = warp & 3;          // TMEM lane group (rows 32g .. 32g+31)
    const int h = (warp - 4) >> 2;   // column half (0: 0..127, 1: 128..255)
    int buf = 0;
    uint32_t tphase = 0;
    // scale ring position: entry sk % kStages, parity sk / kStages
    static_assert((kStages & (kStages - 1)) == 0, "ring position arithmetic");
    uint32_t sk = 0;
    for (int t = blockIdx.x; t < FP8BS_NUM_TILES; t += gridDim.x) {
      const TileCoord tc = tile_coord(t, p, sm);
      const int col0 = tc.n0 + h * 128;
      float2 acc[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = make_float2(0.0f, 0.0f);

      for (int kb = 0; kb < p.KB; ++kb) {
        // the slab's scales, copied ahead into the ring by warps 2 and 3 (rows
        // past M and columns past N carry zero scales, so no guard is needed)
        const uint32_t se = sk & (kStages - 1);
        if (!bounded_wait(&sm.tfull[buf], tphase, abort_flag)) goto epilogue_done;
        if (!bounded_wait(&sm.scl_full[se], sk / kStages, abort_flag)) goto epilogue_done;
        const float sa = sm.scl_sa[se][g * 32 + lane];
        float sb = 0.0f;
        if constexpr (kSb == kSbBlock) sb = sm.scl_sb[se][h];
        tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(g * 32) << 16) +
                               static_cast<uint32_t>(buf * kBN + h * 128);
        uint32_t ra[32], rb[32];
        tmem_ld32(taddr, ra);
        tmem_wait_ld(ra);
        if constexpr (kSb == kSbBlock) {
          const float sc = sa * sb;
          const float2 sc2 = make_float2(sc, sc);
#pragma unroll
          for (int c = 0; c < 4; c += 2) {
            tmem_ld32(taddr + (c + 1) * 32, rb);
            promote32(acc + c * 16, ra, sc2);
            tmem_wait_ld(rb);
            if (c + 2 < 4) tmem_ld32(taddr + (c + 2) * 32, ra);
            promote32(acc + (c + 1) * 16, rb, sc2);
            if (c + 2 < 4) tmem_wait_ld(ra);
          }
        } else {
          const float2 sa2 = make_float2(sa, sa);
          const float* sbs = &sm.scl_sb[se][h * 128];
#pragma unroll
          for (int c = 0; c < 4; c += 2) {
            tmem_ld32(taddr + (c + 1) * 32, rb);
            promote32_percol(acc + c * 16, ra, sbs + c * 32, sa2);
            tmem_wait_ld(rb);
            if (c + 2 < 4) tmem_ld32(taddr + (c + 2) * 32, ra);
            promote32_percol(acc + (c + 1) * 16, rb, sbs + (c + 1) * 32, sa2);
            if (c + 2 < 4) tmem_wait_ld(ra);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sm.tempty[buf]);
          mbar_arrive(&sm.scl_free[se]);
        }
        if (++buf == 2) {
          buf = 0;
          tphase ^= 1u;
        }
        sk = (sk + 1) & (2 * kStages - 1);
      }
      // ---- epilogue: this warp's 32 rows x 128 columns, through TMA stores
      // (rows of a tile never straddle two experts: expert ranges are whole tiles)
      store_rows_tma<kOutBf16>(acc, smem_u32(&sm.epi_stage[warp - 4][0]), lane, &tmap_c, col0,
                               tc.m0 + g * 32);
    }
  epilogue_done:
    if (lane == 0) bulk_wait_all();   // this warp's output stores are complete
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

#undef FP8BS_NUM_TILES

constexpr size_t kProbeSmemBytes = 1024 + (128 + 256) * 128;   // alignment slack + A + B

// Accumulation probe: D[128][256] = A[128][K] * B[256][K]^T over raw E4M3
// codes (no scales), K = 32 * n_mma <= 128, with n_mma tcgen05 kind::f8f6f4
// MMAs (M=128, N=256, K=32) accumulating in TMEM, read back as raw FP32.  The
// operands are copied into shared memory in the 128-byte-swizzled K-major
// layout the MMA descriptors describe (row r's 16-byte chunk j at chunk
// position j ^ (r & 7)); bytes past K are zero.  One CTA of 128 threads.
__global__ void __launch_bounds__(128, 1) fp8bs_mma_probe_kernel(const uint8_t* __restrict__ a,
                                                                 const uint8_t* __restrict__ b,
                                                                 int K, float* __restrict__ d) {
  extern __shared__ __align__(1024) unsigned char probe_smem_raw[];   // kProbeSmemBytes
  unsigned char* op = probe_smem_raw + ((1024u - (smem_u32(probe_smem_raw) & 1023u)) & 1023u);
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < (128 + 256) * 8; i += 128) {   // 16-byte chunks
    const int r = i / 8, j = i % 8;
    const uint8_t* src = r < 128 ? a + static_cast<int64_t>(r) * K : b + static_cast<int64_t>(r - 128) * K;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t v = 0;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int k = j * 16 + q * 4 + t;
        if (k < K) v |= static_cast<uint32_t>(src[k]) << (8 * t);
      }
      w[q] = v;
    }
    const int rr = r < 128 ? r : r - 128;
    unsigned char* base = op + (r < 128 ? 0 : 128 * 128);
    *reinterpret_cast<uint4*>(base + rr * 128 + ((j ^ (rr & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (tid == 0) {
    mbar_init(&bar, 1);
    abort_s = 0;
    fence_mbarrier_init();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 0) tmem_alloc(&tmem_base_s, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base_s;
  if (tid == 0) {
    const uint64_t adesc = smem_desc_k_sw128(smem_u32(op));
    const uint64_t bdesc = smem_desc_k_sw128(smem_u32(op + 128 * 128));
    for (int kk = 0; kk < K / 32; ++kk)
      mma_f8f6f4(tb, adesc + 2u * kk, bdesc + 2u * kk, idesc_e4m3_f32(128, 256), kk > 0 ? 1u : 0u);
    mma_commit(&bar);
  }
  __syncwarp();
  const bool ok = bounded_wait(&bar, 0, &abort_s);
  tc_fence_after();
  if (ok) {
    uint32_t r[32];
#pragma unroll 1
    for (int c = 0; c < 256; c += 32) {
      tmem_ld32(tb + (static_cast<uint32_t>(warp * 32) << 16) + c, r);
      tmem_wait_ld(r);
      float* row = d + static_cast<int64_t>(warp * 32 + lane) * 256 + c;
#pragma unroll
      for (int i = 0; i < 32; ++i) row[i] = __uint_as_float(r[i]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tb, 256);
}

// One CTA waits on a barrier that nothing arrives at, with a time limit; the
// wait gives up, records a timeout in the device error word and returns.
__global__ void fp8bs_timeout_probe_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) bounded_wait_noabort(&bar, 0, limit_ns);
}

}  // namespace fp8bs
