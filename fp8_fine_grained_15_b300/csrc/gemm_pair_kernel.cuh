// Block-scaled FP8 GEMM on CTA pairs (tcgen05 cta_group::2): the dense path of
// fp8bs_gemm.
//
// Same method as gemm_kernel.cuh ("Should Fixing Deepseek Take 60 Steps?",
// Figure 6 and Figure 7 (a) passages; untitled page at jp-study.kr, Figure 7 (b)
// passage): every 128-deep K-slab is multiplied on the tensor cores and its
// partial sum is promoted into FP32 registers on CUDA cores with the row scale
// and the column-block (or column) scale of that slab.
//
// Why pairs: with one CTA per 128x256 tile each SM pulls 48 KB of operands per
// slab from L2 and only four such stages fit in shared memory; measured, the
// TMA round trip (~2900 cycles at that load) then bounds the slab rate.  A
// cluster of two CTAs computes a 256 x BN tile with one pair MMA: each CTA
// stages its own 128 rows of A and one half (BN/2 rows) of B.
//
// Tile width BN: 256 (32 KB per SM and slab, a 6-stage ring of which the
// block modes keep 5 and the per-column mode 4, parking output in the rest,
// and two 256-column TMEM slab buffers) is what the library launches.  BN = 128 (24 KB, 8 stages, four
// 128-column buffers) compiles and passes the parity tests; pair MMAs with
// N = 128 stream at 97 % of the N = 256 rate in isolation, but with 45 % more
// operand bytes per FLOP the whole kernel measured 1.4-2x slower on the
// layer's GEMMs, so it is not instantiated.
//
// Roles (384 threads per CTA, both CTAs of the pair):
//   warp 0      TMA producer: this CTA's A rows and B half of each slab; the
//               loads complete on the even CTA's `full` barrier.
//   warp 1      even CTA only: issues 4 x tcgen05.mma.cta_group::2 (M=256,
//               N=256, K=32) per slab into one of two 256-column TMEM buffers,
//               then one commit that arrives on `done[stage]` in both CTAs:
//               the stage may be refilled and the TMEM slab may be read.
//   warps 2, 3  scale loaders: every slab's A scales (this CTA's 128 rows)
//               and B scales (the tile's columns or column blocks) into a
//               shared-memory ring, one entry per operand stage, with cp.async
//               that arrives on the entry's `scl_full` barrier.
//   warps 4..11 promotion + epilogue of this CTA's 128 rows (as in the
//               single-CTA kernel); each warp releases its TMEM columns by
//               arriving on the even CTA's `tmem_free` barrier (16 arrivals)
//               and its scale entry on `scl_free`.
//               The epilogue goes out through TMA stores: each warp writes a
//               32-row x 64-byte chunk of its rows into a 2 KB shared buffer
//               (64-byte swizzle, conflict-free) and one lane stores the box;
//               half of the tile is parked in ring stages given up for it
//               and drains during the next tile.
//               (Stores straight from registers, one row per lane, hit 32
//               cache lines per instruction: ~13k cycles per FP32 tile.)
#pragma once
#include "gemm_kernel.cuh"

namespace fp8bs {

constexpr int kPairTileM = 2 * kBM;             // rows of a pair tile
constexpr int kPairRingBytes = 6 * 32768;       // operand ring per CTA

// kPark: ring stages given up to park half of each warp's finished tile (its
// TMA stores then drain while the next tile runs).
template <int BN, int kPark = 0>
struct PairCfg {
  static_assert(BN == 128 || BN == 256, "pair tile width");
  static constexpr int kStageA = kBM * kBK;              // this CTA's 128 rows of A, one slab
  static constexpr int kStageB = (BN / 2) * kBK;         // this CTA's half of the B tile
  static constexpr int kStageBytes = kStageA + kStageB;
  static constexpr int kStages = kPairRingBytes / kStageBytes - kPark;   // 6 or 8, less kPark
  static constexpr int kBufs = kTmemCols / BN;           // TMEM slab buffers: 2 or 4
  static constexpr int kWarpCols = BN / 2;               // columns per promotion warp
  static constexpr int kChunks = kWarpCols / 32;         // x32 TMEM loads per warp and slab
  // parking area of a promotion warp: its share of the stages given up
  static constexpr int kParkWarpBytes = kPark * kStageBytes / kEpiWarps;
  // the last columns of a warp that fit its parking area (32 rows of
  // kOutBytes-byte outputs), in whole 64-byte boxes
  template <int kOutBytes>
  static constexpr int park_cols() {
    return kParkWarpBytes / (32 * kOutBytes) < kWarpCols ? kParkWarpBytes / (32 * kOutBytes)
                                                         : kWarpCols;
  }
};

// Ring stages each mode gives up for parking: the per-column mode (Wgrad:
// FP32 output, short K, the largest epilogue per slab) and the block modes
// (BF16 output: one stage parks half a tile; measured ~0.5 % on Fprop and
// Dgrad, two stages no better).
constexpr int kPairParkPerCol = 2;
constexpr int kPairParkBlock = 1;
// Scale ring of the pair kernel: warps 2 and 3 of each CTA load every slab's
// A and B scales into shared memory ahead of the promotion warps (one entry
// per operand stage, so both rings advance together), so that no global load
// latency lies on the promotion's path.
constexpr int kPairScaleThreads = 64;

// Register split of the pair kernel: its role warpgroup (TMA and MMA issue
// loops, scale loads) keeps 56 per thread and the promotion warpgroups 224
// (128 x 56 + 256 x 224 = 64512 = 168 x 384); no spills in either.
constexpr uint32_t kPairProducerRegs = 56;
constexpr uint32_t kPairEpilogueRegs = 224;
static_assert(128 * kPairProducerRegs + 256 * kPairEpilogueRegs <= 168 * kGemmThreads,
              "register split exceeds the launch budget");

template <int BN>
struct PairSmem {
  alignas(1024) unsigned char epi_stage[kEpiWarps][kEpiStageBytes];
  uint64_t full[PairCfg<BN>::kStages];   // even CTA: both CTAs' loads of a slab have landed
  uint64_t done[PairCfg<BN>::kStages];   // both CTAs: the slab's MMAs are complete
  uint64_t tmem_free[PairCfg<BN>::kBufs];  // even CTA: 16 promotion warps released a buffer
  uint64_t drain;
  uint64_t scl_full[PairCfg<BN>::kStages];   // this CTA: the scale loaders filled an entry
  uint64_t scl_free[PairCfg<BN>::kStages];   // this CTA: its promotion warps read an entry
  uint32_t tmem_base;
  int32_t abort_flag;
  // per slab, in a ring of one entry per operand stage: the A scales of this
  // CTA's 128 rows, and the B scales of the tile's BN columns (per-column
  // mode) or of its BN / 128 column blocks (block modes)
  alignas(16) float scl_sa[PairCfg<BN>::kStages][kBM];
  alignas(16) float scl_sb[PairCfg<BN>::kStages][BN];
};

template <int BN>
constexpr size_t pair_smem_bytes() {
  return 1024 /* alignment slack */ + static_cast<size_t>(kPairRingBytes) + sizeof(PairSmem<BN>);
}

// Output tile t of the walk -> (m tile, n tile): groups of p.group_m m tiles,
// within a group m fastest, then n.  A wave of clusters then covers about
// group_m x (clusters / group_m) tiles, so both its A and its B panels stay in
// L2 (with all m tiles in one group, the wave's A panels are all of A and are
// re-read from DRAM every wave when A and a wave's B exceed L2).
__device__ __forceinline__ void pair_tile_mn(int t, const GemmParams& p, int& mt, int& nt) {
  const int per_group = p.group_m * p.num_n_tiles;
  const int first = (t / per_group) * p.group_m;
  const int rows = p.num_m_tiles - first < p.group_m ? p.num_m_tiles - first : p.group_m;
  const int l = t - (t / per_group) * per_group;
  mt = first + l % rows;
  nt = l / rows;
}

// Work unit u of the persistent walk: a whole tile, or one K-range of a tail
// tile (the tiles of the last, partial wave are split along K so that every
// cluster has work; their FP32 partials are summed by split_fixup_kernel).
struct PairUnit {
  int tile, kb0, kb1;
  int slot;   // < 0: whole tile, stored to C; else the partial's workspace slot
  int rev;    // slabs taken last to first
};

__device__ __forceinline__ PairUnit pair_unit(int u, const GemmParams& p) {
  PairUnit w;
  if (u < p.full_tiles) {
    w.tile = u;
    w.kb0 = 0;
    w.kb1 = p.KB;
    w.slot = -1;
    w.rev = p.k_order == kKOrderSerpentine && ((u / static_cast<int>(gridDim.x >> 1)) & 1);
  } else {
    const int v = u - p.full_tiles;
    const int sp = v % p.splits;
    w.tile = p.full_tiles + v / p.splits;
    w.kb0 = (sp * p.KB) / p.splits;
    w.kb1 = ((sp + 1) * p.KB) / p.splits;
    w.slot = v;
    w.rev = 0;
  }
  return w;
}

// K slab of the unit's i-th step (kb0 <= i <= kb1; i = kb1 gives the slab
// after the last one, whose scales are prefetched and not used: kb1, or kb0 - 1
// when reversed, either of which the scale loads treat as out of range when it
// lies outside [0, KB)).
__device__ __forceinline__ int pair_kb(const PairUnit& w, int i) {
  return w.rev ? w.kb1 - 1 - (i - w.kb0) : i;
}

// Sum of the K-range partials of the tail tiles, in split order, converted to
// the output type (kAcc: added to the FP32 values already in C).  One thread
// per 4 columns of one row of one tail tile.
template <int BN, bool kOutBf16, bool kAcc = false>
__global__ void __launch_bounds__(256) split_fixup_kernel(const float* __restrict__ ws,
                                                          GemmParams p, int tail_tiles) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int q = static_cast<int>(idx % (BN / 4));
  const int r = static_cast<int>((idx / (BN / 4)) % kPairTileM);
  const int64_t tt = idx / ((BN / 4) * kPairTileM);
  if (tt >= tail_tiles) return;
  const int tile = p.full_tiles + static_cast<int>(tt);
  int mt, nt;
  pair_tile_mn(tile, p, mt, nt);
  const int row = mt * kPairTileM + r;
  const int col = nt * BN + q * 4;
  if (row >= p.M || col >= p.N) return;   // N is a multiple of 16: col..col+3 < N
  float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int sp = 0; sp < p.splits; ++sp) {
    const float4 v = __ldcs(reinterpret_cast<const float4*>(
        ws + ((tt * p.splits + sp) * kPairTileM + r) * static_cast<int64_t>(BN) + q * 4));
    sum.x += v.x;
    sum.y += v.y;
    sum.z += v.z;
    sum.w += v.w;
  }
  if constexpr (kOutBf16) {
    __nv_bfloat16* c = reinterpret_cast<__nv_bfloat16*>(p.C) + static_cast<int64_t>(row) * p.ldc + col;
    *reinterpret_cast<uint2*>(c) = make_uint2(pack_bf16x2(sum.x, sum.y), pack_bf16x2(sum.z, sum.w));
  } else {
    float4* c = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.C) +
                                          static_cast<int64_t>(row) * p.ldc + col);
    if constexpr (kAcc) {
      const float4 old = *c;
      sum = make_float4(old.x + sum.x, old.y + sum.y, old.z + sum.z, old.w + sum.w);
    }
    *c = sum;
  }
}

// p.num_m_tiles counts 256-row pair tiles here.  kAcc (FP32 output only):
// C += A * B^T, the tiles added into C by TMA reduce-add.
template <int BN, int kSb, bool kOutBf16, bool kAcc = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    fp8bs_gemm_pair_kernel(const __grid_constant__ GemmParams p,
                           const __grid_constant__ CUtensorMap tmap_a,
                           const __grid_constant__ CUtensorMap tmap_b,
                           const __grid_constant__ CUtensorMap tmap_c,
                           const __grid_constant__ CUtensorMap tmap_ws) {
  extern __shared__ __align__(1024) unsigned char pair_smem_raw[];
  const uint32_t raw_addr = smem_u32(pair_smem_raw);
  unsigned char* ring = pair_smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  constexpr int kPark = kSb == kSbPerCol ? kPairParkPerCol : kPairParkBlock;
  using Cfg = PairCfg<BN, kPark>;
  PairSmem<BN>& sm = *reinterpret_cast<PairSmem<BN>*>(ring + static_cast<size_t>(kPairRingBytes));
  const uint32_t ring_addr = smem_u32(ring);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();   // 0: the CTA that issues the MMAs
  // (tile bounds and strides are recomputed from the parameters and special
  // registers rather than held: the promotion warps have no registers to spare)
#define PAIR_FIRST static_cast<int>(blockIdx.x >> 1)
#define PAIR_STRIDE static_cast<int>(gridDim.x >> 1)
  volatile int* abort_flag = &sm.abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.done[s], 1);
    }
    for (int b = 0; b < Cfg::kBufs; ++b) mbar_init(&sm.tmem_free[b], 2 * kEpiWarps);
    for (int e = 0; e < Cfg::kStages; ++e) {
      mbar_init(&sm.scl_full[e], kPairScaleThreads);
      mbar_init(&sm.scl_free[e], kEpiWarps);
    }
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
    tma_prefetch_desc(&tmap_c);
  }
  if (warp == 1) tmem_alloc_pair(&sm.tmem_base, kTmemCols);
  tc_fence_before();
  __syncwarp();
  cluster_sync();   // barriers of both CTAs initialised, TMEM allocated in both
  tc_fence_after();
  const uint32_t tmem_base = sm.tmem_base;

  if (warp < 4) {
    regs_dealloc<kPairProducerRegs>();
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------------- TMA
      // A rows are re-read by every wave of the m-fastest walk (keep them in
      // L2); a B panel is consumed by the CTAs of one wave (measured: Fprop
      // 0.488 -> 0.438 ms against evict_last for both; evict_normal for B
      // then measured 0.5-1 % faster than evict_first on Fprop).
      const uint64_t policy_a = l2_policy_evict_last();
      const uint64_t policy_b = l2_policy_evict_normal();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, parity_mask = 0;
      bool aborted = false;
      for (int u = PAIR_FIRST; u < p.units && !aborted; u += PAIR_STRIDE) {
        const PairUnit w = pair_unit(u, p);
        int mt, nt;
        pair_tile_mn(w.tile, p, mt, nt);
        const int a_row = mt * kPairTileM + static_cast<int>(rank) * kBM;
        const int b_row = nt * BN + static_cast<int>(rank) * (BN / 2);
        for (int i = w.kb0; i < w.kb1; ++i) {
          const int kb = pair_kb(w, i);
          if (!bounded_wait(&sm.done[stage], phase ^ 1u, abort_flag)) {
            aborted = true;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(&sm.full[stage], 2 * Cfg::kStageBytes);
          const uint32_t full_bar = mapa_shared(smem_u32(&sm.full[stage]), 0);
          const uint32_t dst = ring_addr + stage * Cfg::kStageBytes;
          tma_load_2d_pair(dst, &tmap_a, kb * kBK, a_row, full_bar, policy_a);
          tma_load_2d_pair(dst + Cfg::kStageA, &tmap_b, kb * kBK, b_row, full_bar, policy_b);
          issued_mask |= 1u << stage;
          parity_mask = (parity_mask & ~(1u << stage)) | (phase << stage);
          if (++stage == Cfg::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every load issued must land before either CTA may exit.  The even CTA
      // sees both CTAs' bytes on its `full` barriers; the odd CTA cannot wait
      // on them, so after an abort it gives its own copies time to land.
      if (rank == 0) {
        for (int s = 0; s < Cfg::kStages; ++s)
          if (issued_mask & (1u << s))
            bounded_wait_noabort(&sm.full[s], (parity_mask >> s) & 1u, kSpinLimitNs);
      } else if (aborted) {
        __nanosleep(100000);
      }
    } else if (warp == 1 && lane == 0 && rank == 0) {
      // ---------------------------------------------------------------- MMA
      constexpr uint32_t idesc = idesc_e4m3_f32(kPairTileM, BN);
      int stage = 0, buf = 0;
      uint32_t phase = 0, tphase = 0;
      bool issued = false;
      for (int u = PAIR_FIRST; u < p.units; u += PAIR_STRIDE) {
        const PairUnit w = pair_unit(u, p);
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!bounded_wait(&sm.full[stage], phase, abort_flag)) goto mma_done;
          if (!bounded_wait(&sm.tmem_free[buf], tphase ^ 1u, abort_flag)) goto mma_done;
          tc_fence_after();
          const uint32_t a_addr = ring_addr + stage * Cfg::kStageBytes;
          const uint64_t adesc = smem_desc_k_sw128(a_addr);
          const uint64_t bdesc = smem_desc_k_sw128(a_addr + Cfg::kStageA);
          const uint32_t d = tmem_base + static_cast<uint32_t>(buf * BN);
#pragma unroll
          for (int kk = 0; kk < kBK / 32; ++kk)  // 32 bytes = 32 E4M3 values per MMA
            mma_f8f6f4_pair(d, adesc + 2u * kk, bdesc + 2u * kk, idesc, kk > 0 ? 1u : 0u);
          mma_commit_pair(&sm.done[stage], 0x3);
          issued = true;
          if (++stage == Cfg::kStages) {
            stage = 0;
            phase ^= 1u;
          }
          if (++buf == Cfg::kBufs) {
            buf = 0;
            tphase ^= 1u;
          }
        }
      }
    mma_done:
      if (issued) {  // all MMAs must finish before TMEM is released in either CTA
        mma_commit_pair(&sm.drain, 0x1);
        bounded_wait_noabort(&sm.drain, 0, kSpinLimitNs);
      }
    } else if (warp >= 2) {
      // ------------------------------------------------------------ scales
      // Every slab's scales into the next free ring entry with asynchronous
      // copies that arrive on the entry's barrier when they land, so that the
      // loads of several slabs are in flight at once: thread lt copies the A
      // scales of rows lt and 64 + lt, and 4 B scales (per-column mode) or one
      // column block's scale (block modes, BN / 128 threads).  Rows past M and
      // columns past N get zeros.
      const int lt = static_cast<int>(threadIdx.x) - 64;
      int e = 0;
      uint32_t ephase = 0;
      for (int u = PAIR_FIRST; u < p.units; u += PAIR_STRIDE) {
        const PairUnit w = pair_unit(u, p);
        int mt, nt;
        pair_tile_mn(w.tile, p, mt, nt);
        const int row0 = mt * kPairTileM + static_cast<int>(rank) * kBM;
        const int n0 = nt * BN;
        // block modes: this thread's column block (threads 0 .. BN/128 - 1)
        const int cb = n0 / 128 + (lt < BN / 128 ? lt : 0);
        const bool cb_ok = cb * 128 < p.N;
        const float* sb_k = p.sb + static_cast<int64_t>(cb_ok ? cb : 0) * p.sb_n_stride;
        const uint32_t cb_bytes = cb_ok ? 4u : 0u;
        for (int i = w.kb0; i < w.kb1; ++i) {
          const int kb = pair_kb(w, i);
          if (!bounded_wait(&sm.scl_free[e], ephase ^ 1u, abort_flag)) goto scales_done;
          const float* sa_k = p.sa + static_cast<int64_t>(kb) * p.ldsa;
#pragma unroll
          for (int r = lt; r < kBM; r += kPairScaleThreads) {
            const bool ok = row0 + r < p.M;
            cp_async_4(smem_u32(&sm.scl_sa[e][r]), sa_k + (ok ? row0 + r : 0), ok ? 4u : 0u);
          }
          if constexpr (kSb == kSbPerCol) {
#pragma unroll
            for (int j = lt * 4; j < BN; j += 4 * kPairScaleThreads) {
              // N is a multiple of 16: columns n0+j .. n0+j+3 are all in or all out
              const bool ok = n0 + j < p.N;
              cp_async_16(smem_u32(&sm.scl_sb[e][j]),
                          p.sb + static_cast<int64_t>(kb) * p.ldsb + (ok ? n0 + j : 0),
                          ok ? 16u : 0u);
            }
          } else {
            if (lt < BN / 128)
              cp_async_4(smem_u32(&sm.scl_sb[e][lt]), sb_k + static_cast<int64_t>(kb) * p.sb_k_stride,
                         cb_bytes);
          }
          cp_async_arrive(&sm.scl_full[e]);
          if (++e == Cfg::kStages) {
            e = 0;
            ephase ^= 1u;
          }
        }
      }
    scales_done:
      cp_async_wait_all();   // this thread's copies have landed before the CTA may exit
    }
  } else {
    regs_alloc<kPairEpilogueRegs>();
    // ------------------------------------------------- promotion + epilogue
    const int g = warp & 3;          // TMEM lane group (rows 32g .. 32g+31 of this CTA)
    const int h = (warp - 4) >> 2;   // column half of the tile (kWarpCols columns each)
    int buf = 0, stage = 0;   // the slab's TMEM buffer; its operand stage and scale entry
    uint32_t phase = 0;
    for (int u = PAIR_FIRST; u < p.units; u += PAIR_STRIDE) {
      const PairUnit w = pair_unit(u, p);
      int mt, nt;
      pair_tile_mn(w.tile, p, mt, nt);
      const int row = mt * kPairTileM + static_cast<int>(rank) * kBM + g * 32 + lane;
      const int col0 = nt * BN + h * Cfg::kWarpCols;
      float2 acc[Cfg::kWarpCols / 2];
#pragma unroll
      for (int i = 0; i < Cfg::kWarpCols / 2; ++i) acc[i] = make_float2(0.0f, 0.0f);

      for (int i = w.kb0; i < w.kb1; ++i) {
        // the slab's scales, loaded ahead into the ring by warps 2 and 3 (rows
        // past M and columns past N carry zero scales, so no guard is needed)
        if (!bounded_wait(&sm.scl_full[stage], phase, abort_flag)) goto epilogue_done;
        const float sa = sm.scl_sa[stage][g * 32 + lane];
        float sb = 0.0f;
        if constexpr (kSb == kSbBlock) sb = sm.scl_sb[stage][(h * Cfg::kWarpCols) / 128];
        if (!bounded_wait(&sm.done[stage], phase, abort_flag)) goto epilogue_done;
        tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(g * 32) << 16) +
                               static_cast<uint32_t>(buf * BN + h * Cfg::kWarpCols);
        uint32_t ra[32], rb[32];
        tmem_ld32(taddr, ra);
        tmem_wait_ld(ra);
        if constexpr (kSb == kSbBlock) {
          const float sc = sa * sb;
          const float2 sc2 = make_float2(sc, sc);
#pragma unroll
          for (int c = 0; c < Cfg::kChunks; c += 2) {
            tmem_ld32(taddr + (c + 1) * 32, rb);
            promote32(acc + c * 16, ra, sc2);
            tmem_wait_ld(rb);
            if (c + 2 < Cfg::kChunks) tmem_ld32(taddr + (c + 2) * 32, ra);
            promote32(acc + (c + 1) * 16, rb, sc2);
            if (c + 2 < Cfg::kChunks) tmem_wait_ld(ra);
          }
        } else {
          const float2 sa2 = make_float2(sa, sa);
          const float* sbs = &sm.scl_sb[stage][h * Cfg::kWarpCols];
#pragma unroll
          for (int c = 0; c < Cfg::kChunks; c += 2) {
            tmem_ld32(taddr + (c + 1) * 32, rb);
            promote32_percol(acc + c * 16, ra, sbs + c * 32, sa2);
            tmem_wait_ld(rb);
            if (c + 2 < Cfg::kChunks) tmem_ld32(taddr + (c + 2) * 32, ra);
            promote32_percol(acc + (c + 1) * 16, rb, sbs + (c + 1) * 32, sa2);
            if (c + 2 < Cfg::kChunks) tmem_wait_ld(ra);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_cluster(mapa_shared(smem_u32(&sm.tmem_free[buf]), 0));
          mbar_arrive(&sm.scl_free[stage]);
        }
        if (++buf == Cfg::kBufs) buf = 0;
        if (++stage == Cfg::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // ---- epilogue: this warp's 32 rows x kWarpCols columns, through TMA
      // stores (addresses are recomputed, not held: the promotion warps have
      // no registers to spare while the accumulators are live)
      const uint32_t stg = smem_u32(&sm.epi_stage[warp - 4][0]);
      if (w.slot < 0) {
        if constexpr (kPark > 0) {
          // the first columns through the staging buffer, the last kParkCols
          // parked (their stores drain while the next tile runs)
          constexpr int kParkCols = Cfg::template park_cols<kOutBf16 ? 2 : 4>();
          constexpr int kStaged = Cfg::kWarpCols - kParkCols;
          static_assert(kParkCols % 32 == 0 && kParkCols > 0, "parked columns: whole boxes");
          if constexpr (kStaged > 0)
            store_rows_tma<kOutBf16, kAcc, kStaged>(acc, stg, lane, &tmap_c, col0, row - lane);
          const uint32_t park = ring_addr + Cfg::kStages * Cfg::kStageBytes +
                                static_cast<uint32_t>(warp - 4) * Cfg::kParkWarpBytes;
          park_rows_tma<kOutBf16, kAcc, kParkCols>(acc + kStaged / 2, park, lane, &tmap_c,
                                                   col0 + kStaged, row - lane);
        } else {
          store_rows_tma<kOutBf16, kAcc, Cfg::kWarpCols>(acc, stg, lane, &tmap_c, col0,
                                                         row - lane);
        }
      } else {
        store_rows_tma<false, false, Cfg::kWarpCols>(
            acc, stg, lane, &tmap_ws, h * Cfg::kWarpCols,
            w.slot * kPairTileM + static_cast<int>(rank) * kBM + g * 32);
      }
    }
  epilogue_done:
    if (lane == 0) bulk_wait_all();   // this warp's output stores are complete
  }

  tc_fence_before();
  __syncwarp();
  cluster_sync();   // no CTA leaves while its peer may still touch its shared memory
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

#undef PAIR_FIRST
#undef PAIR_STRIDE

}  // namespace fp8bs
